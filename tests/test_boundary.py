"""Host-only tests of the C ABI: the library builds and loads, exports every
symbol the header declares, and every argument rule returns its status before
any CUDA call.  No test here touches a GPU (fake, never-dereferenced pointers
are only passed to the checking entry points)."""
import ctypes
import os
import re

import pytest

from kimi_delta_attention_gate_gb300 import _binding as kb
from kimi_delta_attention_gate_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kb.load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_binding_expects():
    assert declared_functions() == sorted(kb.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert kb.kda_abi_version() == 2


def test_status_strings(lib):
    for s in range(8):
        assert kb.kda_status_string(s)
    assert kb.kda_status_string(0) == "ok"


def test_every_header_is_covered():
    assert [os.path.basename(h) for h in HEADERS] == ["kda.h", "kda_bwd.h", "kda_cp.h"]


def test_struct_layout_matches_header():
    # int32 x 9, float x 2, int32 x 5 -> 64 bytes, then 14 pointers and a size_t
    assert kb.kda_fwd_params.q.offset == 64
    assert kb.kda_fwd_params.workspace_bytes.offset == 64 + 14 * 8
    assert ctypes.sizeof(kb.kda_fwd_params) == 64 + 15 * 8
    # the forward block, then 11 pointers and a size_t
    assert kb.kda_bwd_params.d_o.offset == ctypes.sizeof(kb.kda_fwd_params)
    assert kb.kda_bwd_params.workspace_bytes.offset == 184 + 11 * 8
    assert ctypes.sizeof(kb.kda_bwd_params) == 184 + 12 * 8


FAKE = 0x10000  # 16-byte aligned, never dereferenced by the checks


def valid_params(**over):
    p = kb.kda_fwd_params()
    p.B, p.T, p.H, p.HV, p.K, p.V = 2, 100, 2, 4, 128, 64
    p.chunk_size = 64
    p.in_dtype = kb.KDA_BF16
    p.gate_mode = kb.KDA_GATE_SAFE
    p.lower_bound = -5.0
    p.scale = 128 ** -0.5
    p.qk_l2norm = 1
    p.beta_sigmoid = 1
    p.N = 2
    for f in ("q", "k", "v", "g", "beta", "o"):
        setattr(p, f, FAKE)
    for k_, v_ in over.items():
        setattr(p, k_, v_)
    return p


def check(p):
    return kb.kda_fwd_check(p)


def test_valid_params_pass_and_have_workspace(lib):
    p = valid_params()
    assert check(p) == kb.KDA_OK
    assert kb.kda_fwd_workspace_size(p) > 0


@pytest.mark.parametrize("over,status", [
    (dict(gate_mode=kb.KDA_GATE_PLAIN), kb.KDA_ERR_INVALID_ARG),            # A_log required
    (dict(lower_bound=-5.5), kb.KDA_ERR_INVALID_ARG),                        # lb >= -5
    (dict(lower_bound=0.0), kb.KDA_ERR_INVALID_ARG),                         # lb < 0
    (dict(lower_bound=float("nan")), kb.KDA_ERR_INVALID_ARG),
    (dict(chunk_size=16), kb.KDA_ERR_SHAPE),                                 # 32 or 64 only
    (dict(chunk_size=128), kb.KDA_ERR_SHAPE),
    (dict(K=257), kb.KDA_ERR_SHAPE),                                         # K <= 256
    (dict(V=257), kb.KDA_ERR_SHAPE),
    (dict(HV=3), kb.KDA_ERR_SHAPE),                                          # HV % H == 0
    (dict(in_dtype=7), kb.KDA_ERR_DTYPE),
    (dict(gate_mode=9), kb.KDA_ERR_INVALID_ARG),
    (dict(q=0), kb.KDA_ERR_INVALID_ARG),                                     # NULL input
    (dict(o=0), kb.KDA_ERR_INVALID_ARG),
    (dict(k=FAKE + 4), kb.KDA_ERR_INVALID_ARG),                              # misaligned
    (dict(dt_bias=FAKE + 8), kb.KDA_ERR_INVALID_ARG),
    (dict(h_out=FAKE + 4), kb.KDA_ERR_INVALID_ARG),
    (dict(N=3), kb.KDA_ERR_SHAPE),                                           # N == B without varlen
    (dict(qk_l2norm=2), kb.KDA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), kb.KDA_ERR_INVALID_ARG),
    (dict(B=0), kb.KDA_ERR_SHAPE),
    (dict(allow_neg_eigval=1, beta_sigmoid=0), kb.KDA_ERR_INVALID_ARG),   # needs beta sigmoid
    (dict(allow_neg_eigval=2), kb.KDA_ERR_INVALID_ARG),
    (dict(state_v_first=3), kb.KDA_ERR_INVALID_ARG),
])
def test_rule_rejections(lib, over, status):
    p = valid_params(**over)
    assert check(p) == status
    assert kb.kda_last_error() != ""
    assert kb.kda_fwd_workspace_size(p) == 0


def test_plain_gate_with_alog_and_safe_without_alog_pass(lib):
    assert check(valid_params(gate_mode=kb.KDA_GATE_PLAIN, A_log=FAKE)) == kb.KDA_OK
    assert check(valid_params(gate_mode=kb.KDA_GATE_SAFE, A_log=0)) == kb.KDA_OK
    assert check(valid_params(gate_mode=kb.KDA_GATE_PREGATED, lower_bound=0.0)) == kb.KDA_OK


def cu_params(cu, T=200, **over):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    p = valid_params(B=1, T=T, N=len(cu) - 1, cu_seqlens=FAKE, **over)
    p.cu_seqlens_host = ctypes.addressof(arr)
    return p, arr


def test_varlen_rules(lib):
    p, keep = cu_params([0, 5, 64, 200])
    assert check(p) == kb.KDA_OK
    p, keep = cu_params([0, 5, 64, 201])
    assert check(p) == kb.KDA_ERR_SHAPE                                       # beyond T
    p, keep = cu_params([0, 70, 64, 100])
    assert check(p) == kb.KDA_ERR_SHAPE                                       # decreasing
    p, keep = cu_params([1, 5, 64, 100])
    assert check(p) == kb.KDA_ERR_SHAPE                                       # must start at 0
    p, keep = cu_params([0, 5, 64, 100])
    p.B = 2
    assert check(p) == kb.KDA_ERR_SHAPE                                       # B == 1
    p, keep = cu_params([0, 5, 64, 100])
    p.cu_seqlens_host = None
    assert check(p) == kb.KDA_ERR_INVALID_ARG                                 # host copy needed


def test_num_chunks(lib):
    assert kb.kda_fwd_num_chunks(valid_params()) == 2 * 2            # B = 2, T = 100, chunk 64
    p, keep = cu_params([0, 5, 64, 64, 200])                          # 1 + 1 + 0 + 3
    assert kb.kda_fwd_num_chunks(p) == 5
    assert kb.kda_fwd_num_chunks(valid_params(K=300)) == 0            # invalid parameters


def test_workspace_grows_with_chunks(lib):
    a = kb.kda_fwd_workspace_size(valid_params(T=64))
    b = kb.kda_fwd_workspace_size(valid_params(T=65))
    assert b > a > 0
    p, keep = cu_params([0, 1, 2, 3], T=3)
    c = kb.kda_fwd_workspace_size(p)
    assert c > 0


def test_fwd_rejects_small_workspace_before_cuda(lib):
    p = valid_params()
    p.workspace = FAKE
    p.workspace_bytes = 16
    assert kb.kda_fwd(p, 0) == kb.KDA_ERR_WORKSPACE
    p.workspace_bytes = kb.kda_fwd_workspace_size(p)
    p.workspace = FAKE + 16
    assert kb.kda_fwd(p, 0) == kb.KDA_ERR_WORKSPACE                           # 256-byte alignment


def test_fwd_without_gpu_reports_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("would launch on fake pointers; only meaningful without a GPU")
    p = valid_params()
    p.workspace = FAKE
    p.workspace_bytes = kb.kda_fwd_workspace_size(p)
    assert kb.kda_fwd(p, 0) == kb.KDA_ERR_CUDA


def test_python_wrapper_gate_selection():
    from kimi_delta_attention_gate_gb300 import _gate_mode
    assert _gate_mode(False, None, None) == kb.KDA_GATE_PREGATED
    assert _gate_mode(True, None, -5.0) == kb.KDA_GATE_SAFE
    assert _gate_mode(True, None, None) == kb.KDA_GATE_PLAIN
    with pytest.raises(ValueError):
        _gate_mode(True, True, None)


def test_launch_counts_of_the_pipelined_schedule(lib):
    # fp32 or V != 128: CUDA-core stages, one launch each
    p = valid_params()
    assert kb.kda_fwd_num_launches(p) == kb.kda_fwd_num_stages(p) == 2
    # bf16, K = V = 128, 4 heads x 512 chunks: five segments of intra + recurrence
    p = valid_params(B=1, T=64 * 512, H=4, HV=4, V=128, N=1)
    assert kb.kda_fwd_num_stages(p) == 2
    assert kb.kda_fwd_num_launches(p) == 10
    ws_seg = kb.kda_fwd_workspace_size(p)
    blocks = 66048 * 512 * 4
    assert ws_seg >= blocks + 4 * 128 * 128 * 4          # + the fp32 states carried across
    # many recurrences (N * HV > 96): no segments
    p = valid_params(B=1, T=64 * 512, H=128, HV=128, V=128, N=1)
    assert kb.kda_fwd_num_launches(p) == 2
    # varlen adds the chunk-table launch
    p, keep = cu_params([0, 64 * 400, 64 * 600], T=64 * 600, H=4, HV=4, V=128)
    assert kb.kda_fwd_num_launches(p) == 1 + 2 * 6


def test_host_entry_arena_size_and_rejections(lib):
    p = valid_params()
    # device copies of q, k, v, g, beta and o (each 256-byte aligned), then the workspace
    copies = 2 * 102400 + 102400 + 204800 + 1792 + 102400
    assert kb.kda_fwd_host_arena_size(p) == copies + kb.kda_fwd_workspace_size(p)
    fs = valid_params(final_state=FAKE)
    assert kb.kda_fwd_host_arena_size(fs) == kb.kda_fwd_host_arena_size(p) + 2 * 4 * 128 * 64 * 4
    assert kb.kda_fwd_host_arena_size(valid_params(K=300)) == 0
    need = kb.kda_fwd_host_arena_size(p)
    # arena checks come before any CUDA call
    assert kb.kda_fwd_host(p, 0, need, 0) == kb.KDA_ERR_WORKSPACE
    assert kb.kda_fwd_host(p, FAKE, need - 1, 0) == kb.KDA_ERR_WORKSPACE
    assert kb.kda_fwd_host(p, FAKE + 16, need, 0) == kb.KDA_ERR_WORKSPACE
    assert kb.kda_fwd_host(valid_params(q=None), FAKE, need, 0) == kb.KDA_ERR_INVALID_ARG
    # varlen on the host entry is selected by cu_seqlens_host alone
    cu = (ctypes.c_int64 * 3)(0, 150, 200)
    v = valid_params(B=1, T=200, N=2, cu_seqlens_host=ctypes.addressof(cu))
    assert kb.kda_fwd_host_arena_size(v) > 0


def test_make_params_rejects_int32_seqlens():
    """The C ABI reads 8-byte offsets: an int32 cu_seqlens (FLA's usual type) must not be read
    as int64.  make_params refuses it; the kda_fwd wrapper converts before calling it."""
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    q = torch.zeros((1, 16, 1, 8))
    v = torch.zeros((1, 16, 1, 8))
    b = torch.zeros((1, 16, 1))
    for bad in (dict(cu_seqlens=torch.tensor([0, 5, 16], dtype=torch.int32),
                     cu_seqlens_cpu=torch.tensor([0, 5, 16], dtype=torch.int64)),
                dict(cu_seqlens=torch.tensor([0, 5, 16], dtype=torch.int64),
                     cu_seqlens_cpu=torch.tensor([0, 5, 16], dtype=torch.int32))):
        with pytest.raises(ValueError, match="int64"):
            kda.make_params(q, q, v, v, b, lower_bound=-5.0, o=v, **bad)
    from kimi_delta_attention_gate_gb300 import _int64_seqlens
    cu, cu_cpu = _int64_seqlens(torch.tensor([0, 5, 16], dtype=torch.int32), None)
    assert cu.dtype == torch.int64 and cu_cpu.dtype == torch.int64
    assert cu_cpu.tolist() == [0, 5, 16]


def test_make_params_keeps_its_tensors_alive():
    """The parameter block holds raw addresses; it also holds the tensors behind them, so that
    temporaries passed by the caller cannot be freed (and their memory reused) before launch."""
    import gc
    import weakref
    import torch
    import kimi_delta_attention_gate_gb300 as kda
    q = torch.zeros((1, 16, 1, 8))
    v = torch.zeros((1, 16, 1, 8))
    b = torch.zeros((1, 16, 1))
    h0 = torch.ones((1, 1, 8, 8))
    ref = weakref.ref(h0)
    p = kda.make_params(q, q, v, v, b, lower_bound=-5.0, o=v, initial_state=h0,
                        cu_seqlens=torch.tensor([0, 16], dtype=torch.int64),
                        cu_seqlens_cpu=torch.tensor([0, 16], dtype=torch.int64))
    addr = p.h0
    del h0
    gc.collect()
    assert ref() is not None and ref().data_ptr() == addr
    assert any(t.data_ptr() == p.cu_seqlens for t in p._keep)
    del p
    gc.collect()
    assert ref() is None
