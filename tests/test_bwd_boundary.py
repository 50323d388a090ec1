"""Host-only tests of the backward entry points (include/kda_bwd.h): every argument rule
returns its status before any CUDA call, the workspace and launch counts follow the plan.
No test here touches a GPU (fake, never-dereferenced pointers go to the checks only)."""
import ctypes

import pytest

from kimi_delta_attention_gate_gb300 import _binding as kb
from kimi_delta_attention_gate_gb300 import build as kbuild

FAKE = 0x10000  # 16-byte aligned, never dereferenced by the checks


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kb.load()


def params(**over):
    p = kb.kda_bwd_params()
    f = p.fwd
    f.B, f.T, f.H, f.HV, f.K, f.V = 2, 100, 2, 4, 128, 64
    f.chunk_size = 64
    f.in_dtype = kb.KDA_BF16
    f.gate_mode = kb.KDA_GATE_SAFE
    f.lower_bound = -5.0
    f.scale = 128 ** -0.5
    f.qk_l2norm = 1
    f.beta_sigmoid = 1
    f.N = 2
    for name in ("q", "k", "v", "g", "beta"):
        setattr(f, name, FAKE)
    for name in ("d_o", "dq", "dk", "dv", "dg", "dbeta"):
        setattr(p, name, FAKE)
    for key, val in over.items():
        if key.startswith("fwd_"):
            setattr(f, key[4:], val)
        else:
            setattr(p, key, val)
    return p


def test_valid_parameters_pass(lib):
    p = params()
    assert kb.kda_bwd_check(p) == kb.KDA_OK
    assert kb.kda_bwd_workspace_size(p) > 0
    assert kb.kda_bwd_num_launches(p) == 5                     # prep, states, dstate, grads, gate


@pytest.mark.parametrize("over,status", [
    (dict(d_o=0), kb.KDA_ERR_INVALID_ARG),                     # in the place of o
    (dict(dq=0), kb.KDA_ERR_INVALID_ARG),
    (dict(dbeta=0), kb.KDA_ERR_INVALID_ARG),
    (dict(dv=FAKE + 4), kb.KDA_ERR_INVALID_ARG),               # misaligned
    (dict(dh0=FAKE + 8), kb.KDA_ERR_INVALID_ARG),
    (dict(d_final_state=FAKE + 4), kb.KDA_ERR_INVALID_ARG),
    (dict(dA_log=FAKE), kb.KDA_ERR_INVALID_ARG),               # without A_log
    (dict(ddt_bias=FAKE), kb.KDA_ERR_INVALID_ARG),             # without dt_bias
    (dict(dA_log=FAKE, fwd_A_log=FAKE, fwd_gate_mode=kb.KDA_GATE_PREGATED),
     kb.KDA_ERR_INVALID_ARG),                                  # no in-kernel gate
    (dict(fwd_chunk_size=16), kb.KDA_ERR_SHAPE),               # the forward's rules apply
    (dict(fwd_HV=3), kb.KDA_ERR_SHAPE),
    (dict(fwd_lower_bound=-6.0), kb.KDA_ERR_INVALID_ARG),
    (dict(fwd_q=0), kb.KDA_ERR_INVALID_ARG),
])
def test_rule_rejections(lib, over, status):
    p = params(**over)
    assert kb.kda_bwd_check(p) == status
    assert kb.kda_last_error() != ""
    assert kb.kda_bwd_workspace_size(p) == 0
    assert kb.kda_bwd_num_launches(p) == 0


def test_optional_gradients_with_their_inputs_pass(lib):
    p = params(dA_log=FAKE, fwd_A_log=FAKE, ddt_bias=FAKE, fwd_dt_bias=FAKE, dh0=FAKE,
               d_final_state=FAKE)
    assert kb.kda_bwd_check(p) == kb.KDA_OK
    p = params(fwd_gate_mode=kb.KDA_GATE_PLAIN, fwd_A_log=FAKE, dA_log=FAKE)
    assert kb.kda_bwd_check(p) == kb.KDA_OK
    p = params(dh0=FAKE)                                       # the gradient at a zero h0
    assert kb.kda_bwd_check(p) == kb.KDA_OK


def test_output_o_and_states_of_the_forward_block_are_not_needed(lib):
    p = params()
    assert p.fwd.o is None and p.fwd.final_state is None
    assert kb.kda_bwd_check(p) == kb.KDA_OK


def test_workspace_follows_the_chunk_count(lib):
    """Per (chunk, value head): the recomputed intermediates (with Aqk, P and A^T as C x C and
    the block-referenced Q / K rows as three C x K, plus a range flag), then the state before
    and the state gradient after the chunk (K V fp32 each)."""
    C, K, V = 64, 128, 64
    block = 4 * (14 * C * K + 4 * C * V + 3 * C * C + C + K + 4)
    block = (block + 255) // 256 * 256
    per_chunk_head = block + 2 * 4 * K * V
    a = kb.kda_bwd_workspace_size(params(fwd_T=64))            # 2 sequences x 1 chunk x 4 heads
    b = kb.kda_bwd_workspace_size(params(fwd_T=65))            # 2 chunks each
    assert b - a == 2 * 4 * per_chunk_head


def test_varlen_launch_count_and_chunk_table(lib):
    cu = (ctypes.c_int64 * 4)(0, 5, 64, 200)
    p = params(fwd_B=1, fwd_T=200, fwd_N=3, fwd_cu_seqlens=FAKE)
    p.fwd.cu_seqlens_host = ctypes.addressof(cu)
    assert kb.kda_bwd_check(p) == kb.KDA_OK
    assert kb.kda_bwd_num_launches(p) == 6                     # + the chunk table


def test_no_tokens_launches_only_the_state_stages(lib):
    p = params(fwd_T=0)
    for name in ("q", "k", "v", "g", "beta"):
        setattr(p.fwd, name, None)
    for name in ("d_o", "dq", "dk", "dv", "dg", "dbeta"):
        setattr(p, name, None)
    assert kb.kda_bwd_check(p) == kb.KDA_OK
    assert kb.kda_bwd_num_launches(p) == 2


def test_rejects_small_workspace_before_cuda(lib):
    p = params()
    p.workspace = FAKE
    p.workspace_bytes = 16
    assert kb.kda_bwd(p, 0) == kb.KDA_ERR_WORKSPACE
    p.workspace_bytes = kb.kda_bwd_workspace_size(p)
    p.workspace = FAKE + 16
    assert kb.kda_bwd(p, 0) == kb.KDA_ERR_WORKSPACE


def test_without_gpu_reports_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("would launch on fake pointers; only meaningful without a GPU")
    p = params()
    p.workspace = FAKE
    p.workspace_bytes = kb.kda_bwd_workspace_size(p)
    assert kb.kda_bwd(p, 0) == kb.KDA_ERR_CUDA


def test_stage_lists(lib):
    names = lambda p: [kb.kda_bwd_stage_name(p, i) for i in range(kb.kda_bwd_num_stages(p))]
    assert names(params()) == ["zero_outputs", "bwd_prep", "bwd_states", "bwd_dstate", "bwd_grads",
                               "bwd_gate"]
    cu = (ctypes.c_int64 * 4)(0, 5, 64, 200)
    p = params(fwd_B=1, fwd_T=200, fwd_N=3, fwd_cu_seqlens=FAKE)
    p.fwd.cu_seqlens_host = ctypes.addressof(cu)
    assert names(p) == ["zero_outputs", "chunk_table", "bwd_prep", "bwd_states", "bwd_dstate",
                        "bwd_grads", "bwd_gate"]
    assert kb.kda_bwd_num_launches(p) == kb.kda_bwd_num_stages(p) - 1
    assert kb.kda_bwd_stage_name(params(), 6) == "" and kb.kda_bwd_stage_name(params(), -1) == ""
    assert kb.kda_bwd_num_stages(params(dq=0)) == 0
    # bf16 at K = V = 128, chunk 64: the products over v get a tensor-core stage of their own
    assert names(params(fwd_V=128)) == ["zero_outputs", "bwd_prep", "bwd_states", "bwd_dstate",
                                        "bwd_vprod", "bwd_grads", "bwd_gate"]
    assert "bwd_vprod" not in names(params(fwd_V=128, fwd_in_dtype=kb.KDA_F32))


def test_stage_rejects_small_workspace_before_cuda(lib):
    p = params()
    p.workspace = FAKE
    p.workspace_bytes = 16
    assert kb.kda_bwd_stage(p, 0, 1) == kb.KDA_ERR_WORKSPACE
