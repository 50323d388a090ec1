"""ctypes view of the C ABI in ``include/kda.h``, ``include/kda_bwd.h`` and
``include/kda_cp.h`` (argument marshalling only).

Loading fails loudly when the CUDA library has not been built: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkda_gb300.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_SHAPE = 2
KDA_ERR_DTYPE = 3
KDA_ERR_UNSUPPORTED = 4
KDA_ERR_CUDA = 5
KDA_ERR_DEVICE_STATUS = 6
KDA_ERR_WORKSPACE = 7

KDA_GATE_PREGATED = 0
KDA_GATE_PLAIN = 1
KDA_GATE_SAFE = 2

KDA_BF16 = 0
KDA_F32 = 1

KDA_DEV_BAD_SEQLENS = 0x1
KDA_DEV_TIMEOUT = 0x2

# Every symbol the header declares.
EXPORTED = ("kda_fwd_workspace_size", "kda_fwd_check", "kda_fwd", "kda_fwd_num_launches",
            "kda_fwd_num_chunks", "kda_fused_recurrent_fwd", "kda_fwd_host_arena_size",
            "kda_fwd_host",
            "kda_fwd_num_stages",
            "kda_fwd_stage_name", "kda_fwd_stage", "kda_get_device_status", "kda_status_string",
            "kda_last_error", "kda_abi_version", "kda_fwd_noalloc",
            "kda_bwd_check", "kda_bwd_workspace_size", "kda_bwd_num_launches", "kda_bwd",
            "kda_bwd_num_stages", "kda_bwd_stage_name", "kda_bwd_stage",
            "kda_state_affine_apply")

# Size of the static device scratch behind kda_fwd_noalloc (KDA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class kda_fwd_params(ctypes.Structure):
    """Mirror of ``struct kda_fwd_params`` (field order and types must match the header)."""

    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("HV", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("chunk_size", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32), ("lower_bound", ctypes.c_float),
        ("scale", ctypes.c_float), ("qk_l2norm", ctypes.c_int32),
        ("beta_sigmoid", ctypes.c_int32), ("N", ctypes.c_int32),
        ("allow_neg_eigval", ctypes.c_int32), ("state_v_first", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p), ("h0", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
        ("cu_seqlens_host", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p), ("h_out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class kda_bwd_params(ctypes.Structure):
    """Mirror of ``struct kda_bwd_params`` (include/kda_bwd.h)."""

    _fields_ = [
        ("fwd", kda_fwd_params), ("d_o", ctypes.c_void_p), ("d_final_state", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p), ("dA_log", ctypes.c_void_p),
        ("ddt_bias", ctypes.c_void_p), ("dh0", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kda status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load ``libkda_gb300.so`` (once).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built; run kimi_delta_attention_gate_gb300.build.build() "
                    "(nvcc, sm_103a).  There is no fallback path.")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(kda_fwd_params)
            lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
            lib.kda_fwd_workspace_size.argtypes = [P]
            lib.kda_fwd_check.restype = ctypes.c_int
            lib.kda_fwd_check.argtypes = [P]
            lib.kda_fwd.restype = ctypes.c_int
            lib.kda_fwd.argtypes = [P, ctypes.c_void_p]
            lib.kda_fwd_noalloc.restype = ctypes.c_int
            lib.kda_fwd_noalloc.argtypes = [P, ctypes.c_void_p]
            lib.kda_fwd_num_launches.restype = ctypes.c_int32
            lib.kda_fwd_num_launches.argtypes = [P]
            lib.kda_fwd_num_chunks.restype = ctypes.c_int64
            lib.kda_fwd_num_chunks.argtypes = [P]
            lib.kda_fused_recurrent_fwd.restype = ctypes.c_int
            lib.kda_fused_recurrent_fwd.argtypes = [P, ctypes.c_void_p]
            lib.kda_fwd_host_arena_size.restype = ctypes.c_size_t
            lib.kda_fwd_host_arena_size.argtypes = [P]
            lib.kda_fwd_host.restype = ctypes.c_int
            lib.kda_fwd_host.argtypes = [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
            lib.kda_fwd_num_stages.restype = ctypes.c_int32
            lib.kda_fwd_num_stages.argtypes = [P]
            lib.kda_fwd_stage_name.restype = ctypes.c_char_p
            lib.kda_fwd_stage_name.argtypes = [P, ctypes.c_int32]
            lib.kda_fwd_stage.restype = ctypes.c_int
            lib.kda_fwd_stage.argtypes = [P, ctypes.c_void_p, ctypes.c_int32]
            lib.kda_get_device_status.restype = ctypes.c_uint32
            lib.kda_get_device_status.argtypes = [ctypes.c_void_p]
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [ctypes.c_int]
            lib.kda_last_error.restype = ctypes.c_char_p
            lib.kda_last_error.argtypes = []
            lib.kda_abi_version.restype = ctypes.c_int32
            lib.kda_abi_version.argtypes = []
            PB = ctypes.POINTER(kda_bwd_params)
            lib.kda_bwd_check.restype = ctypes.c_int
            lib.kda_bwd_check.argtypes = [PB]
            lib.kda_bwd_workspace_size.restype = ctypes.c_size_t
            lib.kda_bwd_workspace_size.argtypes = [PB]
            lib.kda_bwd_num_launches.restype = ctypes.c_int32
            lib.kda_bwd_num_launches.argtypes = [PB]
            lib.kda_bwd.restype = ctypes.c_int
            lib.kda_bwd.argtypes = [PB, ctypes.c_void_p]
            lib.kda_bwd_num_stages.restype = ctypes.c_int32
            lib.kda_bwd_num_stages.argtypes = [PB]
            lib.kda_bwd_stage_name.restype = ctypes.c_char_p
            lib.kda_bwd_stage_name.argtypes = [PB, ctypes.c_int32]
            lib.kda_bwd_stage.restype = ctypes.c_int
            lib.kda_bwd_stage.argtypes = [PB, ctypes.c_void_p, ctypes.c_int32]
            lib.kda_state_affine_apply.restype = ctypes.c_int
            lib.kda_state_affine_apply.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            _lib = lib
    return _lib


def kda_fwd_workspace_size(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_workspace_size(ctypes.byref(p)))


def kda_fwd_check(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_check(ctypes.byref(p)))


def kda_fwd(p: kda_fwd_params, stream: int = 0) -> int:
    return int(load().kda_fwd(ctypes.byref(p), ctypes.c_void_p(stream)))


def kda_fwd_noalloc(p: kda_fwd_params, stream: int = 0) -> int:
    return int(load().kda_fwd_noalloc(ctypes.byref(p), ctypes.c_void_p(stream)))


def kda_fwd_host_arena_size(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_host_arena_size(ctypes.byref(p)))


def kda_fwd_host(p: kda_fwd_params, arena: int, arena_bytes: int, stream: int) -> int:
    return int(load().kda_fwd_host(ctypes.byref(p), ctypes.c_void_p(arena), ctypes.c_size_t(arena_bytes),
                                   ctypes.c_void_p(stream)))


def kda_fused_recurrent_fwd(p: kda_fwd_params, stream: int) -> int:
    return int(load().kda_fused_recurrent_fwd(ctypes.byref(p), ctypes.c_void_p(stream)))


def kda_fwd_num_chunks(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_num_chunks(ctypes.byref(p)))


def kda_fwd_num_launches(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_num_launches(ctypes.byref(p)))


def kda_fwd_num_stages(p: kda_fwd_params) -> int:
    return int(load().kda_fwd_num_stages(ctypes.byref(p)))


def kda_fwd_stage_name(p: kda_fwd_params, stage: int) -> str:
    return load().kda_fwd_stage_name(ctypes.byref(p), int(stage)).decode()


def kda_fwd_stage(p: kda_fwd_params, stream: int, stage: int) -> int:
    return int(load().kda_fwd_stage(ctypes.byref(p), ctypes.c_void_p(stream), int(stage)))


def kda_get_device_status(stream: int = 0) -> int:
    return int(load().kda_get_device_status(ctypes.c_void_p(stream)))


def kda_status_string(s: int) -> str:
    return load().kda_status_string(int(s)).decode()


def kda_last_error() -> str:
    return load().kda_last_error().decode()


def kda_abi_version() -> int:
    return int(load().kda_abi_version())


def kda_bwd_check(p: kda_bwd_params) -> int:
    return int(load().kda_bwd_check(ctypes.byref(p)))


def kda_bwd_workspace_size(p: kda_bwd_params) -> int:
    return int(load().kda_bwd_workspace_size(ctypes.byref(p)))


def kda_bwd_num_launches(p: kda_bwd_params) -> int:
    return int(load().kda_bwd_num_launches(ctypes.byref(p)))


def kda_bwd(p: kda_bwd_params, stream: int = 0) -> int:
    return int(load().kda_bwd(ctypes.byref(p), ctypes.c_void_p(stream)))


def kda_bwd_num_stages(p: kda_bwd_params) -> int:
    return int(load().kda_bwd_num_stages(ctypes.byref(p)))


def kda_bwd_stage_name(p: kda_bwd_params, stage: int) -> str:
    return load().kda_bwd_stage_name(ctypes.byref(p), int(stage)).decode()


def kda_bwd_stage(p: kda_bwd_params, stream: int, stage: int) -> int:
    return int(load().kda_bwd_stage(ctypes.byref(p), ctypes.c_void_p(stream), int(stage)))


def kda_state_affine_apply(P: int, R: int, S_in, S_out: int, nmaps: int, K: int, V: int,
                           state_v_first: int, stream: int = 0) -> int:
    return int(load().kda_state_affine_apply(ctypes.c_void_p(P), ctypes.c_void_p(R),
                                             ctypes.c_void_p(S_in), ctypes.c_void_p(S_out),
                                             int(nmaps), int(K), int(V), int(state_v_first),
                                             ctypes.c_void_p(stream)))


def raise_for(status: int) -> None:
    if status != KDA_OK:
        raise KdaError(status, kda_last_error() or kda_status_string(status))
