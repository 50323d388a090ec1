"""GPU unit tests of the tcgen05 primitives (tc_common.cuh) the tensor-core
kernels are built from: shared-memory descriptors for 128-byte-swizzled K-major
and MN-major operands, the instruction descriptor (M, N, negate), MMA chains over
K, and the TMEM lane layout of the accumulator.  Inputs are small multiples of
1/4, so every product and sum is exact in fp32 and the check is exact."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "tc_probe.cu")
OUT = os.path.join(HERE, "_build", "libtc_probe.so")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    csrc = os.path.join(ROOT, "kimi_delta_attention_gate_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-I", csrc, "-I", os.path.join(ROOT, "include"),
                    SRC, "-o", OUT], check=True)
    lib = ctypes.CDLL(OUT)
    lib.tc_probe_run.restype = ctypes.c_int
    return lib


def bf16_bits(x):
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def run(lib, M, N, K, a_mn=0, b_mn=0, neg_a=0, seed=0, a_tmem=0):
    r = np.random.default_rng(seed)
    A = r.integers(-4, 5, size=(M, K)).astype(np.float32) / 4
    B = r.integers(-4, 5, size=(N, K)).astype(np.float32) / 4
    out = np.zeros((128, N), np.float32)
    rc = lib.tc_probe_run(M, N, K, a_mn, b_mn, neg_a, a_tmem,
                          bf16_bits(A).ctypes.data_as(ctypes.c_void_p),
                          bf16_bits(B).ctypes.data_as(ctypes.c_void_p),
                          out.ctypes.data_as(ctypes.c_void_p))
    assert rc == 0, rc
    ref = (A.astype(np.float64) @ B.T.astype(np.float64)) * (-1.0 if neg_a else 1.0)
    return out, ref


@pytest.mark.parametrize("M,N,K", [(128, 64, 64), (128, 128, 128), (128, 16, 128), (128, 32, 128),
                                   (128, 48, 128), (128, 256, 64), (128, 64, 16)])
def test_kmajor(probe, M, N, K):
    out, ref = run(probe, M, N, K)
    assert np.array_equal(out[:M], ref)


@pytest.mark.parametrize("a_mn,b_mn", [(1, 0), (0, 1), (1, 1)])
def test_mn_major(probe, a_mn, b_mn):
    out, ref = run(probe, 128, 128, 64, a_mn=a_mn, b_mn=b_mn, seed=3)
    assert np.array_equal(out[:128], ref)


def test_negate_a(probe):
    out, ref = run(probe, 128, 64, 64, neg_a=1, seed=4)
    assert np.array_equal(out, ref)


def test_m64_lane_layout(probe):
    """M = 64: row r of D sits in TMEM lane 32*(r // 16) + r % 16."""
    out, ref = run(probe, 64, 64, 64, seed=5)
    lanes = np.array([32 * (r // 16) + r % 16 for r in range(64)])
    found = {r: [int(l) for l in range(128) if np.array_equal(out[l], ref[r])] for r in range(64)}
    assert np.array_equal(out[lanes], ref), f"row -> lanes holding it: {found}"


@pytest.mark.parametrize("N,K,b_mn", [(64, 128, 0), (128, 64, 0), (192, 64, 0), (128, 128, 1)])
def test_a_from_tensor_memory(probe, N, K, b_mn):
    """A in TMEM (row m in lane m, bf16 pairs along the columns, lower K index in the low
    half), B from shared memory."""
    out, ref = run(probe, 128, N, K, b_mn=b_mn, a_tmem=1, seed=7 + N + K)
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("b_mn", [0, 1])
def test_m64_n32_k32(probe, b_mn):
    """The small solve products: M = 64, N = 32, K = 32 (two K steps of a 64-wide tile), B
    K-major or MN-major (half of one 64-element panel)."""
    out, ref = run(probe, 64, 32, 32, b_mn=b_mn, seed=9 + b_mn)
    lanes = np.array([32 * (r // 16) + r % 16 for r in range(64)])
    assert np.array_equal(out[lanes], ref)
