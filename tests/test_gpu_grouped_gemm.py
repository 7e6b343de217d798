"""The tcgen05 grouped GEMM on its own (moe_grouped_gemm), against a plain fp64
reference of the same op on the stored bf16 values."""
import numpy as np
import pytest
import scipy.special as sp
import torch

import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import to_dev, to_host_f32

pytestmark = pytest.mark.gpu


def _ref(A, B, B3, bias, offsets, act):
    A = si.as_f32(A).astype(np.float64)
    B = si.as_f32(B).astype(np.float64)
    out = np.zeros((A.shape[0], B.shape[2]))
    for g in range(B.shape[0]):
        lo, hi = offsets[g], offsets[g + 1]
        z = A[lo:hi] @ B[g]
        if act == moe.SWIGLU:
            u = A[lo:hi] @ si.as_f32(B3).astype(np.float64)[g]
            z = z * sp.expit(z) * u
        else:
            if bias is not None:
                z = z + si.as_f32(bias).astype(np.float64)[g]
            if act == moe.RELU:
                z = np.maximum(z, 0)
            elif act == moe.GELU:
                z = 0.5 * z * sp.erfc(-z / np.sqrt(2))
        out[lo:hi] = z
    return out


@pytest.mark.parametrize("single_cta", [False, True], ids=["cta_pair", "one_cta"])
@pytest.mark.parametrize("act", [moe.NONE, moe.RELU, moe.GELU, moe.SWIGLU])
@pytest.mark.parametrize("shape", [(5, 256, 192), (3, 64, 320), (2, 1024, 256), (4, 128, 640)])
def test_grouped_gemm_bf16(act, shape, single_cta):
    G, K, N = shape
    rng = np.random.default_rng(G * 7 + K + N + act)
    sizes = rng.integers(0, 600, size=G)
    sizes[rng.integers(0, G)] = 0                       # an empty group
    offsets = np.concatenate([[7], 7 + np.cumsum(sizes)]).astype(np.int32)   # rows before the first group
    M = int(offsets[-1]) + 5                            # and after the last
    A = si.normal(M * K, 11, 1, dtype=si.BF16).reshape(M, K)
    B = si.normal(G * K * N, 11, 2, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N)
    B3 = si.normal(G * K * N, 11, 3, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N) if act == moe.SWIGLU else None
    bias = si.normal(G * N, 11, 4, std=0.1, dtype=si.BF16).reshape(G, N) if act in (moe.NONE, moe.GELU) else None
    C0 = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")   # sentinel outside the groups
    C, ws = moe.grouped_gemm(moe.BF16, act, to_dev(offsets), to_dev(A), to_dev(B), to_dev(B3), to_dev(bias), C=C0,
                             single_cta=single_cta)
    assert moe.check_device_errors(ws) == 0
    got = to_host_f32(C).astype(np.float64)
    ref = _ref(A, B, B3, bias, offsets, act)
    inside = np.zeros(M, bool)
    inside[offsets[0]:offsets[-1]] = True
    assert np.all(got[~inside] == 3.0), "rows outside every group were written"
    g, r = got[inside], ref[inside]
    # bf16 output rounding (2^-8 relative) plus fp32 accumulation error
    tol = 2 ** -8 * np.abs(r) + 1e-3 * np.sqrt(np.mean(r ** 2))
    bad = np.abs(g - r) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; max err {np.abs(g - r).max():.3e}"


def test_grouped_gemm_rejects_bad_offsets_on_device():
    G, K, N = 2, 64, 64
    M = 100
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((G, K, N), dtype=torch.bfloat16, device="cuda")
    C0 = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([0, 80, 150], dtype=torch.int32, device="cuda")    # past M
    C, ws = moe.grouped_gemm(moe.BF16, moe.NONE, offs, A, B, C=C0)
    assert moe.check_device_errors(ws) == 6          # MOE_ERR_DEVICE
    assert torch.all(C == 3.0)
