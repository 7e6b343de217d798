"""moe_grouped_gemm_noalloc: the grouped GEMM for callers that cannot allocate
device memory at call time (planned-memory hosts, framework plugins, loops
that must not call cudaMalloc); its scratch is a fixed device array inside the
library.  Checked through the C ABI against moe_grouped_gemm, which takes a
caller workspace, on two calls in a row: the second call reuses the same
scratch with different groups and shapes, so anything left over from the first
would show.  Collected last on purpose; passes alone or after the rest."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import to_dev, to_host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def _case(seed, G, K, N, act):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(0, 260, size=G)
    offsets = np.concatenate([[3], 3 + np.cumsum(sizes)]).astype(np.int32)
    M = int(offsets[-1]) + 9
    A = si.normal(M * K, seed, 1, dtype=si.BF16).reshape(M, K)
    B = si.normal(G * K * N, seed, 2, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N)
    B3 = si.normal(G * K * N, seed, 3, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N) \
        if act == moe.SWIGLU else None
    bias = si.normal(G * N, seed, 4, std=0.1, dtype=si.BF16).reshape(G, N) if act == moe.GELU else None
    return offsets, M, to_dev(A), to_dev(B), to_dev(B3), to_dev(bias)


def _tol(ref):
    # the grouped-GEMM tests' bound: bf16 output rounding plus fp32 accumulation
    return 2 ** -8 * np.abs(ref) + 1e-3 * np.sqrt(np.mean(ref ** 2))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [(21, 6, 256, 192, moe.GELU), (22, 3, 128, 320, moe.SWIGLU)]
    for seed, G, K, N, act in cases:
        offsets, M, A, B, B3, bias = _case(seed, G, K, N, act)
        offs = to_dev(offsets)
        C_ref = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        C_ref, ws = moe.grouped_gemm(moe.BF16, act, offs, A, B, B3, bias, C=C_ref)
        assert moe.check_device_errors(ws) == 0
        C_na = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        moe.grouped_gemm_noalloc(moe.BF16, act, offs, A, B, B3, bias, C=C_na)
        torch.cuda.synchronize()
        ref = to_host_f32(C_ref).astype(np.float64)
        got = to_host_f32(C_na).astype(np.float64)
        assert np.all(np.abs(got - ref) <= _tol(ref)), f"case {seed}: max diff {np.abs(got - ref).max():.3e}"
        assert np.all(got[: offsets[0]] == 5.0) and np.all(got[offsets[-1]:] == 5.0)


def test_noalloc_rejects_more_groups_than_its_scratch_holds():
    K = N = 64
    G = 265
    A = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((G, K, N), dtype=torch.bfloat16, device="cuda")
    offs = torch.zeros((G + 1,), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.grouped_gemm_noalloc(moe.BF16, moe.NONE, offs, A, B)
    assert e.value.status == 2       # MOE_ERR_UNSUPPORTED
