"""moe_grouped_gemm_noalloc: the grouped GEMM for callers that cannot allocate
device memory at call time (planned-memory hosts, framework plugins, loops
that must not call cudaMalloc); its scratch is a fixed device array inside the
library.

Checked through the C ABI on calls in a row that share that scratch:
- bitwise equal to moe_grouped_gemm (which takes a caller workspace) on the
  same inputs: both run the same deterministic kernels;
- element by element against a plain fp64 evaluation of the same op;
- at the array's limit of 264 groups;
- with options forwarded (the one-CTA kernel, a wait limit, stage events);
- invalid offsets leave C as it was, and the next valid call is unaffected
  (no status or table of the failed call leaks into it).
Collected last on purpose; passes alone or after the rest."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import to_dev, to_host_f32
from test_gpu_grouped_gemm import _ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def _case(seed, G, K, N, act, max_rows=260):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(0, max_rows, size=G)
    offsets = np.concatenate([[3], 3 + np.cumsum(sizes)]).astype(np.int32)
    M = int(offsets[-1]) + 9
    A = si.normal(M * K, seed, 1, dtype=si.BF16).reshape(M, K)
    B = si.normal(G * K * N, seed, 2, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N)
    B3 = si.normal(G * K * N, seed, 3, std=1 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N) \
        if act == moe.SWIGLU else None
    bias = si.normal(G * N, seed, 4, std=0.1, dtype=si.BF16).reshape(G, N) if act == moe.GELU else None
    return offsets, M, (A, B, B3, bias)


def _bits(t):
    return t.view(torch.int16).cpu()


def _check_against_fp64(host, offsets, act, got):
    A, B, B3, bias = host
    ref = _ref(A, B, B3, bias, offsets, act)
    g = to_host_f32(got).astype(np.float64)
    inside = slice(int(offsets[0]), int(offsets[-1]))
    r, gg = ref[inside], g[inside]
    # bf16 output rounding (2^-8 relative) plus fp32 accumulation error, as the
    # grouped-GEMM tests bound it
    tol = 2 ** -8 * np.abs(r) + 1e-3 * np.sqrt(np.mean(r ** 2))
    bad = np.abs(gg - r) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; max err {np.abs(gg - r).max():.3e}"
    assert np.all(g[: offsets[0]] == 5.0) and np.all(g[offsets[-1]:] == 5.0), "rows outside every group written"


CASES = [(21, 6, 256, 192, moe.GELU, 260), (22, 3, 128, 320, moe.SWIGLU, 260),
         (23, 264, 64, 64, moe.NONE, 12)]          # the scratch's limit: 264 groups


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row():
    for seed, G, K, N, act, max_rows in CASES:
        offsets, M, host = _case(seed, G, K, N, act, max_rows)
        A, B, B3, bias = (to_dev(h) for h in host)
        offs = to_dev(offsets)
        C_ref = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        C_ref, ws = moe.grouped_gemm(moe.BF16, act, offs, A, B, B3, bias, C=C_ref)
        assert moe.check_device_errors(ws) == 0
        C_na = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        moe.grouped_gemm_noalloc(moe.BF16, act, offs, A, B, B3, bias, C=C_na)
        torch.cuda.synchronize()
        assert torch.equal(_bits(C_na), _bits(C_ref)), f"case {seed}: not bitwise equal to moe_grouped_gemm"
        _check_against_fp64(host, offsets, act, C_na)


def test_noalloc_forwards_options():
    seed, G, K, N, act, max_rows = CASES[0]
    offsets, M, host = _case(seed, G, K, N, act, max_rows)
    A, B, B3, bias = (to_dev(h) for h in host)
    offs = to_dev(offsets)
    C_ref = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    C_ref, ws = moe.grouped_gemm(moe.BF16, act, offs, A, B, B3, bias, C=C_ref, single_cta=True)
    assert moe.check_device_errors(ws) == 0
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    C_na = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    moe.grouped_gemm_noalloc(moe.BF16, act, offs, A, B, B3, bias, C=C_na, single_cta=True,
                             timeout_ns=500_000_000, stage_events=ev)
    torch.cuda.synchronize()
    assert ev[0].elapsed_time(ev[1]) >= 0.0           # both stage events were recorded around the GEMM
    assert torch.equal(_bits(C_na), _bits(C_ref)), "one-CTA kernel: not bitwise equal to moe_grouped_gemm"
    _check_against_fp64(host, offsets, act, C_na)


def test_noalloc_bad_offsets_leave_C_and_do_not_leak_into_the_next_call():
    seed, G, K, N, act, max_rows = CASES[1]
    offsets, M, host = _case(seed, G, K, N, act, max_rows)
    A, B, B3, bias = (to_dev(h) for h in host)
    for bad in (np.array([0, 40, 30, 50], np.int32),             # decreasing
                np.array([0, 10, 20, M + 1], np.int32),          # past M
                np.array([-1, 10, 20, 30], np.int32)):           # negative
        C_bad = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        moe.grouped_gemm_noalloc(moe.BF16, act, to_dev(bad), A, B, B3, bias, C=C_bad)
        torch.cuda.synchronize()
        assert torch.all(C_bad == 5.0), f"offsets {bad.tolist()}: C was written"
        # the next call, with valid offsets, on the same scratch
        C_ok = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        moe.grouped_gemm_noalloc(moe.BF16, act, to_dev(offsets), A, B, B3, bias, C=C_ok)
        C_ref = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        C_ref, ws = moe.grouped_gemm(moe.BF16, act, to_dev(offsets), A, B, B3, bias, C=C_ref)
        assert moe.check_device_errors(ws) == 0
        assert torch.equal(_bits(C_ok), _bits(C_ref))


def test_noalloc_rejects_more_groups_than_its_scratch_holds():
    K = N = 64
    G = 265
    A = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((G, K, N), dtype=torch.bfloat16, device="cuda")
    offs = torch.zeros((G + 1,), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.grouped_gemm_noalloc(moe.BF16, moe.NONE, offs, A, B)
    assert e.value.status == 2       # MOE_ERR_UNSUPPORTED
