"""Failure detection on the device without a GPU fault: a wait limit far
shorter than a TMA copy makes the first bounded mbarrier wait run out.  The
kernel records MOE_ERR_TIMEOUT in the workspace status word and stops cleanly
(its copies in flight drained, its TMEM freed); every later stage sees the
word and skips its work.  The host reads the status, and the next call on the
same workspace and context runs normally.

The one-CTA expert GEMM is selected: its copies complete on its own barriers,
which it drains before exiting.  In a CTA pair, copies complete on the
leader's barriers, so a one-sided abort is not exercised here."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import check_routing, check_y, device_inputs, run

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def test_wait_limit_reports_timeout_and_the_next_call_runs():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=512, d=256, f=512)
    inp = si.layer_inputs(cfg, seed=41)
    dinp = device_inputs(inp)
    out = run(cfg, dinp, timeout_ns=1, gemm_single_cta=True)
    assert moe.check_device_errors(out.workspace) == MOE_ERR_TIMEOUT
    # the same workspace and context, default limit: a normal, correct call
    out2 = run(cfg, dinp, workspace=out.workspace, gemm_single_cta=True)
    assert moe.check_device_errors(out2.workspace) == 0
    ref, gl, _ = check_routing(cfg, inp, out2)
    check_y(cfg, inp, out2, gl, np.arange(cfg.T))


def test_grouped_gemm_wait_limit_reports_timeout():
    G, M, K, N = 3, 600, 256, 256
    A = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    B = (torch.randn(G, K, N, device="cuda") / 16).to(torch.bfloat16)
    offs = torch.tensor([0, 200, 450, 600], dtype=torch.int32, device="cuda")
    ws = torch.empty((moe.lib().moe_grouped_gemm_workspace_size(G),), dtype=torch.uint8, device="cuda")
    moe.grouped_gemm(moe.BF16, moe.NONE, offs, A, B, workspace=ws, timeout_ns=1, single_cta=True)
    assert moe.check_device_errors(ws) == MOE_ERR_TIMEOUT
    C, _ = moe.grouped_gemm(moe.BF16, moe.NONE, offs, A, B, workspace=ws, single_cta=True)
    assert moe.check_device_errors(ws) == 0
    ref = torch.cat([A[offs[g]:offs[g + 1]].float() @ B[g].float() for g in range(G)])
    err = (C.float() - ref).abs().max().item()
    assert err <= 2e-2 * ref.abs().max().item()
