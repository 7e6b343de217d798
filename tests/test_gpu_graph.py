"""The layer captured in a CUDA graph (ForwardGraph) and replayed: bitwise the
same outputs as direct calls, also after the input is changed in place."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import device_inputs, run

pytestmark = pytest.mark.gpu

FIELDS = ("y", "topk_idx", "topk_w", "expert_counts", "dropped_mask", "f", "P", "L_aux", "route_stats")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def _same(a, b):
    for n in FIELDS:
        assert torch.equal(getattr(a, n), getattr(b, n)), n


@pytest.mark.parametrize("base,over", [
    ("gpt2_top2_gelu_bf16", dict(T=300, d=256, f=512)),
    ("skew_capacity_gelu_bf16", dict(T=500, d=256, f=384)),
    ("deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320)),
    ("tiny_top1_relu_f32", {}),
], ids=["gpt2", "skew", "deepseek", "tiny_f32"])
def test_graph_replay_matches_direct_calls(base, over):
    cfg = si.CONFIGS[base].replace(**over)
    inp = si.layer_inputs(cfg, seed=51)
    d = device_inputs(inp)
    g = moe.ForwardGraph(cfg, d["x"], d["W_g"], d["b_g"], d["W1"], d["b1"], d["W2"], d["b2"], d["W3"])
    out = g.replay()
    torch.cuda.synchronize()
    _same(out, run(cfg, d, debug=False))
    # a new batch written into the captured input buffer
    x2 = device_inputs({"x": si.layer_inputs(cfg, seed=52)["x"]})["x"]
    d["x"].copy_(x2)
    out = g.replay()
    torch.cuda.synchronize()
    assert moe.check_device_errors(out.workspace) == 0
    _same(out, run(cfg, d, debug=False))


def test_graph_replay_fp8():
    cfg = si.CONFIGS["mixtral_swiglu_bf16"].replace(T=260, d=512, f=1024)
    inp = si.layer_inputs(cfg, seed=53)
    d = device_inputs(inp)
    ex = moe.quantize_experts_fp8(d["W1"], d["W2"], d["W3"])
    g = moe.ForwardGraph(cfg, d["x"], d["W_g"], d["b_g"], experts=ex)
    out = g.replay()
    torch.cuda.synchronize()
    ref = moe.forward_fp8(cfg, d["x"], d["W_g"], d["b_g"], ex)
    torch.cuda.synchronize()
    _same(out, ref)
