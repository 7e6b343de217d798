"""Expert-choice routing on the GPU against the fp64 oracle.

Integer decisions (the chosen tokens of every expert) are compared bit for bit
with the oracle's selection taken on the GPU's own fp32 scores; the scores
themselves, the statistics and y within tolerance (y's weights are the
oracle's own fp64 gate probabilities)."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import Y_TOL, device_inputs, half_ulp_bf16, run, to_host_f32

pytestmark = pytest.mark.gpu

CASES = [
    ("gpt2_softmax_bias", "gpt2_top2_gelu_bf16", dict(T=300, expert_choice=True)),
    ("gpt2_cf_1", "gpt2_top2_gelu_bf16", dict(T=333, expert_choice=True, capacity_factor=1.0)),
    ("mixtral_swiglu", "mixtral_swiglu_bf16", dict(T=260, d=512, f=1024, expert_choice=True)),
    ("deepseek_sigmoid_shared", "deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320, expert_choice=True)),
    ("skew_cf", "skew_capacity_gelu_bf16", dict(T=500, f=1024, expert_choice=True)),
    ("tiny_f32", "tiny_top1_relu_f32", dict(expert_choice=True, k=2)),
    ("many_experts", "deepseek_shared_sigmoid_bf16", dict(T=700, E=40, k=3, S=0, d=256, f=192, expert_choice=True)),
    ("max_E_shared", "deepseek_shared_sigmoid_bf16", dict(T=300, E=256, k=8, S=2, d=256, f=192, expert_choice=True)),
    # one token: every expert chooses it (C = 1)
    ("one_token", "mixtral_swiglu_bf16", dict(T=1, d=256, f=256, expert_choice=True)),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def _check(cfg, inp, out):
    T, E = cfg.T, cfg.E
    C = moe.capacity(cfg)
    assert C == oracle.ec_capacity(T, E, cfg.k, cfg.capacity_factor)
    gs = out.router_logits.cpu().numpy().astype(np.float64)          # the scores the experts chose on
    ref = oracle.ec_forward(cfg, inp, scores=gs)
    np.testing.assert_allclose(gs, ref["probs"], rtol=2e-3, atol=1e-7)
    perm = out.perm_token.cpu().numpy()[:E * C].reshape(E, C)
    assert np.array_equal(perm, ref["perm"])
    assert np.all(out.expert_counts.cpu().numpy() == C)
    np.testing.assert_allclose(out.f.cpu().numpy(), ref["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(out.P.cpu().numpy(), ref["P"], rtol=1e-5, atol=1e-9)
    la = float(out.L_aux.cpu().numpy()[0])
    assert abs(la - ref["L_aux"]) <= 1e-5 * abs(ref["L_aux"]) + 1e-12
    np.testing.assert_allclose(out.route_stats.cpu().numpy(), [np.log(E), 0.0, 0.0], rtol=1e-6, atol=1e-7)
    # y: tokens no expert chose (and no shared expert) are exactly 0
    y = to_host_f32(out.y).astype(np.float64)
    yr = ref["y"]
    chosen = np.zeros(T, bool)
    chosen[np.unique(ref["perm"])] = True
    skipped = ~chosen if cfg.S == 0 else np.zeros(T, bool)
    assert np.all(y[skipped] == 0.0)
    live = ~skipped
    rms = float(np.sqrt(np.mean(yr[live] ** 2)))
    bound = Y_TOL[cfg.dtype] * rms
    if out.y.dtype == torch.bfloat16:
        bound = bound + half_ulp_bf16(yr[live])
    dy = np.abs(y[live] - yr[live])
    assert np.all(dy <= bound), f"max|dy| {dy.max():.3e}, tol*rms {Y_TOL[cfg.dtype] * rms:.3e}"
    return ref


@pytest.mark.parametrize("label,base,over", CASES, ids=[c[0] for c in CASES])
def test_expert_choice_layer(label, base, over):
    cfg = si.CONFIGS[base].replace(**over)
    inp = si.layer_inputs(cfg, seed=11)
    out = run(cfg, device_inputs(inp))
    assert moe.check_device_errors(out.workspace) == 0
    ref = _check(cfg, inp, out)
    if cfg.capacity_factor > 0 and cfg.capacity_factor < cfg.k:
        chosen = np.zeros(cfg.T, bool)
        chosen[np.unique(ref["perm"])] = True
        assert (~chosen).any()                     # the case really has tokens no expert chose


def test_expert_choice_ties_go_to_the_lower_token():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=200, d=128, f=128, E=4, k=1, expert_choice=True)
    inp = si.layer_inputs(cfg, seed=12)
    inp["W_g"] = np.zeros_like(inp["W_g"])
    inp["b_g"] = np.zeros_like(inp["b_g"])
    out = run(cfg, device_inputs(inp))
    C = moe.capacity(cfg)
    perm = out.perm_token.cpu().numpy()[:cfg.E * C].reshape(cfg.E, C)
    assert np.all(perm == np.arange(C)[None, :])
    _check(cfg, inp, out)


def test_expert_choice_with_router_noise_and_host_buffers():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=300, expert_choice=True)
    inp = si.layer_inputs(cfg, seed=13)
    inp["noise"] = si.router_noise(cfg, seed=13, std=1.0)
    dinp = device_inputs(inp)
    out = run(cfg, dinp)
    _check(cfg, inp, out)
    torch.cuda.synchronize()
    host = moe.forward_host(cfg, dinp["x"].cpu().pin_memory(), dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"],
                            dinp["W2"], dinp["b2"], dinp["W3"], router_noise_host=dinp["noise"].cpu().pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(host.y.view(torch.int16), out.y.cpu().view(torch.int16))
    assert torch.equal(host.expert_counts, out.expert_counts.cpu())


def test_expert_choice_empty_batch():
    """T = 0: nothing is chosen; the statistics are zero and nothing is launched
    that reads a token (also with FP8 experts, and in the backward pass)."""
    cfg = si.CONFIGS["deepseek_shared_sigmoid_bf16"].replace(T=0, d=256, f=192, expert_choice=True)
    inp = si.layer_inputs(cfg.replace(T=1), seed=14)
    dinp = device_inputs(inp)
    x = dinp["x"][:0]
    out = moe.forward(cfg, x, dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], dinp["W3"])
    torch.cuda.synchronize()
    assert moe.check_device_errors(out.workspace) == 0
    assert np.all(out.expert_counts.cpu().numpy() == 0) and float(out.L_aux.cpu()[0]) == 0.0
    ex = moe.quantize_experts_fp8(dinp["W1"], dinp["W2"], dinp["W3"])
    o8 = moe.forward_fp8(cfg, x, dinp["W_g"], dinp["b_g"], ex, dinp["b1"], dinp["b2"])
    torch.cuda.synchronize()
    assert moe.check_device_errors(o8.workspace) == 0
    g = moe.backward(cfg, x, dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], dinp["W3"], x)
    torch.cuda.synchronize()
    for name in ("dW_g", "dW1", "dW2", "dW3"):
        assert torch.all(getattr(g, name) == 0), name


@pytest.mark.parametrize("name", ["mixtral_swiglu_bf16", "deepseek_shared_sigmoid_bf16"])
def test_expert_choice_full_size_sampled(name):
    """The workload shapes at full size, in the bench's launch configuration:
    every expert's choice bit for bit (on the GPU's own probabilities), the
    statistics, and y of sampled tokens against the oracle."""
    cfg = si.CONFIGS[name].replace(expert_choice=True)
    inp = si.layer_inputs(cfg, seed=0)
    out = run(cfg, device_inputs(inp))
    assert moe.check_device_errors(out.workspace) == 0
    T, E = cfg.T, cfg.E
    C = moe.capacity(cfg)
    gs = out.router_logits.cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(15)
    perm = out.perm_token.cpu().numpy()[:E * C].reshape(E, C)
    # sampled tokens: some chosen by several experts, some by none, the ends
    counts = np.bincount(perm.reshape(-1), minlength=T)
    rows = {0, T - 1, int(np.argmax(counts))}
    unchosen = np.flatnonzero(counts == 0)
    if unchosen.size:
        rows.add(int(unchosen[0]))
    while len(rows) < 8:
        rows.add(int(rng.integers(0, T)))
    rows = np.array(sorted(rows))
    ref = oracle.ec_forward(cfg, inp, rows=rows, scores=gs)
    assert np.array_equal(perm, ref["perm"])
    np.testing.assert_allclose(gs, ref["probs"], rtol=2e-3, atol=1e-7)
    np.testing.assert_allclose(out.P.cpu().numpy(), ref["P"], rtol=1e-5, atol=1e-9)
    assert abs(float(out.L_aux.cpu().numpy()[0]) - ref["L_aux"]) <= 1e-5 * abs(ref["L_aux"])
    y = to_host_f32(out.y)[rows].astype(np.float64)
    yr = ref["y"]
    live = np.ones(rows.size, bool) if cfg.S else counts[rows] > 0
    assert np.all(y[~live] == 0.0)
    # RMS over the rows the experts produce, as in the small cases
    rms = float(np.sqrt(np.mean(yr[live] ** 2)))
    dy = np.abs(y[live] - yr[live])
    assert np.all(dy <= Y_TOL[cfg.dtype] * rms + half_ulp_bf16(yr[live])), float(dy.max())
