"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the worked
top-k example printed in "手撕一个极简 MoE-FFN" §三, brute force over all subsets,
closed forms (uniform routing gives L_aux = alpha), hand-derived capacity cases,
and special cases that reduce to library routines (numpy matmul, numpy
lexsort, scipy erf / expit).  They are chosen so that a dropped term, a wrong
sign or index, or a transposed operand anywhere in the oracle fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sp

import oracle
import seeded_inputs as si

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _cfg(**kw):
    base = dict(name="pin", T=9, d=16, f=24, E=4, k=2, S=0, act=si.RELU, gating=si.SOFTMAX, dtype=si.F32)
    base.update(kw)
    return si.LayerConfig(**base)


def _rand_inputs(cfg, seed=3):
    return si.layer_inputs(cfg, seed)


# ---- routing --------------------------------------------------------------------

def test_worked_example_topk():
    g = json.load(open(os.path.join(GOLD, "topk_worked_example.json")))
    idx = oracle.topk_row(g["scores"], g["k"])
    assert idx.tolist() == g["indices"]
    # The scores are softmax probabilities: their logarithms are logits that give
    # them back under softmax, so the weights go through the oracle's own gating.
    logits = np.log(np.array([g["scores"]], np.float64))
    w = oracle.topk_weights(logits, idx[None, :], oracle.SOFTMAX)[0]
    np.testing.assert_allclose(w, g["weights"], rtol=0, atol=1e-15)
    assert oracle.topk(logits, g["k"])[0].tolist() == g["indices"]


def _brute_topk(v, k):
    """The unique k-subset S with (v_i > v_j) or (v_i == v_j and i < j) for all
    i in S, j not in S, listed by descending value then ascending index."""
    E = len(v)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all((v[i] > v[j]) or (v[i] == v[j] and i < j) for i in S for j in rest):
            winners.append(S)
    assert len(winners) == 1
    return sorted(winners[0], key=lambda i: (-v[i], i))


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8])
def test_topk_brute_force(E):
    rng = np.random.default_rng(E)
    for trial in range(200):
        k = int(rng.integers(1, E + 1))
        # few distinct values so that ties are common
        v = rng.integers(-3, 4, size=E).astype(np.float64) * 0.25
        if trial % 3 == 0:
            v = rng.standard_normal(E)
        assert oracle.topk_row(v, k).tolist() == _brute_topk(v.tolist(), k)


def test_topk_ties_go_to_lower_index():
    assert oracle.topk_row([0.0] * 8, 3).tolist() == [0, 1, 2]
    assert oracle.topk_row([1.0, 2.0, 2.0, 1.0, 2.0], 2).tolist() == [1, 2]
    assert oracle.topk_row([5.0, 1.0, 5.0, 5.0], 4).tolist() == [0, 2, 3, 1]


def test_k1_weight_is_exactly_one():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((50, 7)) * 3
    for gating in (oracle.SOFTMAX, oracle.SIGMOID_NORM):
        idx = oracle.topk(logits, 1)
        w = oracle.topk_weights(logits, idx, gating)
        assert np.all(w == 1.0)
        assert np.array_equal(idx[:, 0], np.argmax(logits, axis=1))


def test_softmax_probs_sum_to_one_and_match_library():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((40, 16)) * 4
    p = oracle.gate_probs(logits, oracle.SOFTMAX)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(p, sp.softmax(logits, axis=1), rtol=1e-14, atol=0)


def test_softmax_renormalised_topk_is_softmax_of_selected_logits():
    # closed form: p_j / sum_sel p = exp(l_j) / sum_sel exp(l)
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((60, 12)) * 2
    idx = oracle.topk(logits, 4)
    w = oracle.topk_weights(logits, idx, oracle.SOFTMAX)
    sel = np.take_along_axis(logits, idx.astype(np.int64), 1)
    np.testing.assert_allclose(w, sp.softmax(sel, axis=1), rtol=1e-14, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)          # listed in descending order


def test_normalised_sigmoid_gating():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((30, 64)) * 3
    p = oracle.gate_probs(logits, oracle.SIGMOID_NORM)
    s = sp.expit(logits)
    np.testing.assert_allclose(p, s / s.sum(1, keepdims=True), rtol=1e-14, atol=0)
    idx = oracle.topk(logits, 6)
    w = oracle.topk_weights(logits, idx, oracle.SIGMOID_NORM)
    ssel = np.take_along_axis(s, idx.astype(np.int64), 1)
    np.testing.assert_allclose(w, ssel / ssel.sum(1, keepdims=True), rtol=1e-14, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", [si.F32, si.BF16])
@pytest.mark.parametrize("bias", [True, False])
def test_router_logits_match_library_matmul(dtype, bias):
    cfg = _cfg(T=33, d=48, E=5, dtype=dtype, router_bias=bias)
    inp = _rand_inputs(cfg)
    l = oracle.router_logits(inp["x"], inp["W_g"], inp["b_g"], dtype)
    x = si.as_f32(inp["x"]).astype(np.float64)
    W = si.as_f32(inp["W_g"]).astype(np.float64)
    ref = x @ W
    if bias:
        ref = ref + si.as_f32(inp["b_g"]).astype(np.float64)[None, :]
    np.testing.assert_allclose(l, ref, rtol=1e-13, atol=1e-13)


# ---- activations ----------------------------------------------------------------

def test_activation_values():
    assert oracle.act(oracle.RELU, -2.5) == 0.0 and oracle.act(oracle.RELU, 1.75) == 1.75
    # GELU(z) = z * Phi(z); Phi(1) = 0.841344746068543 (standard normal table)
    assert oracle.act(oracle.GELU, 0.0) == 0.0
    assert abs(oracle.act(oracle.GELU, 1.0) - 0.841344746068543) < 1e-14
    assert abs(oracle.act(oracle.GELU, -1.0) + (1 - 0.841344746068543)) < 1e-14
    assert abs(oracle.act(oracle.GELU, 12.0) - 12.0) < 1e-15
    assert abs(oracle.act(oracle.GELU, -12.0)) < 1e-30
    z = np.linspace(-8, 8, 97)
    g = np.array([oracle.act(oracle.GELU, v) for v in z])
    # 1 + erf(z / sqrt 2) cancels for z << 0: allow fp64 cancellation, |z| * 2^-52
    np.testing.assert_allclose(g, z * 0.5 * sp.erfc(-z / np.sqrt(2)), rtol=1e-13, atol=8 * 2.0 ** -52)
    s = np.array([oracle.act(oracle.SWIGLU, v) for v in z])
    np.testing.assert_allclose(s, z * sp.expit(z), rtol=1e-14, atol=1e-300)


# ---- experts and the weighted sum ------------------------------------------------

def _dense_ffn(cfg, inp, g, x):
    """Expert g on all rows of x with library matmuls (numpy, fp64)."""
    f64 = lambda a: None if a is None else si.as_f32(a).astype(np.float64)
    W1, W2 = f64(inp["W1"])[g], f64(inp["W2"])[g]
    if cfg.act == si.SWIGLU:
        W3 = f64(inp["W3"])[g]
        a = x @ W1
        return (a * sp.expit(a) * (x @ W3)) @ W2
    h = x @ W1
    if inp["b1"] is not None:
        h = h + f64(inp["b1"])[g]
    h = np.maximum(h, 0) if cfg.act == si.RELU else 0.5 * h * sp.erfc(-h / np.sqrt(2))
    o = h @ W2
    if inp["b2"] is not None:
        o = o + f64(inp["b2"])[g]
    return o


@pytest.mark.parametrize("act", [si.RELU, si.GELU, si.SWIGLU])
@pytest.mark.parametrize("dtype", [si.F32, si.BF16])
def test_identical_experts_with_k_equal_E_is_the_dense_ffn(act, dtype):
    cfg = _cfg(T=11, d=16, f=40, E=4, k=4, act=act, dtype=dtype, ffn_bias=(act != si.SWIGLU))
    inp = _rand_inputs(cfg)
    for name in ("W1", "W2", "W3", "b1", "b2"):
        if inp[name] is not None:
            inp[name] = np.ascontiguousarray(np.broadcast_to(inp[name][:1], inp[name].shape))
    out = oracle.forward(cfg, inp)
    x = si.as_f32(inp["x"]).astype(np.float64)
    np.testing.assert_allclose(out["y"], _dense_ffn(cfg, inp, 0, x), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act,gating,cf,S", [
    (si.RELU, si.SOFTMAX, 0.0, 0),
    (si.GELU, si.SOFTMAX, 1.0, 0),
    (si.SWIGLU, si.SIGMOID_NORM, 0.0, 2),
    (si.SWIGLU, si.SOFTMAX, 0.75, 1),
])
def test_sparse_equals_dense_masked(act, gating, cf, S):
    """Run every expert on every token and mask afterwards (the dense-masked
    formulation of the MoELayer in "Mixture of Experts混合专家模型架构原理与路由策略实现"), with capacity drops and shared
    experts; it must equal the oracle's sparse grouped result."""
    cfg = _cfg(T=23, d=16, f=32, E=6, k=3, S=S, act=act, gating=gating, capacity_factor=cf,
               ffn_bias=(act != si.SWIGLU), dtype=si.BF16)
    inp = _rand_inputs(cfg, seed=7)
    out = oracle.forward(cfg, inp)
    x = si.as_f32(inp["x"]).astype(np.float64)
    y = np.zeros((cfg.T, cfg.d))
    gate = np.zeros((cfg.T, cfg.E))
    for t in range(cfg.T):
        for j in range(cfg.k):
            if not out["dropped"][t, j]:
                gate[t, out["topk_idx"][t, j]] += out["topk_w"][t, j]
    for e in range(cfg.E):
        y += gate[:, e:e + 1] * _dense_ffn(cfg, inp, e, x)
    for s in range(S):
        y += _dense_ffn(cfg, inp, cfg.E + s, x)
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)
    if cf > 0:
        assert out["dropped"].sum() > 0      # the case really exercises drops


# ---- capacity, drops, grouped order ------------------------------------------------

def test_capacity_formula():
    assert oracle.capacity(8192, 16, 1.25) == 640
    assert oracle.capacity(10, 3, 1.0) == 4
    assert oracle.capacity(8, 2, 1.0) == 4
    assert oracle.capacity(100, 8, 0.0) == -1
    assert oracle.capacity(100, 8, -1.0) == -1


def test_capacity_hand_cases():
    g = json.load(open(os.path.join(GOLD, "capacity_hand_cases.json")))
    for c in g["cases"]:
        C = oracle.capacity(c["T"], c["E"], c["capacity_factor"])
        assert C == c["capacity"], c["name"]
        d = oracle.dispatch(np.array(c["topk_idx"], np.int32), c["E"], C)
        for key in ("n_pre", "counts", "offsets", "dropped", "slot", "perm"):
            assert d[key].tolist() == c[key], (c["name"], key)


@pytest.mark.parametrize("cf", [0.0, 0.5, 1.0, 1.25, 3.0])
def test_dispatch_invariants(cf):
    rng = np.random.default_rng(11)
    T, E, k = 257, 9, 3
    logits = rng.standard_normal((T, E)) + np.linspace(0, 2.5, E)   # skewed
    idx = oracle.topk(logits, k)
    C = oracle.capacity(T, E, cf)
    d = oracle.dispatch(idx, E, C)
    assert np.array_equal(d["n_pre"], np.bincount(idx.ravel(), minlength=E))
    expect_counts = d["n_pre"] if C < 0 else np.minimum(d["n_pre"], C)
    assert np.array_equal(d["counts"], expect_counts)
    assert d["counts"].sum() == T * k - d["dropped"].sum()
    if C < 0:
        assert d["dropped"].sum() == 0
    assert np.array_equal(d["offsets"], np.concatenate([[0], np.cumsum(d["counts"])]))
    # grouped order: the kept (expert, token) keys sorted stably (library lexsort)
    kept = d["dropped"] == 0
    tok = np.repeat(np.arange(T), k).reshape(T, k)[kept]
    exp = idx[kept]
    order = np.lexsort((tok, exp))
    assert np.array_equal(d["perm"], tok[order])
    # slot is a bijection from kept assignments onto 0..total-1, consistent with perm
    s = d["slot"][kept]
    assert np.array_equal(np.sort(s), np.arange(d["counts"].sum()))
    assert np.array_equal(d["perm"][s], tok)
    assert np.all(d["slot"][~kept] == -1)
    # kept are exactly the first C arrivals of each expert in token order
    if C >= 0:
        for e in range(E):
            arrivals = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
            for r, (t, j) in enumerate(arrivals):
                assert d["dropped"][t, j] == (1 if r >= C else 0)


# ---- balance statistics -------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("gating", [si.SOFTMAX, si.SIGMOID_NORM])
def test_laux_is_alpha_under_uniform_router(k, gating):
    """All-zero router: every P_i = 1/E; ties send every token to experts
    0..k-1, so f_i = 1/k there.  Then L_aux = alpha * E * k * (1/k)(1/E) = alpha."""
    E, T, alpha = 8, 64, 0.01
    cfg = _cfg(T=T, d=16, E=E, k=k, gating=gating, alpha=alpha)
    inp = _rand_inputs(cfg)
    inp["W_g"] = np.zeros_like(inp["W_g"])
    inp["b_g"] = np.zeros_like(inp["b_g"])
    r = oracle.routing(cfg, oracle.router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype))
    assert np.all(r["topk_idx"] == np.arange(k))
    np.testing.assert_allclose(r["P"], 1.0 / E, rtol=0, atol=1e-16)
    np.testing.assert_allclose(r["f"][:k], 1.0 / k, rtol=0, atol=0)
    assert abs(r["L_aux"] - alpha) <= 1e-17


def test_laux_is_alpha_when_f_is_uniform():
    """Each expert chosen equally often => f_i = 1/E, so sum_i f_i P_i = 1/E for
    any P that sums to one, and L_aux = alpha."""
    rng = np.random.default_rng(5)
    E, k = 6, 1
    T = 4 * E
    logits = rng.standard_normal((T, E))
    logits[np.arange(T), np.arange(T) % E] += 50.0         # token t picks t mod E
    for gating in (si.SOFTMAX, si.SIGMOID_NORM):
        cfg = _cfg(T=T, E=E, k=k, gating=gating, alpha=0.02)
        r = oracle.routing(cfg, logits)
        np.testing.assert_allclose(r["f"], 1.0 / E, rtol=0, atol=0)
        assert abs(r["L_aux"] - 0.02) <= 1e-16
        np.testing.assert_allclose(r["P"].sum(), 1.0, rtol=0, atol=1e-15)


def test_f_counts_selections_before_the_capacity_cut():
    g = json.load(open(os.path.join(GOLD, "capacity_hand_cases.json")))["cases"][0]
    T, E, k = g["T"], g["E"], g["k"]
    idx = np.array(g["topk_idx"], np.int32)
    probs = np.full((T, E), 1.0 / E)
    d = oracle.dispatch(idx, E, g["capacity"])
    f, P, L = oracle.balance(d["n_pre"], probs, k, 1.0)
    np.testing.assert_allclose(f, [6 / 8, 2 / 8], rtol=0, atol=0)
    assert abs(L - 1.0) < 1e-15           # uniform P: alpha * E * sum f / E = alpha


def test_empty_batch():
    cfg = _cfg(T=0, d=16, E=4, k=2)
    r = oracle.routing(cfg, np.zeros((0, 4)))
    assert r["counts"].tolist() == [0, 0, 0, 0] and r["L_aux"] == 0.0
    assert np.all(r["f"] == 0) and np.all(r["P"] == 0)


# ---- router noise and routing-health statistics ------------------------------------

def test_noise_alone_decides_routing_when_the_router_is_flat():
    """All-zero W_g and b_g: the noisy scores are the noise itself, so top-k is
    the k largest noise values (library argsort, ties impossible with
    continuous noise) and the weights are the softmax of the selected noise."""
    cfg = _cfg(T=40, d=16, E=7, k=3)
    inp = _rand_inputs(cfg)
    inp["W_g"] = np.zeros_like(inp["W_g"])
    inp["b_g"] = np.zeros_like(inp["b_g"])
    inp["noise"] = si.router_noise(cfg, seed=2, std=1.5)
    out = oracle.forward(cfg, inp, rows=[0])
    nz = inp["noise"].astype(np.float64)
    expect = np.argsort(-nz, axis=1, kind="stable")[:, :3]
    assert np.array_equal(out["topk_idx"], expect)
    sel = np.take_along_axis(nz, expect, 1)
    np.testing.assert_allclose(out["topk_w"], sp.softmax(sel, axis=1), rtol=1e-13, atol=0)
    np.testing.assert_allclose(out["P"], sp.softmax(nz, axis=1).mean(0), rtol=1e-13, atol=0)


def test_zero_noise_changes_nothing_and_noise_shifts_logits_exactly():
    cfg = _cfg(T=25, d=16, E=5, k=2, dtype=si.BF16)
    inp = _rand_inputs(cfg)
    clean = oracle.forward(cfg, inp)
    inp0 = dict(inp, noise=np.zeros((cfg.T, cfg.E), np.float32))
    zero = oracle.forward(cfg, inp0)
    for key in ("topk_idx", "topk_w", "counts", "f", "P", "y"):
        assert np.array_equal(np.asarray(zero[key]), np.asarray(clean[key])), key
    nz = si.router_noise(cfg, seed=4, std=0.7)
    noisy = oracle.forward(cfg, dict(inp, noise=nz))
    np.testing.assert_allclose(noisy["logits"], clean["logits"] + nz.astype(np.float64), rtol=0, atol=1e-15)


def test_route_health_closed_forms():
    E, k, T = 8, 2, 64
    # uniform selections: entropy ln E, variance 0, CV 0
    h = oracle.route_health(np.full(E, T * k // E, np.int32), T, k)
    np.testing.assert_allclose(h, [np.log(E), 0.0, 0.0], rtol=1e-15, atol=1e-15)
    # every selection on one expert (k = 1): entropy 0, CV = sqrt(E - 1)
    n = np.zeros(E, np.int32)
    n[3] = T
    h = oracle.route_health(n, T, 1)
    assert h[0] == 0.0
    np.testing.assert_allclose(h[2], np.sqrt(E - 1), rtol=1e-14)
    np.testing.assert_allclose(h[1], ((1 - 1 / E) ** 2 + (E - 1) / E ** 2) / E, rtol=1e-14)
    # against library routines on random counts
    rng = np.random.default_rng(9)
    n = rng.integers(0, 50, size=E).astype(np.int32)
    n[0] += 1
    T = int(n.sum())
    h = oracle.route_health(n, T, 1)
    f = n / n.sum()
    np.testing.assert_allclose(h[0], sp.entr(f).sum(), rtol=1e-13)
    np.testing.assert_allclose(h[1], np.var(f), rtol=1e-13)
    np.testing.assert_allclose(h[2], np.std(n) / np.mean(n), rtol=1e-13)
    assert np.all(oracle.route_health(np.zeros(E, np.int32), 0, 2) == 0.0)


# ---- expert-choice routing ------------------------------------------------------------

def test_ec_capacity():
    assert oracle.ec_capacity(16384, 8, 2, 0.0) == 4096
    assert oracle.ec_capacity(100, 8, 2, 1.25) == 16          # ceil(100 * 1.25 / 8)
    assert oracle.ec_capacity(10, 2, 3, 0.0) == 10            # capped at T


def test_ec_select_brute_force():
    rng = np.random.default_rng(12)
    for trial in range(60):
        T, E = int(rng.integers(1, 12)), int(rng.integers(1, 6))
        C = int(rng.integers(0, T + 1))
        sc = rng.integers(0, 4, size=(T, E)).astype(np.float64) * 0.25     # many ties
        if trial % 2:
            sc = rng.random((T, E))
        perm = oracle.ec_select(sc, C)
        for e in range(E):
            best = sorted(range(T), key=lambda t: (-sc[t, e], t))[:C]
            assert perm[e].tolist() == sorted(best)


def test_ec_flat_router_takes_the_first_tokens():
    cfg = _cfg(T=20, d=16, E=4, k=2)
    inp = _rand_inputs(cfg)
    inp["W_g"] = np.zeros_like(inp["W_g"])
    inp["b_g"] = np.zeros_like(inp["b_g"])
    out = oracle.ec_forward(cfg, inp, rows=[0])
    C = oracle.ec_capacity(cfg.T, cfg.E, cfg.k, 0.0)
    assert C == 10
    assert np.all(out["perm"] == np.arange(C)[None, :])
    assert np.all(out["counts"] == C)
    assert abs(out["L_aux"] - cfg.alpha) < 1e-17        # f = 1/E and P sums to 1


@pytest.mark.parametrize("act", [si.GELU, si.SWIGLU])
def test_ec_every_token_to_every_expert_is_the_dense_soft_mixture(act):
    """C = T: every expert takes every token, so y = sum_e s[t,e] FFN_e(x_t)
    (numpy matmuls); with identical experts and softmax scores that is FFN(x)."""
    cfg = _cfg(T=9, d=16, f=24, E=3, k=2, act=act, capacity_factor=5.0, ffn_bias=(act != si.SWIGLU))
    inp = _rand_inputs(cfg, seed=5)
    out = oracle.ec_forward(cfg, inp)
    assert out["capacity"] == cfg.T
    x = si.as_f32(inp["x"]).astype(np.float64)
    y = sum(out["probs"][:, e:e + 1] * _dense_ffn(cfg, inp, e, x) for e in range(cfg.E))
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)
    for name in ("W1", "W2", "W3", "b1", "b2"):
        if inp[name] is not None:
            inp[name] = np.ascontiguousarray(np.broadcast_to(inp[name][:1], inp[name].shape))
    out = oracle.ec_forward(cfg, inp)
    np.testing.assert_allclose(out["y"], _dense_ffn(cfg, inp, 0, x), rtol=1e-12, atol=1e-12)


def test_ec_orphan_tokens_get_only_the_shared_experts():
    cfg = _cfg(T=12, d=16, f=24, E=3, k=1, S=1, act=si.SWIGLU, ffn_bias=False, capacity_factor=0.5)
    inp = _rand_inputs(cfg, seed=6)
    out = oracle.ec_forward(cfg, inp)
    chosen = np.zeros(cfg.T, bool)
    chosen[np.unique(out["perm"])] = True
    assert (~chosen).sum() > 0
    x = si.as_f32(inp["x"]).astype(np.float64)
    shared = _dense_ffn(cfg, inp, cfg.E, x)
    np.testing.assert_allclose(out["y"][~chosen], shared[~chosen], rtol=1e-12, atol=1e-12)
    routed = out["y"] - shared
    for t in np.nonzero(chosen)[0]:
        expect = sum(out["probs"][t, e] * _dense_ffn(cfg, inp, e, x[t:t + 1])[0]
                     for e in range(cfg.E) if t in out["perm"][e])
        np.testing.assert_allclose(routed[t], expect, rtol=1e-12, atol=1e-12)
