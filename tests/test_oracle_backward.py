"""The oracle's backward pass against central finite differences of its own
forward pass, in fp64 on tiny layers.

The scalar is L = sum_t <dy_t, y_t> + dL_aux * L_aux.  Routing (top-k and the
capacity cut) is piecewise constant, so a coordinate is only checked when its
perturbation leaves every routing decision unchanged.  Inputs are stored in
fp32, so each perturbed value is the fp32 neighbour actually stored, and the
difference quotient divides by that stored difference."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si


def _cfg(**kw):
    base = dict(name="bwd", T=7, d=8, f=12, E=4, k=2, S=0, act=si.GELU, gating=si.SOFTMAX, dtype=si.F32)
    base.update(kw)
    return si.LayerConfig(**base)


def _loss(cfg, inp, dy, dL_aux):
    out = oracle.forward(cfg, inp)
    return float(np.sum(dy * out["y"]) + dL_aux * out["L_aux"]), out


def _fd_check(cfg, inp, dy, dL_aux, names, n_coords=5, seed=0, h=2.0 ** -10):
    g = oracle.backward(cfg, inp, dy, dL_aux)
    _, base = _loss(cfg, inp, dy, dL_aux)
    rng = np.random.default_rng(seed)
    key = {"x": "dx", "W_g": "dW_g", "b_g": "db_g", "W1": "dW1", "b1": "db1", "W2": "dW2", "b2": "db2", "W3": "dW3"}
    checked = 0
    for name in names:
        arr = inp[name]
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, size=min(n_coords, flat.size), replace=False):
            v0 = flat[i]
            vp, vm = np.float32(v0 + h), np.float32(v0 - h)
            flat[i] = vp
            lp, op = _loss(cfg, inp, dy, dL_aux)
            flat[i] = vm
            lm, om = _loss(cfg, inp, dy, dL_aux)
            flat[i] = v0
            same = all(np.array_equal(o["topk_idx"], base["topk_idx"]) and np.array_equal(o["dropped"], base["dropped"])
                       for o in (op, om))
            if not same:
                continue
            fd = (lp - lm) / (float(vp) - float(vm))
            an = g[key[name]].reshape(-1)[i]
            scale = max(1.0, np.abs(g[key[name]]).max())
            assert abs(fd - an) <= 2e-5 * scale, (name, i, fd, an)
            checked += 1
    assert checked >= len(names) * n_coords // 2
    return g


def test_backward_gelu_softmax_capacity_bias_noise():
    cfg = _cfg(capacity_factor=0.9, router_bias_std=0.5)
    inp = si.layer_inputs(cfg, seed=3)
    inp["noise"] = si.router_noise(cfg, seed=3, std=0.3)
    dy = np.random.default_rng(1).standard_normal((cfg.T, cfg.d))
    g = _fd_check(cfg, inp, dy, 0.7, ["x", "W_g", "b_g", "W1", "b1", "W2", "b2"])
    assert g["routing"]["dropped"].sum() > 0          # the capacity cut is exercised


def test_backward_swiglu_sigmoid_shared():
    cfg = _cfg(act=si.SWIGLU, gating=si.SIGMOID_NORM, S=1, k=3, E=5, ffn_bias=False)
    inp = si.layer_inputs(cfg, seed=4)
    dy = np.random.default_rng(2).standard_normal((cfg.T, cfg.d))
    _fd_check(cfg, inp, dy, 1.3, ["x", "W_g", "b_g", "W1", "W2", "W3"], seed=1)


def test_backward_only_aux_reaches_only_the_router():
    """dy = 0: the expert weights get no gradient, the router only through L_aux."""
    cfg = _cfg(act=si.SWIGLU, ffn_bias=False)
    inp = si.layer_inputs(cfg, seed=5)
    g = oracle.backward(cfg, inp, np.zeros((cfg.T, cfg.d)), 1.0)
    for key in ("dW1", "dW2", "dW3"):
        assert np.all(g[key] == 0.0)
    assert np.abs(g["dW_g"]).max() > 0
    g0 = oracle.backward(cfg, inp, np.zeros((cfg.T, cfg.d)), 0.0)
    assert np.all(g0["dW_g"] == 0.0) and np.all(g0["dx"] == 0.0)


# ---- expert-choice routing --------------------------------------------------------

def _ec_loss(cfg, inp, dy, dL_aux):
    out = oracle.ec_forward(cfg, inp)
    return float(np.sum(dy * out["y"]) + dL_aux * out["L_aux"]), out


def _ec_fd_check(cfg, inp, dy, dL_aux, names, n_coords=5, seed=0, h=2.0 ** -10):
    g = oracle.ec_backward(cfg, inp, dy, dL_aux)
    _, base = _ec_loss(cfg, inp, dy, dL_aux)
    assert np.array_equal(g["perm"], base["perm"])
    rng = np.random.default_rng(seed)
    key = {"x": "dx", "W_g": "dW_g", "b_g": "db_g", "W1": "dW1", "b1": "db1", "W2": "dW2", "b2": "db2", "W3": "dW3"}
    checked = 0
    for name in names:
        flat = inp[name].reshape(-1)
        for i in rng.choice(flat.size, size=min(n_coords, flat.size), replace=False):
            v0 = flat[i]
            vp, vm = np.float32(v0 + h), np.float32(v0 - h)
            flat[i] = vp
            lp, op = _ec_loss(cfg, inp, dy, dL_aux)
            flat[i] = vm
            lm, om = _ec_loss(cfg, inp, dy, dL_aux)
            flat[i] = v0
            if not all(np.array_equal(o["perm"], base["perm"]) for o in (op, om)):
                continue                                # the choice moved: not differentiable here
            fd = (lp - lm) / (float(vp) - float(vm))
            an = g[key[name]].reshape(-1)[i]
            scale = max(1.0, np.abs(g[key[name]]).max())
            assert abs(fd - an) <= 2e-5 * scale, (name, i, fd, an)
            checked += 1
    assert checked >= len(names) * n_coords // 2
    return g


def test_ec_backward_gelu_softmax_bias_noise_unchosen_tokens():
    cfg = _cfg(T=9, expert_choice=True, capacity_factor=0.5, router_bias_std=0.5)
    inp = si.layer_inputs(cfg, seed=6)
    inp["noise"] = si.router_noise(cfg, seed=6, std=0.3)
    dy = np.random.default_rng(3).standard_normal((cfg.T, cfg.d))
    g = _ec_fd_check(cfg, inp, dy, 0.7, ["x", "W_g", "b_g", "W1", "b1", "W2", "b2"])
    chosen = np.zeros(cfg.T, bool)
    chosen[np.unique(g["perm"])] = True
    assert (~chosen).any()                              # a token no expert chose: dx from nothing
    t = int(np.flatnonzero(~chosen)[0])
    # an unchosen token's only path to the loss is the aux term, whose gradient vanishes
    assert np.abs(g["dx"][t]).max() <= 1e-12


def test_ec_backward_swiglu_sigmoid_shared():
    cfg = _cfg(act=si.SWIGLU, gating=si.SIGMOID_NORM, S=1, k=2, E=5, ffn_bias=False, expert_choice=True)
    inp = si.layer_inputs(cfg, seed=7)
    dy = np.random.default_rng(4).standard_normal((cfg.T, cfg.d))
    _ec_fd_check(cfg, inp, dy, 1.3, ["x", "W_g", "b_g", "W1", "W2", "W3"], seed=2)


@pytest.mark.parametrize("gating", [si.SOFTMAX, si.SIGMOID_NORM])
def test_ec_backward_with_every_token_chosen_is_the_top_E_token_choice_backward(gating):
    """C = T: every expert chooses every token, so y = sum_e p_e o_e, which is
    token choice with k = E (the top-E weights renormalised over all E are p
    itself) and f_e = 1/E in both: the two independently written backward
    passes must agree."""
    cfg = _cfg(T=6, E=3, k=3, S=1, gating=gating, act=si.GELU, router_bias_std=0.3)
    inp = si.layer_inputs(cfg, seed=8)
    dy = np.random.default_rng(5).standard_normal((cfg.T, cfg.d))
    tc = oracle.backward(cfg, inp, dy, 0.9)
    ec = oracle.ec_backward(cfg.replace(expert_choice=True, capacity_factor=float(cfg.E)), inp, dy, 0.9)
    assert ec["capacity"] == cfg.T
    for key in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2"):
        np.testing.assert_allclose(ec[key], tc[key], rtol=1e-10, atol=1e-12 * max(1.0, np.abs(tc[key]).max()))


def test_ec_aux_loss_is_constant_so_it_carries_no_gradient():
    """With expert choice f_e = 1/E, so L_aux = alpha sum_e P_e = alpha for any
    logits: dy = 0 leaves every gradient at rounding level."""
    cfg = _cfg(act=si.SWIGLU, ffn_bias=False, expert_choice=True, gating=si.SIGMOID_NORM)
    inp = si.layer_inputs(cfg, seed=9)
    assert abs(oracle.ec_forward(cfg, inp)["L_aux"] - cfg.alpha) <= 1e-15
    g = oracle.ec_backward(cfg, inp, np.zeros((cfg.T, cfg.d)), 1.0)
    for key in ("dW1", "dW2", "dW3"):
        assert np.all(g[key] == 0.0)
    assert np.abs(g["dW_g"]).max() <= 1e-15 and np.abs(g["dx"]).max() <= 1e-15


# ---- dx of single tokens (the sampled full-size checks use these) ------------------

@pytest.mark.parametrize("over", [dict(capacity_factor=0.9), dict(act=si.SWIGLU, gating=si.SIGMOID_NORM, S=1,
                                                                  k=3, E=5, ffn_bias=False)])
def test_dx_rows_equal_the_backward_pass_without_the_aux_term(over):
    cfg = _cfg(**over)
    inp = si.layer_inputs(cfg, seed=10)
    dy = np.random.default_rng(6).standard_normal((cfg.T, cfg.d))
    g = oracle.backward(cfg, inp, dy, 0.0)
    r = g["routing"]
    rows = [0, 3, cfg.T - 1]
    lg = oracle.router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype)
    dx = oracle.dx_rows(cfg, inp, rows, dy[rows], lg[rows], r["topk_idx"][rows], r["topk_w"][rows],
                        r["dropped"][rows])
    np.testing.assert_allclose(dx, g["dx"][rows], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("over", [dict(capacity_factor=0.5, router_bias_std=0.5),
                                  dict(act=si.SWIGLU, gating=si.SIGMOID_NORM, S=1, E=5, ffn_bias=False)])
def test_ec_dx_rows_equal_the_expert_choice_backward_without_the_aux_term(over):
    cfg = _cfg(T=9, expert_choice=True, **over)
    inp = si.layer_inputs(cfg, seed=11)
    dy = np.random.default_rng(7).standard_normal((cfg.T, cfg.d))
    g = oracle.ec_backward(cfg, inp, dy, 0.0)
    chose = np.zeros((cfg.T, cfg.E), np.uint8)
    for e in range(cfg.E):
        chose[g["perm"][e], e] = 1
    rows = [1, 4, 8]
    dx = oracle.ec_dx_rows(cfg, inp, rows, dy[rows], g["logits"][rows], chose[rows])
    np.testing.assert_allclose(dx, g["dx"][rows], rtol=1e-12, atol=1e-14)
