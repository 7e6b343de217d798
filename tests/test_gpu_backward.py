"""moe_backward on the GPU against the oracle's fp64 backward pass, with
token-choice and expert-choice routing.

Both route on the GPU's own fp32 logits (taken from a forward call, which
computes the very same logits), so every routing decision agrees; with expert
choice both choose on the GPU's own fp32 probabilities.  At the full workload
sizes the oracle computes dx of sampled tokens one at a time (dL_aux = 0).  The GPU
keeps several bf16 intermediates (dO, the pre-activations, H, dA, dU) like the
forward keeps H.  Checks:
- the expert-weight gradients (dW1, dW2, dW3, db1, db2) element by element,
  |error| <= 2 x the first-order error that bf16 storage of those
  intermediates and fp32 accumulation can put in the entry (see
  expert_grad_bounds);
- dx and the router gradients by max-abs error (<= 5e-2 RMS);
- every gradient tensor also by its relative Frobenius error (<= 1e-2; <= 2e-2
  for every expert slab of a weight gradient)."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import device_inputs, run

pytestmark = pytest.mark.gpu

CASES = [
    ("gelu_bias_capacity", "gpt2_top2_gelu_bf16", dict(T=300, d=256, f=512, capacity_factor=1.0), 0.0),
    ("swiglu_mixtral", "mixtral_swiglu_bf16", dict(T=260, d=512, f=1024), 0.0),
    ("sigmoid_shared_fine", "deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320), 0.0),
    ("relu_noise", "gpt2_top2_gelu_bf16", dict(T=200, d=192, f=448, act=si.RELU, E=5, k=3), 0.8),
    ("one_token", "mixtral_swiglu_bf16", dict(T=1, d=256, f=256, S=1), 0.0),
    # the widest routing: 256 experts (8 mask words, 8 tokens per dx warp), k = 8
    ("max_E_and_k", "deepseek_shared_sigmoid_bf16", dict(T=150, E=256, k=8, S=1, d=256, f=192), 0.0),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


# Element-wise bound on the expert-weight gradients: |error| <= 2 x the
# first-order error that the GPU's storage and arithmetic can put in the entry
# (expert_grad_bounds); the factor 2 covers second-order terms.
EW_MARGIN = 2.0


def expert_grad_bounds(cfg, inp, dy, groups):
    """Per expert slab, the first-order worst-case error of each weight-gradient
    entry, in fp64.  ``groups[g] = (tokens, weights)``: the token rows of slab g
    and the gate weight of each (1 for shared experts).

    The GPU keeps bf16 copies (relative error r = 2^-8 each) of dO = w dy, of
    H and of the pre-activations a = x W1 + b1, u = x W3, and of dA and dU; its
    dot products accumulate in fp32 (error <= n 2^-24 sum|terms| over n terms).
    Propagated to first order, with S = |dO| |W2|^T and s = silu, g = gelu:
      e_a = d 2^-24 |x||W1|,  e_u = d 2^-24 |x||W3|        (fp32 a, u)
      E_a = r|a| + e_a,  E_u = r|u| + e_u                  (stored a, u)
      E_H = r|H| + |dH/da| e_a + |dH/du| e_u               (stored H)
      E_dH = (r + d 2^-24) S,  E_dO = r|dO|
      SwiGLU: E_dA = r|dA| + E_dH|u s'| + |dH s'| E_u + |dH u s''| E_a
              E_dU = r|dU| + E_dH|s| + |dH s'| E_a
      GELU:   E_dA = r|dA| + E_dH|g'| + |dH g''| E_a
      ReLU:   E_dA = r|dA| + E_dH [a > 0]
    and dW2 = H^T dO, dW1 = X^T dA, dW3 = X^T dU, db1 = sum dA, db2 = sum dO:
      |dW2 err| <= E_H^T |dO| + |H|^T E_dO,  |dW1 err| <= |X|^T E_dA,
      |dW3 err| <= |X|^T E_dU,  |db1 err| <= sum E_dA,  |db2 err| <= sum E_dO,
    each plus the fp32 accumulation over the slab's rows."""
    import scipy.special as sp
    r = 2.0 ** -8
    x = si.as_f32(inp["x"]).astype(np.float64)
    dyf = np.asarray(dy, np.float64)
    W1 = si.as_f32(inp["W1"]).astype(np.float64)
    W2 = si.as_f32(inp["W2"]).astype(np.float64)
    W3 = si.as_f32(inp["W3"]).astype(np.float64) if inp["W3"] is not None else None
    b1 = si.as_f32(inp["b1"]).astype(np.float64) if inp["b1"] is not None else None
    G = len(groups)
    f, d = cfg.f, cfg.d
    gd = d * 2.0 ** -24
    out = {"dW1": np.zeros((G, d, f)), "dW2": np.zeros((G, f, d)), "db1": np.zeros((G, f)), "db2": np.zeros((G, d))}
    if cfg.act == si.SWIGLU:
        out["dW3"] = np.zeros((G, d, f))
    for g, (tt, w) in enumerate(groups):
        if len(tt) == 0:
            continue
        n = len(tt)
        ga = n * 2.0 ** -24                       # fp32 accumulation over the slab's rows
        X = x[tt]
        aX = np.abs(X)
        dO = np.asarray(w, np.float64)[:, None] * dyf[tt]
        a = X @ W1[g] + (b1[g] if b1 is not None else 0.0)
        e_a = gd * (aX @ np.abs(W1[g]))
        E_a = r * np.abs(a) + e_a
        dH = dO @ W2[g].T
        E_dH = (r + gd) * (np.abs(dO) @ np.abs(W2[g]).T)
        if cfg.act == si.SWIGLU:
            u = X @ W3[g]
            e_u = gd * (aX @ np.abs(W3[g]))
            E_u = r * np.abs(u) + e_u
            sg = sp.expit(a)
            s0 = a * sg
            s1 = sg * (1 + a * (1 - sg))
            s2 = sg * (1 - sg) * (2 + a * (1 - 2 * sg))
            H = s0 * u
            E_H = r * np.abs(H) + np.abs(s1 * u) * e_a + np.abs(s0) * e_u
            dA, dU = dH * u * s1, dH * s0
            E_dA = r * np.abs(dA) + E_dH * np.abs(u * s1) + np.abs(dH * s1) * E_u + np.abs(dH * u * s2) * E_a
            E_dU = r * np.abs(dU) + E_dH * np.abs(s0) + np.abs(dH * s1) * E_a
            out["dW3"][g] = aX.T @ E_dU + ga * (aX.T @ np.abs(dU))
        elif cfg.act == si.GELU:
            phi = np.exp(-0.5 * a * a) / np.sqrt(2 * np.pi)
            g1 = 0.5 * sp.erfc(-a / np.sqrt(2)) + a * phi
            g2 = phi * (2 - a * a)
            H = a * 0.5 * sp.erfc(-a / np.sqrt(2))
            E_H = r * np.abs(H) + np.abs(g1) * e_a
            dA = dH * g1
            E_dA = r * np.abs(dA) + E_dH * np.abs(g1) + np.abs(dH * g2) * E_a
        else:
            pos = (a > 0).astype(np.float64)
            H = np.maximum(a, 0.0)
            E_H = r * np.abs(H) + pos * e_a
            dA = dH * pos
            E_dA = r * np.abs(dA) + E_dH * pos
        out["dW1"][g] = aX.T @ E_dA + ga * (aX.T @ np.abs(dA))
        out["db1"][g] = E_dA.sum(axis=0) + ga * np.abs(dA).sum(axis=0)
        out["dW2"][g] = E_H.T @ np.abs(dO) + r * (np.abs(H).T @ np.abs(dO)) + ga * (np.abs(H).T @ np.abs(dO))
        out["db2"][g] = (r + ga) * np.abs(dO).sum(axis=0)
    return out


def token_choice_groups(cfg, routing):
    idx, w, dropped = routing["topk_idx"], routing["topk_w"], routing["dropped"]
    groups = []
    for e in range(cfg.E):
        tt, jj = np.nonzero((idx == e) & (dropped == 0))
        groups.append((tt, w[tt, jj]))
    for _ in range(cfg.S):
        groups.append((np.arange(cfg.T), np.ones(cfg.T)))
    return groups


def check_expert_grads_elementwise(g, ref, bounds):
    for name, eb in bounds.items():
        got = getattr(g, name)
        if got is None:
            continue
        got = got.cpu().numpy().astype(np.float64)
        err = np.abs(got - ref[name])
        rel = err / np.maximum(eb, 1e-300)
        ratio = float(rel.max())
        w = np.unravel_index(int(np.argmax(rel)), rel.shape)
        print(f"{name}: max |error| / first-order bound = {ratio:.3e} (allowed {EW_MARGIN:.1f}) at "
              f"{tuple(int(i) for i in w)}: got {got[w]:.6e} ref {ref[name][w]:.6e} bound {eb[w]:.3e}")
        assert np.all(err <= EW_MARGIN * eb), f"{name}: max |error| / bound = {ratio:.3e} at {tuple(int(i) for i in w)}"


def _close(name, got, ref, fro_tol=1e-2, max_tol=5e-2):
    """Relative Frobenius error of the whole tensor <= fro_tol.  Stacked weight
    gradients (one slab per expert): also each slab's relative Frobenius error
    <= 2 fro_tol, so one wrong slab or tile cannot hide in the total.  A slab
    entry is a sum of x_r dA_r over the expert's rows, so with few rows the
    entries are heavy-tailed products and a max-abs bound against the RMS says
    little; dx, dW_g, db_g get max-abs error <= max_tol RMS."""
    got = got.cpu().numpy().astype(np.float64)
    if np.sqrt(np.mean(ref ** 2)) == 0.0:
        assert np.all(got == 0.0), name
        return
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert fro <= fro_tol, f"{name}: rel. Frobenius {fro:.2e}"
    if name in ("dW1", "dW2", "dW3", "db1", "db2"):
        for g, (gs, rs) in enumerate(zip(got.reshape(got.shape[0], -1), ref.reshape(ref.shape[0], -1))):
            nr = np.linalg.norm(rs)
            if nr == 0.0:
                assert np.all(gs == 0.0), (name, g)
                continue
            sf = float(np.linalg.norm(gs - rs) / nr)
            assert sf <= 2 * fro_tol, f"{name}[{g}]: rel. Frobenius {sf:.2e}"
    else:
        mx = float(np.abs(got - ref).max()) / float(np.sqrt(np.mean(ref ** 2)))
        assert mx <= max_tol, f"{name}: max/RMS {mx:.2e}"


# The router's logit gradient of a token with k = 2 is w0 w1 (dw0 - dw1), with
# dw_j = <dy, O_j>: when the two dot products nearly cancel, the bf16-level
# error of O (about 2^-9 of |dw|) becomes a large part of the difference.  Over
# many tokens that averages out; for a handful of tokens the router gradients
# (dW_g, db_g) get a 5x looser relative bound.
FEW_TOKENS = 32


@pytest.mark.parametrize("label,base,over,noise", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(label, base, over, noise):
    cfg = si.CONFIGS[base].replace(**over)
    inp = si.layer_inputs(cfg, seed=21)
    if noise:
        inp["noise"] = si.router_noise(cfg, seed=21, std=noise)
    dinp = device_inputs(inp)
    dy = si.normal(cfg.T * cfg.d, 21, 30, dtype=si.BF16).reshape(cfg.T, cfg.d)
    fwd = run(cfg, dinp)                               # the GPU's own logits
    gl = fwd.router_logits.cpu().numpy().astype(np.float64)
    g = moe.backward(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"],
                     dinp["W3"], device_inputs({"dy": dy})["dy"], dL_aux=1.0, router_noise=dinp.get("noise"))
    assert moe.check_device_errors(g.workspace) == 0
    ref = oracle.backward(cfg, inp, si.as_f32(dy).astype(np.float64), 1.0, logits=gl)
    for name in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW3"):
        if getattr(g, name) is None:          # the layer has no such parameter
            continue
        loose = name in ("dW_g", "db_g") and cfg.T < FEW_TOKENS
        _close(name, getattr(g, name), ref[name], *((5e-2, 2.5e-1) if loose else ()))
    check_expert_grads_elementwise(g, ref, expert_grad_bounds(cfg, inp, si.as_f32(dy),
                                                              token_choice_groups(cfg, ref["routing"])))
    if cfg.capacity_factor > 0:
        assert ref["routing"]["dropped"].sum() > 0


def test_backward_is_deterministic():
    cfg = si.CONFIGS["deepseek_shared_sigmoid_bf16"].replace(T=300, d=512, f=320)
    dinp = device_inputs(si.layer_inputs(cfg, seed=22))
    dy = device_inputs({"dy": si.normal(cfg.T * cfg.d, 22, 30, dtype=si.BF16).reshape(cfg.T, cfg.d)})["dy"]
    args = [dinp[n] for n in ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W3")]
    a = moe.backward(cfg, *args, dy)
    b = moe.backward(cfg, *args, dy)
    torch.cuda.synchronize()
    for name in ("dx", "dW_g", "dW1", "dW2", "dW3"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_backward_empty_batch_gives_zero_weight_gradients():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=0, d=128, f=128)
    inp = si.layer_inputs(cfg.replace(T=1), seed=23)
    dinp = device_inputs(inp)
    x = dinp["x"][:0]
    g = moe.backward(cfg, x, dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"], None, x)
    torch.cuda.synchronize()
    for name in ("dW_g", "db_g", "dW1", "db1", "dW2", "db2"):
        assert torch.all(getattr(g, name) == 0), name


# ---- expert-choice routing --------------------------------------------------------

EC_CASES = [
    # C = 75: every expert's rows padded to 128 in the weight-gradient layout;
    # with cf 1 some tokens are chosen by no expert
    ("gelu_softmax_bias_unchosen", "gpt2_top2_gelu_bf16", dict(T=300, d=256, f=512, capacity_factor=1.0), 0.0),
    ("swiglu_mixtral", "mixtral_swiglu_bf16", dict(T=260, d=512, f=1024), 0.0),
    ("sigmoid_shared_fine", "deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320), 0.0),
    ("many_experts_noise", "deepseek_shared_sigmoid_bf16", dict(T=400, E=40, k=3, S=0, d=256, f=192), 0.5),
    ("max_E_shared", "deepseek_shared_sigmoid_bf16", dict(T=300, E=256, k=8, S=2, d=256, f=192), 0.0),
    # one token, chosen by every expert: C = 1 row in each 128-row padded segment
    ("one_token_shared", "mixtral_swiglu_bf16", dict(T=1, d=256, f=256, S=1), 0.0),
]


@pytest.mark.parametrize("label,base,over,noise", EC_CASES, ids=[c[0] for c in EC_CASES])
def test_expert_choice_backward_matches_oracle(label, base, over, noise):
    """The experts choose on the GPU's own fp32 probabilities (from a forward
    call); the oracle takes the gradient at its own fp64 logits."""
    cfg = si.CONFIGS[base].replace(expert_choice=True, **over)
    inp = si.layer_inputs(cfg, seed=24)
    if noise:
        inp["noise"] = si.router_noise(cfg, seed=24, std=noise)
    dinp = device_inputs(inp)
    dy = si.normal(cfg.T * cfg.d, 24, 30, dtype=si.BF16).reshape(cfg.T, cfg.d)
    fwd = run(cfg, dinp)
    gs = fwd.router_logits.cpu().numpy().astype(np.float64)          # the probabilities the experts chose on
    g = moe.backward(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"],
                     dinp["W3"], device_inputs({"dy": dy})["dy"], dL_aux=1.0, router_noise=dinp.get("noise"))
    assert moe.check_device_errors(g.workspace) == 0
    ref = oracle.ec_backward(cfg, inp, si.as_f32(dy).astype(np.float64), 1.0, scores=gs)
    assert np.array_equal(fwd.perm_token.cpu().numpy()[:cfg.E * ref["capacity"]].reshape(cfg.E, -1), ref["perm"])
    for name in ("dx", "dW_g", "db_g", "dW1", "db1", "dW2", "db2", "dW3"):
        if getattr(g, name) is None:
            continue
        # the logit gradient p (dp - <p, dp>) cancels like the token-choice one
        loose = name in ("dW_g", "db_g") and cfg.T < FEW_TOKENS
        _close(name, getattr(g, name), ref[name], *((5e-2, 2.5e-1) if loose else ()))
    # expert e's rows: its chosen tokens, weighted by the oracle's gate probabilities
    groups = [(ref["perm"][e], ref["probs"][ref["perm"][e], e]) for e in range(cfg.E)]
    groups += [(np.arange(cfg.T), np.ones(cfg.T)) for _ in range(cfg.S)]
    check_expert_grads_elementwise(g, ref, expert_grad_bounds(cfg, inp, si.as_f32(dy), groups))
    if label.endswith("unchosen"):
        chosen = np.zeros(cfg.T, bool)
        chosen[np.unique(ref["perm"])] = True
        assert (~chosen).any()


def test_expert_choice_backward_is_deterministic():
    cfg = si.CONFIGS["mixtral_swiglu_bf16"].replace(T=260, d=256, f=512, expert_choice=True)
    dinp = device_inputs(si.layer_inputs(cfg, seed=25))
    dy = device_inputs({"dy": si.normal(cfg.T * cfg.d, 25, 30, dtype=si.BF16).reshape(cfg.T, cfg.d)})["dy"]
    args = [dinp[n] for n in ("x", "W_g", "b_g", "W1", "b1", "W2", "b2", "W3")]
    a = moe.backward(cfg, *args, dy)
    b = moe.backward(cfg, *args, dy)
    torch.cuda.synchronize()
    for name in ("dx", "dW_g", "dW1", "dW2", "dW3"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


# ---- full size, sampled ------------------------------------------------------------

@pytest.mark.parametrize("ec", [False, True], ids=["token_choice", "expert_choice"])
@pytest.mark.parametrize("name", ["mixtral_swiglu_bf16", "deepseek_shared_sigmoid_bf16"])
def test_backward_full_size_sampled_dx(name, ec):
    """The workload shapes at full size, in the bench's launch configuration:
    dx of sampled tokens against the oracle's per-token dx.  With dL_aux = 0 a
    token's dx depends on its own routing, logits and dy only, so the oracle
    computes it one token at a time."""
    cfg = si.CONFIGS[name].replace(expert_choice=ec)
    inp = si.layer_inputs(cfg, seed=0)
    dinp = device_inputs(inp)
    dy = si.normal(cfg.T * cfg.d, 26, 30, dtype=si.BF16).reshape(cfg.T, cfg.d)
    fwd = run(cfg, dinp)
    g = moe.backward(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"], dinp["b2"],
                     dinp["W3"], device_inputs({"dy": dy})["dy"], dL_aux=0.0)
    assert moe.check_device_errors(g.workspace) == 0
    T, E = cfg.T, cfg.E
    rng = np.random.default_rng(26)
    n = 3 if name == "mixtral_swiglu_bf16" else 6
    rows = np.array(sorted({0, T - 1} | set(rng.choice(T, size=n - 2, replace=False).tolist())))
    dyr = si.as_f32(dy)[rows].astype(np.float64)
    if not ec:
        gl = fwd.router_logits.cpu().numpy().astype(np.float64)          # the GPU's own logits
        r = oracle.routing(cfg, gl)
        ref = oracle.dx_rows(cfg, inp, rows, dyr, gl[rows], r["topk_idx"][rows], r["topk_w"][rows],
                             r["dropped"][rows])
    else:
        C = moe.capacity(cfg)
        perm = fwd.perm_token.cpu().numpy()[:E * C].reshape(E, C)     # the GPU's choice (bit-exact elsewhere)
        chose = np.zeros((T, E), np.uint8)
        for e in range(E):
            chose[perm[e], e] = 1
        lg = oracle.router_logits(np.ascontiguousarray(inp["x"][rows]), inp["W_g"], inp["b_g"], cfg.dtype)
        ref = oracle.ec_dx_rows(cfg, inp, rows, dyr, lg, chose[rows])
    got = g.dx.cpu().numpy()[rows].astype(np.float64)
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert fro <= 1e-2, fro
    assert float(np.abs(got - ref).max()) <= 5e-2 * float(np.sqrt(np.mean(ref ** 2)))
    assert np.isfinite(g.dW1.cpu().numpy()).all()
