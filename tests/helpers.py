"""Shared test plumbing: host <-> device copies of stored values and the
parity checks of the CUDA path against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe

# Bounds on y: max |y_gpu - y_ref| <= TOL * RMS(y_ref) over the compared rows.
Y_TOL = {si.F32: 1e-4, si.BF16: 2e-2}
# Logits: |l_gpu - l_ref| <= 1e-5 * sum_i |x_i W_g[i,e]| + 1e-6 |b_e| (the scale of
# the dot product's rounding; a plain relative bound is undefined near zero).
LOGIT_REL = 1e-5
TOPK_W_RTOL = 1e-6
LAUX_RTOL = 1e-5


def to_dev(a, device="cuda"):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_f32(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def device_inputs(inp):
    return {k: to_dev(v) for k, v in inp.items()}


def run(cfg, dinp, debug=True, **kw):
    return moe.forward(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], dinp["W1"], dinp["b1"], dinp["W2"],
                       dinp["b2"], dinp["W3"], router_noise=dinp.get("noise"), debug=debug, **kw)


def logit_scale(inp):
    x = si.as_f32(inp["x"]).astype(np.float64)
    W = si.as_f32(inp["W_g"]).astype(np.float64)
    s = LOGIT_REL * (np.abs(x) @ np.abs(W))
    if inp["b_g"] is not None:
        s += 1e-6 * np.abs(si.as_f32(inp["b_g"]).astype(np.float64))[None, :]
    if inp.get("noise") is not None:       # one more fp32 addition
        s += 1e-6 * np.abs(inp["noise"].astype(np.float64))
    return s + 1e-30


def check_routing(cfg, inp, out, own_logits=None):
    """Logits within tolerance; every integer decision bitwise equal to the
    oracle's decisions taken on the GPU's own fp32 logits; flips against the
    oracle's own fp64 logits only where the k-th and (k+1)-th logits nearly tie."""
    T, E, k = cfg.T, cfg.E, cfg.k
    gl = out.router_logits.cpu().numpy().astype(np.float64)
    if own_logits is None:
        own_logits = oracle.router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype)
        if inp.get("noise") is not None:
            own_logits = oracle.add_noise(own_logits, inp["noise"])
    scale = logit_scale(inp)
    err = np.abs(gl - own_logits)
    assert np.all(err <= scale), f"logit error {err.max():.3e}, ratio {(err / scale).max():.3f}"

    ref = oracle.routing(cfg, gl)
    assert np.array_equal(out.topk_idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(out.topk_w.cpu().numpy(), ref["topk_w"], rtol=TOPK_W_RTOL, atol=1e-7)
    assert np.array_equal(out.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(out.dropped_mask.cpu().numpy(), ref["dropped"])
    nk = int(ref["offsets"][-1])
    assert np.array_equal(out.perm_token.cpu().numpy()[:nk], ref["perm"])
    assert np.array_equal(out.slot.cpu().numpy(), ref["slot"])
    np.testing.assert_allclose(out.f.cpu().numpy(), ref["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(out.P.cpu().numpy(), ref["P"], rtol=1e-5, atol=1e-9)
    la = float(out.L_aux.cpu().numpy()[0])
    assert abs(la - ref["L_aux"]) <= LAUX_RTOL * abs(ref["L_aux"]) + 1e-12, (la, ref["L_aux"])
    assert int(out.expert_counts.sum()) == T * k - int(out.dropped_mask.sum())
    if out.route_stats is not None:
        np.testing.assert_allclose(out.route_stats.cpu().numpy(), ref["health"], rtol=2e-6, atol=1e-7)

    own_idx = oracle.topk(own_logits, k)
    diff = np.nonzero(np.any(own_idx != ref["topk_idx"], axis=1))[0]
    if diff.size:
        srt = -np.sort(-own_logits[diff], axis=1)
        gap = srt[:, k - 1] - (srt[:, k] if k < E else -np.inf)
        assert np.all(gap <= 2 * scale[diff].max(axis=1)), "routing differs away from a near-tie"
    return ref, gl, diff.size


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v|: the error of storing v in bf16."""
    _, e = np.frexp(np.abs(v))            # |v| = m 2^e, m in [0.5, 1)
    return np.where(v == 0, 0.0, np.ldexp(1.0, e - 9))


def check_y(cfg, inp, out, gl, rows, literal=None):
    """y against the oracle on the compared rows; returns (max|dy| / RMS over
    all compared rows, max|dy| / RMS over the live rows).

    A row whose every routed choice was cut by the capacity limit (and that
    has no shared expert) skips the layer: its y is exactly 0 by definition,
    and it is checked to be exactly 0 on both sides.

    y in fp32 (``literal`` None or True): the bound as it stands,
    max |y - y_ref| <= TOL * RMS(y_ref), RMS over every compared row.

    y in the storage dtype bf16, or ``literal=False``: RMS(y_ref) is taken
    over the live rows only, so that a batch in which the capacity cut zeroes
    most tokens does not shrink the bound of the rows that are computed; with
    bf16 y its own final rounding (half a bf16 spacing at y_ref) is added, as a
    bf16 number cannot sit closer to the exact value than that.  Both margins
    are printed."""
    ref = oracle.forward(cfg, inp, rows=rows, logits=gl)
    y = to_host_f32(out.y)[rows].astype(np.float64)
    yr = ref["y"]
    skipped = np.asarray(ref["dropped"])[rows].all(axis=1) if cfg.S == 0 else np.zeros(len(rows), bool)
    assert np.all(y[skipped] == 0.0) and np.all(yr[skipped] == 0.0), "a row that skipped the layer is not 0"
    live = ~skipped
    dy = np.abs(y - yr)
    tol = Y_TOL[cfg.dtype]
    rms_all = float(np.sqrt(np.mean(yr ** 2)))
    rms_live = float(np.sqrt(np.mean(yr[live] ** 2))) if live.any() else 0.0
    m_all = float(dy.max()) / rms_all if rms_all > 0 else 0.0
    m_live = float(dy.max()) / rms_live if rms_live > 0 else 0.0
    y_f32 = out.y.dtype == torch.float32
    print(f"{cfg.name} T={cfg.T} y {'fp32' if y_f32 else 'bf16'}: max|dy|/RMS(all {len(rows)} rows) = {m_all:.3e}, "
          f"/RMS(live {int(live.sum())} rows) = {m_live:.3e}, tol {tol:.0e}")
    if not live.any():
        return m_all, m_live
    if y_f32 and literal is not False:
        assert np.all(dy <= tol * rms_all), f"max|dy| = {dy.max():.4e}, TOL * RMS = {tol * rms_all:.4e}"
        return m_all, m_live
    bound = tol * rms_live
    if not y_f32:
        bound = bound + half_ulp_bf16(yr[live])
    assert np.all(dy[live] <= bound), f"max|dy| = {dy.max():.4e}, TOL * RMS(live) = {tol * rms_live:.4e}"
    return m_all, m_live
