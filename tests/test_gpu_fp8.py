"""FP8 (E4M3) experts on the GPU against the oracle's FP8 layer.

Every quantisation is an integer decision and is compared bit for bit:
- the weight codes and scales, against the oracle's quantisation of the same
  bf16 weights;
- the codes and scales of the grouped x rows, against the oracle's
  quantisation of x;
- the codes of the hidden activations, against the oracle's quantisation of
  the kernel's own bf16 H (the decision in the kernel's precision, as routing
  is checked on the kernel's own logits).

The floating-point stages are checked against the oracle's fp64 arithmetic on
the same codes:
- H, within its bf16 rounding plus the fp32 accumulation;
- the expert outputs O, within the fp32 accumulation's bound;
- y, against the combine of those expert outputs (the bf16 bound).

End to end, y is checked against the oracle's own FP8 layer element by
element, with the bf16 layer's bound max|dy| <= 2e-2 RMS(y_ref) (with y
stored in bf16, plus half a bf16 spacing at y_ref for its own rounding); only
the rare quantisation decisions that the fp32 and fp64 paths take differently
separate the two (an E4M3 step of one hidden element moves y by about 0.4% of
RMS(y); measured at most 4.3e-4 with fp32 y).  Beside it: the relative
Frobenius error <= 5e-3, and the unquantised layer within 8% (the bound
derived from E4M3's precision)."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
import sparse_mixture_experts_48_b300 as moe
from helpers import Y_TOL, check_routing, device_inputs, half_ulp_bf16, to_host_f32

pytestmark = pytest.mark.gpu

CASES = [
    ("gpt2_gelu_bias", "gpt2_top2_gelu_bf16", dict(T=300, d=256, f=512)),
    ("skew_capacity_drops", "skew_capacity_gelu_bf16", dict(T=500, d=256, f=384)),
    ("relu_k_tail", "gpt2_top2_gelu_bf16", dict(T=200, d=192, f=320, act=si.RELU, E=5, k=3)),
    ("mixtral_swiglu", "mixtral_swiglu_bf16", dict(T=260, d=512, f=1024)),
    ("deepseek_shared_sigmoid", "deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320)),
    ("max_E_and_k", "deepseek_shared_sigmoid_bf16", dict(T=150, E=256, k=8, S=1, d=256, f=192)),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_48_b300 import build
    build.build()


def _region(cfg, ws, region, dtype, shape):
    off, n = moe.workspace_region(cfg, region)
    t = ws[off:off + n].view(dtype)
    return t.reshape(shape)


def _np_bf16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def run_fp8(cfg, inp, **kw):
    dinp = device_inputs(inp)
    ex = moe.quantize_experts_fp8(dinp["W1"], dinp["W2"], dinp.get("W3"))
    out = moe.forward_fp8(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], ex, dinp["b1"], dinp["b2"],
                          router_noise=dinp.get("noise"), debug=True, **kw)
    torch.cuda.synchronize()
    assert moe.check_device_errors(out.workspace) == 0
    return ex, out


def check_weights(ex, wq):
    assert np.array_equal(ex.W1.cpu().numpy(), wq["W1q"]) and np.array_equal(ex.s1.cpu().numpy(), wq["s1"])
    assert np.array_equal(ex.W2.cpu().numpy(), wq["W2q"]) and np.array_equal(ex.s2.cpu().numpy(), wq["s2"])
    if "W3q" in wq:
        assert np.array_equal(ex.W3.cpu().numpy(), wq["W3q"]) and np.array_equal(ex.s3.cpu().numpy(), wq["s3"])


def row_expert(ref, cfg, r):
    """Expert (slab) and token of grouped row r."""
    off = np.asarray(ref["offsets"])
    T = cfg.T
    rows_tk = T * cfg.k
    if r < rows_tk:
        return int(np.searchsorted(off, r, side="right") - 1), int(ref["perm"][r])
    s, t = divmod(r - rows_tk, T)
    return cfg.E + s, t


def check_y_elementwise(y, yr, y_bf16):
    """max|y - y_ref| <= 2e-2 RMS(y_ref) (+ half a bf16 spacing at y_ref when y is bf16)."""
    rms = float(np.sqrt(np.mean(yr ** 2)))
    bound = Y_TOL[si.BF16] * rms + (half_ulp_bf16(yr) * 1.01 if y_bf16 else 0.0)
    dy = np.abs(y - yr)
    print(f"FP8 y {'bf16' if y_bf16 else 'fp32'}: max|dy|/RMS = {dy.max() / rms:.3e}")
    assert np.all(dy <= bound), f"max|dy|/RMS = {dy.max() / rms:.3e}"


def check_layer(cfg, inp, ex, out, rows=None, stages=True):
    cfg8 = cfg.replace(fp8_experts=True)
    ref_route, gl, _ = check_routing(cfg8, inp, out)
    wq = oracle.quantize_experts(cfg, inp)
    check_weights(ex, wq)
    ref = oracle.fp8_forward(cfg, inp, rows=rows, logits=gl, wq=wq)
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    nk = int(ref["offsets"][-1])
    rows_tk, rows_all = T * k, T * k + S * T
    ws = out.workspace
    xp = _region(cfg8, ws, moe.REGION_XPERM, torch.uint8, (rows_tk, d)).cpu().numpy()
    xs = _region(cfg8, ws, moe.REGION_X_SCALE, torch.float32, (rows_tk,)).cpu().numpy()
    perm = ref["perm"]
    assert np.array_equal(xp[:nk], ref["xq"][perm]) and np.array_equal(xs[:nk], ref["xs"][perm])
    live = np.concatenate([np.arange(nk), rows_tk + np.arange(S * T)]).astype(np.int64)
    if rows is not None:                     # the grouped rows of the sampled tokens only
        want = set(int(t) for t in rows)
        live = np.array([r for r in live if row_expert(ref, cfg, r)[1] in want], np.int64)
    if stages:
        H = _region(cfg8, ws, moe.REGION_H, torch.bfloat16, (rows_all, f))
        Hb = _np_bf16(H)[live]
        Hq = _region(cfg8, ws, moe.REGION_H_CODES, torch.uint8, (rows_all, f)).cpu().numpy()[live]
        Hs = _region(cfg8, ws, moe.REGION_H_SCALE, torch.float32, (rows_all,)).cpu().numpy()[live]
        O = _region(cfg8, ws, moe.REGION_O, torch.float32, (rows_all, d)).cpu().numpy()[live]
        # the kernel's quantisation of its own H, bit for bit
        q, s = oracle.quantize_rows(Hb)
        assert np.array_equal(q, Hq) and np.array_equal(s, Hs)
        Hf = si.as_f32(Hb).astype(np.float64)
        W2d = oracle.e4m3_values(wq["W2q"]) * wq["s2"][:, :, None]          # [G, d, f]
        for i, r in enumerate(live):
            g, t = row_expert(ref, cfg, int(r))
            h = oracle.fp8_hidden(cfg, g, ref["xq"][t], ref["xs"][t], wq, inp)
            bound = half_ulp_bf16(h) * 1.01 + 1e-5 * np.abs(h).max()
            assert np.all(np.abs(Hf[i] - h) <= bound), (int(r), float(np.abs(Hf[i] - h).max()))
            o = oracle.fp8_out(cfg, g, Hq[i], Hs[i], wq, inp)
            hd = oracle.e4m3_values(Hq[i]) * float(Hs[i])
            scale = np.abs(W2d[g]) @ np.abs(hd)
            assert np.all(np.abs(O[i] - o) <= 1e-5 * scale + 1e-30), (int(r), float(np.abs(O[i] - o).max()))
    # y end to end against the oracle's own FP8 layer and the unquantised layer
    rr = ref["rows"]
    y = to_host_f32(out.y)[rr].astype(np.float64)
    yr = ref["y"]
    skipped = np.asarray(ref["dropped"])[rr].all(axis=1) if S == 0 else np.zeros(len(rr), bool)
    assert np.all(y[skipped] == 0.0)
    check_y_elementwise(y, yr, out.y.dtype == torch.bfloat16)
    rel = float(np.linalg.norm(y - yr) / np.linalg.norm(yr))
    assert rel <= 5e-3, rel
    y16 = oracle.forward(cfg, inp, rows=rr, logits=gl)["y"]
    rel16 = float(np.linalg.norm(y - y16) / np.linalg.norm(y16))
    assert rel16 <= 8e-2, rel16
    return rel, rel16


@pytest.mark.parametrize("y_f32", [False, True], ids=["y_bf16", "y_f32"])
@pytest.mark.parametrize("label,base,over", CASES, ids=[c[0] for c in CASES])
def test_fp8_layer(label, base, over, y_f32):
    cfg = si.CONFIGS[base].replace(**over)
    inp = si.layer_inputs(cfg, seed=31)
    ex, out = run_fp8(cfg, inp, y_f32=y_f32)
    check_layer(cfg, inp, ex, out)
    # y against the combine of the kernel's own expert outputs (bf16 bound)
    cfg8 = cfg.replace(fp8_experts=True)
    T, d, k, S = cfg.T, cfg.d, cfg.k, cfg.S
    O = _region(cfg8, out.workspace, moe.REGION_O, torch.float32, (T * k + S * T, d)).cpu().numpy()
    O = O.astype(np.float64)
    slot = out.slot.cpu().numpy()
    w = out.topk_w.cpu().numpy().astype(np.float64)
    yc = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                yc[t] += w[t, j] * O[slot[t, j]]
        for s in range(S):
            yc[t] += O[T * k + s * T + t]
    y = to_host_f32(out.y).astype(np.float64)
    rms = float(np.sqrt(np.mean(yc ** 2)))
    assert np.all(np.abs(y - yc) <= 1e-5 * rms + (half_ulp_bf16(yc) * 1.01 if not y_f32 else 0.0))


def test_fp8_router_noise():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=256, d=256, f=256)
    inp = si.layer_inputs(cfg, seed=32)
    inp["noise"] = si.router_noise(cfg, seed=32, std=0.5)
    ex, out = run_fp8(cfg, inp)
    check_layer(cfg, inp, ex, out)


def test_fp8_empty_batch():
    cfg = si.CONFIGS["mixtral_swiglu_bf16"].replace(T=0, d=256, f=256)
    inp = si.layer_inputs(cfg.replace(T=1), seed=1)
    dinp = device_inputs(inp)
    ex = moe.quantize_experts_fp8(dinp["W1"], dinp["W2"], dinp["W3"])
    x = torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    out = moe.forward_fp8(cfg, x, dinp["W_g"], dinp["b_g"], ex, None, None)
    torch.cuda.synchronize()
    assert moe.check_device_errors(out.workspace) == 0
    assert np.all(out.expert_counts.cpu().numpy() == 0) and float(out.L_aux.cpu()[0]) == 0.0


def test_fp8_deterministic():
    cfg = si.CONFIGS["deepseek_shared_sigmoid_bf16"].replace(T=400, d=256, f=192)
    inp = si.layer_inputs(cfg, seed=33)
    _, a = run_fp8(cfg, inp)
    _, b = run_fp8(cfg, inp)
    assert torch.equal(a.y, b.y)


@pytest.mark.parametrize("shape", [(1, 16), (7, 64), (300, 1024), (33, 14336)])
def test_quantize_rows_bit_exact(shape):
    rows, cols = shape
    x = si.normal(rows * cols, 5, 40, dtype=si.BF16).reshape(rows, cols)
    xf = si.as_f32(x).copy()
    if rows > 3:                      # a zero row, a huge row, a tiny row
        xf[1] = 0.0
        xf[2] *= 1e30
        xf[3] *= 1e-30
    xb = (xf.view(np.uint32) >> 16).astype(np.uint16)     # exact: already bf16 values
    q, s = moe.quantize_rows_fp8(device_inputs({"x": xb})["x"])
    torch.cuda.synchronize()
    qr, sr = oracle.quantize_rows(xb)
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr)


@pytest.mark.parametrize("shape", [(3, 64, 96), (2, 4096, 256), (1, 512, 1408)])
def test_quantize_weights_bit_exact(shape):
    G, K, N = shape
    W = si.normal(G * K * N, 6, 41, std=1.0 / np.sqrt(K), dtype=si.BF16).reshape(G, K, N)
    q, s = moe.quantize_weights_fp8(device_inputs({"W": W})["W"])
    torch.cuda.synchronize()
    qr, sr = oracle.quantize_weights(W)
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr)


def test_fp8_full_size_sampled():
    """The Mixtral-shaped layer (T=16384, d=4096, f=14336, E=8, k=2) in the
    launch configuration the FP8 bench times; y on sampled tokens, every
    routing decision on all tokens."""
    cfg = si.CONFIGS["mixtral_swiglu_bf16"]
    inp = si.layer_inputs(cfg, seed=0)
    ex, out = run_fp8(cfg, inp)
    rows = np.random.default_rng(7).choice(cfg.T, size=6, replace=False)
    check_layer(cfg, inp, ex, out, rows=rows, stages=False)


def test_fp8_host_buffers_match_device_call():
    """moe_forward_fp8_host (x in, outputs out through pinned host memory)
    gives bitwise the outputs of moe_forward_fp8 on device buffers."""
    cfg = si.CONFIGS["deepseek_shared_sigmoid_bf16"].replace(T=300, d=256, f=192)
    inp = si.layer_inputs(cfg, seed=34)
    inp["noise"] = si.router_noise(cfg, seed=34, std=0.3)
    dinp = device_inputs(inp)
    ex = moe.quantize_experts_fp8(dinp["W1"], dinp["W2"], dinp.get("W3"))
    dev = moe.forward_fp8(cfg, dinp["x"], dinp["W_g"], dinp["b_g"], ex, dinp["b1"], dinp["b2"],
                          router_noise=dinp["noise"])
    x_host = dinp["x"].cpu().pin_memory()
    host = moe.forward_fp8_host(cfg, x_host, dinp["W_g"], dinp["b_g"], ex, dinp["b1"], dinp["b2"],
                                router_noise_host=dinp["noise"].cpu().pin_memory())
    torch.cuda.synchronize()
    assert moe.check_device_errors(host.workspace) == 0
    for n in ("y", "topk_idx", "topk_w", "expert_counts", "dropped_mask", "f", "P", "L_aux", "route_stats"):
        assert torch.equal(getattr(dev, n).cpu(), getattr(host, n)), n


EC_CASES = [
    ("gpt2_softmax_bias", "gpt2_top2_gelu_bf16", dict(T=300, d=256, f=512)),
    ("mixtral_swiglu", "mixtral_swiglu_bf16", dict(T=260, d=512, f=1024)),
    ("deepseek_sigmoid_shared", "deepseek_shared_sigmoid_bf16", dict(T=300, d=512, f=320)),
    ("skew_cf_unchosen", "skew_capacity_gelu_bf16", dict(T=500, d=256, f=384)),
    ("max_E_shared", "deepseek_shared_sigmoid_bf16", dict(T=300, E=256, k=8, S=2, d=256, f=192)),
    ("one_token", "mixtral_swiglu_bf16", dict(T=1, d=256, f=256)),
]


@pytest.mark.parametrize("label,base,over", EC_CASES, ids=[c[0] for c in EC_CASES])
def test_fp8_expert_choice_layer(label, base, over):
    """Expert choice with FP8 experts: the choice bit for bit on the GPU's own
    scores, the chosen rows' codes and scales bit for bit against the oracle's
    quantisation of x, the hidden codes bit for bit on the kernel's own H, and
    y against the oracle's FP8 expert-choice layer and the unquantised one."""
    cfg = si.CONFIGS[base].replace(expert_choice=True, **over)
    inp = si.layer_inputs(cfg, seed=34)
    ex, out = run_fp8(cfg, inp)
    cfg8 = cfg.replace(fp8_experts=True)
    T, d, f, E, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.S
    C = moe.capacity(cfg8)
    gs = out.router_logits.cpu().numpy().astype(np.float64)
    wq = oracle.quantize_experts(cfg, inp)
    check_weights(ex, wq)
    ref = oracle.fp8_ec_forward(cfg, inp, scores=gs, wq=wq)
    assert ref["capacity"] == C
    perm = out.perm_token.cpu().numpy()[:E * C]
    assert np.array_equal(perm.reshape(E, C), ref["perm"])
    assert np.all(out.expert_counts.cpu().numpy() == C)
    rows_tk = E * C
    ws = out.workspace
    xp = _region(cfg8, ws, moe.REGION_XPERM, torch.uint8, (rows_tk, d)).cpu().numpy()
    xs = _region(cfg8, ws, moe.REGION_X_SCALE, torch.float32, (rows_tk,)).cpu().numpy()
    assert np.array_equal(xp, ref["xq"][perm]) and np.array_equal(xs, ref["xs"][perm])
    rows_all = rows_tk + S * T
    H = _np_bf16(_region(cfg8, ws, moe.REGION_H, torch.bfloat16, (rows_all, f)))
    Hq = _region(cfg8, ws, moe.REGION_H_CODES, torch.uint8, (rows_all, f)).cpu().numpy()
    Hs = _region(cfg8, ws, moe.REGION_H_SCALE, torch.float32, (rows_all,)).cpu().numpy()
    q, s = oracle.quantize_rows(H)
    assert np.array_equal(q, Hq) and np.array_equal(s, Hs)
    y = to_host_f32(out.y).astype(np.float64)
    yr = ref["y"]
    chosen = np.zeros(T, bool)
    chosen[np.unique(ref["perm"])] = True
    skipped = ~chosen if S == 0 else np.zeros(T, bool)
    assert np.all(y[skipped] == 0.0)
    check_y_elementwise(y, yr, out.y.dtype == torch.bfloat16)
    rel = float(np.linalg.norm(y - yr) / np.linalg.norm(yr))
    assert rel <= 5e-3, rel
    y16 = oracle.ec_forward(cfg, inp, scores=gs)["y"]
    rel16 = float(np.linalg.norm(y - y16) / np.linalg.norm(y16))
    assert rel16 <= 8e-2, rel16
    if label == "skew_cf_unchosen":
        assert skipped.any()


def test_fp8_expert_choice_host_buffers_equal_the_device_call():
    cfg = si.CONFIGS["mixtral_swiglu_bf16"].replace(T=260, d=256, f=512, expert_choice=True)
    inp = si.layer_inputs(cfg, seed=35)
    ex, out = run_fp8(cfg, inp)
    dinp = device_inputs(inp)
    host = moe.forward_fp8_host(cfg, dinp["x"].cpu().pin_memory(), dinp["W_g"], dinp["b_g"], ex,
                                dinp["b1"], dinp["b2"])
    torch.cuda.synchronize()
    assert torch.equal(host.y.view(torch.int16), out.y.cpu().view(torch.int16))
    assert torch.equal(host.expert_counts, out.expert_counts.cpu())


def test_fp8_expert_choice_full_size_sampled():
    """Expert choice with FP8 experts on the Mixtral-shaped layer in the
    launch configuration the bench times: every expert's choice bit for bit,
    the weight codes bit for bit, the chosen rows' codes and scales, and y of
    sampled tokens against the oracle's FP8 expert-choice layer."""
    cfg = si.CONFIGS["mixtral_swiglu_bf16"].replace(expert_choice=True)
    inp = si.layer_inputs(cfg, seed=0)
    ex, out = run_fp8(cfg, inp)
    cfg8 = cfg.replace(fp8_experts=True)
    T, d, E = cfg.T, cfg.d, cfg.E
    C = moe.capacity(cfg8)
    gs = out.router_logits.cpu().numpy().astype(np.float64)
    wq = oracle.quantize_experts(cfg, inp)
    check_weights(ex, wq)
    rows = np.array(sorted(set(np.random.default_rng(16).choice(T, size=6, replace=False).tolist()) | {0, T - 1}))
    ref = oracle.fp8_ec_forward(cfg, inp, rows=rows, scores=gs, wq=wq)
    perm = out.perm_token.cpu().numpy()[:E * C]
    assert np.array_equal(perm.reshape(E, C), ref["perm"])
    xp = _region(cfg8, out.workspace, moe.REGION_XPERM, torch.uint8, (E * C, d)).cpu().numpy()
    xs = _region(cfg8, out.workspace, moe.REGION_X_SCALE, torch.float32, (E * C,)).cpu().numpy()
    sel = np.random.default_rng(17).choice(E * C, size=64, replace=False)
    assert np.array_equal(xp[sel], ref["xq"][perm[sel]]) and np.array_equal(xs[sel], ref["xs"][perm[sel]])
    y = to_host_f32(out.y)[rows].astype(np.float64)
    yr = ref["y"]
    check_y_elementwise(y, yr, out.y.dtype == torch.bfloat16)
    rel = float(np.linalg.norm(y - yr) / np.linalg.norm(yr))
    assert rel <= 5e-3, rel
