"""Pins of the oracle's FP8 (E4M3) expert path, against the format's
definition, a library codec (torch's CPU float8_e4m3fn and bfloat16 casts),
closed forms, and numpy matmuls on the decoded operands.

E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, subnormals, no
infinities, largest finite 448, S.1111.111 is NaN."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si


def _torch_e4m3(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_format_points():
    # values fixed by the format: exponent bias 7, 3 mantissa bits, subnormal quantum 2^-9
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6          # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert oracle.e4m3_value(0x3F) == 1.875
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))


def test_decode_matches_library_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = oracle.e4m3_values(codes)
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(lib[~nan], ours[~nan])


def test_encode_of_every_value_is_its_code():
    for c in range(256):
        v = oracle.e4m3_value(c)
        if np.isnan(v):
            continue
        assert oracle.e4m3_encode(np.array([v], np.float32))[0] == c, hex(c)


def test_encode_matches_library_in_range():
    rng = np.random.default_rng(3)
    mags = np.exp2(rng.uniform(-12, np.log2(448.0), size=200000))
    v = (mags * rng.choice([-1.0, 1.0], size=mags.size)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), _torch_e4m3(v))


def test_midpoints_round_to_even_and_overflow_saturates():
    pos = [c for c in range(0x7F)]                       # 0 .. 448, ascending
    vals = [oracle.e4m3_value(c) for c in pos]
    mids = np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])], np.float32)
    got = oracle.e4m3_encode(mids)
    want = [c if c % 2 == 0 else c + 1 for c in pos[:-1]]    # the even code of each pair
    assert np.array_equal(got, np.array(want, np.uint8))
    assert np.array_equal(got, _torch_e4m3(mids))
    big = np.array([448.0, 464.0, 500.0, 1e30, np.inf, -1e30, -np.inf], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_bf16_round_matches_library():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(100000) * np.exp2(rng.uniform(-20, 20, 100000))).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    ours = np.array([oracle.bf16_round(float(x)) for x in v])
    assert np.array_equal(lib.astype(np.float64), ours)


def test_quantize_rows_hand_case():
    q, s = oracle.quantize_rows(np.array([[1.0, -2.0, 0.5, 0.0]], np.float32))
    # a = 2: r = 224, s = 2/448; 224 = 1.75 2^7, -448, 112 = 1.75 2^6, 0
    assert s[0] == np.float32(2.0) / np.float32(448.0)
    assert list(q[0]) == [0x76, 0xFE, 0x6E, 0x00]


def test_quantize_rows_properties():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 300)) * np.exp2(rng.integers(-8, 8, (64, 1)))).astype(np.float32)
    x[3] = 0.0
    q, s = oracle.quantize_rows(x)
    # the largest magnitude of a row maps to +-448
    big = np.abs(x).argmax(axis=1)
    for r in range(64):
        if r == 3:
            assert np.all(q[r] == 0)
            continue
        assert q[r, big[r]] & 0x7F == 0x7E
        assert s[r] == np.float32(np.abs(x[r]).max()) / np.float32(448.0)
    # decoded values within half a quantum (relative 2^-4 for normals, 2^-10 s for subnormals)
    dec = oracle.e4m3_values(q) * s[:, None].astype(np.float64)
    err = np.abs(dec - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_quantize_weights_is_per_output_unit_and_transposed():
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=4, d=64, f=96, E=3)
    inp = si.layer_inputs(cfg, seed=2)
    Wq, s = oracle.quantize_weights(inp["W1"])
    assert Wq.shape == (3, 96, 64) and s.shape == (3, 96)
    Wf = si.as_f32(inp["W1"])
    for g in range(3):
        qg, sg = oracle.quantize_rows(np.ascontiguousarray(Wf[g].T))
        assert np.array_equal(qg, Wq[g]) and np.array_equal(sg, s[g])


def _bf16_round_array(a):
    return np.vectorize(oracle.bf16_round)(a)


@pytest.mark.parametrize("act", [si.RELU, si.GELU, si.SWIGLU])
def test_identical_experts_with_k_equal_E_is_the_dense_fp8_ffn(act):
    """k = E with identical experts: y is one expert's output (the weights sum to
    1), computed here with numpy matmuls on the decoded operands."""
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=6, d=64, f=80, E=3, k=3, S=0, act=act,
                                                   capacity_factor=0.0)
    inp = si.layer_inputs(cfg, seed=7)
    for name in ("W1", "W2", "W3", "b1", "b2"):
        if inp.get(name) is not None:
            inp[name] = np.ascontiguousarray(np.repeat(inp[name][:1], cfg.E, axis=0))
    if act == si.SWIGLU:
        inp["b1"] = inp["b2"] = None
    ref = oracle.fp8_forward(cfg, inp)
    wq = oracle.quantize_experts(cfg, inp)
    xd = oracle.e4m3_values(ref["xq"]) * ref["xs"][:, None]
    W1d = (oracle.e4m3_values(wq["W1q"][0]) * wq["s1"][0][:, None]).T          # [d, f]
    a = xd @ W1d
    if act == si.SWIGLU:
        W3d = (oracle.e4m3_values(wq["W3q"][0]) * wq["s3"][0][:, None]).T
        h = a / (1.0 + np.exp(-a)) * (xd @ W3d)
    else:
        a = a + si.as_f32(inp["b1"])[0]
        from scipy.special import erf
        h = np.maximum(a, 0.0) if act == si.RELU else 0.5 * a * (1.0 + erf(a / np.sqrt(2.0)))
    hq, hs = oracle.quantize_rows(_bf16_round_array(h).astype(np.float32))
    hd = oracle.e4m3_values(hq) * hs[:, None].astype(np.float64)
    W2d = (oracle.e4m3_values(wq["W2q"][0]) * wq["s2"][0][:, None]).T          # [f, d]
    o = hd @ W2d
    if act != si.SWIGLU:
        o = o + si.as_f32(inp["b2"])[0]
    np.testing.assert_allclose(ref["y"], o, rtol=1e-9, atol=1e-12 * np.abs(o).max())


@pytest.mark.parametrize("base", ["gpt2_top2_gelu_bf16", "mixtral_swiglu_bf16", "deepseek_shared_sigmoid_bf16"])
def test_fp8_layer_is_close_to_the_unquantised_layer(base):
    """E4M3 keeps 4 significant bits: rounding a value with significand m in
    [1, 2) errs by up to 2^-4/m, uniformly, so the RMS relative error of one
    quantised operand is sqrt(2^-8 E[m^-2] / 3) = 2.65% for log-uniform m.  A
    GEMM output carries its two operands' errors, sqrt(2) 2.65% = 3.75%; the
    second GEMM adds h's and W2's quantisation: sqrt(3.75^2 + 2 2.65^2) = 5.3%
    for one gated product, and with SwiGLU's two (silu(a) u) 6.5%.  The layer
    output is within 8% in relative Frobenius norm of the unquantised layer's
    (about 20% above the derived 6.5%), and not identical to it."""
    cfg = si.CONFIGS[base].replace(T=24, d=128, f=192)
    inp = si.layer_inputs(cfg, seed=11)
    y8 = oracle.fp8_forward(cfg, inp)["y"]
    y = oracle.forward(cfg, inp)["y"]
    rel = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    assert 1e-3 < rel < 8e-2, rel


@pytest.mark.parametrize("act", [si.GELU, si.SWIGLU])
def test_fp8_expert_halves_against_numpy(act):
    """fp8_hidden and fp8_out (the two halves of one FP8 expert) against numpy
    matmuls on the decoded operands, repeated while other arrays are allocated
    and freed: the wrappers' argument buffers (the fp32 biases are converted
    on the fly) must stay alive through each call."""
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=4, d=128, f=192, E=3, act=act)
    inp = si.layer_inputs(cfg, seed=12)
    if act == si.SWIGLU:
        inp["b1"] = inp["b2"] = None
    wq = oracle.quantize_experts(cfg, inp)
    xq, xs = oracle.quantize_rows(inp["x"])
    g = 2
    W1d = oracle.e4m3_values(wq["W1q"][g]) * wq["s1"][g][:, None]             # [f, d]
    a = W1d @ (oracle.e4m3_values(xq[1]) * float(xs[1]))
    if act == si.SWIGLU:
        u = (oracle.e4m3_values(wq["W3q"][g]) * wq["s3"][g][:, None]) @ (oracle.e4m3_values(xq[1]) * float(xs[1]))
        h_ref = a / (1.0 + np.exp(-a)) * u
    else:
        from scipy.special import erf
        a = a + si.as_f32(inp["b1"])[g]
        h_ref = 0.5 * a * (1.0 + erf(a / np.sqrt(2.0)))
    hq, hs = oracle.quantize_rows(_bf16_round_array(h_ref).astype(np.float32))
    o_ref = (oracle.e4m3_values(wq["W2q"][g]) * wq["s2"][g][:, None]) @ (oracle.e4m3_values(hq[0]) * float(hs[0]))
    if act != si.SWIGLU:
        o_ref = o_ref + si.as_f32(inp["b2"])[g]
    for i in range(50):
        churn = [np.ones(500 + 7 * i) for _ in range(4)]
        h = oracle.fp8_hidden(cfg, g, xq[1], xs[1], wq, inp)
        o = oracle.fp8_out(cfg, g, hq[0], hs[0], wq, inp)
        del churn
        np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)


def test_fp8_expert_choice_every_token_to_every_expert_is_the_fp8_soft_mixture():
    """C = T: every expert takes every token, so y = sum_e p_e FFN8_e(x), each
    FP8 expert output composed here from fp8_hidden, the bf16 rounding of h,
    its quantisation and fp8_out."""
    cfg = si.CONFIGS["gpt2_top2_gelu_bf16"].replace(T=5, d=64, f=96, E=3, k=3, expert_choice=True,
                                                   capacity_factor=3.0)
    inp = si.layer_inputs(cfg, seed=13)
    ref = oracle.fp8_ec_forward(cfg, inp)
    assert ref["capacity"] == cfg.T
    wq = oracle.quantize_experts(cfg, inp)
    xq, xs = oracle.quantize_rows(inp["x"])
    for t in range(cfg.T):
        want = np.zeros(cfg.d)
        for e in range(cfg.E):
            h = oracle.fp8_hidden(cfg, e, xq[t], xs[t], wq, inp)
            hq, hs = oracle.quantize_rows(_bf16_round_array(h).astype(np.float32))
            want += ref["probs"][t, e] * oracle.fp8_out(cfg, e, hq[0], hs[0], wq, inp)
        np.testing.assert_allclose(ref["y"][t], want, rtol=1e-12, atol=1e-14)
