"""The seeded input generator: published SplitMix64 outputs, determinism,
moments of the normal draws, and bf16 rounding against torch's conversion."""
import numpy as np
import torch

import seeded_inputs as si


def test_splitmix64_published_outputs():
    # SplitMix64 with initial state 0 (S. Vigna's reference generator)
    assert si.splitmix_raw(0, 0) == 0xE220A8397B1DCDAF
    assert si.splitmix_raw(0, 1) == 0x6E789E6AA1B965F4
    assert si.splitmix_raw(0, 2) == 0x06C45D188009454F


def test_deterministic_and_counter_based():
    a = si.normal(10000, 3, 1)
    b = si.normal(10000, 3, 1)
    assert np.array_equal(a, b)
    c = si.normal(100, 3, 1, offset=5000)
    assert np.array_equal(a[5000:5100], c)
    assert not np.array_equal(a[:100], si.normal(100, 4, 1))
    assert not np.array_equal(a[:100], si.normal(100, 3, 2))
    np.testing.assert_allclose(a[:10], [si.normal_f64(3, 1, i) for i in range(10)], rtol=1e-7)


def test_normal_moments():
    n = 1 << 20
    z = si.normal(n, 0, 1).astype(np.float64)
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.std() - 1) < 0.005
    assert abs((z ** 4).mean() - 3) < 0.05          # kurtosis of a normal
    w = si.normal(n, 1, 2, mean=0.5, std=2.0).astype(np.float64)
    assert abs(w.mean() - 0.5) < 5 * 2 / np.sqrt(n) and abs(w.std() - 2) < 0.01


def test_bf16_rounding_matches_torch():
    v = si.normal(1 << 16, 9, 1, std=3.0)
    ours = si.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    bits = si.normal(1 << 16, 9, 1, std=3.0, dtype=si.BF16)
    assert np.array_equal(bits, ref)
    back = si.bf16_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_layer_inputs_shapes():
    cfg = si.CONFIGS["deepseek_shared_sigmoid_bf16"].replace(T=8, d=64, f=64)
    inp = si.layer_inputs(cfg)
    G = cfg.E + cfg.S
    assert inp["x"].shape == (8, 64) and inp["W_g"].shape == (64, cfg.E)
    assert inp["W1"].shape == (G, 64, 64) and inp["W3"].shape == (G, 64, 64)
    assert inp["W2"].shape == (G, 64, 64)
    assert inp["b_g"] is None and inp["b1"] is None and inp["b2"] is None
