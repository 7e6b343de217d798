"""The expert GEMM epilogue's GELU, checked on the host.

The bf16 tensor-core epilogues evaluate the erf GELU x Phi(x) with the erf
approximation of Abramowitz and Stegun, Handbook of Mathematical Functions,
eq. 7.1.26 (|error| <= 1.5e-7).  The constants are read from the kernel header
itself, so that a mistyped digit there fails here; the formula is evaluated in
fp64 against scipy's erfc over a dense grid.  (On the device, the approximate
reciprocal and exponential add a few ulp of the small term; the GPU GEMM tests
bound the whole epilogue element by element.)"""
import os
import re

import numpy as np
import scipy.special as sp

HDR = os.path.join(os.path.dirname(__file__), "..", "sparse_mixture_experts_48_b300", "csrc", "tcgen05.cuh")


def _constants():
    src = open(HDR).read()
    body = src[src.index("__device__ __forceinline__ float gelu_erf"):]
    p = float(re.search(r"kP = ([0-9.]+)f \* 0\.70710678118654752f", body).group(1))
    a = [float(re.search(rf"kA{i} = 0\.5f \* (-?[0-9.]+)f", body).group(1)) for i in range(1, 6)]
    return p, a


def test_gelu_epilogue_constants_are_the_published_ones():
    p, a = _constants()
    assert p == 0.3275911
    assert a == [0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429]


def test_gelu_epilogue_within_the_approximation_bound():
    p, a = _constants()
    x = np.linspace(-12.0, 12.0, 2_000_001)
    t = 1.0 / (1.0 + p / np.sqrt(2.0) * np.abs(x))
    h = 0.5 * t * (a[0] + t * (a[1] + t * (a[2] + t * (a[3] + t * a[4])))) * np.exp(-0.5 * x * x)
    g = x * np.where(x >= 0, 1.0 - h, h)
    exact = 0.5 * x * sp.erfc(-x / np.sqrt(2.0))
    # |erf error| <= 1.5e-7 gives |GELU error| <= 0.5 |x| 1.5e-7
    assert np.all(np.abs(g - exact) <= 0.5 * np.abs(x) * 1.5e-7 + 1e-15)
    # the sign branch: Phi(0) = 1/2 from both sides, Phi(-x) = 1 - Phi(x)
    assert abs(g[len(x) // 2]) == 0.0
    assert np.allclose(g - g[::-1], x, atol=1e-6)
