"""Seeded synthetic workloads for the MoE-FFN layer.

This module only produces inputs: the five layer configurations (shapes and
options) and, for each, seeded tensors drawn by the counter-based generator in
``gen.c`` (SplitMix64 -> Box-Muller in fp64 -> round to fp32 / bf16).  It holds
none of the layer's arithmetic, so the oracle's callers and the CUDA path's
callers can share it without sharing any computation.

Recipe (the pages train on no public dataset; everything is synthetic):
  x ~ N(0, 1); W_g, W1, W3 ~ N(0, 1/d); W2 ~ N(0, 1/f) (std = 1/sqrt(fan_in));
  biases b_g, b1, b2 ~ N(0, 0.01) read as std 0.01; the skewed-routing
  configuration draws b_g ~ N(0, 2.0) read as std 2.0.

Tensor layouts (row-major, ``[in, out]`` weights as in the gate formula
Gate(x) = softmax(W_g x) with W_g of shape [d_model, num_experts]):
  x [T, d], W_g [d, E], b_g [E], W1 / W3 [E+S, d, f], b1 [E+S, f],
  W2 [E+S, f, d], b2 [E+S, d].  Routed experts are 0..E-1, shared E..E+S-1.
bf16 tensors are returned as ``numpy.uint16`` arrays of raw bf16 bits.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libseeded.so")

TAG = {"x": 1, "W_g": 2, "b_g": 3, "W1": 4, "b1": 5, "W2": 6, "b2": 7, "W3": 8, "noise": 9}

RELU, GELU, SWIGLU = 0, 1, 2
SOFTMAX, SIGMOID_NORM = 0, 1
F32, BF16 = 0, 1


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    S: int
    act: int
    gating: int
    dtype: int
    capacity_factor: float = 0.0      # <= 0: no capacity limit
    alpha: float = 0.01
    router_bias: bool = True
    ffn_bias: bool = True
    router_bias_std: float = 0.01
    bias_std: float = 0.01
    expert_choice: bool = False       # each expert chooses its tokens instead
    fp8_experts: bool = False         # expert weights held as E4M3 codes

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)

    @property
    def n_mats(self) -> int:
        return 3 if self.act == SWIGLU else 2


# The five workloads of the layer (shapes from the pages' examples: the
# MiniMind-style top-1 model, GPT-2 FFN width, capacity with skew, the
# Mixtral 8x7B layer shape, fine-grained + shared DeepSeekMoE-style experts).
CONFIGS: Dict[str, LayerConfig] = {
    "tiny_top1_relu_f32": LayerConfig("tiny_top1_relu_f32", T=256, d=64, f=256, E=4, k=1, S=0,
                                      act=RELU, gating=SOFTMAX, dtype=F32),
    "gpt2_top2_gelu_bf16": LayerConfig("gpt2_top2_gelu_bf16", T=4096, d=768, f=3072, E=8, k=2, S=0,
                                       act=GELU, gating=SOFTMAX, dtype=BF16),
    "skew_capacity_gelu_bf16": LayerConfig("skew_capacity_gelu_bf16", T=8192, d=1024, f=4096, E=16, k=2,
                                           S=0, act=GELU, gating=SOFTMAX, dtype=BF16,
                                           capacity_factor=1.25, router_bias_std=2.0),
    "mixtral_swiglu_bf16": LayerConfig("mixtral_swiglu_bf16", T=16384, d=4096, f=14336, E=8, k=2, S=0,
                                       act=SWIGLU, gating=SOFTMAX, dtype=BF16,
                                       router_bias=False, ffn_bias=False),
    "deepseek_shared_sigmoid_bf16": LayerConfig("deepseek_shared_sigmoid_bf16", T=16384, d=2048, f=1408,
                                                E=64, k=6, S=2, act=SWIGLU, gating=SIGMOID_NORM,
                                                dtype=BF16, router_bias=False, ffn_bias=False),
}
CONFIG_ORDER = list(CONFIGS)


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", _SO, src, "-lm"])
    return _SO


_lib: Optional[ctypes.CDLL] = None


def _L() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.seeded_u64.restype = u64
        lib.seeded_u64.argtypes = [u64, u64, u64]
        lib.seeded_splitmix_raw.restype = u64
        lib.seeded_splitmix_raw.argtypes = [u64, u64]
        lib.seeded_normal_f64.restype = dbl
        lib.seeded_normal_f64.argtypes = [u64, u64, u64]
        for fn in (lib.seeded_normal_f32, lib.seeded_normal_bf16):
            fn.restype = None
            fn.argtypes = [u64, u64, dbl, dbl, u64, i64, vp]
        lib.seeded_bf16_to_f32.argtypes = [vp, i64, vp]
        lib.seeded_f32_to_bf16.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def normal(n: int, seed: int, tag: int, mean: float = 0.0, std: float = 1.0, dtype: int = F32,
           offset: int = 0, out: Optional[np.ndarray] = None) -> np.ndarray:
    """n seeded normals; float32 array for F32, uint16 bf16 bits for BF16."""
    lib = _L()
    if dtype == F32:
        out = np.empty(n, np.float32) if out is None else out
        lib.seeded_normal_f32(seed, tag, mean, std, offset, n, out.ctypes.data)
    else:
        out = np.empty(n, np.uint16) if out is None else out
        lib.seeded_normal_bf16(seed, tag, mean, std, offset, n, out.ctypes.data)
    return out


def u64(seed: int, tag: int, c: int) -> int:
    return int(_L().seeded_u64(seed, tag, c))


def splitmix_raw(state: int, c: int) -> int:
    return int(_L().seeded_splitmix_raw(state, c))


def normal_f64(seed: int, tag: int, i: int) -> float:
    return float(_L().seeded_normal_f64(seed, tag, i))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    _L().seeded_bf16_to_f32(bits.ctypes.data, bits.size, out.ctypes.data)
    return out


def f32_to_bf16(vals: np.ndarray) -> np.ndarray:
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    out = np.empty(vals.shape, np.uint16)
    _L().seeded_f32_to_bf16(vals.ctypes.data, vals.size, out.ctypes.data)
    return out


def layer_inputs(cfg: LayerConfig, seed: int = 0) -> Dict[str, Optional[np.ndarray]]:
    """All input tensors of one layer configuration, seeded, in stored dtype."""
    T, d, f, E, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.S
    G = E + S
    dt = cfg.dtype

    def draw(name, shape, std, mean=0.0):
        n = int(np.prod(shape))
        return normal(n, seed, TAG[name], mean, std, dt).reshape(shape)

    inp: Dict[str, Optional[np.ndarray]] = {}
    inp["x"] = draw("x", (T, d), 1.0)
    inp["W_g"] = draw("W_g", (d, E), 1.0 / np.sqrt(d))
    inp["b_g"] = draw("b_g", (E,), cfg.router_bias_std) if cfg.router_bias else None
    inp["W1"] = draw("W1", (G, d, f), 1.0 / np.sqrt(d))
    inp["W3"] = draw("W3", (G, d, f), 1.0 / np.sqrt(d)) if cfg.act == SWIGLU else None
    inp["W2"] = draw("W2", (G, f, d), 1.0 / np.sqrt(f))
    inp["b1"] = draw("b1", (G, f), cfg.bias_std) if cfg.ffn_bias else None
    inp["b2"] = draw("b2", (G, d), cfg.bias_std) if cfg.ffn_bias else None
    return inp


def router_noise(cfg: LayerConfig, seed: int = 0, std: float = 1.0) -> np.ndarray:
    """Scaled Gaussian router noise, fp32 [T, E]: std * N(0, 1)."""
    return normal(cfg.T * cfg.E, seed, TAG["noise"], 0.0, std, F32).reshape(cfg.T, cfg.E)


def x_only(cfg: LayerConfig, seed: int = 0) -> np.ndarray:
    return normal(cfg.T * cfg.d, seed, TAG["x"], 0.0, 1.0, cfg.dtype).reshape(cfg.T, cfg.d)


def as_f32(a: Optional[np.ndarray]) -> Optional[np.ndarray]:
    """Stored values widened to fp32 (exact for both stored dtypes)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return bf16_to_f32(a)
    return a
