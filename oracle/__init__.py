"""fp64 CPU oracle of the MoE-FFN forward layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It is the checker, not the product: the product
path (``sparse_mixture_experts_48_b300``) never imports it and shares no code
with it.  The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C,
fp64); this file only builds it, marshals arrays and chains its steps in the
order the pages give them:

  logits -> gate probabilities -> top-k on the logits -> renormalised weights
  -> capacity / drops / grouped order -> expert FFNs + gate-weighted sum (+
  shared experts) -> balance statistics f, P, L_aux.

``fp8_forward`` runs the same layer with E4M3 expert weights and activations
(per-output-unit weight scales, per-row activation scales) for the FP8 path.

Every function takes the STORED input values (fp32 arrays, or uint16 arrays
of bf16 bits) and widens them to double itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libmoe_oracle.so")

RELU, GELU, SWIGLU = 0, 1, 2
SOFTMAX, SIGMOID_NORM = 0, 1
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "moe_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        # -O2, no fast-math: the C library's exp/erf in double, IEEE order of operations.
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _SO, src, "-lm"])
    return _SO


_lib: Optional[ctypes.CDLL] = None


def _L() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_router_logits.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp]
        lib.oracle_gate_probs.argtypes = [i64, i32, i32, vp, vp]
        lib.oracle_topk_row.argtypes = [i32, i32, vp, vp]
        lib.oracle_topk.argtypes = [i64, i32, i32, vp, vp]
        lib.oracle_topk_weights.argtypes = [i64, i32, i32, i32, vp, vp, vp]
        lib.oracle_capacity.restype = i64
        lib.oracle_capacity.argtypes = [i64, i32, dbl]
        lib.oracle_dispatch.argtypes = [i64, i32, i32, i64, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_act.restype = dbl
        lib.oracle_act.argtypes = [i32, dbl]
        lib.oracle_expert_ffn.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_layer_rows.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, i64, vp, vp, vp, vp,
                                          vp, vp, vp, vp, vp, vp]
        lib.oracle_balance.argtypes = [i64, i32, i32, dbl, vp, vp, vp, vp, vp]
        lib.oracle_add_noise.argtypes = [i64, i32, vp, vp]
        lib.oracle_route_health.argtypes = [i64, i32, i32, vp, vp]
        lib.oracle_backward.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32, i32, dbl, dbl] + [vp] * 21
        lib.oracle_ec_backward.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32, dbl, dbl, i64] + [vp] * 18
        lib.oracle_dx_rows.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32, i32] + [vp] * 13
        lib.oracle_ec_dx_rows.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32] + [vp] * 10
        lib.oracle_ec_capacity.restype = i64
        lib.oracle_ec_capacity.argtypes = [i64, i32, i32, dbl]
        lib.oracle_ec_select.argtypes = [i64, i32, i64, vp, vp]
        lib.oracle_ec_layer_rows.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, vp, i64, vp, vp, vp, vp, vp,
                                             vp, vp, vp, vp]
        u8 = ctypes.c_uint8
        lib.oracle_bf16_round.restype = dbl
        lib.oracle_bf16_round.argtypes = [dbl]
        lib.oracle_e4m3_value.restype = dbl
        lib.oracle_e4m3_value.argtypes = [u8]
        lib.oracle_e4m3_encode.argtypes = [i64, vp, vp]
        lib.oracle_quantize_rows.argtypes = [i64, i64, vp, vp, vp]
        lib.oracle_fp8_layer_rows.argtypes = [i32, i32, i32, i32, i32, i32, vp, i64] + [vp] * 14
        lib.oracle_fp8_hidden.argtypes = [i32, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp]
        lib.oracle_fp8_out.argtypes = [i32, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp, vp]
        lib.oracle_fp8_ec_layer_rows.argtypes = [i32, i32, i32, i32, i32, i64, i64, vp, i64] + [vp] * 13
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    """Pointer to a's data that keeps a alive for the call: arguments such as
    _p(np.ascontiguousarray(v, np.int32)) may be temporaries, whose buffers
    would otherwise be freed before the C function reads them."""
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _stored(a: Optional[np.ndarray], dtype: int) -> Optional[np.ndarray]:
    if a is None:
        return None
    want = np.float32 if dtype == F32 else np.uint16
    if a.dtype != want:
        raise TypeError(f"oracle expects stored {want.__name__} values, got {a.dtype}")
    return np.ascontiguousarray(a)


# ---- single steps -----------------------------------------------------------

def router_logits(x, W_g, b_g, dtype: int) -> np.ndarray:
    x, W_g, b_g = _stored(x, dtype), _stored(W_g, dtype), _stored(b_g, dtype)
    T, d = x.shape
    E = W_g.shape[1]
    out = np.empty((T, E), np.float64)
    _L().oracle_router_logits(T, d, E, dtype, _p(x), _p(W_g), _p(b_g), _p(out))
    return out


def gate_probs(logits: np.ndarray, gating: int) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float64)
    T, E = logits.shape
    out = np.empty((T, E), np.float64)
    _L().oracle_gate_probs(T, E, gating, _p(logits), _p(out))
    return out


def topk_row(values: Sequence[float], k: int) -> np.ndarray:
    v = np.ascontiguousarray(values, np.float64)
    idx = np.empty(k, np.int32)
    _L().oracle_topk_row(v.size, k, _p(v), _p(idx))
    return idx


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float64)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    _L().oracle_topk(T, E, k, _p(logits), _p(idx))
    return idx


def topk_weights(logits: np.ndarray, idx: np.ndarray, gating: int) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float64)
    idx = np.ascontiguousarray(idx, np.int32)
    T, E = logits.shape
    k = idx.shape[1]
    w = np.empty((T, k), np.float64)
    _L().oracle_topk_weights(T, E, k, gating, _p(logits), _p(idx), _p(w))
    return w


def capacity(T: int, E: int, capacity_factor: float) -> int:
    return int(_L().oracle_capacity(T, E, capacity_factor))


def dispatch(idx: np.ndarray, E: int, C: int) -> Dict[str, np.ndarray]:
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    n_pre = np.empty(E, np.int32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    dropped = np.empty((T, k), np.uint8)
    slot = np.empty((T, k), np.int32)
    perm = np.full(max(T * k, 1), -1, np.int32)
    _L().oracle_dispatch(T, E, k, C, _p(idx), _p(n_pre), _p(counts), _p(offsets), _p(dropped), _p(slot),
                         _p(perm))
    return dict(n_pre=n_pre, counts=counts, offsets=offsets, dropped=dropped, slot=slot,
                perm=perm[: int(offsets[E])])


def act(kind: int, z: float) -> float:
    return float(_L().oracle_act(kind, z))


def expert_ffn(xrow: np.ndarray, g: int, cfg, W1, b1, W2, b2, W3) -> np.ndarray:
    dt = cfg.dtype
    xr = np.ascontiguousarray(xrow, np.float64)
    out = np.empty(cfg.d, np.float64)
    _L().oracle_expert_ffn(cfg.d, cfg.f, cfg.act, dt, g, _p(xr), _p(_stored(W1, dt)), _p(_stored(b1, dt)),
                           _p(_stored(W2, dt)), _p(_stored(b2, dt)), _p(_stored(W3, dt)), _p(out))
    return out


def layer_rows(cfg, rows: Sequence[int], inp: Dict, idx: np.ndarray, w: np.ndarray,
               dropped: np.ndarray) -> np.ndarray:
    dt = cfg.dtype
    rows = np.ascontiguousarray(rows, np.int64)
    y = np.empty((rows.size, cfg.d), np.float64)
    _L().oracle_layer_rows(cfg.d, cfg.f, cfg.E, idx.shape[1], cfg.S, cfg.act, dt, _p(rows), rows.size,
                           _p(_stored(inp["x"], dt)), _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)),
                           _p(_stored(inp["W2"], dt)), _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                           _p(np.ascontiguousarray(idx, np.int32)), _p(np.ascontiguousarray(w, np.float64)),
                           _p(np.ascontiguousarray(dropped, np.uint8)), _p(y))
    return y


def balance(n_pre: np.ndarray, probs: np.ndarray, k: int, alpha: float):
    n_pre = np.ascontiguousarray(n_pre, np.int32)
    probs = np.ascontiguousarray(probs, np.float64)
    T, E = probs.shape
    f = np.empty(E, np.float64)
    P = np.empty(E, np.float64)
    L = np.empty(1, np.float64)
    _L().oracle_balance(T, E, k, alpha, _p(n_pre), _p(probs), _p(f), _p(P), _p(L))
    return f, P, float(L[0])


def add_noise(logits: np.ndarray, noise: np.ndarray) -> np.ndarray:
    """logits + noise (noise: fp32 [T, E], the scaled Gaussian router noise)."""
    out = np.array(logits, dtype=np.float64, order="C", copy=True)
    nz = np.ascontiguousarray(noise, np.float32)
    if nz.shape != out.shape:
        raise ValueError("noise must have the logits' shape")
    _L().oracle_add_noise(out.shape[0], out.shape[1], _p(out), _p(nz))
    return out


def route_health(n_pre: np.ndarray, T: int, k: int):
    """(entropy of the selection shares, their variance, CV of the counts)."""
    n = np.ascontiguousarray(n_pre, np.int32)
    out = np.empty(3, np.float64)
    _L().oracle_route_health(T, n.size, k, _p(n), _p(out))
    return out


# ---- the layer, chained ---------------------------------------------------------

def routing(cfg, logits: np.ndarray) -> Dict[str, np.ndarray]:
    """Steps after the logits up to the grouped order, on the given logits."""
    probs = gate_probs(logits, cfg.gating)
    idx = topk(logits, cfg.k)
    w = topk_weights(logits, idx, cfg.gating)
    C = capacity(logits.shape[0], cfg.E, cfg.capacity_factor)
    disp = dispatch(idx, cfg.E, C)
    f, P, L_aux = balance(disp["n_pre"], probs, cfg.k, cfg.alpha)
    out = dict(probs=probs, topk_idx=idx, topk_w=w, capacity=C, f=f, P=P, L_aux=L_aux,
               health=route_health(disp["n_pre"], logits.shape[0], cfg.k))
    out.update(disp)
    return out


def forward(cfg, inp: Dict, rows: Optional[Sequence[int]] = None,
            logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The whole layer.  ``rows``: token rows whose output y is computed (all
    when None; routing and statistics always cover every token).  ``logits``:
    route on these logits instead of the oracle's own (used to compare the
    integer decisions on the very fp32 logits another implementation made;
    they already contain any router noise).  ``inp["noise"]`` (optional):
    router noise added to the oracle's own logits."""
    own = router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype) if logits is None else None
    if own is not None and inp.get("noise") is not None:
        own = add_noise(own, inp["noise"])
    lg = own if logits is None else np.ascontiguousarray(logits, np.float64)
    out = routing(cfg, lg)
    out["logits"] = lg
    rows = np.arange(cfg.T) if rows is None else np.asarray(rows, np.int64)
    out["rows"] = rows
    out["y"] = layer_rows(cfg, rows, inp, out["topk_idx"], out["topk_w"], out["dropped"])
    return out


# ---- expert-choice routing ------------------------------------------------------------

def ec_capacity(T: int, E: int, k: int, capacity_factor: float) -> int:
    return int(_L().oracle_ec_capacity(T, E, k, capacity_factor))


def ec_select(scores: np.ndarray, C: int) -> np.ndarray:
    """[E, C] chosen tokens per expert (ascending), by score, ties to the lower token."""
    sc = np.ascontiguousarray(scores, np.float64)
    T, E = sc.shape
    perm = np.empty((E, max(C, 0)), np.int32)
    _L().oracle_ec_select(T, E, C, _p(sc), _p(perm))
    return perm


def ec_forward(cfg, inp: Dict, rows: Optional[Sequence[int]] = None,
               scores: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The layer with expert-choice routing.  ``scores``: select on these gate
    probabilities [T, E] instead of the oracle's own (to compare decisions on
    the very fp32 scores another implementation made); the weights of the sum
    are the oracle's own fp64 gate probabilities either way."""
    dt = cfg.dtype
    lg = router_logits(inp["x"], inp["W_g"], inp["b_g"], dt)
    if inp.get("noise") is not None:
        lg = add_noise(lg, inp["noise"])
    probs = gate_probs(lg, cfg.gating)
    T = lg.shape[0]
    C = ec_capacity(T, cfg.E, cfg.k, cfg.capacity_factor)
    perm = ec_select(probs if scores is None else scores, C)
    counts = np.full(cfg.E, C, np.int32)
    P = probs.mean(axis=0) if T > 0 else np.zeros(cfg.E)
    f = np.full(cfg.E, 1.0 / cfg.E) if T > 0 else np.zeros(cfg.E)
    L_aux = cfg.alpha * cfg.E * float(np.sum(f * P))
    rows = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    rows = np.ascontiguousarray(rows, np.int64)
    y = np.empty((rows.size, cfg.d), np.float64)
    _L().oracle_ec_layer_rows(cfg.d, cfg.f, cfg.E, cfg.S, cfg.act, dt, T, C, _p(rows), rows.size,
                              _p(_stored(inp["x"], dt)), _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)),
                              _p(_stored(inp["W2"], dt)), _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                              _p(np.ascontiguousarray(perm, np.int32)), _p(np.ascontiguousarray(probs)), _p(y))
    return dict(logits=lg, probs=probs, capacity=C, perm=perm, counts=counts, f=f, P=P, L_aux=L_aux, rows=rows, y=y)


# ---- backward pass ------------------------------------------------------------------

def backward(cfg, inp: Dict, dy: np.ndarray, dL_aux: float = 1.0,
             logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Gradients of sum_t <dy_t, y_t> + dL_aux * L_aux (token choice), fp64.
    ``logits``: route on (and differentiate the gating at) these logits instead
    of the oracle's own, as in forward()."""
    dt = cfg.dtype
    if logits is None:
        lg = router_logits(inp["x"], inp["W_g"], inp["b_g"], dt)
        if inp.get("noise") is not None:
            lg = add_noise(lg, inp["noise"])
    else:
        lg = np.ascontiguousarray(logits, np.float64)
    r = routing(cfg, lg)
    T, d, f, E, S, k = cfg.T, cfg.d, cfg.f, cfg.E, cfg.S, cfg.k
    G = E + S
    out = dict(dx=np.empty((T, d)), dW_g=np.empty((d, E)), db_g=np.empty(E), dW1=np.empty((G, d, f)),
               db1=np.empty((G, f)), dW2=np.empty((G, f, d)), db2=np.empty((G, d)),
               dW3=np.empty((G, d, f)) if cfg.act == SWIGLU else None)
    dyc = np.ascontiguousarray(dy, np.float64)
    _L().oracle_backward(T, d, f, E, k, S, cfg.act, cfg.gating, dt, cfg.alpha, dL_aux,
                         _p(_stored(inp["x"], dt)), _p(_stored(inp["W_g"], dt)), _p(np.ascontiguousarray(lg)),
                         _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)), _p(_stored(inp["W2"], dt)),
                         _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                         _p(np.ascontiguousarray(r["topk_idx"], np.int32)), _p(np.ascontiguousarray(r["topk_w"])),
                         _p(np.ascontiguousarray(r["dropped"], np.uint8)), _p(np.ascontiguousarray(r["n_pre"], np.int32)),
                         _p(dyc), _p(out["dx"]), _p(out["dW_g"]), _p(out["db_g"]), _p(out["dW1"]), _p(out["db1"]),
                         _p(out["dW2"]), _p(out["db2"]), _p(out["dW3"]))
    out["routing"] = r
    return out


def ec_backward(cfg, inp: Dict, dy: np.ndarray, dL_aux: float = 1.0,
                scores: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Gradients of sum_t <dy_t, y_t> + dL_aux * L_aux with expert-choice
    routing, fp64.  ``scores``: the experts choose on these gate probabilities
    [T, E] (as in ec_forward); the gradient is taken at the oracle's own
    logits either way."""
    dt = cfg.dtype
    lg = router_logits(inp["x"], inp["W_g"], inp["b_g"], dt)
    if inp.get("noise") is not None:
        lg = add_noise(lg, inp["noise"])
    probs = gate_probs(lg, cfg.gating)
    T, d, f, E, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.S
    C = ec_capacity(T, E, cfg.k, cfg.capacity_factor)
    perm = ec_select(probs if scores is None else scores, C)
    G = E + S
    out = dict(dx=np.empty((T, d)), dW_g=np.empty((d, E)), db_g=np.empty(E), dW1=np.empty((G, d, f)),
               db1=np.empty((G, f)), dW2=np.empty((G, f, d)), db2=np.empty((G, d)),
               dW3=np.empty((G, d, f)) if cfg.act == SWIGLU else None)
    _L().oracle_ec_backward(T, d, f, E, S, cfg.act, cfg.gating, dt, cfg.alpha, dL_aux, C,
                            _p(np.ascontiguousarray(perm, np.int32)), _p(_stored(inp["x"], dt)),
                            _p(_stored(inp["W_g"], dt)), _p(np.ascontiguousarray(lg)),
                            _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)), _p(_stored(inp["W2"], dt)),
                            _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                            _p(np.ascontiguousarray(dy, np.float64)), _p(out["dx"]), _p(out["dW_g"]),
                            _p(out["db_g"]), _p(out["dW1"]), _p(out["db1"]), _p(out["dW2"]), _p(out["db2"]),
                            _p(out["dW3"]))
    out.update(perm=perm, capacity=C, probs=probs, logits=lg)
    return out


def dx_rows(cfg, inp: Dict, rows: Sequence[int], dy_rows: np.ndarray, logits_rows: np.ndarray,
            idx_rows: np.ndarray, w_rows: np.ndarray, dropped_rows: np.ndarray) -> np.ndarray:
    """dx of the listed tokens with dL_aux = 0 (token choice), without the
    parameter gradients: each token's routing row, logits row and dy row are
    given (from a routing over the whole batch)."""
    rows = np.asarray(rows, np.int64)
    n, dt = rows.size, cfg.dtype
    x = np.ascontiguousarray(inp["x"][rows])
    dx = np.empty((n, cfg.d))
    _L().oracle_dx_rows(n, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S, cfg.act, cfg.gating, dt, _p(_stored(x, dt)),
                        _p(_stored(inp["W_g"], dt)), _p(np.ascontiguousarray(logits_rows, np.float64)),
                        _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)), _p(_stored(inp["W2"], dt)),
                        _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                        _p(np.ascontiguousarray(idx_rows, np.int32)), _p(np.ascontiguousarray(w_rows, np.float64)),
                        _p(np.ascontiguousarray(dropped_rows, np.uint8)),
                        _p(np.ascontiguousarray(dy_rows, np.float64)), _p(dx))
    return dx


def ec_dx_rows(cfg, inp: Dict, rows: Sequence[int], dy_rows: np.ndarray, logits_rows: np.ndarray,
               chose_rows: np.ndarray) -> np.ndarray:
    """dx of the listed tokens with dL_aux = 0 (expert choice): chose_rows
    [n, E] marks the experts that chose each token (from a selection over the
    whole batch)."""
    rows = np.asarray(rows, np.int64)
    n, dt = rows.size, cfg.dtype
    x = np.ascontiguousarray(inp["x"][rows])
    dx = np.empty((n, cfg.d))
    _L().oracle_ec_dx_rows(n, cfg.d, cfg.f, cfg.E, cfg.S, cfg.act, cfg.gating, dt, _p(_stored(x, dt)),
                           _p(_stored(inp["W_g"], dt)), _p(np.ascontiguousarray(logits_rows, np.float64)),
                           _p(_stored(inp["W1"], dt)), _p(_stored(inp["b1"], dt)), _p(_stored(inp["W2"], dt)),
                           _p(_stored(inp["b2"], dt)), _p(_stored(inp["W3"], dt)),
                           _p(np.ascontiguousarray(chose_rows, np.uint8)),
                           _p(np.ascontiguousarray(dy_rows, np.float64)), _p(dx))
    return dx


# ---- FP8 (E4M3) experts ----------------------------------------------------------

def _as_f32_values(a: np.ndarray) -> np.ndarray:
    """Stored values as fp32 (bf16 bits widen exactly)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(a, np.float32)


def bf16_round(v: float) -> float:
    """Nearest bf16 value (ties to even) of a double."""
    return float(_L().oracle_bf16_round(float(v)))


def e4m3_value(code: int) -> float:
    return float(_L().oracle_e4m3_value(int(code)))


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp32 values -> E4M3 codes (nearest, ties to even, saturating at 448)."""
    x = np.ascontiguousarray(v, np.float32)
    q = np.empty(x.shape, np.uint8)
    _L().oracle_e4m3_encode(x.size, _p(x), _p(q))
    return q


def quantize_rows(v: np.ndarray):
    """Per-row E4M3 quantisation of a [rows, cols] matrix of stored values (fp32,
    or uint16 bf16 bits): (codes uint8 [rows, cols], decoding scales fp32 [rows])."""
    x = np.ascontiguousarray(_as_f32_values(np.asarray(v)))
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty(rows, np.float32)
    _L().oracle_quantize_rows(rows, cols, _p(x), _p(q), _p(s))
    return q, s


def quantize_weights(W: np.ndarray):
    """Stacked [G, in, out] weights -> (codes [G, out, in], scales [G, out]): one
    scale per output unit of each expert."""
    G, K, N = W.shape
    Wt = np.ascontiguousarray(np.swapaxes(_as_f32_values(W), 1, 2)).reshape(G * N, K)
    q, s = quantize_rows(Wt)
    return q.reshape(G, N, K), s.reshape(G, N)


def quantize_experts(cfg, inp: Dict) -> Dict[str, np.ndarray]:
    out = {}
    out["W1q"], out["s1"] = quantize_weights(inp["W1"])
    out["W2q"], out["s2"] = quantize_weights(inp["W2"])
    if inp.get("W3") is not None:
        out["W3q"], out["s3"] = quantize_weights(inp["W3"])
    return out


def _bias_f32(inp: Dict, name: str):
    return None if inp.get(name) is None else np.ascontiguousarray(_as_f32_values(inp[name]))


def fp8_hidden(cfg, g: int, xq_row: np.ndarray, xs: float, wq: Dict[str, np.ndarray], inp: Dict) -> np.ndarray:
    """Hidden activations [f] (fp64, before the bf16 rounding) of FP8 expert g
    on one quantised row."""
    h = np.empty(cfg.f, np.float64)
    xr = np.ascontiguousarray(xq_row, np.uint8)
    _L().oracle_fp8_hidden(cfg.d, cfg.f, cfg.act, int(g), _p(xr), float(xs), _p(wq["W1q"]), _p(wq["s1"]),
                           _p(wq.get("W3q")), _p(wq.get("s3")), _p(_bias_f32(inp, "b1")), _p(h))
    return h


def fp8_out(cfg, g: int, hq_row: np.ndarray, hs: float, wq: Dict[str, np.ndarray], inp: Dict) -> np.ndarray:
    """Output [d] of FP8 expert g from one quantised hidden row."""
    o = np.empty(cfg.d, np.float64)
    hr = np.ascontiguousarray(hq_row, np.uint8)
    _L().oracle_fp8_out(cfg.d, cfg.f, cfg.act, int(g), _p(hr), float(hs), _p(wq["W2q"]), _p(wq["s2"]),
                        _p(_bias_f32(inp, "b2")), _p(o))
    return o


def fp8_forward(cfg, inp: Dict, rows: Optional[Sequence[int]] = None, logits: Optional[np.ndarray] = None,
                wq: Optional[Dict[str, np.ndarray]] = None) -> Dict[str, np.ndarray]:
    """The layer with FP8 experts: routing, statistics and gate weights exactly as
    ``forward`` (on the bf16 inputs); the expert FFNs on per-token quantised x,
    per-(expert, output unit) quantised weights (``wq``: the oracle's own
    ``quantize_experts`` when None) and per-row quantised h."""
    own = router_logits(inp["x"], inp["W_g"], inp["b_g"], cfg.dtype) if logits is None else None
    if own is not None and inp.get("noise") is not None:
        own = add_noise(own, inp["noise"])
    lg = own if logits is None else np.ascontiguousarray(logits, np.float64)
    out = routing(cfg, lg)
    out["logits"] = lg
    wq = quantize_experts(cfg, inp) if wq is None else wq
    xq, xs = quantize_rows(inp["x"])
    rows = np.arange(cfg.T) if rows is None else np.asarray(rows, np.int64)
    rows = np.ascontiguousarray(rows, np.int64)
    out["rows"] = rows
    y = np.empty((rows.size, cfg.d), np.float64)
    b1, b2 = _bias_f32(inp, "b1"), _bias_f32(inp, "b2")
    _L().oracle_fp8_layer_rows(cfg.d, cfg.f, cfg.E, cfg.k, cfg.S, cfg.act, _p(rows), rows.size, _p(xq), _p(xs),
                               _p(wq["W1q"]), _p(wq["s1"]), _p(wq.get("W3q")), _p(wq.get("s3")), _p(b1),
                               _p(wq["W2q"]), _p(wq["s2"]), _p(b2),
                               _p(np.ascontiguousarray(out["topk_idx"], np.int32)),
                               _p(np.ascontiguousarray(out["topk_w"], np.float64)),
                               _p(np.ascontiguousarray(out["dropped"], np.uint8)), _p(y))
    out["y"] = y
    out["xq"], out["xs"] = xq, xs
    return out


def fp8_ec_forward(cfg, inp: Dict, rows: Optional[Sequence[int]] = None, scores: Optional[np.ndarray] = None,
                   wq: Optional[Dict[str, np.ndarray]] = None) -> Dict[str, np.ndarray]:
    """Expert-choice routing (as ``ec_forward``) with FP8 experts (as
    ``fp8_forward``): the choosing experts' outputs from the token's quantised
    row, weighted by the oracle's own fp64 gate probabilities."""
    ref = ec_forward(cfg, inp, rows=[], scores=scores)
    wq = quantize_experts(cfg, inp) if wq is None else wq
    xq, xs = quantize_rows(inp["x"])
    T = ref["probs"].shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    rows = np.ascontiguousarray(rows, np.int64)
    y = np.empty((rows.size, cfg.d), np.float64)
    b1, b2 = _bias_f32(inp, "b1"), _bias_f32(inp, "b2")
    _L().oracle_fp8_ec_layer_rows(cfg.d, cfg.f, cfg.E, cfg.S, cfg.act, T, ref["capacity"], _p(rows), rows.size,
                                  _p(xq), _p(xs), _p(wq["W1q"]), _p(wq["s1"]), _p(wq.get("W3q")), _p(wq.get("s3")),
                                  _p(b1), _p(wq["W2q"]), _p(wq["s2"]), _p(b2),
                                  _p(np.ascontiguousarray(ref["perm"], np.int32)),
                                  _p(np.ascontiguousarray(ref["probs"])), _p(y))
    ref.update(rows=rows, y=y, xq=xq, xs=xs)
    return ref
