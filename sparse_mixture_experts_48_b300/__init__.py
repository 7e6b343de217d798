"""B300-native forward pass of a token-choice Mixture-of-Experts FFN layer.

A thin ctypes binding over ``libmoe.so`` (C ABI in ``include/moe.h``).  Every
step of the layer runs in the library's CUDA kernels; this module only checks
tensor shapes, allocates outputs and workspace through PyTorch, and passes raw
device pointers and the current CUDA stream.  There is no fallback: if the
library is missing, or no CUDA device is present, calls raise.

    import sparse_mixture_experts_48_b300 as moe
    cfg = moe.MoEConfig(T=4096, d=768, f=3072, E=8, k=2, S=0, act=moe.GELU,
                        gating=moe.SOFTMAX, dtype=moe.BF16)
    out = moe.forward(cfg, x, W_g, b_g, W1, b1, W2, b2)      # torch CUDA tensors
    out.y, out.topk_idx, out.topk_w, out.expert_counts, out.L_aux ...

bf16 tensors may be passed as torch.bfloat16 or as int16/uint16 raw bits.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

RELU, GELU, SWIGLU, NONE = 0, 1, 2, 3
FLAG_Y_F32 = 1
FLAG_EXPERT_CHOICE = 2
FLAG_FP8_EXPERTS = 4
REGION_XPERM, REGION_X_SCALE, REGION_H, REGION_H_CODES, REGION_H_SCALE, REGION_O = 1, 2, 3, 4, 5, 6
SOFTMAX, SIGMOID_NORM = 0, 1
F32, BF16 = 0, 1
NUM_STAGES = 6
STAGE_NAMES = ("router", "select", "gather", "expert_gemm1", "expert_gemm2", "combine")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    T: int
    d: int
    f: int
    E: int
    k: int
    S: int = 0
    act: int = SWIGLU
    gating: int = SOFTMAX
    dtype: int = BF16
    capacity_factor: float = 0.0
    alpha: float = 0.01
    y_f32: bool = False        # write y in fp32 whatever dtype is
    expert_choice: bool = False  # each expert chooses its tokens (see moe.h)
    fp8_experts: bool = False    # E4M3 expert weights (forward_fp8)


class _CConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("act", ctypes.c_int32), ("gating", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("capacity_factor", ctypes.c_double), ("alpha", ctypes.c_double), ("flags", ctypes.c_int64)]


class _COpts(ctypes.Structure):
    _fields_ = [("stage_events", ctypes.POINTER(ctypes.c_void_p)), ("wait_timeout_ns", ctypes.c_int64),
                ("flags", ctypes.c_int64)]


class _CFp8(ctypes.Structure):
    _fields_ = [("W1", ctypes.c_void_p), ("s1", ctypes.c_void_p), ("W3", ctypes.c_void_p),
                ("s3", ctypes.c_void_p), ("W2", ctypes.c_void_p), ("s2", ctypes.c_void_p)]


OPT_GEMM_SINGLE_CTA = 1


_lib_handle: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so.  Raises if it has not been built."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m sparse_mixture_experts_48_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    cfgp = ctypes.POINTER(_CConfig)
    optp = ctypes.POINTER(_COpts)
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_validate_config.restype = ctypes.c_int
    L.moe_validate_config.argtypes = [cfgp]
    L.moe_workspace_size.restype = sz
    L.moe_workspace_size.argtypes = [cfgp]
    L.moe_capacity.restype = i64
    L.moe_capacity.argtypes = [cfgp]
    L.moe_forward.restype = ctypes.c_int
    L.moe_forward.argtypes = [cfgp] + [vp] * 9 + [vp] * 12 + [vp, sz, vp, optp]
    L.moe_forward_host_workspace_size.restype = sz
    L.moe_forward_host_workspace_size.argtypes = [cfgp]
    L.moe_forward_host.restype = ctypes.c_int
    L.moe_forward_host.argtypes = [cfgp] + [vp] * 9 + [vp] * 9 + [vp, sz, vp, optp]
    L.moe_backward_workspace_size.restype = sz
    L.moe_backward_workspace_size.argtypes = [cfgp]
    L.moe_backward.restype = ctypes.c_int
    L.moe_backward.argtypes = [cfgp] + [vp] * 10 + [ctypes.c_float] + [vp] * 9 + [sz, vp, optp]
    L.moe_check_device_errors.restype = ctypes.c_int
    L.moe_check_device_errors.argtypes = [vp, vp]
    L.moe_grouped_gemm_workspace_size.restype = sz
    L.moe_grouped_gemm_workspace_size.argtypes = [i32]
    L.moe_grouped_gemm.restype = ctypes.c_int
    L.moe_grouped_gemm.argtypes = [i32, i32, i32, vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp, optp]
    L.moe_grouped_gemm_noalloc.restype = ctypes.c_int
    L.moe_grouped_gemm_noalloc.argtypes = [i32, i32, i32, vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, optp]
    L.moe_quantize_weights_fp8.restype = ctypes.c_int
    L.moe_quantize_weights_fp8.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.moe_quantize_rows_fp8.restype = ctypes.c_int
    L.moe_quantize_rows_fp8.argtypes = [vp, i64, i64, vp, vp, vp]
    L.moe_forward_fp8.restype = ctypes.c_int
    L.moe_forward_fp8.argtypes = [cfgp] + [vp] * 4 + [ctypes.POINTER(_CFp8)] + [vp] * 2 + [vp] * 12 + [vp, sz, vp,
                                                                                                       optp]
    L.moe_forward_fp8_host.restype = ctypes.c_int
    L.moe_forward_fp8_host.argtypes = [cfgp] + [vp] * 4 + [ctypes.POINTER(_CFp8)] + [vp] * 2 + [vp] * 9 + [vp, sz,
                                                                                                           vp, optp]
    L.moe_workspace_region.restype = ctypes.c_int
    L.moe_workspace_region.argtypes = [cfgp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    _lib_handle = L
    return L


def exported_symbols() -> Sequence[str]:
    return ("moe_status_string", "moe_validate_config", "moe_workspace_size", "moe_capacity", "moe_forward",
            "moe_forward_host_workspace_size", "moe_forward_host", "moe_backward_workspace_size", "moe_backward",
            "moe_check_device_errors",
            "moe_grouped_gemm_workspace_size", "moe_grouped_gemm", "moe_grouped_gemm_noalloc",
            "moe_quantize_weights_fp8", "moe_quantize_rows_fp8", "moe_forward_fp8", "moe_forward_fp8_host",
            "moe_workspace_region")


def c_config(cfg, y_f32: Optional[bool] = None) -> _CConfig:
    yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
    flags = (FLAG_Y_F32 if yf else 0) | (FLAG_EXPERT_CHOICE if getattr(cfg, "expert_choice", False) else 0)
    flags |= FLAG_FP8_EXPERTS if getattr(cfg, "fp8_experts", False) else 0
    return _CConfig(int(cfg.T), int(cfg.d), int(cfg.f), int(cfg.E), int(cfg.k), int(cfg.S), int(cfg.act),
                    int(cfg.gating), int(cfg.dtype), float(cfg.capacity_factor), float(cfg.alpha), flags)


def validate(cfg) -> int:
    return int(lib().moe_validate_config(ctypes.byref(c_config(cfg))))


def workspace_size(cfg) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(c_config(cfg))))


def capacity(cfg) -> int:
    return int(lib().moe_capacity(ctypes.byref(c_config(cfg))))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _opts(stage_events, timeout_ns: int, flags: int = 0):
    if stage_events is None and not timeout_ns and not flags:
        return None, None
    arr = None
    if stage_events is not None:
        for e in stage_events:
            if not e.cuda_event:       # torch creates the CUDA event on its first record
                e.record()
        arr = (ctypes.c_void_p * len(stage_events))(*[ctypes.c_void_p(e.cuda_event) for e in stage_events])
    o = _COpts(ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)) if arr is not None else None, int(timeout_ns),
               int(flags))
    return o, arr


_STORE = {F32: (torch.float32,), BF16: (torch.bfloat16, torch.int16, torch.uint16)}


def _check(t: Optional[torch.Tensor], name: str, shape, dtypes, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")


@dataclasses.dataclass
class MoEOutput:
    y: torch.Tensor
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    expert_counts: torch.Tensor
    dropped_mask: torch.Tensor
    f: torch.Tensor
    P: torch.Tensor
    L_aux: torch.Tensor
    route_stats: Optional[torch.Tensor] = None   # entropy, variance, CV of the selection shares
    router_logits: Optional[torch.Tensor] = None
    perm_token: Optional[torch.Tensor] = None
    slot: Optional[torch.Tensor] = None
    workspace: Optional[torch.Tensor] = None


def alloc_outputs(cfg, device, debug: bool = False, y_f32: bool = False) -> MoEOutput:
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    yd = torch.float32 if (cfg.dtype == F32 or y_f32) else torch.bfloat16
    out = MoEOutput(
        y=torch.empty((T, d), dtype=yd, device=device),
        topk_idx=torch.empty((T, k), dtype=torch.int32, device=device),
        topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
        expert_counts=torch.empty((E,), dtype=torch.int32, device=device),
        dropped_mask=torch.empty((T, k), dtype=torch.uint8, device=device),
        f=torch.empty((E,), dtype=torch.float32, device=device),
        P=torch.empty((E,), dtype=torch.float32, device=device),
        L_aux=torch.empty((1,), dtype=torch.float32, device=device),
        route_stats=torch.empty((3,), dtype=torch.float32, device=device))
    if debug:
        rows = T * k
        if getattr(cfg, "expert_choice", False):
            rows = max(rows, E * capacity(cfg))
        out.router_logits = torch.empty((T, E), dtype=torch.float32, device=device)
        out.perm_token = torch.full((max(rows, 1),), -1, dtype=torch.int32, device=device)
        out.slot = torch.empty((T, k), dtype=torch.int32, device=device)
    return out


def alloc_workspace(cfg, device) -> torch.Tensor:
    n = workspace_size(cfg)
    if n == 0:
        raise MoEError(validate(cfg), "moe_workspace_size")
    return torch.empty((n,), dtype=torch.uint8, device=device)


def forward(cfg, x, W_g, b_g, W1, b1, W2, b2, W3=None, *, router_noise: Optional[torch.Tensor] = None,
            out: Optional[MoEOutput] = None,
            workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
            debug: bool = False, stage_events=None, timeout_ns: int = 0,
            y_f32: Optional[bool] = None, gemm_single_cta: bool = False) -> MoEOutput:
    """Enqueue the layer's forward pass on ``stream`` (default: the current one).

    ``y_f32``: write y in fp32 (default: the config's ``y_f32``, else its dtype).
    ``gemm_single_cta``: bf16 expert GEMMs on the one-CTA tile kernel instead
    of the default CTA-pair kernel.
    ``router_noise``: fp32 [T, E] CUDA tensor added to the router logits before
    gating and top-k (scaled Gaussian noise drawn by the caller).

    Asynchronous: returns once the kernels are enqueued.  Host-detected errors
    raise MoEError; device-side ones are reported by check_device_errors()."""
    if not torch.cuda.is_available():
        raise RuntimeError("the MoE layer runs on a CUDA device; none is available")
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    G = E + S
    st = _STORE[cfg.dtype]
    _check(x, "x", (T, d), st)
    _check(W_g, "W_g", (d, E), st)
    _check(b_g, "b_g", (E,), st, required=False)
    _check(W1, "W1", (G, d, f), st)
    _check(W3, "W3", (G, d, f), st, required=cfg.act == SWIGLU)
    _check(W2, "W2", (G, f, d), st)
    _check(b1, "b1", (G, f), st, required=False)
    _check(b2, "b2", (G, d), st, required=False)
    _check(router_noise, "router_noise", (T, E), (torch.float32,), required=False)
    dev = x.device
    yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
    if out is None:
        out = alloc_outputs(cfg, dev, debug=debug, y_f32=yf)
    want = torch.float32 if (cfg.dtype == F32 or yf) else torch.bfloat16
    if out.y.dtype != want or tuple(out.y.shape) != (T, d):
        raise ValueError(f"y must be {want} of shape {(T, d)}")
    if workspace is None:
        workspace = out.workspace if out.workspace is not None else alloc_workspace(cfg, dev)
    out.workspace = workspace
    opts, keep = _opts(stage_events, timeout_ns, OPT_GEMM_SINGLE_CTA if gemm_single_cta else 0)
    ccfg = c_config(cfg, y_f32=yf)
    with torch.cuda.device(dev):
        status = lib().moe_forward(
            ctypes.byref(ccfg), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(router_noise), _ptr(W1), _ptr(b1), _ptr(W2),
            _ptr(b2), _ptr(W3), _ptr(out.y), _ptr(out.topk_idx), _ptr(out.topk_w), _ptr(out.expert_counts),
            _ptr(out.dropped_mask), _ptr(out.f), _ptr(out.P), _ptr(out.L_aux), _ptr(out.route_stats),
            _ptr(out.router_logits), _ptr(out.perm_token), _ptr(out.slot), _ptr(workspace), workspace.numel(),
            _stream_handle(stream),
            ctypes.byref(opts) if opts is not None else None)
    del keep
    if status != 0:
        raise MoEError(status, "moe_forward")
    return out


def alloc_host_outputs(cfg, y_f32: bool = False) -> MoEOutput:
    """Page-locked host tensors for the outputs of forward_host."""
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    yd = torch.float32 if (cfg.dtype == F32 or y_f32) else torch.bfloat16
    pin = dict(pin_memory=True)
    return MoEOutput(
        y=torch.empty((T, d), dtype=yd, **pin), topk_idx=torch.empty((T, k), dtype=torch.int32, **pin),
        topk_w=torch.empty((T, k), dtype=torch.float32, **pin),
        expert_counts=torch.empty((E,), dtype=torch.int32, **pin),
        dropped_mask=torch.empty((T, k), dtype=torch.uint8, **pin), f=torch.empty((E,), dtype=torch.float32, **pin),
        P=torch.empty((E,), dtype=torch.float32, **pin), L_aux=torch.empty((1,), dtype=torch.float32, **pin),
        route_stats=torch.empty((3,), dtype=torch.float32, **pin))


def host_workspace_size(cfg, y_f32: Optional[bool] = None) -> int:
    return int(lib().moe_forward_host_workspace_size(ctypes.byref(c_config(cfg, y_f32=y_f32))))


def forward_host(cfg, x_host: torch.Tensor, W_g, b_g, W1, b1, W2, b2, W3=None, *,
                 router_noise_host: Optional[torch.Tensor] = None, out: Optional[MoEOutput] = None,
                 workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                 y_f32: Optional[bool] = None, gemm_single_cta: bool = False) -> MoEOutput:
    """The layer on a host batch: x_host (page-locked CPU tensor) in, host
    outputs back (moe_forward_host).  Weights are CUDA tensors.  Asynchronous:
    the host outputs are valid once ``stream`` is synchronised.  Alternating
    two workspaces on two streams overlaps one batch's copies with another's
    kernels."""
    if not torch.cuda.is_available():
        raise RuntimeError("the MoE layer runs on a CUDA device; none is available")
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    G = E + S
    st = _STORE[cfg.dtype]
    if x_host.is_cuda or not x_host.is_contiguous() or tuple(x_host.shape) != (T, d) or x_host.dtype not in st:
        raise ValueError("x_host must be a contiguous CPU tensor of shape (T, d) in the config's dtype")
    _check(W_g, "W_g", (d, E), st)
    _check(b_g, "b_g", (E,), st, required=False)
    _check(W1, "W1", (G, d, f), st)
    _check(W3, "W3", (G, d, f), st, required=cfg.act == SWIGLU)
    _check(W2, "W2", (G, f, d), st)
    _check(b1, "b1", (G, f), st, required=False)
    _check(b2, "b2", (G, d), st, required=False)
    if router_noise_host is not None and (router_noise_host.is_cuda or tuple(router_noise_host.shape) != (T, E)
                                          or router_noise_host.dtype != torch.float32
                                          or not router_noise_host.is_contiguous()):
        raise ValueError("router_noise_host must be a contiguous fp32 CPU tensor of shape (T, E)")
    yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
    if out is None:
        out = alloc_host_outputs(cfg, y_f32=yf)
    dev = W1.device
    if workspace is None:
        workspace = torch.empty((host_workspace_size(cfg, yf),), dtype=torch.uint8, device=dev)
    out.workspace = workspace
    opts, keep = _opts(None, 0, OPT_GEMM_SINGLE_CTA if gemm_single_cta else 0)
    ccfg = c_config(cfg, y_f32=yf)
    with torch.cuda.device(dev):
        status = lib().moe_forward_host(
            ctypes.byref(ccfg), _ptr(x_host), _ptr(W_g), _ptr(b_g), _ptr(router_noise_host), _ptr(W1), _ptr(b1),
            _ptr(W2), _ptr(b2), _ptr(W3), _ptr(out.y), _ptr(out.topk_idx), _ptr(out.topk_w), _ptr(out.expert_counts),
            _ptr(out.dropped_mask), _ptr(out.f), _ptr(out.P), _ptr(out.L_aux), _ptr(out.route_stats),
            _ptr(workspace), workspace.numel(), _stream_handle(stream),
            ctypes.byref(opts) if opts is not None else None)
    del keep
    if status != 0:
        raise MoEError(status, "moe_forward_host")
    return out


@dataclasses.dataclass
class MoEGrads:
    dx: torch.Tensor
    dW_g: torch.Tensor
    db_g: Optional[torch.Tensor]
    dW1: torch.Tensor
    db1: Optional[torch.Tensor]
    dW2: torch.Tensor
    db2: Optional[torch.Tensor]
    dW3: Optional[torch.Tensor]
    workspace: Optional[torch.Tensor] = None


def backward(cfg, x, W_g, b_g, W1, b1, W2, b2, W3, dy, dL_aux: float = 1.0, *,
             router_noise: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> MoEGrads:
    """Gradients of sum <dy, y> + dL_aux * L_aux (moe_backward; fp32 outputs),
    with token-choice or expert-choice routing (cfg.expert_choice).
    Recomputes the forward pass inside; asynchronous like forward()."""
    if not torch.cuda.is_available():
        raise RuntimeError("the MoE layer runs on a CUDA device; none is available")
    T, d, f, E, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.S
    G = E + S
    st = _STORE[cfg.dtype]
    _check(x, "x", (T, d), st)
    _check(dy, "dy", (T, d), st)
    _check(W_g, "W_g", (d, E), st)
    _check(b_g, "b_g", (E,), st, required=False)
    _check(W1, "W1", (G, d, f), st)
    _check(W3, "W3", (G, d, f), st, required=cfg.act == SWIGLU)
    _check(W2, "W2", (G, f, d), st)
    _check(b1, "b1", (G, f), st, required=False)
    _check(b2, "b2", (G, d), st, required=False)
    _check(router_noise, "router_noise", (T, E), (torch.float32,), required=False)
    dev = W1.device
    z = dict(dtype=torch.float32, device=dev)
    g = MoEGrads(dx=torch.empty((T, d), **z), dW_g=torch.empty((d, E), **z),
                 db_g=torch.empty((E,), **z) if b_g is not None else None, dW1=torch.empty((G, d, f), **z),
                 db1=torch.empty((G, f), **z) if b1 is not None else None, dW2=torch.empty((G, f, d), **z),
                 db2=torch.empty((G, d), **z) if b2 is not None else None,
                 dW3=torch.empty((G, d, f), **z) if cfg.act == SWIGLU else None)
    ccfg = c_config(cfg)
    if workspace is None:
        n = int(lib().moe_backward_workspace_size(ctypes.byref(ccfg)))
        if n == 0:
            raise MoEError(2, "moe_backward_workspace_size")
        workspace = torch.empty((n,), dtype=torch.uint8, device=dev)
    g.workspace = workspace
    with torch.cuda.device(dev):
        status = lib().moe_backward(
            ctypes.byref(ccfg), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(router_noise), _ptr(W1), _ptr(b1), _ptr(W2),
            _ptr(b2), _ptr(W3), _ptr(dy), float(dL_aux), _ptr(g.dx), _ptr(g.dW_g), _ptr(g.db_g), _ptr(g.dW1),
            _ptr(g.db1), _ptr(g.dW2), _ptr(g.db2), _ptr(g.dW3), _ptr(workspace), workspace.numel(),
            _stream_handle(stream), None)
    if status != 0:
        raise MoEError(status, "moe_backward")
    return g


def check_device_errors(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise ``stream`` and return the device status of the last call."""
    return int(lib().moe_check_device_errors(_ptr(workspace), _stream_handle(stream)))


def grouped_gemm(dtype: int, act: int, seg_offsets: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                 B3: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                 C: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None, stage_events=None, timeout_ns: int = 0,
                 single_cta: bool = False):
    """C[r] = epilogue(A[r] @ B[g]) for the rows r of each group g (see moe.h)."""
    G, K, N = B.shape
    M = A.shape[0]
    if seg_offsets.dtype != torch.int32 or tuple(seg_offsets.shape) != (G + 1,) or not seg_offsets.is_cuda:
        raise ValueError("seg_offsets must be a CUDA int32 tensor of G+1 entries")
    if A.shape[1] != K:
        raise ValueError("A and B disagree on K")
    st = _STORE[dtype]
    _check(A, "A", (M, K), st)
    _check(B, "B", (G, K, N), st)
    _check(B3, "B3", (G, K, N), st, required=act == SWIGLU)
    _check(bias, "bias", (G, N), st, required=False)
    if C is None:
        C = torch.zeros((M, N), dtype=A.dtype, device=A.device)
    if workspace is None:
        workspace = torch.empty((lib().moe_grouped_gemm_workspace_size(G),), dtype=torch.uint8, device=A.device)
    opts, keep = _opts(stage_events, timeout_ns, OPT_GEMM_SINGLE_CTA if single_cta else 0)
    with torch.cuda.device(A.device):
        status = lib().moe_grouped_gemm(dtype, act, G, _ptr(seg_offsets), M, K, N, _ptr(A), _ptr(B), _ptr(B3),
                                        _ptr(bias), _ptr(C), _ptr(workspace), workspace.numel(),
                                        _stream_handle(stream), ctypes.byref(opts) if opts is not None else None)
    del keep
    if status != 0:
        raise MoEError(status, "moe_grouped_gemm")
    return C, workspace


def grouped_gemm_noalloc(dtype: int, act: int, seg_offsets: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                         B3: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                         C: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                         stage_events=None, timeout_ns: int = 0, single_cta: bool = False):
    """grouped_gemm without a workspace, for callers that cannot allocate at
    call time: the library's own fixed device scratch is used instead (see
    moe.h).  Pass C to avoid any allocation here; if it is omitted, torch (not
    the library) allocates it."""
    G, K, N = B.shape
    M = A.shape[0]
    if seg_offsets.dtype != torch.int32 or tuple(seg_offsets.shape) != (G + 1,) or not seg_offsets.is_cuda:
        raise ValueError("seg_offsets must be a CUDA int32 tensor of G+1 entries")
    st = _STORE[dtype]
    _check(A, "A", (M, K), st)
    _check(B, "B", (G, K, N), st)
    _check(B3, "B3", (G, K, N), st, required=act == SWIGLU)
    _check(bias, "bias", (G, N), st, required=False)
    if C is None:
        C = torch.zeros((M, N), dtype=A.dtype, device=A.device)
    opts, keep = _opts(stage_events, timeout_ns, OPT_GEMM_SINGLE_CTA if single_cta else 0)
    with torch.cuda.device(A.device):
        status = lib().moe_grouped_gemm_noalloc(dtype, act, G, _ptr(seg_offsets), M, K, N, _ptr(A), _ptr(B),
                                                _ptr(B3), _ptr(bias), _ptr(C), _stream_handle(stream),
                                                ctypes.byref(opts) if opts is not None else None)
    del keep
    if status != 0:
        raise MoEError(status, "moe_grouped_gemm_noalloc")
    return C


# ---- FP8 (E4M3) experts ------------------------------------------------------------

@dataclasses.dataclass
class Fp8Experts:
    """Expert weights as E4M3 codes, K-major, with one fp32 decoding scale per
    (expert, output unit): W1/W3 [E+S, f, d] with s1/s3 [E+S, f]; W2 [E+S, d, f]
    with s2 [E+S, d]."""
    W1: torch.Tensor
    s1: torch.Tensor
    W2: torch.Tensor
    s2: torch.Tensor
    W3: Optional[torch.Tensor] = None
    s3: Optional[torch.Tensor] = None


def quantize_weights_fp8(W: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """bf16 weight slabs [G, K, N] -> (codes uint8 [G, N, K], scales fp32 [G, N])."""
    if W.dim() != 3:
        raise ValueError("W must be [G, K, N]")
    _check(W, "W", tuple(W.shape), _STORE[BF16])
    G, K, N = W.shape
    Q = torch.empty((G, N, K), dtype=torch.uint8, device=W.device)
    sc = torch.empty((G, N), dtype=torch.float32, device=W.device)
    with torch.cuda.device(W.device):
        st = lib().moe_quantize_weights_fp8(_ptr(W), G, K, N, _ptr(Q), _ptr(sc), _stream_handle(stream))
    if st != 0:
        raise MoEError(st, "moe_quantize_weights_fp8")
    return Q, sc


def quantize_rows_fp8(X: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """bf16 rows [rows, cols] -> (codes uint8 [rows, cols], scales fp32 [rows])."""
    if X.dim() != 2:
        raise ValueError("X must be [rows, cols]")
    _check(X, "X", tuple(X.shape), _STORE[BF16])
    rows, cols = X.shape
    Q = torch.empty((rows, cols), dtype=torch.uint8, device=X.device)
    sc = torch.empty((rows,), dtype=torch.float32, device=X.device)
    with torch.cuda.device(X.device):
        st = lib().moe_quantize_rows_fp8(_ptr(X), rows, cols, _ptr(Q), _ptr(sc), _stream_handle(stream))
    if st != 0:
        raise MoEError(st, "moe_quantize_rows_fp8")
    return Q, sc


def quantize_experts_fp8(W1: torch.Tensor, W2: torch.Tensor, W3: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> Fp8Experts:
    q1, s1 = quantize_weights_fp8(W1, stream)
    q2, s2 = quantize_weights_fp8(W2, stream)
    q3, s3 = quantize_weights_fp8(W3, stream) if W3 is not None else (None, None)
    return Fp8Experts(W1=q1, s1=s1, W2=q2, s2=s2, W3=q3, s3=s3)


def _fp8_cfg(cfg):
    return dataclasses.replace(cfg, fp8_experts=True) if not getattr(cfg, "fp8_experts", False) else cfg


def forward_fp8(cfg, x, W_g, b_g, experts: Fp8Experts, b1=None, b2=None, *,
                router_noise: Optional[torch.Tensor] = None, out: Optional[MoEOutput] = None,
                workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                debug: bool = False, stage_events=None, timeout_ns: int = 0,
                y_f32: Optional[bool] = None) -> MoEOutput:
    """The layer with FP8 experts (moe_forward_fp8): routing as forward(), the
    expert GEMMs on E4M3 codes.  ``stage_events``: NUM_STAGES + 2 events (the
    last one after the hidden activations' quantisation)."""
    if not torch.cuda.is_available():
        raise RuntimeError("the MoE layer runs on a CUDA device; none is available")
    cfg = _fp8_cfg(cfg)
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    G = E + S
    st = _STORE[cfg.dtype]
    u8, f32 = (torch.uint8,), (torch.float32,)
    _check(x, "x", (T, d), st)
    _check(W_g, "W_g", (d, E), st)
    _check(b_g, "b_g", (E,), st, required=False)
    _check(experts.W1, "W1 codes", (G, f, d), u8)
    _check(experts.s1, "s1", (G, f), f32)
    _check(experts.W2, "W2 codes", (G, d, f), u8)
    _check(experts.s2, "s2", (G, d), f32)
    _check(experts.W3, "W3 codes", (G, f, d), u8, required=cfg.act == SWIGLU)
    _check(experts.s3, "s3", (G, f), f32, required=cfg.act == SWIGLU)
    _check(b1, "b1", (G, f), st, required=False)
    _check(b2, "b2", (G, d), st, required=False)
    _check(router_noise, "router_noise", (T, E), (torch.float32,), required=False)
    dev = x.device
    yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
    if out is None:
        out = alloc_outputs(cfg, dev, debug=debug, y_f32=yf)
    if workspace is None:
        workspace = out.workspace if out.workspace is not None else alloc_workspace(cfg, dev)
    out.workspace = workspace
    opts, keep = _opts(stage_events, timeout_ns, 0)
    ccfg = c_config(cfg, y_f32=yf)
    w = _fp8_struct(experts)
    with torch.cuda.device(dev):
        status = lib().moe_forward_fp8(
            ctypes.byref(ccfg), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(router_noise), ctypes.byref(w), _ptr(b1),
            _ptr(b2), _ptr(out.y), _ptr(out.topk_idx), _ptr(out.topk_w), _ptr(out.expert_counts),
            _ptr(out.dropped_mask), _ptr(out.f), _ptr(out.P), _ptr(out.L_aux), _ptr(out.route_stats),
            _ptr(out.router_logits), _ptr(out.perm_token), _ptr(out.slot), _ptr(workspace), workspace.numel(),
            _stream_handle(stream), ctypes.byref(opts) if opts is not None else None)
    del keep
    if status != 0:
        raise MoEError(status, "moe_forward_fp8")
    return out


def _fp8_struct(experts: Fp8Experts) -> _CFp8:
    return _CFp8(experts.W1.data_ptr(), experts.s1.data_ptr(),
                 experts.W3.data_ptr() if experts.W3 is not None else None,
                 experts.s3.data_ptr() if experts.s3 is not None else None,
                 experts.W2.data_ptr(), experts.s2.data_ptr())


def forward_fp8_host(cfg, x_host: torch.Tensor, W_g, b_g, experts: Fp8Experts, b1=None, b2=None, *,
                     router_noise_host: Optional[torch.Tensor] = None, out: Optional[MoEOutput] = None,
                     workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                     y_f32: Optional[bool] = None) -> MoEOutput:
    """forward_fp8 on a host batch (moe_forward_fp8_host): x_host and the
    outputs are page-locked CPU tensors, the weights CUDA tensors."""
    if not torch.cuda.is_available():
        raise RuntimeError("the MoE layer runs on a CUDA device; none is available")
    cfg = _fp8_cfg(cfg)
    T, d = cfg.T, cfg.d
    if x_host.is_cuda or not x_host.is_contiguous() or tuple(x_host.shape) != (T, d) or \
            x_host.dtype not in _STORE[cfg.dtype]:
        raise ValueError("x_host must be a contiguous CPU tensor of shape (T, d) in the config's dtype")
    yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
    if out is None:
        out = alloc_host_outputs(cfg, y_f32=yf)
    dev = experts.W1.device
    if workspace is None:
        workspace = torch.empty((host_workspace_size(cfg, yf),), dtype=torch.uint8, device=dev)
    out.workspace = workspace
    ccfg = c_config(cfg, y_f32=yf)
    w = _fp8_struct(experts)
    with torch.cuda.device(dev):
        status = lib().moe_forward_fp8_host(
            ctypes.byref(ccfg), _ptr(x_host), _ptr(W_g), _ptr(b_g), _ptr(router_noise_host), ctypes.byref(w),
            _ptr(b1), _ptr(b2), _ptr(out.y), _ptr(out.topk_idx), _ptr(out.topk_w), _ptr(out.expert_counts),
            _ptr(out.dropped_mask), _ptr(out.f), _ptr(out.P), _ptr(out.L_aux), _ptr(out.route_stats),
            _ptr(workspace), workspace.numel(), _stream_handle(stream), None)
    if status != 0:
        raise MoEError(status, "moe_forward_fp8_host")
    return out


def workspace_region(cfg, region: int):
    """(offset, bytes) of an intermediate in the workspace of ``cfg``'s call."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib().moe_workspace_region(ctypes.byref(c_config(cfg)), int(region), ctypes.byref(off), ctypes.byref(n))
    if st != 0:
        raise MoEError(st, "moe_workspace_region")
    return int(off.value), int(n.value)


# ---- CUDA graphs ------------------------------------------------------------------

class ForwardGraph:
    """One whole forward pass (forward() or, with ``experts``, forward_fp8())
    captured once in a CUDA graph and replayed: every kernel of the layer runs
    again on the same buffers without host-side launch work, which is what
    bounds small layers.  Update the inputs in place (``x.copy_(...)``) before
    ``replay()``; the outputs are in ``out``.

    The capture runs one warm-up call first (first-use kernel attributes and
    the device's cluster occupancy are queried then, outside the capture)."""

    def __init__(self, cfg, x, W_g, b_g, W1=None, b1=None, W2=None, b2=None, W3=None, *,
                 experts: Optional[Fp8Experts] = None, router_noise: Optional[torch.Tensor] = None,
                 debug: bool = False, y_f32: Optional[bool] = None, gemm_single_cta: bool = False):
        self.cfg = _fp8_cfg(cfg) if experts is not None else cfg
        self.stream = torch.cuda.Stream(device=x.device)
        yf = bool(getattr(cfg, "y_f32", False)) if y_f32 is None else bool(y_f32)
        self.out = alloc_outputs(self.cfg, x.device, debug=debug, y_f32=yf)
        self.out.workspace = alloc_workspace(self.cfg, x.device)
        if experts is not None:
            def call():
                forward_fp8(self.cfg, x, W_g, b_g, experts, b1, b2, router_noise=router_noise, out=self.out,
                            workspace=self.out.workspace, stream=self.stream, y_f32=yf)
        else:
            def call():
                forward(self.cfg, x, W_g, b_g, W1, b1, W2, b2, W3, router_noise=router_noise, out=self.out,
                        workspace=self.out.workspace, stream=self.stream, y_f32=yf,
                        gemm_single_cta=gemm_single_cta)
        self.stream.wait_stream(torch.cuda.current_stream(x.device))
        with torch.cuda.stream(self.stream):
            call()
        self.stream.synchronize()
        status = check_device_errors(self.out.workspace, self.stream)
        if status != 0:
            raise MoEError(status, "ForwardGraph warm-up")
        self.graph = torch.cuda.CUDAGraph()
        # relaxed: the launchers set kernel attributes (not stream work) while capturing
        with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="relaxed"):
            call()

    def replay(self) -> MoEOutput:
        """Enqueue the captured forward on the graph's stream, ordered after
        the current stream's work (and the current stream after it)."""
        cur = torch.cuda.current_stream(self.stream.device)
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        cur.wait_stream(self.stream)
        return self.out
