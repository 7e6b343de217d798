"""The C-ABI library: it loads, exports every entry point include/moe.h
declares, and its host-side checks answer before anything touches a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_mixture_experts_48_b300 as moe
import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_mixture_experts_48_b300 import build
    build.build()
    return moe.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_entry_point(L):
    declared = _declared()
    assert declared, "no entry points parsed from moe.h"
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(declared) <= exported, set(declared) - exported
    assert set(declared) == set(moe.exported_symbols())
    for name in declared:
        assert hasattr(L, name)


def test_config_struct_layout():
    assert ctypes.sizeof(moe._CConfig) == 64
    assert moe._CConfig.capacity_factor.offset == 40 and moe._CConfig.flags.offset == 56


def test_status_strings(L):
    for code, name in moe.STATUS.items():
        assert L.moe_status_string(code).decode() == name


def _cfg(**kw):
    base = dict(T=4096, d=768, f=3072, E=8, k=2, S=0, act=moe.GELU, gating=moe.SOFTMAX, dtype=moe.BF16)
    base.update(kw)
    return moe.MoEConfig(**base)


@pytest.mark.parametrize("name", si.CONFIG_ORDER)
def test_the_five_workloads_are_valid(L, name):
    c = si.CONFIGS[name]
    assert moe.validate(c) == 0
    assert moe.workspace_size(c) > 0


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), 1), (dict(k=9, E=16), 2), (dict(k=3, E=2), 1), (dict(E=0), 1), (dict(E=257), 2),
    (dict(d=0), 1), (dict(T=-1), 1), (dict(act=7), 1), (dict(gating=2), 1), (dict(dtype=3), 1),
    (dict(d=96), 2), (dict(f=100), 2), (dict(S=9), 2), (dict(S=-1), 1),
    (dict(dtype=moe.F32, d=66), 2), (dict(capacity_factor=float("nan")), 1),
])
def test_invalid_configs(L, kw, status):
    c = _cfg(**kw)
    assert moe.validate(c) == status
    assert moe.workspace_size(c) == 0


def test_capacity_formula_matches_the_pages_reading(L):
    c = si.CONFIGS["skew_capacity_gelu_bf16"]
    assert moe.capacity(c) == 640            # ceil(8192 * 1.25 / 16)
    assert moe.capacity(_cfg(T=10, E=3, capacity_factor=1.0)) == 4
    assert moe.capacity(_cfg(capacity_factor=0.0)) == -1


def test_empty_batch_is_valid(L):
    c = _cfg(T=0)
    assert moe.validate(c) == 0 and moe.workspace_size(c) > 0


def _call_forward(L, cfg, **over):
    """moe_forward with fake, aligned, never-dereferenced pointers: every case
    here is rejected by the host checks before any CUDA call."""
    P = ctypes.c_void_p
    args = dict(x=P(0x10000), W_g=P(0x20000), b_g=None, noise=None, W1=P(0x30000), b1=None, W2=P(0x40000),
                b2=None, W3=None, y=P(0x50000000), topk_idx=P(0x60000), topk_w=P(0x70000), counts=P(0x80000),
                dropped=P(0x90000), f=P(0xA0000), Pp=P(0xB0000), L_aux=P(0xC0000), stats=None, logits=None,
                perm=None, slot=None, ws=P(0x100000), ws_bytes=moe.workspace_size(cfg))
    args.update(over)
    c = moe.c_config(cfg)
    return L.moe_forward(ctypes.byref(c), args["x"], args["W_g"], args["b_g"], args["noise"], args["W1"],
                         args["b1"], args["W2"], args["b2"], args["W3"], args["y"], args["topk_idx"], args["topk_w"],
                         args["counts"], args["dropped"], args["f"], args["Pp"], args["L_aux"], args["stats"],
                         args["logits"], args["perm"], args["slot"], args["ws"], args["ws_bytes"], None, None)


def test_forward_host_checks(L):
    c = _cfg()
    P = ctypes.c_void_p
    assert _call_forward(L, c, x=None) == 1
    assert _call_forward(L, c, L_aux=None) == 1
    assert _call_forward(L, c, W3=P(0xD0000)) == 1                  # W3 without SwiGLU
    assert _call_forward(L, _cfg(act=moe.SWIGLU)) == 1             # SwiGLU without W3
    assert _call_forward(L, c, x=P(0x10008)) == 1                   # misaligned
    assert _call_forward(L, c, noise=P(0xE0004)) == 1               # misaligned noise
    assert _call_forward(L, c, y=P(0x10000 + 64)) == 1              # y overlaps x
    assert _call_forward(L, c, ws_bytes=moe.workspace_size(c) - 1) == 3
    assert _call_forward(L, c, ws=None) == 3
    assert _call_forward(L, c, ws=P(0x100080)) == 3                 # workspace not 256-byte aligned
    assert _call_forward(L, _cfg(k=9, E=16)) == 2
    # T == 0: the per-token tensors are empty and may be NULL (the host checks
    # pass; without a GPU the first CUDA call then reports MOE_ERR_CUDA).
    e = _cfg(T=0)
    assert _call_forward(L, e, x=None, y=None, topk_idx=None, topk_w=None, dropped=None) in (0, 4)
    assert _call_forward(L, e, W_g=None) == 1


def test_grouped_gemm_host_checks(L):
    P = ctypes.c_void_p
    ws = moe.lib().moe_grouped_gemm_workspace_size(4)
    assert ws > 0
    f = L.moe_grouped_gemm
    assert f(moe.BF16, moe.NONE, 4, None, 256, 128, 128, P(0x1000), P(0x2000), None, None, P(0x3000),
             P(0x100000), ws, None, None) == 1
    assert f(moe.BF16, moe.NONE, 4, P(0x800), 256, 100, 128, P(0x1000), P(0x2000), None, None, P(0x3000),
             P(0x100000), ws, None, None) == 2
    assert f(moe.BF16, moe.SWIGLU, 4, P(0x800), 256, 128, 128, P(0x1000), P(0x2000), None, None, P(0x3000),
             P(0x100000), ws, None, None) == 1
    assert f(moe.BF16, moe.NONE, 4, P(0x800), 256, 128, 128, P(0x1000), P(0x2000), None, None, P(0x3000),
             P(0x100000), ws - 1, None, None) == 3


def test_fp8_config_rules(L):
    c8 = _cfg(fp8_experts=True)
    assert moe.validate(c8) == 0
    assert moe.workspace_size(c8) > 0 and moe.workspace_size(c8) != moe.workspace_size(_cfg())
    assert moe.validate(_cfg(fp8_experts=True, dtype=moe.F32, d=64, f=64)) == 2
    ce8 = _cfg(fp8_experts=True, expert_choice=True)
    assert moe.validate(ce8) == 0
    # expert choice keeps x's codes per token as well as per grouped row
    assert moe.workspace_size(ce8) > moe.workspace_size(_cfg(expert_choice=True))
    # FP8 regions exist only with the flag
    assert moe.workspace_region(c8, moe.REGION_H_CODES)[1] == (4096 * 2) * 3072
    with pytest.raises(moe.MoEError):
        moe.workspace_region(_cfg(), moe.REGION_H_CODES)
    assert moe.workspace_region(_cfg(), moe.REGION_H)[1] == (4096 * 2) * 3072 * 2
    # the flag routes to moe_forward_fp8: moe_forward refuses it, the host path and the backward too
    assert _call_forward(L, c8, ws_bytes=moe.workspace_size(c8)) == 1
    assert L.moe_forward_host_workspace_size(ctypes.byref(moe.c_config(c8))) > moe.workspace_size(c8)
    assert L.moe_backward_workspace_size(ctypes.byref(moe.c_config(c8))) == 0


def test_backward_workspace_with_expert_choice(L):
    ce = _cfg(expert_choice=True)
    n = L.moe_backward_workspace_size(ctypes.byref(moe.c_config(ce)))
    assert n > 0
    # every expert's C rows are padded to whole 128-row blocks: C = 75 and
    # C = 128 take the same grouped rows, C = 129 one block more
    sz = [L.moe_backward_workspace_size(ctypes.byref(moe.c_config(_cfg(T=T, expert_choice=True,
                                                                         capacity_factor=1.0)))) for T in
          (600, 1024, 1032)]
    assert 0 < sz[0] <= sz[1] < sz[2]
    assert sz[2] - sz[1] >= 8 * 128 * 768 * 2
    assert L.moe_backward_workspace_size(ctypes.byref(moe.c_config(_cfg(expert_choice=True, fp8_experts=True)))) == 0


def _call_forward_fp8(L, cfg, w, **over):
    P = ctypes.c_void_p
    args = dict(x=P(0x10000), W_g=P(0x20000), y=P(0x50000000), ws=P(0x100000), ws_bytes=moe.workspace_size(cfg))
    args.update(over)
    c = moe.c_config(cfg)
    wp = ctypes.byref(w) if w is not None else None
    return L.moe_forward_fp8(ctypes.byref(c), args["x"], args["W_g"], None, None, wp, None, None, args["y"],
                             P(0x60000), P(0x70000), P(0x80000), P(0x90000), P(0xA0000), P(0xB0000), P(0xC0000),
                             None, None, None, None, args["ws"], args["ws_bytes"], None, None)


def test_forward_fp8_host_checks(L):
    c8 = _cfg(fp8_experts=True)
    w = moe._CFp8(0x30000, 0x31000, None, None, 0x40000, 0x41000)
    assert _call_forward_fp8(L, c8, None) == 1                            # no weights
    assert _call_forward_fp8(L, _cfg(), w, ws_bytes=moe.workspace_size(_cfg())) == 1   # flag missing
    assert _call_forward_fp8(L, c8, moe._CFp8(0x30000, None, None, None, 0x40000, 0x41000)) == 1  # no s1
    assert _call_forward_fp8(L, c8, moe._CFp8(0x30000, 0x31004, None, None, 0x40000, 0x41000)) == 1  # misaligned
    assert _call_forward_fp8(L, c8, w, ws_bytes=moe.workspace_size(c8) - 1) == 3
    assert _call_forward_fp8(L, c8, w, x=None) == 1


def test_quantize_host_checks(L):
    P = ctypes.c_void_p
    assert L.moe_quantize_weights_fp8(P(0x1000), 2, 100, 64, P(0x2000), P(0x3000), None) == 2     # K % 16
    assert L.moe_quantize_weights_fp8(P(0x1000), 2, 64, 64, None, P(0x3000), None) == 1
    assert L.moe_quantize_weights_fp8(P(0x1008), 2, 64, 64, P(0x2000), P(0x3000), None) == 1       # misaligned
    assert L.moe_quantize_weights_fp8(None, 0, 64, 64, None, None, None) == 0                      # empty
    assert L.moe_quantize_rows_fp8(P(0x1000), 4, 40, P(0x2000), P(0x3000), None) == 2              # cols % 16
    assert L.moe_quantize_rows_fp8(P(0x1000), -1, 64, P(0x2000), P(0x3000), None) == 1
    assert L.moe_quantize_rows_fp8(None, 0, 64, None, None, None) == 0


def _call_backward(L, cfg, **over):
    """moe_backward with fake, aligned, never-dereferenced pointers: every case
    here is rejected by the host checks before any CUDA call."""
    P = ctypes.c_void_p
    sw = cfg.act == moe.SWIGLU
    args = dict(x=P(0x10000), W_g=P(0x20000), b_g=None, noise=None, W1=P(0x30000), b1=None, W2=P(0x40000),
                b2=None, W3=P(0x50000) if sw else None, dy=P(0x60000), dL_aux=1.0, dx=P(0x70000),
                dW_g=P(0x80000), db_g=None, dW1=P(0x90000), db1=None, dW2=P(0xA0000), db2=None,
                dW3=P(0xB0000) if sw else None, ws=P(0x100000),
                ws_bytes=L.moe_backward_workspace_size(ctypes.byref(moe.c_config(cfg))))
    args.update(over)
    c = moe.c_config(cfg)
    return L.moe_backward(ctypes.byref(c), args["x"], args["W_g"], args["b_g"], args["noise"], args["W1"],
                          args["b1"], args["W2"], args["b2"], args["W3"], args["dy"], args["dL_aux"], args["dx"],
                          args["dW_g"], args["db_g"], args["dW1"], args["db1"], args["dW2"], args["db2"], args["dW3"],
                          args["ws"], args["ws_bytes"], None, None)


@pytest.mark.parametrize("ec", [False, True], ids=["token_choice", "expert_choice"])
def test_backward_host_checks(L, ec):
    P = ctypes.c_void_p
    c = _cfg(expert_choice=ec)
    assert _call_backward(L, c, dy=None) == 1
    assert _call_backward(L, c, dx=None) == 1
    assert _call_backward(L, c, dW1=None) == 1
    assert _call_backward(L, c, b_g=P(0xC0000)) == 1                 # b_g without db_g
    assert _call_backward(L, c, db1=P(0xD0000)) == 1                 # db1 without b1
    assert _call_backward(L, c, W3=P(0xE0000)) == 1                  # W3 without SwiGLU
    assert _call_backward(L, _cfg(act=moe.SWIGLU, expert_choice=ec), dW3=None) == 1
    assert _call_backward(L, _cfg(act=moe.SWIGLU, expert_choice=ec), b1=P(0xC1000), db1=P(0xC2000)) == 1
    assert _call_backward(L, c, dL_aux=float("nan")) == 1
    assert _call_backward(L, c, dy=P(0x60008)) == 1                  # misaligned
    assert _call_backward(L, c, ws_bytes=L.moe_backward_workspace_size(ctypes.byref(moe.c_config(c))) - 1) == 3
    assert _call_backward(L, c, ws=P(0x100040)) == 3                 # workspace not 256-byte aligned
    # fp32 layers and FP8 experts have no backward pass here
    assert _call_backward(L, _cfg(dtype=moe.F32, d=64, f=64, expert_choice=ec), ws_bytes=1 << 30) == 2
    assert _call_backward(L, _cfg(fp8_experts=True, expert_choice=ec), ws_bytes=1 << 30) == 2
    # T == 0: x, dy and dx may be NULL (the host checks pass; without a GPU
    # the first CUDA call then reports MOE_ERR_CUDA)
    e = _cfg(T=0, expert_choice=ec)
    assert _call_backward(L, e, x=None, dy=None, dx=None) in (0, 4)
