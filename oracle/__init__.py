"""Oracle for one sparse MoE layer forward: TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement of the layer (``moe_oracle.cpp``, fp64
accumulation), wrapped with ctypes. It runs on one thread; ``moe_forward``
can also split its token list over several threads, each running the same
per-token code, which gives bit-identical outputs (used to check full-size
layers in reasonable time). Only ``tests/``, the smoke check and
the benchmark's CPU-baseline leg may import this package. It shares no code
with the CUDA library and never imports it.

Arrays are numpy (or CPU torch tensors, converted here). bf16 data travels as
its raw 16-bit patterns (``uint16``); int4 weights as packed bytes plus bf16
scales. dtype codes: 0 = f32, 1 = bf16, 2 = int4 with 128-wide groups,
3 = MXFP8 (E4M3 bytes), 4 = MXFP4 (E2M1 nibbles), both with E8M0 scale bytes
per 32 reduction indices.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, I4G128, MXFP8, MXFP4 = 0, 1, 2, 3, 4
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_handle = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (portable C++17, no intrinsics, no FMA
    contraction so x86 and Arm hosts give the same bits)."""
    stale = not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            build()
            h = ctypes.CDLL(_LIB)
            vp, i, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            h.oracle_version.restype = i
            h.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
            h.oracle_bf16_to_float.restype = ctypes.c_float
            h.oracle_float_to_bf16.argtypes = [ctypes.c_float]
            h.oracle_float_to_bf16.restype = ctypes.c_uint16
            h.oracle_weight_at.argtypes = [vp, vp, i, i, i, i, i, i]
            h.oracle_weight_at.restype = f64
            h.oracle_mx_element.argtypes = [i, i]
            h.oracle_mx_element.restype = f64
            h.oracle_router_logits.argtypes = [vp, i, vp, vp, i, i, i, _f32p]
            h.oracle_select_topk.argtypes = [_f32p, i, i, i, _i32p, _f32p, vp, vp]
            h.oracle_dispatch.argtypes = [_i32p, i, i, i, _i32p, _i32p, vp, vp]
            h.oracle_expert_ffn.argtypes = [vp, i, i, vp, vp, vp, vp, vp, vp, i, i, i, i,
                                            _f64p]
            h.oracle_combine.argtypes = [_f32p, _i32p, _f32p, i, i, i, i, vp, vp]
            h.oracle_moe_forward.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, vp, vp,
                                             vp, i, i, vp, i, vp, vp, vp, vp, vp]
            h.oracle_moe_forward_mt.argtypes = h.oracle_moe_forward.argtypes + [i]
            for name in ("oracle_router_logits", "oracle_select_topk", "oracle_dispatch",
                         "oracle_expert_ffn", "oracle_combine", "oracle_moe_forward",
                         "oracle_moe_forward_mt"):
                getattr(h, name).restype = i
            _handle = h
    return _handle


def to_np(a):
    """CPU torch tensor or numpy array -> contiguous numpy (bf16 -> uint16 bits)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16)
            return a.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def bf16_to_float(bits: int) -> float:
    return float(_lib().oracle_bf16_to_float(int(bits)))


def float_to_bf16(v: float) -> int:
    return int(_lib().oracle_float_to_bf16(float(v)))


def weight_at(w, s, w_dt, e, rows, cols, r, c) -> float:
    w, s = to_np(w), to_np(s)
    return float(_lib().oracle_weight_at(_ptr(w), _ptr(s), w_dt, e, rows, cols, r, c))


def mx_element(w_dt, code) -> float:
    """Value of one E4M3 (w_dt MXFP8) or E2M1 (MXFP4) code, or of an E8M0
    scale code (any other w_dt)."""
    return float(_lib().oracle_mx_element(w_dt, int(code)))


def router_logits(x, act_dt, w_r, b_r, T, d, E):
    x, w_r, b_r = to_np(x), to_np(w_r), to_np(b_r)
    if b_r is not None:
        b_r = np.ascontiguousarray(b_r, dtype=np.float32)
    out = np.empty((T, E), np.float32)
    _check(_lib().oracle_router_logits(_ptr(x), act_dt, _ptr(w_r), _ptr(b_r), T, d, E, out),
           "router_logits")
    return out


def select_topk(logits, k):
    logits = np.ascontiguousarray(to_np(logits), dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    gap = np.empty(T, np.float32)
    inner = np.empty(T, np.float32)
    _check(_lib().oracle_select_topk(logits, T, E, k, idx, w, _ptr(gap), _ptr(inner)),
           "select_topk")
    return idx, w, gap, inner


def dispatch(topk_idx, E):
    topk_idx = np.ascontiguousarray(to_np(topk_idx), dtype=np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_token = np.empty(T * k, np.int32)
    assign_row = np.empty(T * k, np.int32)
    _check(_lib().oracle_dispatch(topk_idx, T, k, E, counts, offsets, _ptr(row_token),
                                  _ptr(assign_row)), "dispatch")
    return counts, offsets, row_token, assign_row


def expert_ffn(x_rows, act_dt, layer, e, d, f, w_dt):
    """FFN of expert ``e`` on the rows of ``x_rows`` -> float64 [n][d]."""
    x_rows = to_np(x_rows)
    n = x_rows.shape[0]
    y = np.empty((n, d), np.float64)
    ws = [to_np(layer.get(k)) for k in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")]
    _check(_lib().oracle_expert_ffn(_ptr(x_rows), act_dt, n, *[_ptr(a) for a in ws], w_dt, e,
                                    d, f, y), "expert_ffn")
    return y


def combine(y_perm, assign_row, topk_w, T, k, d, out_dt):
    y_perm = np.ascontiguousarray(to_np(y_perm), dtype=np.float32)
    assign_row = np.ascontiguousarray(to_np(assign_row), dtype=np.int32)
    topk_w = np.ascontiguousarray(to_np(topk_w), dtype=np.float32)
    y64 = np.empty((T, d), np.float64)
    yo = np.empty((T, d), np.float32 if out_dt == F32 else np.uint16)
    _check(_lib().oracle_combine(y_perm, assign_row, topk_w, T, k, d, out_dt, _ptr(y64),
                                 _ptr(yo)), "combine")
    return y64, yo


def moe_forward(layer, act_dt, w_dt, T, d, E, k, f, tokens=None, threads=1):
    """Whole layer for ``tokens`` (all when None). Returns a dict with y_f64
    [n][d], y (act dtype: float32 or uint16 bf16 bits), topk_idx, topk_w, gap.
    ``threads`` > 1 splits the token list into that many contiguous ranges,
    one thread each, with bit-identical results."""
    x, w_r, b_r = to_np(layer["x"]), to_np(layer["w_router"]), to_np(layer.get("b_router"))
    if b_r is not None:
        b_r = np.ascontiguousarray(b_r, dtype=np.float32)
    ws = [to_np(layer.get(key)) for key in ("w_gate", "w_up", "w_down", "s_gate", "s_up",
                                           "s_down")]
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tok is None else len(tok)
    y64 = np.empty((n, d), np.float64)
    yo = np.empty((n, d), np.float32 if act_dt == F32 else np.uint16)
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    gap = np.empty(n, np.float32)
    args = (_ptr(x), act_dt, T, d, _ptr(w_r), _ptr(b_r), E, k, *[_ptr(a) for a in ws], w_dt, f,
            _ptr(tok), 0 if tok is None else len(tok), _ptr(y64), _ptr(yo), _ptr(idx), _ptr(w),
            _ptr(gap))
    if threads > 1:
        rc = _lib().oracle_moe_forward_mt(*args, int(threads))
    else:
        rc = _lib().oracle_moe_forward(*args)
    _check(rc, "moe_forward")
    return {"y_f64": y64, "y": yo, "topk_idx": idx, "topk_w": w, "gap": gap}
