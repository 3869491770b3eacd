"""GB300-native forward pass of one sparse Mixture-of-Experts layer.

Thin ctypes binding over ``libcoli_moe.so`` (the C ABI in
``include/coli_moe.h``). Every function keeps the C name and argument order;
tensors are passed as device pointers, ``None`` as NULL. Marshalling only:
every step of the layer runs in the library's CUDA kernels, and calling any
of these without the built library raises instead of falling back.

Build with ``mixture_experts_gb300.build()`` (nvcc, sm_103a).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

F32, BF16, I4G128, MXFP8, MXFP4 = 0, 1, 2, 3, 4
PATH_AUTO, PATH_DECODE, PATH_PREFILL = 0, 1, 2
STATUS = {0: "COLI_OK", -1: "COLI_EINVAL", -2: "COLI_ENOMEM", -3: "COLI_ECUDA",
          -4: "COLI_EUNSUPPORTED", -5: "COLI_EDEVICE", -6: "COLI_ETIMEOUT"}
COLI_OK, COLI_EINVAL, COLI_ENOMEM, COLI_ECUDA = 0, -1, -2, -3
COLI_EUNSUPPORTED, COLI_EDEVICE, COLI_ETIMEOUT = -4, -5, -6
COLI_PERMUTE_STATIC_SCRATCH_BYTES = 65536

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcoli_moe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "coli_moe.h")
_lock = threading.Lock()
_lib = None


class ColiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class coli_moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d_model", "d_ff", "n_experts", "top_k", "max_tokens", "act_dtype", "weight_dtype",
        "has_router_bias", "path", "expert_slots", "max_promotions")]


class coli_moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "b_router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")]


def build(force: bool = False) -> str:
    from ._build import build as _b
    return _b(force=force)


_SIGS = {
    # name: (restype, [argtypes])  — P pointer, I int32, Z size_t
    "coli_version": ("s", []),
    "coli_status_string": ("s", ["I"]),
    "coli_last_error": ("s", []),
    "coli_device_status": ("I", ["P", "P", "Z"]),
    "coli_moe_create": ("I", ["P", "P", "P", "P", "P", "Z"]),
    "coli_moe_forward": ("I", ["P", "P", "I", "P", "P", "P", "Z"]),
    "coli_moe_forward_host": ("I", ["P", "P", "I", "P", "P", "P", "Z"]),
    "coli_moe_device_status": ("I", ["P", "P", "P", "Z"]),
    "coli_moe_debug_buffers": ("I", ["P"] * 8),
    "coli_moe_copy_debug": ("I", ["P", "I", "P", "P", "P", "P", "P", "P", "P", "P"]),
    "coli_moe_path_for": ("I", ["P", "I"]),
    "coli_moe_residency": ("I", ["P", "P", "P", "P"]),
    "coli_moe_set_timing": ("I", ["P", "I"]),
    "coli_moe_stage_times": ("I", ["P", "P", "I", "P", "P"]),
    "coli_moe_destroy": (None, ["P"]),
    "coli_route_scratch_bytes": ("Z", ["I", "I", "I"]),
    "coli_route_topk": ("I", ["P", "P", "P", "I", "I", "I", "I", "I", "P", "P", "P", "P", "Z",
                              "P"]),
    "coli_permute_scratch_bytes": ("Z", ["I", "I", "I"]),
    "coli_permute": ("I", ["P", "P", "I", "I", "I", "I", "I", "P", "P", "P", "P", "P", "P", "Z",
                           "P"]),
    "coli_expert_ffn": ("I", ["P", "P", "P", "I", "P", "P"]),
    "coli_combine": ("I", ["P", "P", "P", "I", "I", "I", "I", "P", "P"]),
    "coli_selftest_bounded_wait": ("I", ["I", "P"]),
    "coli_permute_noalloc": ("I", ["P", "P", "I", "I", "I", "I", "I", "P", "P", "P", "P", "P",
                                   "P"]),
}
_CT = {"P": ctypes.c_void_p, "I": ctypes.c_int32, "Z": ctypes.c_size_t, "s": ctypes.c_char_p,
       None: None}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run mixture_experts_gb300.build()")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = _CT[res]
                fn.argtypes = [_CT[a] for a in args]
            _lib = h
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/coli_moe.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coli_\w+)\s*\(", text)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if isinstance(t, ctypes.c_void_p):
        return t.value
    raise TypeError(f"cannot pass {type(t)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        if not torch.cuda.is_available():
            return 0  # argument validation still runs; nothing is launched
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str, msg: str | None = None):
    if rc != 0:
        raise ColiError(rc, f"{what}: {msg if msg is not None else last_error()}")


def last_error() -> str:
    return lib().coli_last_error().decode()


# ---- same names as the C ABI ------------------------------------------------------
def coli_version() -> str:
    return lib().coli_version().decode()


def coli_status_string(status: int) -> str:
    return lib().coli_status_string(status).decode()


def coli_device_status(stream=None) -> int:
    buf = ctypes.create_string_buffer(256)
    return lib().coli_device_status(_stream(stream), buf, 256)


def coli_route_scratch_bytes(T: int, d: int, E: int) -> int:
    return lib().coli_route_scratch_bytes(T, d, E)


def coli_route_topk(x, w_router, b_router, T, d, E, k, act, topk_idx, topk_w, gap=None,
                    scratch=None, scratch_bytes=0, stream=None) -> int:
    return lib().coli_route_topk(_ptr(x), _ptr(w_router), _ptr(b_router), T, d, E, k, act,
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(gap), _ptr(scratch),
                                 scratch_bytes, _stream(stream))


def coli_permute_scratch_bytes(T: int, k: int, E: int) -> int:
    return lib().coli_permute_scratch_bytes(T, k, E)


def coli_permute(topk_idx, x, T, d, E, k, act, counts, offsets, row_token, assign_row, x_perm,
                 scratch=None, scratch_bytes=0, stream=None) -> int:
    return lib().coli_permute(_ptr(topk_idx), _ptr(x), T, d, E, k, act, _ptr(counts),
                              _ptr(offsets), _ptr(row_token), _ptr(assign_row), _ptr(x_perm),
                              _ptr(scratch), scratch_bytes, _stream(stream))


def coli_expert_ffn(h, x_perm, offsets, n_rows, y_perm, stream=None) -> int:
    return lib().coli_expert_ffn(_ptr(h), _ptr(x_perm), _ptr(offsets), n_rows, _ptr(y_perm),
                                 _stream(stream))


def coli_combine(y_perm, assign_row, topk_w, T, k, d, out, y, stream=None) -> int:
    return lib().coli_combine(_ptr(y_perm), _ptr(assign_row), _ptr(topk_w), T, k, d, out, _ptr(y),
                              _stream(stream))


def coli_moe_create(cfg: coli_moe_config, weights: coli_moe_weights, stream=None):
    """Returns (status, handle, message)."""
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(512)
    rc = lib().coli_moe_create(ctypes.byref(cfg), ctypes.byref(weights), _stream(stream),
                               ctypes.byref(h), buf, 512)
    return rc, h, buf.value.decode()


def coli_moe_forward(h, x, T, y, stream=None) -> int:
    return lib().coli_moe_forward(_ptr(h), _ptr(x), T, _ptr(y), _stream(stream), None, 0)


def coli_moe_forward_host(h, x_host, T, y_host, stream=None) -> int:
    return lib().coli_moe_forward_host(_ptr(h), _ptr(x_host), T, _ptr(y_host), _stream(stream),
                                       None, 0)


def coli_moe_device_status(h, stream=None) -> int:
    return lib().coli_moe_device_status(_ptr(h), _stream(stream), None, 0)


def coli_moe_copy_debug(h, T, topk_idx=None, topk_w=None, gap=None, counts=None, offsets=None,
                        row_token=None, assign_row=None, stream=None) -> int:
    return lib().coli_moe_copy_debug(_ptr(h), T, _ptr(topk_idx), _ptr(topk_w), _ptr(gap),
                                     _ptr(counts), _ptr(offsets), _ptr(row_token),
                                     _ptr(assign_row), _stream(stream))


def coli_moe_residency(h, n_experts: int, stream=None):
    """(status, slot of each expert (-1: read from host memory), promotions
    since create) of a handle's residency tier; synchronises the stream."""
    slots = (ctypes.c_int32 * n_experts)()
    n = ctypes.c_int64()
    rc = lib().coli_moe_residency(_ptr(h), slots, ctypes.byref(n), _stream(stream))
    return rc, list(slots), n.value


def coli_moe_path_for(h, T) -> int:
    return lib().coli_moe_path_for(_ptr(h), T)


def coli_moe_set_timing(h, enable: bool) -> int:
    return lib().coli_moe_set_timing(_ptr(h), int(bool(enable)))


def coli_moe_stage_times(h):
    """(per-stage ms summed over timed forwards, forwards, kernel launches)."""
    ms = (ctypes.c_float * 5)()
    nf = ctypes.c_int32()
    nl = ctypes.c_int64()
    _check(lib().coli_moe_stage_times(_ptr(h), ms, 5, ctypes.byref(nf), ctypes.byref(nl)),
           "coli_moe_stage_times")
    return list(ms), nf.value, nl.value


def coli_moe_destroy(h) -> None:
    lib().coli_moe_destroy(_ptr(h))


def coli_permute_noalloc(topk_idx, x, T, d, E, k, act, counts, offsets, row_token, assign_row,
                         x_perm, stream=None) -> int:
    """coli_permute without caller scratch, for callers that cannot allocate
    device memory at the call site; its scratch is a fixed area inside the
    library (COLI_PERMUTE_STATIC_SCRATCH_BYTES), shared by all calls."""
    return lib().coli_permute_noalloc(_ptr(topk_idx), _ptr(x), T, d, E, k, act, _ptr(counts),
                                      _ptr(offsets), _ptr(row_token), _ptr(assign_row),
                                      _ptr(x_perm), _stream(stream))


def coli_selftest_bounded_wait(spin_limit: int, stream=None) -> int:
    return lib().coli_selftest_bounded_wait(spin_limit, _stream(stream))


# ---- convenience -------------------------------------------------------------------
class MoELayer:
    """One MoE layer on the current CUDA device (weights copied at creation).

    ``weights``: dict with w_router, b_router (or None), w_gate, w_up, w_down
    and for int4 s_gate, s_up, s_down — CUDA tensors in the canonical layouts.
    """

    def __init__(self, d_model, d_ff, n_experts, top_k, max_tokens, act_dtype, weight_dtype,
                 weights: dict, path: int = PATH_AUTO, stream=None, expert_slots: int = 0,
                 max_promotions: int = 0):
        import torch
        self.cfg = coli_moe_config(d_model, d_ff, n_experts, top_k, max_tokens, act_dtype,
                                   weight_dtype, int(weights.get("b_router") is not None), path,
                                   expert_slots, max_promotions)
        w = coli_moe_weights(*[_ptr(weights.get(n)) for n in (
            "w_router", "b_router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")])
        rc, h, msg = coli_moe_create(self.cfg, w, stream)
        _check(rc, "coli_moe_create", msg)
        self.h = h
        self._torch = torch
        self.act_torch = torch.float32 if act_dtype == F32 else torch.bfloat16

    def forward(self, x, y=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = self._torch.empty_like(x)
        _check(coli_moe_forward(self.h, x, T, y, stream), "coli_moe_forward")
        return y

    __call__ = forward

    def forward_host(self, x_host, y_host, stream=None):
        _check(coli_moe_forward_host(self.h, x_host, x_host.shape[0], y_host, stream),
               "coli_moe_forward_host")
        return y_host

    def debug(self, T: int, stream=None) -> dict:
        torch = self._torch
        c = self.cfg
        dev = torch.device("cuda")
        out = {
            "topk_idx": torch.empty(T, c.top_k, dtype=torch.int32, device=dev),
            "topk_w": torch.empty(T, c.top_k, dtype=torch.float32, device=dev),
            "gap": torch.empty(T, dtype=torch.float32, device=dev),
            "counts": torch.empty(c.n_experts, dtype=torch.int32, device=dev),
            "offsets": torch.empty(c.n_experts + 1, dtype=torch.int32, device=dev),
            "row_token": torch.empty(T * c.top_k, dtype=torch.int32, device=dev),
            "assign_row": torch.empty(T * c.top_k, dtype=torch.int32, device=dev),
        }
        _check(coli_moe_copy_debug(self.h, T, out["topk_idx"], out["topk_w"], out["gap"],
                                   out["counts"], out["offsets"], out["row_token"],
                                   out["assign_row"], stream), "coli_moe_copy_debug")
        return out

    def path_for(self, T: int) -> int:
        return coli_moe_path_for(self.h, T)

    def residency(self, stream=None):
        """(slot of each expert, -1 = host memory; promotions since create)."""
        rc, slots, n = coli_moe_residency(self.h, self.cfg.n_experts, stream)
        _check(rc, "coli_moe_residency")
        return slots, n

    def status(self, stream=None) -> int:
        return coli_moe_device_status(self.h, stream)

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            coli_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
