"""ctypes declarations of the C ABI (include/moe_decode.h) and thin wrappers.

The wrappers keep the C names. They turn torch tensors into pointers, and
status codes into MoeError. Every step of the decode path runs in
libmoe_decode.so; nothing here computes any part of it. If the library is
missing, the first call raises RuntimeError. There is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Any, Dict, Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_decode.so")

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_TIMEOUT,
 MOE_ERR_RANGE) = range(7)
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_FLAG_F32_DEBUG = 1 << 0
MOE_FLAG_TRACE = 1 << 1
MOE_FLAG_PHASE_TIMES = 1 << 2
MOE_FLAG_GROUPED_COHORTS = 1 << 3
MOE_FLAG_TEST_STALL = 1 << 8
MOE_ACT_SWIGLU, MOE_ACT_GEGLU, MOE_ACT_GEGLU_TANH, MOE_ACT_SWIGLU_CLAMPED = range(4)

EXPORTED = (
    "moe_abi_version", "moe_status_str", "moe_plan_workspace_bytes", "moe_plan_create",
    "moe_decode_forward", "moe_decode_forward_host", "moe_plan_check", "moe_get_routing",
    "moe_get_phase_times", "moe_plan_launch_count", "moe_plan_free", "moe_decode_forward_noalloc",
    "moe_decode_forward_layers",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {moe_status_str(status)} ({status})")


class moe_config(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("top_k", ctypes.c_int), ("D", ctypes.c_int),
                ("Dff", ctypes.c_int), ("bits", ctypes.c_int), ("group_size", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("x_dtype", ctypes.c_int),
                ("router_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("flags", ctypes.c_uint), ("mma_min_tokens", ctypes.c_int),
                ("activation", ctypes.c_int), ("act_limit", ctypes.c_float),
                ("down_bits", ctypes.c_int), ("expert_begin", ctypes.c_int),
                ("expert_end", ctypes.c_int)]


PLANE_FIELDS = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")


class moe_expert_planes(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in PLANE_FIELDS]


class moe_layer_io(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("planes", moe_expert_planes), ("out", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run quantized_moe_decode_softmax_gb300.build.build(). "
                "There is no fallback path.")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
        L.moe_abi_version.restype = i32
        L.moe_status_str.argtypes = [i32]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_plan_workspace_bytes.argtypes = [P(moe_config), P(ctypes.c_size_t)]
        L.moe_plan_create.argtypes = [P(moe_config), P(vp)]
        L.moe_decode_forward.argtypes = [vp, vp, vp, vp, P(moe_expert_planes), i32, i32, vp, vp]
        L.moe_decode_forward_host.argtypes = [vp, vp, vp, vp, P(moe_expert_planes), i32, i32, vp, vp]
        L.moe_plan_check.argtypes = [vp]
        L.moe_get_routing.argtypes = [vp] + [vp] * 8
        L.moe_plan_launch_count.argtypes = [vp, P(ctypes.c_uint64)]
        L.moe_get_phase_times.argtypes = [vp, vp, i32, P(i32)]
        L.moe_plan_free.argtypes = [vp]
        L.moe_decode_forward_layers.argtypes = [vp, P(moe_layer_io), i32, i32, i32, vp]
        for name in ("moe_plan_workspace_bytes", "moe_plan_create", "moe_decode_forward",
                     "moe_decode_forward_host", "moe_plan_check", "moe_get_routing", "moe_plan_launch_count",
                     "moe_get_phase_times", "moe_plan_free", "moe_decode_forward_layers"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _ptr(t: Any) -> Optional[int]:
    """Device or host address of a torch tensor, numpy array, int or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(stream: Any) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoeError(st, what)


def make_config(E, top_k, D, Dff, max_tokens, x_dtype=MOE_DTYPE_BF16, router_dtype=None,
                out_dtype=None, flags=0, mma_min_tokens=0, bits=4, group_size=64,
                activation=MOE_ACT_SWIGLU, act_limit=0.0, down_bits=0, expert_begin=0,
                expert_end=0) -> moe_config:
    router_dtype = x_dtype if router_dtype is None else router_dtype
    out_dtype = x_dtype if out_dtype is None else out_dtype
    return moe_config(E, top_k, D, Dff, bits, group_size, max_tokens, x_dtype, router_dtype,
                      out_dtype, flags, mma_min_tokens, activation, act_limit, down_bits,
                      expert_begin, expert_end)


def make_planes(planes: Any) -> moe_expert_planes:
    """moe_expert_planes from an object or dict holding the nine device tensors."""
    get = planes.__getitem__ if isinstance(planes, dict) else (lambda f: getattr(planes, f))
    return moe_expert_planes(*[_ptr(get(f)) for f in PLANE_FIELDS])


# --- the C entry points, same names --------------------------------------------

def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_status_str(st: int) -> str:
    return lib().moe_status_str(int(st)).decode()


def moe_plan_workspace_bytes(cfg: moe_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_plan_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "moe_plan_workspace_bytes")
    return n.value


def moe_plan_create(cfg: moe_config) -> int:
    h = ctypes.c_void_p(None)
    _check(lib().moe_plan_create(ctypes.byref(cfg), ctypes.byref(h)), "moe_plan_create")
    return h.value


def moe_decode_forward(plan: int, x, router_w, router_bias, planes, n_tokens: int, top_k: int,
                       out, stream=None) -> None:
    pl = planes if isinstance(planes, moe_expert_planes) else make_planes(planes)
    st = lib().moe_decode_forward(plan, _ptr(x), _ptr(router_w), _ptr(router_bias),
                                  ctypes.byref(pl), int(n_tokens), int(top_k), _ptr(out),
                                  _stream(stream))
    _check(st, "moe_decode_forward")


def moe_decode_forward_layers(plan: int, layers, n_tokens: int, top_k: int, stream=None) -> None:
    """layers: sequence of (x, router_w, router_bias, planes, out)."""
    arr = (moe_layer_io * len(layers))()
    for i, (x, rw, rb, planes, out) in enumerate(layers):
        pl = planes if isinstance(planes, moe_expert_planes) else make_planes(planes)
        arr[i] = moe_layer_io(_ptr(x), _ptr(rw), _ptr(rb), pl, _ptr(out))
    st = lib().moe_decode_forward_layers(plan, arr, len(layers), int(n_tokens), int(top_k), _stream(stream))
    _check(st, "moe_decode_forward_layers")


def moe_decode_forward_host(plan: int, x_host, router_w, router_bias, planes, n_tokens: int,
                            top_k: int, out_host, stream=None) -> None:
    pl = planes if isinstance(planes, moe_expert_planes) else make_planes(planes)
    st = lib().moe_decode_forward_host(plan, _ptr(x_host), _ptr(router_w), _ptr(router_bias),
                                       ctypes.byref(pl), int(n_tokens), int(top_k),
                                       _ptr(out_host), _stream(stream))
    _check(st, "moe_decode_forward_host")


def moe_decode_forward_noalloc(cfg: moe_config, x, router_w, router_bias, planes, n_tokens: int,
                               top_k: int, out, stream=None) -> None:
    """The decode step without a plan and without device allocation (see the
    header): scratch lives in a static device array of the library."""
    L = lib()
    fn = L.moe_decode_forward_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(moe_config), vp, vp, vp, ctypes.POINTER(moe_expert_planes),
                   ctypes.c_int, ctypes.c_int, vp, vp]
    fn.restype = ctypes.c_int
    pl = planes if isinstance(planes, moe_expert_planes) else make_planes(planes)
    st = fn(ctypes.byref(cfg), _ptr(x), _ptr(router_w), _ptr(router_bias), ctypes.byref(pl),
            int(n_tokens), int(top_k), _ptr(out), _stream(stream))
    _check(st, "moe_decode_forward_noalloc")


def moe_plan_check(plan: int) -> None:
    _check(lib().moe_plan_check(plan), "moe_plan_check")


def moe_get_routing(plan: int, n_tokens: int, E: int, top_k: int) -> Dict[str, Any]:
    S = n_tokens * top_k
    r = dict(topk_idx=np.empty((n_tokens, top_k), np.int32), topk_w=np.empty((n_tokens, top_k), np.float32),
             counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
             slot_token=np.empty(S, np.int32), slot_k=np.empty(S, np.int32),
             unique=np.empty(E, np.int32), U=np.zeros(1, np.int32))
    order = ("topk_idx", "topk_w", "counts", "offsets", "slot_token", "slot_k", "unique", "U")
    _check(lib().moe_get_routing(plan, *[r[k].ctypes.data for k in order]), "moe_get_routing")
    u = int(r["U"][0])
    r["U"] = u
    r["unique"] = r["unique"][:u].copy()
    return r


def moe_plan_launch_count(plan: int) -> int:
    c = ctypes.c_uint64(0)
    _check(lib().moe_plan_launch_count(plan, ctypes.byref(c)), "moe_plan_launch_count")
    return c.value


PHASES = ("start", "router", "barrier1", "routing", "gate_up", "barrier2", "down", "end",
          "a_wait", "a_compute", "b_wait", "b_compute", "reserved", "a_chunks", "b_tiles",
          "reserved")


def moe_get_phase_times(plan: int) -> np.ndarray:
    """[ctas, 16] int64 of the plan's last fused step (see PHASES and the header)."""
    buf = np.zeros(16 * 1024, np.uint64)
    ctas = ctypes.c_int(0)
    _check(lib().moe_get_phase_times(plan, buf.ctypes.data, buf.size, ctypes.byref(ctas)),
           "moe_get_phase_times")
    return buf[: 16 * ctas.value].reshape(ctas.value, 16).astype(np.int64)


def moe_plan_free(plan: int) -> None:
    _check(lib().moe_plan_free(plan), "moe_plan_free")
