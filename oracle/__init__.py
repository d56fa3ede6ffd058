"""CPU oracle for the quantized MoE decode step (ctypes over moe_oracle.c).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and the CPU-baseline
leg of bench.py may import this package. The CUDA library never calls it.

The C file states what is computed and which passages it follows. This
wrapper only marshals numpy arrays. Inputs are float values for x and the
router (already widened from bf16 where the workload stores bf16), uint32
planes and uint16 (bf16 bits) scales and biases.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


# activation kinds (moe_oracle.c oracle_options)
ACT_SWIGLU, ACT_GEGLU, ACT_GEGLU_TANH, ACT_SWIGLU_CLAMPED = 0, 1, 2, 3


class _Options(ctypes.Structure):
    _fields_ = [("activation", ctypes.c_int), ("limit", ctypes.c_float), ("down_bits", ctypes.c_int)]


class _Planes(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")]


def _load(path: str):
    L = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.oracle_set_threads.argtypes = [i32]
    L.oracle_set_threads.restype = i32
    L.oracle_dequant.argtypes = [vp, vp, vp, i32, i32, vp]
    L.oracle_route.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    L.oracle_group.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    L.oracle_dequant6.argtypes = [vp, vp, vp, i32, i32, vp]
    L.oracle_expert_mlp.argtypes = [i32, i32, vp] + [vp] * 9 + [vp, vp]
    L.oracle_expert_mlp_opt.argtypes = [i32, i32, vp] + [vp] * 9 + [ctypes.POINTER(_Options), vp, vp]
    L.oracle_moe_forward.argtypes = [i32] * 5 + [vp, vp, vp, ctypes.POINTER(_Planes)] + [vp] * 10
    L.oracle_moe_forward.restype = i32
    L.oracle_moe_forward_opt.argtypes = [i32] * 5 + [vp, vp, vp, ctypes.POINTER(_Planes),
                                                     ctypes.POINTER(_Options)] + [vp] * 10
    L.oracle_moe_forward_opt.restype = i32
    L.oracle_round_bf16.argtypes = [vp, vp, ctypes.c_size_t]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(build())
    return _lib


@contextlib.contextmanager
def using(path: str):
    """Temporarily route every call in this module to another build of the
    oracle source (used by the tests that plant a mistake in a copy of it)."""
    global _lib
    old = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = old


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> int:
    return lib().oracle_set_threads(int(n))


def dequant(q, s, b) -> np.ndarray:
    """Dequantise one plane [rows, cols]: q uint32 [rows, cols/8], s/b uint16 bits."""
    q, s, b = _c(q, np.uint32), _c(s, np.uint16), _c(b, np.uint16)
    rows, cols = q.shape[0], q.shape[1] * 8
    out = np.empty((rows, cols), np.float32)
    lib().oracle_dequant(_p(q), _p(s), _p(b), rows, cols, _p(out))
    return out


def dequant6(q, s, b) -> np.ndarray:
    """Dequantise one 6-bit plane [rows, cols]: q uint8 [rows, 3*cols/4] (bit
    stream, code j at bits 6j..6j+5), s/b uint16 bits [rows, cols/64]."""
    q, s, b = _c(q, np.uint8), _c(s, np.uint16), _c(b, np.uint16)
    rows, cols = q.shape[0], q.shape[1] * 4 // 3
    out = np.empty((rows, cols), np.float32)
    lib().oracle_dequant6(_p(q), _p(s), _p(b), rows, cols, _p(out))
    return out


def _options(activation=ACT_SWIGLU, limit=0.0, down_bits=4):
    return _Options(int(activation), float(limit), int(down_bits))


def route(x, router_w, bias, k):
    """-> (topk_idx [n,k] int32, topk_w [n,k] f32, logits [n,E] f32, probs [n,E] f32)."""
    x, wr = _c(x, np.float32), _c(router_w, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    n, D = x.shape
    E = wr.shape[0]
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    lg = np.empty((n, E), np.float32)
    pr = np.empty((n, E), np.float32)
    lib().oracle_route(n, E, D, k, _p(x), _p(wr), _p(bias), _p(idx), _p(w), _p(lg), _p(pr))
    return idx, w, lg, pr


def group(topk_idx, E):
    """-> dict(counts, offsets, slot_token, slot_k, unique, U)."""
    idx = _c(topk_idx, np.int32)
    n, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    st = np.empty(n * k, np.int32)
    sk = np.empty(n * k, np.int32)
    uq = np.empty(E, np.int32)
    U = np.zeros(1, np.int32)
    lib().oracle_group(n, E, k, _p(idx), _p(counts), _p(offsets), _p(st), _p(sk), _p(uq), _p(U))
    u = int(U[0])
    return dict(counts=counts, offsets=offsets, slot_token=st, slot_k=sk, unique=uq[:u].copy(), U=u)


def expert_mlp(x_t, planes, e, activation=ACT_SWIGLU, limit=0.0, down_bits=4):
    """One expert's gated MLP on one token -> (h [F], y [D]). The default is
    SwiGLU with 4-bit down planes; down_bits=6 takes uint8 down codes."""
    x_t = _c(x_t, np.float32)
    D = x_t.shape[0]
    F = planes.gate_q.shape[1]
    arrs = [_c(a[e], a.dtype) for a in planes.arrays()]
    h = np.empty(F, np.float32)
    y = np.empty(D, np.float32)
    opt = _options(activation, limit, down_bits)
    lib().oracle_expert_mlp_opt(D, F, _p(x_t), *[_p(a) for a in arrs], ctypes.byref(opt), _p(h), _p(y))
    return h, y


def moe_forward(x, router_w, bias, planes, k, want_bf16: bool = False, activation=ACT_SWIGLU,
                limit=0.0, down_bits=4):
    """The whole decode step. Returns a dict with routing, grouping and out.
    activation / limit / down_bits select the layer variant (moe_oracle.c
    oracle_options); the default is SwiGLU with 4-bit down planes."""
    x, wr = _c(x, np.float32), _c(router_w, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    n, D = x.shape
    E = wr.shape[0]
    F = planes.gate_q.shape[1]
    arrs = [np.ascontiguousarray(a) for a in planes.arrays()]
    pl = _Planes(*[a.ctypes.data for a in arrs])
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    st = np.empty(n * k, np.int32)
    sk = np.empty(n * k, np.int32)
    uq = np.empty(E, np.int32)
    U = np.zeros(1, np.int32)
    out = np.empty((n, D), np.float32)
    out16 = np.empty((n, D), np.uint16) if want_bf16 else None
    opt = _options(activation, limit, down_bits)
    rc = lib().oracle_moe_forward_opt(E, k, D, F, n, _p(x), _p(wr), _p(bias), ctypes.byref(pl),
                                      ctypes.byref(opt), _p(idx), _p(w), _p(counts), _p(offsets),
                                      _p(st), _p(sk), _p(uq), _p(U), _p(out), _p(out16))
    if rc != 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    u = int(U[0])
    return dict(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, slot_token=st,
                slot_k=sk, unique=uq[:u].copy(), U=u, out=out, out_bf16=out16)


def round_bf16(a) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().oracle_round_bf16(_p(a), _p(out), a.size)
    return out
