"""ctypes front end of ``forward.c`` (TEST INFRASTRUCTURE ONLY).

``build()`` compiles the C oracle with gcc (OpenMP) into ``oracle/_lib``.
``decode_step`` runs one decode step of a Llama-style decoder on host arrays:
weights and KV caches are bf16 bit patterns (``numpy.uint16``), the cache is
appended in place.  ``precision=64`` is the reference arithmetic; ``32`` is
the same code in float, only for timing the CPU baseline.

The argmax is taken on the logits rounded to float32, lowest index on ties,
so that the decision is made in the precision the GPU path computes in.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    src = [os.path.join(_HERE, "forward.c")]
    deps = src + [os.path.join(_HERE, "forward_impl.h")]
    if not force and os.path.exists(_LIB_PATH) and all(
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(p) for p in deps):
        return _LIB_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp] + src + ["-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Shape(C.Structure):
    _fields_ = [("L", C.c_int), ("H", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int),
                ("F", C.c_int), ("V", C.c_int), ("qk_norm", C.c_int), ("eps", C.c_double), ("theta", C.c_double)]


_PP = C.POINTER(C.c_void_p)


class _Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("norm_final", C.c_void_p)] + [
        (n, _PP) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm_attn", "norm_mlp", "qnorm", "knorm")] + [
        ("fp8", C.c_int), ("w8", _PP * 7), ("s8", _PP * 7)]


PROJ = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")  # the seven projections, in the C oracle's matrix order


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        d = C.POINTER(C.c_double)
        u16 = C.POINTER(C.c_uint16)
        _lib.orc_rmsnorm.argtypes = [d, C.c_int, u16, C.c_double, d]
        _lib.orc_matvec.argtypes = [u16, C.c_int, C.c_int, d, d]
        _lib.orc_rope.argtypes = [d, C.c_int, C.c_int, C.c_double]
        _lib.orc_attend.argtypes = [d, u16, u16, C.c_int, C.c_int, d]
        _lib.orc_to_bf16.argtypes = [d, u16, C.c_long]
        _lib.orc_matvec8.argtypes = [C.POINTER(C.c_uint8), C.POINTER(C.c_float), C.c_int, C.c_int, d, d]
        _lib.e4m3_to_double.argtypes = [C.c_uint8]
        _lib.e4m3_to_double.restype = C.c_double
        _lib.bf16_to_double.argtypes = [C.c_uint16]
        _lib.bf16_to_double.restype = C.c_double
        for nm in ("orc_decode_step_f64", "orc_decode_step_f32"):
            getattr(_lib, nm).argtypes = [C.POINTER(_Shape), C.POINTER(_Weights), u16, u16, C.c_int, C.c_int,
                                          C.POINTER(C.c_int), C.POINTER(C.c_int), C.c_int, C.c_void_p, C.c_void_p]
            getattr(_lib, nm).restype = C.c_int
    return _lib


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _up(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_uint16))


# ---- single ops (double) ----

def rmsnorm(x: np.ndarray, w_bf16: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_dp(x), x.size, _up(np.ascontiguousarray(w_bf16)), eps, _dp(y))
    return y


def matvec(W_bf16: np.ndarray, x: np.ndarray) -> np.ndarray:
    N, K = W_bf16.shape
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty(N)
    lib().orc_matvec(_up(np.ascontiguousarray(W_bf16)), N, K, _dp(x), _dp(y))
    return y


def matvec8(codes: np.ndarray, scales: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x for e4m3 codes [N, K] with fp32 scales [ceil(N/128), K/128] (one per 128 x 128 block)."""
    N, K = codes.shape
    assert K % 128 == 0
    c = np.ascontiguousarray(codes, np.uint8)
    sc = np.ascontiguousarray(scales, np.float32)
    assert sc.shape == ((N + 127) // 128, K // 128)
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty(N)
    lib().orc_matvec8(c.ctypes.data_as(C.POINTER(C.c_uint8)), sc.ctypes.data_as(C.POINTER(C.c_float)), N, K,
                      _dp(x), _dp(y))
    return y


def e4m3_value(code: int) -> float:
    return lib().e4m3_to_double(code)


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, np.float64)
    lib().orc_rope(_dp(v), v.size, pos, theta)
    return v


def attend(q: np.ndarray, K_bf16: np.ndarray, V_bf16: np.ndarray) -> np.ndarray:
    n, D = K_bf16.shape
    q = np.ascontiguousarray(q, np.float64)
    o = np.empty(D)
    lib().orc_attend(_dp(q), _up(np.ascontiguousarray(K_bf16)), _up(np.ascontiguousarray(V_bf16)), n, D, _dp(o))
    return o


def to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty(x.shape, np.uint16)
    lib().orc_to_bf16(_dp(x.reshape(-1)), y.reshape(-1).ctypes.data_as(C.POINTER(C.c_uint16)), x.size)
    return y


def bf16_to_f64(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- whole decode step ----

@dataclass
class Shape:
    L: int
    H: int
    Hq: int
    Hkv: int
    D: int
    F: int
    V: int
    qk_norm: bool
    eps: float
    theta: float


def _ptr_array(arrs: Sequence[np.ndarray]):
    t = (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return C.cast(t, _PP), t


def decode_step(shape: Shape, w: Dict[str, object], kcache: np.ndarray, vcache: np.ndarray,
                pos: Sequence[int], tokens: Sequence[int], precision: int = 64,
                nthreads: Optional[int] = None, want_hidden: bool = True):
    """One decode step for all B sequences.  ``w`` maps names to uint16 arrays:
    embed [V,H], lm_head [V,H], norm_final [H], and per-layer lists wq, wk, wv,
    wo, wg, wu, wd, norm_attn, norm_mlp (+ qnorm, knorm when qk_norm).  With
    ``w["fp8"]`` true the seven projection lists hold (e4m3 codes uint8 [N, K],
    fp32 block scales [ceil(N/128), K/128]) pairs instead.
    ``kcache``/``vcache`` are uint16 [L, B, Hkv, Smax, D], appended in place.
    Returns (logits [B,V], hidden [L,B,H] or None, argmax [B])."""
    L, B = shape.L, len(tokens)
    Smax = kcache.shape[3]
    assert kcache.shape == (L, B, shape.Hkv, Smax, shape.D) and kcache.dtype == np.uint16
    assert kcache.flags.c_contiguous and vcache.flags.c_contiguous
    sh = _Shape(shape.L, shape.H, shape.Hq, shape.Hkv, shape.D, shape.F, shape.V, int(shape.qk_norm),
                shape.eps, shape.theta)
    keep = []
    ws = _Weights()
    for n in ("embed", "lm_head", "norm_final"):
        a = np.ascontiguousarray(w[n])
        keep.append(a)
        setattr(ws, n, a.ctypes.data)
    fp8 = bool(w.get("fp8", False))
    ws.fp8 = int(fp8)
    for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm_attn", "norm_mlp", "qnorm", "knorm"):
        lst = w.get(n)
        if lst is None or (fp8 and n in PROJ):
            lst = [np.zeros(shape.D, np.uint16)] * L
        arrs = [np.ascontiguousarray(a) for a in lst]
        keep.append(arrs)
        p, t = _ptr_array(arrs)
        keep.append(t)
        setattr(ws, n, p)
    if fp8:
        for m, n in enumerate(PROJ):
            codes = [np.ascontiguousarray(c, np.uint8) for c, _ in w[n]]
            scales = [np.ascontiguousarray(sc, np.float32) for _, sc in w[n]]
            for c, sc in zip(codes, scales):  # whole 128-wide column blocks, one scale per 128 x 128 block
                assert c.shape[1] % 128 == 0 and sc.shape == ((c.shape[0] + 127) // 128, c.shape[1] // 128)
            keep.append((codes, scales))
            pc, tc = _ptr_array(codes)
            psc, tsc = _ptr_array(scales)
            keep.append((tc, tsc))
            ws.w8[m] = pc
            ws.s8[m] = psc
    dt = np.float64 if precision == 64 else np.float32
    logits = np.empty((B, shape.V), dt)
    hidden = np.empty((L, B, shape.H), dt) if want_hidden else None
    posa = (C.c_int * B)(*[int(p) for p in pos])
    toka = (C.c_int * B)(*[int(t) for t in tokens])
    fn = lib().orc_decode_step_f64 if precision == 64 else lib().orc_decode_step_f32
    rc = fn(C.byref(sh), C.byref(ws), _up(kcache), _up(vcache), B, Smax, posa, toka,
            nthreads or os.cpu_count() or 1, logits.ctypes.data, hidden.ctypes.data if hidden is not None else None)
    if rc != 0:
        raise RuntimeError(f"oracle decode_step failed with {rc}")
    am = np.argmax(logits.astype(np.float32), axis=1)
    return logits, hidden, am
