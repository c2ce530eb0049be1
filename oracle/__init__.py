"""fp64 CPU oracle of the routed MXFP4 MoE layer — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The product path (the CUDA library and
its binding) never imports it.

This module is argument marshalling over ``oracle.c`` (plain fp64 loops); see
that file for the definition it computes and the passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = os.path.join(_HERE, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None


def build_command(out=_LIBNAME):
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
            os.path.join(_HERE, "oracle.c"), "-o", out, "-lm"]


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIBNAME) and os.path.getmtime(_LIBNAME) >= os.path.getmtime(src):
        return _LIBNAME
    tmp = _LIBNAME + f".tmp{os.getpid()}"
    subprocess.run(build_command(tmp), check=True)
    os.replace(tmp, _LIBNAME)
    return _LIBNAME


class _Expert(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            L = ctypes.CDLL(_LIBNAME)
            i32, i64, vp, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            L.orc_e2m1.restype = dbl
            L.orc_e2m1.argtypes = [i32]
            L.orc_e8m0.restype = dbl
            L.orc_e8m0.argtypes = [i32]
            L.orc_mx_at.restype = dbl
            L.orc_mx_at.argtypes = [vp, vp, i64, i64, i64]
            L.orc_dequant.argtypes = [vp, vp, i64, i64, vp]
            L.orc_router_logits.argtypes = [i32, i32, i32, vp, i32, vp, vp, i32, vp]
            L.orc_topk.argtypes = [i32, i32, i32, vp, vp, vp, vp]
            L.orc_bucket.argtypes = [i32, i32, i32, vp, vp, vp]
            L.orc_expert_mlp.argtypes = [i32, i32, vp, ctypes.POINTER(_Expert), vp]
            L.orc_dense_mlp_bf16.argtypes = [i32, i32, vp, vp, vp, vp, vp]
            L.orc_moe_tokens.argtypes = [i32, i32, i32, i32, i32, vp, i32, vp, vp, ctypes.POINTER(_Expert),
                                         vp, vp, vp, vp, i32, vp, i32, vp, vp, vp]
            L.orc_default_threads.restype = i32
            _LIB = L
    return _LIB


def default_threads() -> int:
    return int(lib().orc_default_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc}")


def e2m1(code: int) -> float:
    return float(lib().orc_e2m1(code))


def e8m0(e: int) -> float:
    return float(lib().orc_e8m0(e))


def dequant(q: np.ndarray, s: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    _check(lib().orc_dequant(q.ctypes.data, s.ctypes.data, rows, cols, out.ctypes.data), "orc_dequant")
    return out


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:
        return 1
    raise TypeError("activations must be float32 or uint16 (bf16 bits)")


def router_logits(x, wr, br=None, nthreads=None):
    x = np.ascontiguousarray(x)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    T, H = x.shape
    E = wr.shape[0]
    br = None if br is None else np.ascontiguousarray(br, dtype=np.float32)
    s = np.empty((T, E), dtype=np.float64)
    _check(lib().orc_router_logits(T, H, E, x.ctypes.data, _dtype_code(x), wr.ctypes.data, _ptr(br),
                                   nthreads or default_threads(), s.ctypes.data), "orc_router_logits")
    return s


def topk(s, k):
    s = np.ascontiguousarray(s, dtype=np.float64)
    T, E = s.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    _check(lib().orc_topk(T, E, k, s.ctypes.data, ids.ctypes.data, w.ctypes.data, margin.ctypes.data), "orc_topk")
    return ids, w, margin


def bucket(ids, E):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    sorted_idx = np.empty(T * k, dtype=np.int32)
    _check(lib().orc_bucket(T, E, k, ids.ctypes.data, offsets.ctypes.data, sorted_idx.ctypes.data), "orc_bucket")
    return offsets, sorted_idx


def _expert_struct(ex: dict) -> _Expert:
    st = _Expert()
    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        a = ex[n]
        assert a.dtype == np.uint8 and a.flags.c_contiguous
        setattr(st, n, a.ctypes.data)
    return st


def expert_mlp(H, I, x, ex: dict):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    st = _expert_struct(ex)
    _check(lib().orc_expert_mlp(H, I, x.ctypes.data, ctypes.byref(st), y.ctypes.data), "orc_expert_mlp")
    return y


def dense_mlp_bf16(H, I, x, wg, wu, wd):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    wg, wu, wd = (np.ascontiguousarray(a, dtype=np.uint16) for a in (wg, wu, wd))
    _check(lib().orc_dense_mlp_bf16(H, I, x.ctypes.data, wg.ctypes.data, wu.ctypes.data, wd.ctypes.data,
                                    y.ctypes.data), "orc_dense_mlp_bf16")
    return y


def moe_tokens(x, wr, br, experts, E, I, k, tokens, shared=None, residual=None, nthreads=None):
    """The layer for the listed tokens.  ``experts`` maps expert id -> dict of
    the six host arrays (only the experts the oracle's own routing selects are
    read; a missing one raises).  Returns (out [n][H] fp64, ids, w)."""
    x = np.ascontiguousarray(x)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    T, H = x.shape
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.size
    br = None if br is None else np.ascontiguousarray(br, dtype=np.float32)
    # Route first (oracle's own routing) so that only the selected experts are
    # materialised on the host.
    s = router_logits(x[tokens], wr, br, nthreads)
    ids, _, _ = topk(s, k)
    table = (_Expert * E)()
    keep = []
    for e in sorted(set(int(v) for v in ids.ravel())):
        ex = experts(e) if callable(experts) else experts[e]
        keep.append(ex)
        table[e] = _expert_struct(ex)
    sg = su = sd = None
    if shared is not None:
        sg, su, sd = (np.ascontiguousarray(a, dtype=np.uint16) for a in shared)
    residual = None if residual is None else np.ascontiguousarray(residual, dtype=np.float32)
    out = np.empty((n, H), dtype=np.float64)
    ids2 = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    _check(lib().orc_moe_tokens(T, H, E, I, k, x.ctypes.data, _dtype_code(x), wr.ctypes.data, _ptr(br), table,
                                _ptr(sg), _ptr(su), _ptr(sd), _ptr(residual), n, tokens.ctypes.data,
                                nthreads or default_threads(), out.ctypes.data, ids2.ctypes.data, w.ctypes.data),
           "orc_moe_tokens")
    del keep
    return out, ids2, w
