"""fp64 CPU oracle for block-diagonal-causal attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / ``--impl reference`` legs may import this package.
The product library never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
output rows); this module builds it with gcc and passes numpy arrays through
ctypes. What it computes is the plain definition of attention restricted to
visible pairs (mlx-train-perf 0.5.1 README, "Sequence packing": a token sees
another only inside the same original sequence, causally; the changelog entry
for ``flash_attention(segments=...)``: the mask comes from a per-token segment
id). See ``oracle.c`` for the formulas.

Every function is pinned by tests/test_oracle_pins.py (finite differences,
library SDPA, the two invariants, closed forms, a hand-worked fixture).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
                ("N", ctypes.c_int64), ("D", ctypes.c_int64), ("scale", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            lib.orc_fwd_rows.argtypes = [ctypes.POINTER(_Dims), P, P, P, P, P, ctypes.c_int64, P, P, P, P]
            lib.orc_dq_rows.argtypes = [ctypes.POINTER(_Dims), P, P, P, P, P, P, P, ctypes.c_int64, P, P]
            lib.orc_dkv_rows.argtypes = [ctypes.POINTER(_Dims), P, P, P, P, P, P, P, ctypes.c_int64, P, P, P]
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(q, k, v, seg, scale):
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, D) or v.shape != k.shape or Hq % Hkv:
        raise ValueError("bad shapes")
    if seg is not None:
        seg = np.ascontiguousarray(seg, dtype=np.int32)
        if seg.shape != (B, N):
            raise ValueError("seg must be (B, N)")
    dims = _Dims(B, Hq, Hkv, N, D, float(scale))
    return q, k, v, seg, dims


def forward(q, k, v, seg, scale, dout=None, rows=None):
    """o, lse (and D = rowsum(dO * o) when dout is given).

    q (B,Hq,N,D), k/v (B,Hkv,N,D), seg (B,N) int32 or None (plain causal).
    rows: optional flat query-row indices into (B,Hq,N); then the outputs are
    (len(rows), D) and (len(rows),) instead of full tensors.
    """
    q, k, v, seg, dims = _prep(q, k, v, seg, scale)
    B, Hq, N, D = q.shape
    dout = None if dout is None else _f64(dout)
    full = rows is None
    rows = np.arange(B * Hq * N, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    n = len(rows)
    out = np.empty((n, D)); lse = np.empty(n); delta = np.empty(n) if dout is not None else None
    _load().orc_fwd_rows(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(seg), _ptr(dout),
                         n, _ptr(rows), _ptr(out), _ptr(lse), _ptr(delta))
    if full:
        out = out.reshape(B, Hq, N, D); lse = lse.reshape(B, Hq, N)
        delta = None if delta is None else delta.reshape(B, Hq, N)
    return out, lse, delta


def dq(q, k, v, seg, scale, dout, lse, delta, rows=None):
    """dq for all query rows, or for flat query-row indices `rows`.
    lse and delta are full (B,Hq,N) arrays (only the entries used are read)."""
    q, k, v, seg, dims = _prep(q, k, v, seg, scale)
    B, Hq, N, D = q.shape
    dout, lse, delta = _f64(dout), _f64(lse), _f64(delta)
    full = rows is None
    rows = np.arange(B * Hq * N, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), D))
    _load().orc_dq_rows(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(seg), _ptr(dout),
                        _ptr(lse), _ptr(delta), len(rows), _ptr(rows), _ptr(out))
    return out.reshape(B, Hq, N, D) if full else out


def dkv(q, k, v, seg, scale, dout, lse, delta, rows=None):
    """dk, dv for all key rows, or for flat key-row indices `rows` into (B,Hkv,N)."""
    q, k, v, seg, dims = _prep(q, k, v, seg, scale)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    dout, lse, delta = _f64(dout), _f64(lse), _f64(delta)
    full = rows is None
    rows = np.arange(B * Hkv * N, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
    dk_ = np.empty((len(rows), D)); dv_ = np.empty((len(rows), D))
    _load().orc_dkv_rows(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(seg), _ptr(dout),
                         _ptr(lse), _ptr(delta), len(rows), _ptr(rows), _ptr(dk_), _ptr(dv_))
    if full:
        return dk_.reshape(B, Hkv, N, D), dv_.reshape(B, Hkv, N, D)
    return dk_, dv_


def attention(q, k, v, seg, scale, dout):
    """Full forward + backward: returns dict o, lse, delta, dq, dk, dv."""
    o, lse, delta = forward(q, k, v, seg, scale, dout)
    dq_ = dq(q, k, v, seg, scale, dout, lse, delta)
    dk_, dv_ = dkv(q, k, v, seg, scale, dout, lse, delta)
    return {"o": o, "lse": lse, "delta": delta, "dq": dq_, "dk": dk_, "dv": dv_}
