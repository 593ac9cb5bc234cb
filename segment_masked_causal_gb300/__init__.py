"""Packed (block-diagonal causal) attention on GB300: Python binding of libpa.

Thin ctypes marshalling over the C ABI in include/pa.h: every function here
has the same name as its C entry point, checks that the torch tensors it is
given have the layout the ABI expects, and passes their device pointers and
the current CUDA stream through. All computation happens in the CUDA kernels
of libpa.so; there is no other code path. If the library has not been built
(``python -m segment_masked_causal_gb300.build``), importing works but every
call raises ``LibraryMissing``.

Semantics (mlx-train-perf changelog, PACKED kernels; 0.5.1 README,
"Sequence packing"): token i attends token j iff j <= i and seg[i] == seg[j].
q/out/dout/dq are (B, Hq, N, D) bf16; k/v/dk/dv are (B, Hkv, N, D) bf16; lse
is (B, Hq, N) fp32; seg is (B, N) int32; D in {64, 96, 128}. The *_strided
calls take (B, H, N, D) views with any strides (last dim contiguous); N need
not be a multiple of 128 except in the single-step calls.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_NULL", 2: "PA_ERR_HEAD_DIM", 3: "PA_ERR_GQA", 4: "PA_ERR_SHAPE",
                5: "PA_ERR_ALIGN", 6: "PA_ERR_WORKSPACE", 7: "PA_ERR_ARCH", 8: "PA_ERR_CUDA", 9: "PA_ERR_DTYPE",
                10: "PA_ERR_HOST_MEMORY"}
PA_IO_BF16, PA_IO_F32 = 0, 1
EXPORTS = ["pa_workspace_bytes", "pa_fwd", "pa_bwd", "pa_fwd_causal", "pa_bwd_causal", "pa_build_tile_table",
           "pa_fwd_tiles", "pa_bwd_delta", "pa_bwd_dq", "pa_bwd_dkv", "pa_bwd_noalloc", "pa_device_status",
           "pa_selftest_wait_timeout", "pa_selftest_exp2_fma", "pa_pack_first_fit", "pa_workspace_bytes_strided", "pa_fwd_strided",
           "pa_bwd_strided", "pa_lce_workspace_bytes", "pa_lce_fwd", "pa_lce_bwd_workspace_bytes", "pa_lce_bwd",
           "pa_bwd_fused_workspace_bytes", "pa_bwd_fused", "pa_status_string"]


class LibraryMissing(RuntimeError):
    pass


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class pa_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("N", ctypes.c_int32), ("D", ctypes.c_int32), ("scale", ctypes.c_float)]


class pa_strides(ctypes.Structure):
    _fields_ = [("q_b", ctypes.c_int64), ("q_h", ctypes.c_int64), ("q_n", ctypes.c_int64),
                ("k_b", ctypes.c_int64), ("k_h", ctypes.c_int64), ("k_n", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libpa.so (ctypes), with argument types declared."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(f"{LIB_PATH} not built; run python -m segment_masked_causal_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            P, S = ctypes.c_void_p, ctypes.c_size_t
            D = ctypes.POINTER(pa_dims)
            L.pa_workspace_bytes.argtypes = [D]
            L.pa_workspace_bytes.restype = S
            L.pa_fwd.argtypes = [D, P, P, P, P, P, P, P, S, P]
            L.pa_fwd_causal.argtypes = [D, P, P, P, P, P, P, S, P]
            L.pa_bwd.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, S, P]
            L.pa_bwd_causal.argtypes = [D, P, P, P, P, P, P, P, P, P, P, S, P]
            L.pa_build_tile_table.argtypes = [D, P, P, S, P]
            L.pa_fwd_tiles.argtypes = [D, P, P, P, P, P, P, P, S, P]
            L.pa_bwd_delta.argtypes = [D, P, P, P, P, S, P]
            L.pa_bwd_dq.argtypes = [D, P, P, P, P, P, P, P, P, S, P]
            L.pa_bwd_dkv.argtypes = [D, P, P, P, P, P, P, P, P, P, S, P]
            for f in ("pa_fwd", "pa_fwd_causal", "pa_bwd", "pa_bwd_causal", "pa_build_tile_table", "pa_fwd_tiles",
                      "pa_bwd_delta", "pa_bwd_dq", "pa_bwd_dkv"):
                getattr(L, f).restype = ctypes.c_int
            L.pa_bwd_fused_workspace_bytes.argtypes = [D]
            L.pa_bwd_fused_workspace_bytes.restype = S
            L.pa_bwd_fused.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, S, P]
            L.pa_bwd_fused.restype = ctypes.c_int
            L.pa_bwd_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P, P, ctypes.POINTER(ctypes.c_uint32), P]
            L.pa_bwd_noalloc.restype = ctypes.c_int
            L.pa_selftest_wait_timeout.argtypes = [P, S, P]
            L.pa_selftest_wait_timeout.restype = ctypes.c_int
            L.pa_selftest_exp2_fma.argtypes = [P, P, ctypes.c_int64, P]
            L.pa_selftest_exp2_fma.restype = ctypes.c_int
            L.pa_device_status.argtypes = [P, P]
            L.pa_device_status.restype = ctypes.c_uint32
            ST = ctypes.POINTER(pa_strides)
            L.pa_workspace_bytes_strided.argtypes = [D]
            L.pa_workspace_bytes_strided.restype = S
            L.pa_fwd_strided.argtypes = [D, ST, ctypes.c_int32, P, P, P, P, P, P, P, S, P]
            L.pa_fwd_strided.restype = ctypes.c_int
            L.pa_bwd_strided.argtypes = [D, ST, ctypes.c_int32, P, P, P, P, P, P, P, P, P, P, P, S, P]
            L.pa_bwd_strided.restype = ctypes.c_int
            I32, U64 = ctypes.c_int32, ctypes.c_uint64
            L.pa_lce_workspace_bytes.argtypes = [I32, I32, I32]
            L.pa_lce_workspace_bytes.restype = S
            L.pa_lce_fwd.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, S, P]
            L.pa_lce_fwd.restype = ctypes.c_int
            L.pa_lce_bwd_workspace_bytes.argtypes = [I32, I32, I32]
            L.pa_lce_bwd_workspace_bytes.restype = S
            L.pa_lce_bwd.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, S, P]
            L.pa_lce_bwd.restype = ctypes.c_int
            L.pa_pack_first_fit.argtypes = [P, P, I32, P, I32, I32, I32, U64, U64, P, P, P, P, P, P, P]
            L.pa_pack_first_fit.restype = ctypes.c_int
            L.pa_status_string.argtypes = [ctypes.c_int]
            L.pa_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def make_dims(B, Hq, Hkv, N, D, scale=0.0) -> pa_dims:
    return pa_dims(int(B), int(Hq), int(Hkv), int(N), int(D), float(scale))


def _check(code: int):
    if code != PA_OK:
        raise PAError(code, lib().pa_status_string(code).decode())


def _ptr(t, dtype=None, name=""):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _dims_of(q, k, scale):
    B, Hq, N, D = q.shape
    return make_dims(B, Hq, k.shape[1], N, D, scale)


def pa_workspace_bytes(B, Hq, Hkv, N, D) -> int:
    d = make_dims(B, Hq, Hkv, N, D)
    return int(lib().pa_workspace_bytes(ctypes.byref(d)))


def pa_workspace_bytes_strided(B, Hq, Hkv, N, D) -> int:
    d = make_dims(B, Hq, Hkv, N, D)
    return int(lib().pa_workspace_bytes_strided(ctypes.byref(d)))


def workspace(q, k, device=None, strided=False):
    """A device workspace sized for q/k (caller-owned torch uint8 tensor);
    strided=True sizes it for pa_fwd_strided / pa_bwd_strided."""
    import torch
    B, Hq, N, D = q.shape
    f = pa_workspace_bytes_strided if strided else pa_workspace_bytes
    n = f(B, Hq, k.shape[1], N, D)
    if n == 0:
        raise PAError(4, "invalid dims")
    return torch.empty(n, dtype=torch.uint8, device=device or q.device)


def _ptr_rows(t, dtype, name, like=None):
    """Device pointer of a (B, H, N, D) CUDA tensor whose last dim is
    contiguous; `like` (if given) must have the same strides."""
    if not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be a 4-d CUDA tensor with a contiguous last dim")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if like is not None and tuple(t.stride()) != tuple(like.stride()):
        raise ValueError(f"{name} must have the strides of its group's first tensor")
    return t.data_ptr()


def _strides_of(q, k):
    return pa_strides(q.stride(0), q.stride(1), q.stride(2), k.stride(0), k.stride(1), k.stride(2))


def _io_dtype(q):
    import torch
    if q.dtype == torch.bfloat16:
        return q.dtype, PA_IO_BF16
    if q.dtype == torch.float32:
        return q.dtype, PA_IO_F32
    raise ValueError(f"q must be bfloat16 or float32, got {q.dtype}")


def pa_fwd_strided(q, k, v, seg, out, lse, ws, scale=0.0, stream=None):
    """pa_fwd on (B, H, N, D) views with any strides (e.g. (B, N, H, D) memory
    transposed), bf16 or fp32 (all tensors alike; fp32 is rounded to bf16 on
    the way in); seg None = plain causal. out must share q's strides."""
    import torch
    bf, io = _io_dtype(q)
    d = _dims_of(q, k, scale)
    st = _strides_of(q, k)
    _check(lib().pa_fwd_strided(ctypes.byref(d), ctypes.byref(st), io, _ptr_rows(q, bf, "q"), _ptr_rows(k, bf, "k"),
                                _ptr_rows(v, bf, "v", k), _ptr(seg, torch.int32, "seg"),
                                _ptr_rows(out, bf, "out", q), _ptr(lse, torch.float32, "lse"),
                                _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_bwd_strided(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale=0.0, stream=None):
    """pa_bwd on strided (B, H, N, D) views, bf16 or fp32 (all alike): out,
    dout and dq share q's strides; v, dk and dv share k's. seg None = plain
    causal."""
    import torch
    bf, io = _io_dtype(q)
    d = _dims_of(q, k, scale)
    st = _strides_of(q, k)
    _check(lib().pa_bwd_strided(ctypes.byref(d), ctypes.byref(st), io, _ptr_rows(q, bf, "q"), _ptr_rows(k, bf, "k"),
                                _ptr_rows(v, bf, "v", k), _ptr_rows(out, bf, "out", q),
                                _ptr_rows(dout, bf, "dout", q), _ptr(lse, torch.float32, "lse"),
                                _ptr(seg, torch.int32, "seg"), _ptr_rows(dq, bf, "dq", q), _ptr_rows(dk, bf, "dk", k),
                                _ptr_rows(dv, bf, "dv", k), _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_fwd(q, k, v, seg, out, lse, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_fwd(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                        _ptr(seg, torch.int32, "seg"), _ptr(out, bf, "out"), _ptr(lse, torch.float32, "lse"),
                        _ptr(ws, None, "ws"), ws.numel() if hasattr(ws, "numel") else 0, _stream(stream)))


def pa_fwd_causal(q, k, v, out, lse, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_fwd_causal(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                               _ptr(out, bf, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws, None, "ws"),
                               ws.numel(), _stream(stream)))


def pa_bwd(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                        _ptr(out, bf, "out"), _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"),
                        _ptr(seg, torch.int32, "seg"), _ptr(dq, bf, "dq"), _ptr(dk, bf, "dk"), _ptr(dv, bf, "dv"),
                        _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_bwd_fused_workspace_bytes(B, Hq, Hkv, N, D) -> int:
    d = make_dims(B, Hq, Hkv, N, D)
    return int(lib().pa_bwd_fused_workspace_bytes(ctypes.byref(d)))


def pa_bwd_fused(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale=0.0, stream=None):
    """The single-pass backward (seg None = plain causal); ws sized by
    pa_bwd_fused_workspace_bytes."""
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd_fused(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                              _ptr(out, bf, "out"), _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"),
                              _ptr(seg, torch.int32, "seg"), _ptr(dq, bf, "dq"), _ptr(dk, bf, "dk"),
                              _ptr(dv, bf, "dv"), _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def backward_fused(q, k, v, out, dout, lse, seg=None, scale=0.0, ws=None):
    """Allocate dq/dk/dv and run the single-pass backward (contiguous bf16,
    N % 128 == 0); dq is not bitwise reproducible from run to run."""
    import torch
    B, Hq, N, D = q.shape
    if ws is None:
        n = pa_bwd_fused_workspace_bytes(B, Hq, k.shape[1], N, D)
        if n == 0:
            raise PAError(4, "invalid dims for the single-pass backward")
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    pa_bwd_fused(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale)
    return dq, dk, dv


def pa_bwd_causal(q, k, v, out, dout, lse, dq, dk, dv, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd_causal(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                               _ptr(out, bf, "out"), _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"),
                               _ptr(dq, bf, "dq"), _ptr(dk, bf, "dk"), _ptr(dv, bf, "dv"), _ptr(ws, None, "ws"),
                               ws.numel(), _stream(stream)))


def pa_build_tile_table(q, k, seg, ws, scale=0.0, stream=None):
    import torch
    d = _dims_of(q, k, scale)
    _check(lib().pa_build_tile_table(ctypes.byref(d), _ptr(seg, torch.int32, "seg"), _ptr(ws, None, "ws"),
                                     ws.numel(), _stream(stream)))


def pa_fwd_tiles(q, k, v, seg, out, lse, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_fwd_tiles(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                              _ptr(seg, torch.int32, "seg"), _ptr(out, bf, "out"), _ptr(lse, torch.float32, "lse"),
                              _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_bwd_delta(q, k, out, dout, lse, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd_delta(ctypes.byref(d), _ptr(out, bf, "out"), _ptr(dout, bf, "dout"),
                              _ptr(lse, torch.float32, "lse"), _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_bwd_dq(q, k, v, dout, lse, seg, dq, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd_dq(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                           _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"), _ptr(seg, torch.int32, "seg"),
                           _ptr(dq, bf, "dq"), _ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_bwd_dkv(q, k, v, dout, lse, seg, dk, dv, ws, scale=0.0, stream=None):
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    _check(lib().pa_bwd_dkv(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                            _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"), _ptr(seg, torch.int32, "seg"),
                            _ptr(dk, bf, "dk"), _ptr(dv, bf, "dv"), _ptr(ws, None, "ws"), ws.numel(),
                            _stream(stream)))


def pa_bwd_noalloc(q, k, v, out, dout, lse, seg, dq, dk, dv, scale=0.0, stream=None, wait_status=False):
    """pa_bwd without a workspace, for callers that cannot allocate device
    memory (the scratch is a fixed 8 MiB array inside the library). Returns the
    device status word when wait_status is true (the call then synchronises),
    else None. Calls that overlap on the GPU share that array and race."""
    import torch
    bf = torch.bfloat16
    d = _dims_of(q, k, scale)
    st = ctypes.c_uint32(0xFFFFFFFF)
    _check(lib().pa_bwd_noalloc(ctypes.byref(d), _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                                _ptr(out, bf, "out"), _ptr(dout, bf, "dout"), _ptr(lse, torch.float32, "lse"),
                                _ptr(seg, torch.int32, "seg"), _ptr(dq, bf, "dq"), _ptr(dk, bf, "dk"),
                                _ptr(dv, bf, "dv"), ctypes.byref(st) if wait_status else None, _stream(stream)))
    return int(st.value) if wait_status else None


def pa_selftest_wait_timeout(ws, stream=None):
    """Launch the bounded-wait self-test into the workspace status word (see
    include/pa.h); read the result with pa_device_status."""
    _check(lib().pa_selftest_wait_timeout(_ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


def pa_selftest_exp2_fma(x, y, stream=None):
    """y = 2^x through the FMA-pipe exponential (see include/pa.h);
    x and y are fp32 CUDA tensors of the same number of elements."""
    import torch
    if x.numel() != y.numel():
        raise ValueError("x and y differ in size")
    _check(lib().pa_selftest_exp2_fma(_ptr(x, torch.float32, "x"), _ptr(y, torch.float32, "y"), x.numel(),
                                      _stream(stream)))


def pa_device_status(ws, stream=None) -> int:
    return int(lib().pa_device_status(_ptr(ws, None, "ws"), _stream(stream)))


def pa_pack_first_fit(lengths, rows, N, seed=0, epoch=0, offsets=None, tokens=None, pad_token=0):
    """Pack sequences into `rows` rows of N tokens (host call; see include/pa.h).

    lengths/offsets: per-sequence token counts and prompt lengths (offsets
    None = all 0); tokens: the sequences' tokens concatenated in input order,
    or None to skip the token rows. Returns a dict of numpy arrays: seg and
    loss_mask (rows, N), row_tokens and row_targets (rows, N) or None,
    placement (count,) int64 flat start index or -1, and the ints rows_used
    and placed_tokens. row_targets holds, where loss_mask is 1, the next token
    of the same sequence, and -1 elsewhere (an ignored target for
    pa_lce_fwd)."""
    import numpy as np
    lengths = np.ascontiguousarray(lengths, dtype=np.int32).reshape(-1)
    count = lengths.size
    off = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int32).reshape(-1)
    if off is not None and off.size != count:
        raise ValueError("offsets must have one entry per sequence")
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
    if tok is not None and tok.size != int(lengths.astype(np.int64).sum()):
        raise ValueError("tokens must hold sum(lengths) values")
    rows, N = int(rows), int(N)
    cells = max(rows, 0) * max(N, 0)
    seg = np.empty(cells, np.int32)
    mask = np.empty(cells, np.uint8)
    row_tokens = np.empty(cells, np.int32) if tok is not None else None
    row_targets = np.empty(cells, np.int32) if tok is not None else None
    placement = np.empty(count, np.int64)
    used, placed = ctypes.c_int32(0), ctypes.c_int64(0)

    def p(a):
        return None if a is None or a.size == 0 else a.ctypes.data

    _check(lib().pa_pack_first_fit(p(lengths), p(off), count, p(tok), int(pad_token), rows, N,
                                   int(seed) & 0xFFFFFFFFFFFFFFFF, int(epoch) & 0xFFFFFFFFFFFFFFFF,
                                   seg.ctypes.data if cells else None, p(mask), p(row_tokens), p(row_targets),
                                   p(placement),
                                   ctypes.byref(used), ctypes.byref(placed)))
    return {"seg": seg.reshape(rows, N), "loss_mask": mask.reshape(rows, N),
            "row_tokens": None if row_tokens is None else row_tokens.reshape(rows, N),
            "row_targets": None if row_targets is None else row_targets.reshape(rows, N),
            "placement": placement, "rows_used": int(used.value), "placed_tokens": int(placed.value)}


def packed_batches(lengths, B, N, seed, epoch, offsets=None, tokens=None, pad_token=0, rank=0, world=1):
    """One epoch of fixed-shape packed batches: pack every sequence with
    pa_pack_first_fit into as many rows as it needs, then yield consecutive
    groups of B rows as dicts of seg, loss_mask, row_tokens and row_targets,
    each (B, N).
    Rows of the last batch that hold no sequence are one padding segment with
    no supervised token. Sequences longer than N are left out.

    Data parallel: with world > 1, every rank packs the same epoch (same seed
    and epoch give the same rows) and takes batches rank, rank + world, ...;
    every rank gets the same number of batches, the missing ones being all
    padding (no supervised token), so ranks that step together never wait on
    one that ran out."""
    import numpy as np
    B, world, rank = int(B), int(world), int(rank)
    if not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    count = len(lengths)
    rows = max(-(-count // B), 1) * B
    r = pa_pack_first_fit(lengths, rows, N, seed, epoch, offsets, tokens, pad_token)
    keys = ("seg", "loss_mask", "row_tokens", "row_targets")
    fill = {"seg": 0, "loss_mask": 0, "row_tokens": pad_token, "row_targets": -1}
    n_batches = -(-r["rows_used"] // B)
    per_rank = -(-n_batches // world)
    for i in range(per_rank):
        b = rank + i * world
        if b < n_batches:
            sl = slice(b * B, (b + 1) * B)
            yield {k: (None if r[k] is None else r[k][sl]) for k in keys}
        else:
            yield {k: (None if r[k] is None else np.full((B, N), fill[k], dtype=r[k].dtype)) for k in keys}


def pa_lce_workspace_bytes(N, V, D) -> int:
    return int(lib().pa_lce_workspace_bytes(int(N), int(V), int(D)))


def pa_lce_fwd(hidden, head, targets, nll, lse, target_logit, ws, stream=None):
    """Fused linear cross-entropy forward (see include/pa.h): hidden (N, D)
    and head (V, D) bf16, targets (N) int32; writes nll, lse and
    target_logit, (N) fp32 each."""
    import torch
    N, D = hidden.shape
    V = head.shape[0]
    if head.shape[1] != D:
        raise ValueError("head must be (V, D) with the hidden states' D")
    f = torch.float32
    _check(lib().pa_lce_fwd(N, V, D, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(head, torch.bfloat16, "head"),
                            _ptr(targets, torch.int32, "targets"), _ptr(nll, f, "nll"), _ptr(lse, f, "lse"),
                            _ptr(target_logit, f, "target_logit"), _ptr(ws, None, "ws"), ws.numel(),
                            _stream(stream)))


def linear_cross_entropy_forward(hidden, head, targets, ws=None):
    """Allocate the outputs (and a workspace) and run pa_lce_fwd; returns
    (nll, lse, target_logit)."""
    import torch
    N, D = hidden.shape
    out = [torch.empty(N, dtype=torch.float32, device=hidden.device) for _ in range(3)]
    if ws is None:
        n = pa_lce_workspace_bytes(N, head.shape[0], D)
        if n == 0:
            raise PAError(4, "invalid linear cross-entropy dims")
        ws = torch.empty(n, dtype=torch.uint8, device=hidden.device)
    pa_lce_fwd(hidden, head, targets, *out, ws)
    return tuple(out)


def pa_lce_bwd_workspace_bytes(N, V, D) -> int:
    return int(lib().pa_lce_bwd_workspace_bytes(int(N), int(V), int(D)))


def pa_lce_bwd(hidden, head, targets, lse, g, dhidden, dhead, ws, stream=None):
    """Fused linear cross-entropy backward (see include/pa.h): writes dhidden
    (N, D) bf16 and, unless dhead is None, dhead (V, D) bf16, for the loss
    sum_i g[i] nll[i] with the forward's lse."""
    import torch
    N, D = hidden.shape
    V = head.shape[0]
    if head.shape[1] != D or tuple(dhidden.shape) != (N, D) or (dhead is not None and tuple(dhead.shape) != (V, D)):
        raise ValueError("hidden/dhidden must be (N, D) and head/dhead (V, D)")
    f, bf = torch.float32, torch.bfloat16
    _check(lib().pa_lce_bwd(N, V, D, _ptr(hidden, bf, "hidden"), _ptr(head, bf, "head"),
                            _ptr(targets, torch.int32, "targets"), _ptr(lse, f, "lse"), _ptr(g, f, "g"),
                            _ptr(dhidden, bf, "dhidden"), _ptr(dhead, bf, "dhead"), _ptr(ws, None, "ws"),
                            ws.numel(), _stream(stream)))


def linear_cross_entropy_backward(hidden, head, targets, lse, g, train_head=True, ws=None):
    """Allocate the outputs (and a workspace) and run pa_lce_bwd; returns
    (dhidden, dhead), dhead None when the head does not train."""
    import torch
    N, D = hidden.shape
    dh = torch.empty_like(hidden)
    dw = torch.empty_like(head) if train_head else None
    if ws is None:
        n = pa_lce_bwd_workspace_bytes(N, head.shape[0], D)
        if n == 0:
            raise PAError(4, "invalid linear cross-entropy dims")
        ws = torch.empty(n, dtype=torch.uint8, device=hidden.device)
    pa_lce_bwd(hidden, head, targets, lse, g, dh, dw, ws)
    return dh, dw


def pa_status_string(code: int) -> str:
    return lib().pa_status_string(code).decode()


# ---------------------------------------------------------------- conveniences
def _all_contiguous(*ts):
    return all(t.is_contiguous() for t in ts)


def forward(q, k, v, seg=None, scale=0.0, ws=None):
    """Allocate out/lse and run pa_fwd (seg given) or pa_fwd_causal (seg None);
    strided q/k/v go through pa_fwd_strided (out then takes q's strides)."""
    import torch
    B, Hq, N, D = q.shape
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if not _all_contiguous(q, k, v) or q.dtype == torch.float32:
        out = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
        ws = workspace(q, k, strided=True) if ws is None else ws
        pa_fwd_strided(q, k, v, seg, out, lse, ws, scale)
        return out, lse
    out = torch.empty_like(q)
    ws = workspace(q, k) if ws is None else ws
    if seg is None:
        pa_fwd_causal(q, k, v, out, lse, ws, scale)
    else:
        pa_fwd(q, k, v, seg, out, lse, ws, scale)
    return out, lse


def backward(q, k, v, out, dout, lse, seg=None, scale=0.0, ws=None):
    """Allocate dq/dk/dv and run pa_bwd (seg given) or pa_bwd_causal (seg None);
    strided tensors go through pa_bwd_strided (dq takes q's strides, dk/dv k's)."""
    import torch
    if not _all_contiguous(q, k, v, out, dout) or q.dtype == torch.float32:
        dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
        dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
        dv = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
        ws = workspace(q, k, strided=True) if ws is None else ws
        pa_bwd_strided(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale)
        return dq, dk, dv
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(q, k) if ws is None else ws
    if seg is None:
        pa_bwd_causal(q, k, v, out, dout, lse, dq, dk, dv, ws, scale)
    else:
        pa_bwd(q, k, v, out, dout, lse, seg, dq, dk, dv, ws, scale)
    return dq, dk, dv
