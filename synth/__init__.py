"""Seeded synthetic inputs for packed block-diagonal-causal attention.

This module is the only code shared by the CUDA path's tests/bench and the
oracle. It holds no attention arithmetic: it draws numbers and lays out
segment ids, nothing else.

Random numbers
--------------
A counter-based generator: element ``n`` of stream ``s`` under seed ``seed`` is
``splitmix64(key(seed, s) + (n + 1) * 0x9E3779B97F4A7C15)``, where
``splitmix64`` is the published finaliser of Steele, Lea and Flood (2014,
"Fast splittable pseudorandom number generators"): xor-shift 30, multiply
0xBF58476D1CE4E5B9, xor-shift 27, multiply 0x94D049BB133111EB, xor-shift 31.
Uniforms in (0, 1] take the top 53 bits plus one ulp; normals use the
Box-Muller transform on consecutive uniform pairs.

Tensors are drawn as N(0, 1) in fp64, narrowed to fp32, then rounded to bf16
with round-to-nearest-even; the same bf16 bit patterns feed the GPU and (widened
to fp64) the oracle.

Segment layouts follow the workloads on the pages (mlx-train-perf 0.5.1
README, "Sequence packing": packed rows of 4,096 tokens holding ~40-50
Alpaca-length sequences with median ~84 tokens; and the same page's
"Training packed" description of a seeded shuffle followed by first-fit
placement into fixed rows).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    base = np.array([(seed * 1_000_003 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(base)[0]


def uint64s(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n raw 64-bit draws of stream `stream`, starting at counter `offset`."""
    ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_key(seed, stream) + ctr * _GOLDEN)


def uniforms(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniforms in (0, 1] (fp64)."""
    u = uint64s(seed, stream, n, offset) >> np.uint64(11)
    return (u.astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normals(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (fp64) by Box-Muller on uniform pairs."""
    m = (n + 1) // 2
    u = uniforms(seed, stream, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = (2.0 * math.pi) * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def bf16_normal(seed: int, stream: int, shape) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws with the given shape."""
    n = int(np.prod(shape))
    return f32_to_bf16_bits(normals(seed, stream, n).astype(np.float32)).reshape(shape)


# --------------------------------------------------------------------------
# segment layouts (per-token int32 ids; ids are consecutive runs per row)
# --------------------------------------------------------------------------

def lengths_to_ids(lengths) -> np.ndarray:
    return np.repeat(np.arange(len(lengths), dtype=np.int32), np.asarray(lengths, dtype=np.int64))


def one_segment(B: int, N: int) -> np.ndarray:
    return np.zeros((B, N), dtype=np.int32)


def cut_points_3(seed: int, N: int) -> list[int]:
    """Three segments: two distinct sorted cut points uniform in [1, N-1]."""
    k = 0
    cuts: list[int] = []
    while len(cuts) < 2:
        c = 1 + int(uint64s(seed, 7, 1, offset=k)[0] % np.uint64(N - 1))
        k += 1
        if c not in cuts:
            cuts.append(c)
    a, b = sorted(cuts)
    return [a, b - a, N - b]


def uniform_lengths(seed: int, N: int, lo: int, hi: int, stream: int = 8) -> list[int]:
    """Lengths uniform in [lo, hi] until the row is full; the last is the remainder."""
    out: list[int] = []
    total, k = 0, 0
    while total < N:
        L = lo + int(uint64s(seed, stream, 1, offset=k)[0] % np.uint64(hi - lo + 1))
        k += 1
        L = min(L, N - total)
        out.append(L)
        total += L
    return out


def lognormal_pool(seed: int, need_tokens: int, median: float = 84.0, sigma: float = 0.8,
                   lo: int = 8, hi: int = 1024) -> list[int]:
    """Lengths round(exp(ln median + sigma z)) clipped to [lo, hi], drawn until
    their sum reaches need_tokens."""
    out: list[int] = []
    total, chunk, k = 0, 256, 0
    while total < need_tokens:
        z = normals(seed, 9 + k, chunk)
        k += 1
        for zz in z:
            L = int(round(math.exp(math.log(median) + sigma * zz)))
            L = max(lo, min(hi, L))
            out.append(L)
            total += L
            if total >= need_tokens:
                break
    return out


def shuffle(seed: int, items: list, stream: int = 5) -> list:
    """Fisher-Yates with the counter-based generator."""
    a = list(items)
    r = uint64s(seed, stream, max(len(a), 1))
    for i in range(len(a) - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        a[i], a[j] = a[j], a[i]
    return a


def first_fit(lengths: list[int], B: int, N: int) -> list[list[int]]:
    """First-fit placement into B rows of capacity N; items that fit no row are dropped."""
    rows: list[list[int]] = [[] for _ in range(B)]
    free = [N] * B
    for L in lengths:
        for r in range(B):
            if L <= free[r]:
                rows[r].append(L)
                free[r] -= L
                break
    return rows


def packed_rows(seed: int, B: int, N: int):
    """Lognormal lengths, seeded shuffle, first-fit into B rows; each row's
    unfilled tail becomes one extra (padding) segment. Returns ids (B, N), the
    per-row length lists (padding last when present) and per-row padding counts."""
    pool = lognormal_pool(seed, int(math.ceil(1.1 * B * N)))
    rows = first_fit(shuffle(seed, pool), B, N)
    ids = np.empty((B, N), dtype=np.int32)
    lens_out, pads = [], []
    for r, lens in enumerate(rows):
        pad = N - sum(lens)
        full = lens + ([pad] if pad > 0 else [])
        lens_out.append(full)
        pads.append(pad)
        ids[r] = lengths_to_ids(full)
    return ids, lens_out, pads


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    seed: int
    seg: np.ndarray                                   # (B, N) int32
    lengths: list = field(default_factory=list)      # per row list of segment lengths
    pad: list = field(default_factory=list)          # per row padding tokens (0: none); the
                                                     # padding, when present, is the last segment

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def tensors(self, with_dout: bool = True) -> dict:
        """bf16 bit patterns (uint16) for q, k, v (and dO)."""
        s = self.seed
        out = {
            "q": bf16_normal(s, 1, (self.B, self.Hq, self.N, self.D)),
            "k": bf16_normal(s, 2, (self.B, self.Hkv, self.N, self.D)),
            "v": bf16_normal(s, 3, (self.B, self.Hkv, self.N, self.D)),
        }
        if with_dout:
            out["do"] = bf16_normal(s, 4, (self.B, self.Hq, self.N, self.D))
        return out


def _seg_lengths(seg_row: np.ndarray) -> list[int]:
    change = np.flatnonzero(np.diff(seg_row)) + 1
    bounds = np.concatenate([[0], change, [len(seg_row)]])
    return [int(x) for x in np.diff(bounds)]


def workload(name: str) -> Workload:
    """Named workloads with their seeds (seed = 1000 + workload index)."""
    if name == "tiny_3seg":
        seed = 1001
        lens = cut_points_3(seed, 256)
        return Workload(name, 1, 2, 2, 256, 64, seed, lengths_to_ids(lens)[None, :], [lens])
    if name == "tiny_fixed_1_100_155":
        lens = [1, 100, 155]
        return Workload(name, 1, 2, 2, 256, 64, 1001, lengths_to_ids(lens)[None, :], [lens])
    if name == "causal_2k_gqa":
        return Workload(name, 1, 32, 8, 2048, 128, 1002, one_segment(1, 2048), [[2048]])
    if name == "packed_4x4096_short":
        ids, lens, pad = packed_rows(1003, 4, 4096)
        return Workload(name, 4, 32, 8, 4096, 128, 1003, ids, lens, pad)
    if name == "8k_one_segment":
        return Workload(name, 1, 32, 8, 8192, 128, 1004, one_segment(1, 8192), [[8192]])
    if name == "8k_packed":
        lens = uniform_lengths(1004, 8192, 256, 2048)
        return Workload(name, 1, 32, 8, 8192, 128, 1004, lengths_to_ids(lens)[None, :], [lens])
    if name == "8k_one_segment_d96":
        return Workload(name, 1, 32, 8, 8192, 96, 1006, one_segment(1, 8192), [[8192]])
    if name == "packed_2x4096_short_d96":
        ids, lens, pad = packed_rows(1007, 2, 4096)
        return Workload(name, 2, 16, 4, 4096, 96, 1007, ids, lens, pad)
    for n in (32768, 65536):
        if name == f"long_{n // 1024}k_one_segment":
            return Workload(name, 1, 8, 8, n, 64, 1005, one_segment(1, n), [[n]])
        if name == f"long_{n // 1024}k_packed":
            lens = uniform_lengths(1005, n, 512, 8192)
            return Workload(name, 1, 8, 8, n, 64, 1005, lengths_to_ids(lens)[None, :], [lens])
    raise KeyError(name)


WORKLOADS = [
    "tiny_3seg", "tiny_fixed_1_100_155", "causal_2k_gqa", "packed_4x4096_short",
    "8k_one_segment", "8k_packed",
    "long_32k_one_segment", "long_32k_packed", "long_64k_one_segment", "long_64k_packed",
    "8k_one_segment_d96", "packed_2x4096_short_d96",
]


def custom(B, Hq, Hkv, N, D, lengths_per_row, seed=7) -> Workload:
    """A small workload with explicit segment lengths per row (tests)."""
    ids = np.stack([lengths_to_ids(l) for l in lengths_per_row]).astype(np.int32)
    assert ids.shape == (B, N)
    return Workload(f"custom_{B}x{N}", B, Hq, Hkv, N, D, seed, ids, [list(l) for l in lengths_per_row])

