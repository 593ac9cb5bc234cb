"""The prologue's integer outputs, bit for bit: the segment-range tile table
and the two work lists, read back from the workspace and compared with a
plain CPU computation of the same definitions.

Table entry of tile t of row b (128 tokens): smallest and largest segment id
in the tile; the first key tile u <= t whose id range overlaps tile t's; the
last query tile u >= t whose id range overlaps. A (query tile, key tile) pair
is visited only when the ranges overlap (changelog entry adding the PACKED
kernels: cross-segment blocks are skipped), and a key tile's query walk ends
at the last overlapping query tile (mlx-train-perf 0.5.1 README, "Sequence
packing", the 0.5.0 dK/dV change). A table that visited too many tiles would
still pass every parity test and only cost time; this test catches it.

Work lists: entries b*T + t ordered by decreasing walk bound (t - kv_lo + 1
for the query tiles of the forward and dQ kernels, q_hi - t + 1 for the key
tiles of dK/dV); equal bounds keep the canonical order (query tiles from the
last down, key tiles from the first up, batch rows increasing).

The workspace layout read here is the one include/pa.h documents: status
word at byte 0, the (B, T) int4 table at byte 256, then the two lists, each
region on a 256-byte boundary.
"""
import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


def _round256(x: int) -> int:
    return (x + 255) // 256 * 256


def expected_table(seg: np.ndarray) -> np.ndarray:
    B, N = seg.shape
    T = N // 128
    out = np.zeros((B, T, 4), np.int64)
    for b in range(B):
        s = seg[b].reshape(T, 128).astype(np.int64)
        lo, hi = s.min(1), s.max(1)
        for t in range(T):
            over = [(lo[u] <= hi[t]) and (lo[t] <= hi[u]) for u in range(T)]
            first = next(u for u in range(t + 1) if over[u])
            last = next(u for u in range(T - 1, t - 1, -1) if over[u])
            out[b, t] = (lo[t], hi[t], first, last)
    return out


def expected_lists(table: np.ndarray):
    B, T, _ = table.shape
    canon_q = [b * T + (T - 1 - e // B) for e in range(B * T) for b in [e % B]]
    canon_k = [b * T + e // B for e in range(B * T) for b in [e % B]]
    cost_q = lambda ent: ent % T - table[ent // T, ent % T, 2] + 1
    cost_k = lambda ent: table[ent // T, ent % T, 3] - ent % T + 1
    # Python's sort is stable: equal costs keep the canonical order
    wq = sorted(canon_q, key=lambda ent: -cost_q(ent))
    wk = sorted(canon_k, key=lambda ent: -cost_k(ent))
    return np.array(wq, np.int64), np.array(wk, np.int64)


def read_back(ws: torch.Tensor, B: int, T: int):
    raw = ws.cpu().numpy()
    off_t = 256
    off_q = off_t + _round256(B * T * 16)
    off_k = off_q + _round256(B * T * 4)
    table = raw[off_t:off_t + B * T * 16].view(np.int32).reshape(B, T, 4).astype(np.int64)
    wq = raw[off_q:off_q + B * T * 4].view(np.int32).astype(np.int64)
    wk = raw[off_k:off_k + B * T * 4].view(np.int32).astype(np.int64)
    return table, wq, wk


def _alternating():
    w = synth.custom(2, 4, 2, 1024, 128, [[1024], [1024]], seed=28)
    w.seg[0] = np.array([(i // 128) % 2 for i in range(1024)], np.int32)
    w.seg[1] = np.array([7 + (i // 96) % 2 for i in range(1024)], np.int32)
    return w


def _noncontig():
    w = synth.custom(1, 2, 2, 512, 128, [[100, 100, 100, 212]], seed=26)
    w.seg[0] = np.array([5] * 100 + [9] * 100 + [5] * 100 + [-3] * 212, np.int32)
    return w


def _many_rows():
    """40 rows of 16,384 tokens (5,120 tiles): more tiles than one CTA of the
    prologue takes, so the table and the lists come from the multi-CTA path."""
    lengths = []
    for b in range(40):
        u = synth.uniforms(31 + b, 1, 64)
        row, left = [], 16384
        for x in u:
            L = min(left, 100 + int(x * 3000))
            row.append(L)
            left -= L
            if left == 0:
                break
        if left:
            row.append(left)
        lengths.append(row)
    return synth.custom(40, 1, 1, 16384, 64, lengths, seed=33)


CASES = {
    "packed_4x4096_short": lambda: synth.workload("packed_4x4096_short"),
    "8k_packed": lambda: synth.workload("8k_packed"),
    "8k_one_segment": lambda: synth.workload("8k_one_segment"),
    "long_64k_packed": lambda: synth.workload("long_64k_packed"),
    "noncontiguous_ids": _noncontig,
    "alternating_blocks": _alternating,
    "many_rows_multi_cta": _many_rows,
}


@pytest.mark.parametrize("name", list(CASES))
def test_table_and_work_lists_exact(name, cuda_dev):
    w = CASES[name]()
    q = torch.zeros((w.B, w.Hq, w.N, w.D), dtype=torch.bfloat16, device=cuda_dev)
    k = torch.zeros((w.B, w.Hkv, w.N, w.D), dtype=torch.bfloat16, device=cuda_dev)
    seg = torch.from_numpy(w.seg).to(cuda_dev)
    ws = pa.workspace(q, k)
    ws.fill_(0xA5)  # whatever the prologue does not write stays visible
    pa.pa_build_tile_table(q, k, seg, ws)
    torch.cuda.synchronize()
    T = w.N // 128
    table, wq, wk = read_back(ws, w.B, T)
    exp = expected_table(w.seg)
    np.testing.assert_array_equal(table, exp)
    eq, ek = expected_lists(exp)
    np.testing.assert_array_equal(wq, eq)
    np.testing.assert_array_equal(wk, ek)
    assert pa.pa_device_status(ws) == 0


def test_one_segment_lists_are_the_causal_order(cuda_dev):
    """With every token in one segment the lists are the longest-causal-walk
    order: query tiles from the last down, key tiles from the first up."""
    B, T = 2, 16
    q = torch.zeros((B, 2, T * 128, 64), dtype=torch.bfloat16, device=cuda_dev)
    ws = pa.workspace(q, q)
    pa.pa_build_tile_table(q, q, None, ws)
    torch.cuda.synchronize()
    _, wq, wk = read_back(ws, B, T)
    np.testing.assert_array_equal(wq, [b * T + t for t in range(T - 1, -1, -1) for b in range(B)])
    np.testing.assert_array_equal(wk, [b * T + t for t in range(T) for b in range(B)])


def test_ragged_n_padded_table(cuda_dev):
    """N = 300 runs on whole tiles: the kernels see 3 tiles whose
    tail tokens repeat the row's last id, and the table describes that
    padded row."""
    w = synth.custom(2, 4, 2, 300, 128, [[150, 150], [1, 298, 1]], seed=32)
    q = torch.zeros((w.B, w.Hq, w.N, w.D), dtype=torch.bfloat16, device=cuda_dev)
    k = torch.zeros((w.B, w.Hkv, w.N, w.D), dtype=torch.bfloat16, device=cuda_dev)
    seg = torch.from_numpy(w.seg).to(cuda_dev)
    ws = pa.workspace(q, k)
    pa.forward(q, k, k, seg, ws=ws)
    torch.cuda.synchronize()
    Np = 384
    padded = np.concatenate([w.seg, np.repeat(w.seg[:, -1:], Np - w.N, axis=1)], axis=1)
    table, wq, wk = read_back(ws, w.B, Np // 128)
    exp = expected_table(padded)
    np.testing.assert_array_equal(table, exp)
    eq, ek = expected_lists(exp)
    np.testing.assert_array_equal(wq, eq)
    np.testing.assert_array_equal(wk, ek)
