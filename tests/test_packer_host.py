"""The host packer: the oracle's restatement pinned to published values, hand
work and properties, then the library's pa_pack_first_fit compared with it
element by element (no GPU needed).

Packed batch iterator: mlx-train-perf changelog, "Added" (seeded per-epoch
shuffle, first-fit placement into fixed rows, per-token segment buffers);
loss masking per segment with the supervised set of an unpacked run:
mlx-train-perf 0.5.1 README, "Sequence packing".
"""
import ctypes
import itertools
import json
import math
import os

import numpy as np
import pytest

import segment_masked_causal_gb300 as pa
import synth
from oracle import packing as opk
from segment_masked_causal_gb300 import build as pabuild

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def L():
    pabuild.build()
    return pa.lib()


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ oracle pins
def test_generator_matches_published_splitmix64_outputs():
    """The stream the shuffle draws from is splitmix64: with the key forced to
    a state x, draw n is the (n+1)-th output from state x."""
    g = golden("splitmix64_vectors.json")
    gamma = int(g["gamma"], 16)

    def outputs(state, n):
        ctr = (state + gamma * np.arange(1, n + 1, dtype=object)) % (1 << 64)
        return [int(v) for v in synth._mix(np.array([int(c) for c in ctr], dtype=np.uint64))]

    assert outputs(0, 1)[0] == int(g["state_0_first"], 16)
    assert outputs(1234567, 5) == [int(s) for s in g["state_1234567_first5"]]


def _perm_counts(order_of, trials=6000):
    counts = {}
    for s in range(trials):
        p = tuple(order_of(s))
        counts[p] = counts.get(p, 0) + 1
    return counts


def _assert_uniform(counts, trials=6000):
    """All 3! orders appear, each within 5 standard deviations of trials/6
    (a Sattolo-style off-by-one gives only the 2 cyclic orders)."""
    assert sorted(counts) == sorted(itertools.permutations(range(3))), counts
    mean = trials / 6
    sd = math.sqrt(trials * (1 / 6) * (5 / 6))
    for p, c in counts.items():
        assert abs(c - mean) < 5 * sd, (p, c)


def test_oracle_shuffle_is_uniform_over_permutations():
    _assert_uniform(_perm_counts(lambda s: opk.shuffled_order(3, s, 0)))


def test_oracle_first_fit_hand_worked():
    g = golden("first_fit_hand_worked.json")
    for ex in (g, g["second"]):
        spots = opk.first_fit(ex["lengths"], rows=len(ex["lengths"]), N=g["capacity"])
        assert [list(s) for s in spots] == ex["row_start"]


def test_oracle_supervision_hand_worked():
    for case in golden("first_fit_hand_worked.json")["supervision"]:
        assert [int(b) for b in opk.supervised(case["L"], case["offset"])] == case["mask"], case["why"]


def _random_dataset(rng, count, lo, hi, N):
    lengths = [int(x) for x in rng.integers(lo, hi + 1, size=count)]
    offsets = [int(rng.integers(0, x + 2)) for x in lengths]
    return lengths, offsets


def _check_pack_properties(res, lengths, offsets, rows, N):
    """Properties any correct first-fit pack has, whatever the order."""
    seg = np.asarray(res["seg"])
    mask = np.asarray(res["loss_mask"])
    fill = np.zeros(rows, np.int64)
    for s, at in enumerate(res["placement"]):
        Ls = lengths[s]
        if at < 0:
            continue
        r, start = divmod(int(at), N)
        assert start + Ls <= N
        run = seg[r, start:start + Ls]
        assert (run == run[0]).all()
        # the sequence is a segment of its own
        assert (seg[r] == run[0]).sum() == Ls
        # supervised count in closed form; no supervised position predicts a
        # token of another segment or of the padding
        assert mask[r, start:start + Ls].sum() == max(0, Ls - max(offsets[s], 1))
        fill[r] += Ls
    assert int(fill.sum()) == res["placed_tokens"]
    # a sequence that was left out fits no row even at the end
    free = N - fill
    for s, at in enumerate(res["placement"]):
        if at < 0:
            assert lengths[s] > free.max()
    # first fit never leaves two rows both at most half full
    used = fill[fill > 0]
    assert (2 * used <= N).sum() <= 1
    # used rows are a prefix
    assert res["rows_used"] == int((fill > 0).sum())
    assert (fill[:res["rows_used"]] > 0).all()
    # every supervised position's next token is in its own segment
    r_idx, t_idx = np.nonzero(mask)
    assert (t_idx + 1 < N).all()
    assert (seg[r_idx, t_idx + 1] == seg[r_idx, t_idx]).all()
    # the padding (the last id of a partly filled row) is never supervised
    for r in range(rows):
        if fill[r] < N:
            pad = seg[r, N - 1]
            assert (seg[r, fill[r]:] == pad).all() and mask[r, fill[r]:].sum() == 0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_pack_properties(seed):
    rng = np.random.default_rng(seed)
    lengths, offsets = _random_dataset(rng, 60, 1, 300, 512)
    res = opk.pack(lengths, 8, 512, seed, 3, offsets)
    _check_pack_properties(res, lengths, offsets, 8, 512)


def test_oracle_pack_supervised_pairs_equal_unpacked():
    """The (input token, target token) pairs the loss sees in the packed rows
    are those of each sequence run alone under the unpacked rule."""
    rng = np.random.default_rng(5)
    lengths, offsets = _random_dataset(rng, 30, 1, 90, 256)
    tokens = [int(t) for t in rng.integers(0, 50000, size=sum(lengths))]
    res = opk.pack(lengths, 6, 256, 11, 0, offsets, tokens, pad_token=-7)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    packed_pairs, alone_pairs = [], []
    rt, m = np.asarray(res["row_tokens"]), np.asarray(res["loss_mask"])
    for r, t in zip(*np.nonzero(m)):
        packed_pairs.append((int(rt[r, t]), int(rt[r, t + 1])))
    for s, at in enumerate(res["placement"]):
        if at < 0:
            continue
        seq = tokens[starts[s]:starts[s] + lengths[s]]
        for p in range(lengths[s] - 1):
            if p + 1 >= offsets[s]:
                alone_pairs.append((seq[p], seq[p + 1]))
    assert sorted(packed_pairs) == sorted(alone_pairs)
    tg = np.asarray(res["row_targets"])
    target_pairs = [(int(rt[r, t]), int(tg[r, t])) for r, t in zip(*np.nonzero(tg >= 0))]
    assert sorted(target_pairs) == sorted(alone_pairs)
    assert ((tg >= 0) == (m == 1)).all()


# ------------------------------------------------------- library vs oracle
def _lib_pack(lengths, rows, N, seed, epoch, offsets=None, tokens=None, pad_token=0):
    return pa.pa_pack_first_fit(lengths, rows, N, seed, epoch, offsets, tokens, pad_token)


def _assert_same(lib_res, orc_res):
    for k in ("seg", "loss_mask", "row_tokens", "row_targets"):
        if orc_res[k] is None:
            assert lib_res[k] is None
            continue
        np.testing.assert_array_equal(lib_res[k], np.asarray(orc_res[k], dtype=lib_res[k].dtype), err_msg=k)
    np.testing.assert_array_equal(lib_res["placement"], np.asarray(orc_res["placement"], np.int64))
    assert lib_res["rows_used"] == orc_res["rows_used"]
    assert lib_res["placed_tokens"] == orc_res["placed_tokens"]


CASES = [
    # name, count, lo, hi, rows, N, seed, epoch
    ("alpaca_like", 120, 8, 400, 4, 1024, 42, 0),
    ("alpaca_like_epoch1", 120, 8, 400, 4, 1024, 42, 1),
    ("some_too_long", 40, 1, 700, 3, 512, 7, 2),
    ("exact_fits", 12, 256, 256, 3, 1024, 3, 0),
    ("all_ones", 300, 1, 1, 2, 128, 9, 4),
    ("one_row", 50, 5, 60, 1, 640, 13, 0),
    ("many_rows_ragged_N", 200, 3, 90, 64, 300, 17, 5),
    ("rows_exceed_need", 10, 10, 20, 16, 256, 1, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_library_matches_oracle(case, L):
    _, count, lo, hi, rows, N, seed, epoch = case
    rng = np.random.default_rng(seed + 100 * epoch)
    lengths, offsets = _random_dataset(rng, count, lo, hi, N)
    tokens = [int(t) for t in rng.integers(-5, 1 << 20, size=sum(lengths))]
    lib_res = _lib_pack(lengths, rows, N, seed, epoch, offsets, tokens, pad_token=-1)
    orc_res = opk.pack(lengths, rows, N, seed, epoch, offsets, tokens, pad_token=-1)
    _assert_same(lib_res, orc_res)
    _check_pack_properties(lib_res, lengths, offsets, rows, N)


def test_library_optional_outputs_and_defaults(L):
    lengths = [3, 9, 4, 4, 1]
    a = _lib_pack(lengths, 2, 12, 5, 0)
    b = opk.pack(lengths, 2, 12, 5, 0)
    _assert_same(a, b)  # offsets None = 0, no tokens
    assert a["row_tokens"] is None


def test_library_empty_dataset(L):
    res = _lib_pack([], 3, 128, 1, 0)
    assert res["rows_used"] == 0 and res["placed_tokens"] == 0
    assert (res["seg"] == 0).all() and res["loss_mask"].sum() == 0
    assert res["placement"].shape == (0,)


def test_library_shuffle_is_uniform_over_permutations(L):
    """Three one-token sequences in one row of three: the row holds them in
    the shuffled order, so the placements give the permutation."""
    def order_of(s):
        at = _lib_pack([1, 1, 1], 1, 3, s, 0)["placement"]
        return list(np.argsort(at))
    _assert_uniform(_perm_counts(order_of))


def test_library_reproduces_the_packed_bench_rows(L):
    """The synthetic packed rows of the attention workloads (lognormal lengths,
    shuffle on stream 5, first-fit into B rows) are exactly the library
    packer's output for epoch 5."""
    for seed, B, N in [(1003, 4, 4096), (42, 2, 8192)]:
        ids, lens, pads = synth.packed_rows(seed, B, N)
        pool = synth.lognormal_pool(seed, int(math.ceil(1.1 * B * N)))
        res = _lib_pack(pool, B, N, seed, 5)
        np.testing.assert_array_equal(res["seg"], ids)
        assert res["placed_tokens"] == B * N - sum(pads)


def test_library_epochs_reshuffle_and_are_deterministic(L):
    rng = np.random.default_rng(0)
    lengths, offsets = _random_dataset(rng, 80, 4, 200, 512)
    e0 = _lib_pack(lengths, 40, 512, 77, 0, offsets)
    e0b = _lib_pack(lengths, 40, 512, 77, 0, offsets)
    e1 = _lib_pack(lengths, 40, 512, 77, 1, offsets)
    np.testing.assert_array_equal(e0["placement"], e0b["placement"])
    assert not np.array_equal(e0["placement"], e1["placement"])
    # every sequence fits, so every epoch places all of them
    assert e0["placed_tokens"] == e1["placed_tokens"] == sum(lengths)


def test_library_large_epoch_properties(L):
    """An epoch of 200k Alpaca-length sequences into 4,096-token rows (the
    max-tree keeps first-fit at O(log rows) per sequence)."""
    lengths = synth.lognormal_pool(3, 200_000 * 90)[:200_000]
    rows = 200_000 * 1024 // 4096
    offsets = [x // 3 for x in lengths]
    res = _lib_pack(lengths, rows, 4096, 3, 0, offsets)
    assert res["placed_tokens"] == sum(lengths)
    # spot-check the properties on a sample of rows (full check is slow in Python)
    fill = np.bincount((res["placement"] // 4096).astype(np.int64), weights=np.asarray(lengths, np.float64),
                       minlength=rows)
    used = fill[fill > 0]
    assert (2 * used <= 4096).sum() <= 1
    assert res["rows_used"] == int((fill > 0).sum())
    assert int(res["loss_mask"].sum()) == sum(max(0, x - max(o, 1)) for x, o in zip(lengths, offsets))


def test_packed_batches_fixed_shapes(L):
    rng = np.random.default_rng(1)
    lengths, offsets = _random_dataset(rng, 150, 4, 600, 1024)
    tokens = list(range(sum(lengths)))
    batches = list(pa.packed_batches(lengths, 3, 1024, 9, 0, offsets, tokens, pad_token=-1))
    assert batches
    seen = 0
    for b in batches:
        assert b["seg"].shape == (3, 1024) and b["loss_mask"].shape == (3, 1024)
        assert b["row_tokens"].shape == (3, 1024)
        seen += int((b["row_tokens"] >= 0).sum())
    assert seen == sum(lengths)
    # fewer sequences than rows in a batch: one batch, the rest padding rows
    few = list(pa.packed_batches([5, 6], 4, 64, 0, 0))
    assert len(few) == 1 and few[0]["seg"].shape == (4, 64)
    assert (few[0]["seg"][1:] == 0).all() and few[0]["loss_mask"][1:].sum() == 0


# --------------------------------------------------------------- refusals
def _raw(L, lengths, count, rows, N, offsets=None, tokens=None, seg=True, row_tokens=False):
    n = max(rows, 1) * max(N, 1)
    seg_buf = np.full(n, 12345, np.int32)
    tok_buf = np.full(n, 12345, np.int32)
    la = None if lengths is None else np.asarray(lengths, np.int32)
    oa = None if offsets is None else np.asarray(offsets, np.int32)
    ta = None if tokens is None else np.asarray(tokens, np.int32)
    code = L.pa_pack_first_fit(None if la is None else la.ctypes.data, None if oa is None else oa.ctypes.data,
                               count, None if ta is None else ta.ctypes.data, 0, rows, N, 0, 0,
                               seg_buf.ctypes.data if seg else None, None,
                               tok_buf.ctypes.data if row_tokens else None, None, None, None, None)
    return code, seg_buf, tok_buf


@pytest.mark.parametrize("kw,code", [
    (dict(lengths=[3, 4], count=2, rows=1, N=8, seg=False), 1),
    (dict(lengths=None, count=2, rows=1, N=8), 1),
    (dict(lengths=[3, 4], count=2, rows=1, N=8, row_tokens=True), 1),
    (dict(lengths=[3, 4], count=-1, rows=1, N=8), 4),
    (dict(lengths=[3, 4], count=2, rows=0, N=8), 4),
    (dict(lengths=[3, 4], count=2, rows=1, N=0), 4),
    (dict(lengths=[3, 0], count=2, rows=1, N=8), 4),
    (dict(lengths=[3, 4], count=2, rows=1, N=8, offsets=[0, -1]), 4),
])
def test_refusals_write_nothing(kw, code, L):
    got, seg_buf, tok_buf = _raw(L, **kw)
    assert got == code
    assert (seg_buf == 12345).all() and (tok_buf == 12345).all()


def test_library_matches_oracle_on_generated_inputs(L):
    """Property-based sweep (small shapes): element-by-element equality with
    the oracle, and the first-fit properties, for generated datasets."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(lengths=st.lists(st.integers(1, 40), min_size=0, max_size=40),
               rows=st.integers(1, 6), N=st.integers(1, 64), seed=st.integers(0, 2**64 - 1),
               epoch=st.integers(0, 2**64 - 1), data=st.data())
    def check(lengths, rows, N, seed, epoch, data):
        offsets = [data.draw(st.integers(0, x + 1)) for x in lengths]
        tokens = list(range(100, 100 + sum(lengths)))
        a = _lib_pack(lengths, rows, N, seed, epoch, offsets, tokens, pad_token=-1)
        b = opk.pack(lengths, rows, N, seed, epoch, offsets, tokens, pad_token=-1)
        _assert_same(a, b)
        _check_pack_properties(a, lengths, offsets, rows, N)

    check()


def test_packed_rows_are_sorted_runs(L):
    """Segment ids come out as nondecreasing runs per row (0, 1, ..., then the
    padding id), the layout the attention kernels' tile skipping is fastest on."""
    rng = np.random.default_rng(3)
    lengths, offsets = _random_dataset(rng, 90, 2, 300, 1024)
    res = _lib_pack(lengths, 8, 1024, 5, 2, offsets)
    seg = res["seg"]
    assert (np.diff(seg, axis=1) >= 0).all()
    assert (np.diff(seg, axis=1) <= 1).all()
    assert (seg[:, 0] == 0).all()


def test_row_targets_are_the_next_token_where_supervised(L):
    """row_targets: the next token of the same sequence where the loss mask
    is 1, else -1 (the ignored target of the fused cross-entropy)."""
    rng = np.random.default_rng(11)
    lengths, offsets = _random_dataset(rng, 70, 1, 200, 512)
    tokens = [int(t) for t in rng.integers(0, 1 << 20, size=sum(lengths))]
    r = _lib_pack(lengths, 12, 512, 3, 1, offsets, tokens, pad_token=-5)
    m, rt, tg, seg = r["loss_mask"], r["row_tokens"], r["row_targets"], r["seg"]
    assert (tg[m == 0] == -1).all()
    rr, tt = np.nonzero(m)
    assert (tg[rr, tt] == rt[rr, tt + 1]).all() and (seg[rr, tt] == seg[rr, tt + 1]).all()
    assert (tg[m == 1] >= 0).all()


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_packed_batches_shard_across_ranks(world, L):
    """Every rank gets the same number of (B, N) batches; together they hold
    each packed batch exactly once, and the extras are all padding."""
    rng = np.random.default_rng(21)
    lengths, offsets = _random_dataset(rng, 130, 4, 500, 1024)
    tokens = list(range(sum(lengths)))
    whole = list(pa.packed_batches(lengths, 2, 1024, 4, 0, offsets, tokens, pad_token=-1))
    per = [list(pa.packed_batches(lengths, 2, 1024, 4, 0, offsets, tokens, pad_token=-1, rank=r, world=world))
           for r in range(world)]
    assert len({len(p) for p in per}) == 1
    seen = []
    for r, batches in enumerate(per):
        for i, b in enumerate(batches):
            idx = r + i * world
            if idx < len(whole):
                for k in ("seg", "loss_mask", "row_tokens", "row_targets"):
                    np.testing.assert_array_equal(b[k], whole[idx][k])
                seen.append(idx)
            else:
                assert b["loss_mask"].sum() == 0 and (b["row_targets"] == -1).all() and (b["seg"] == 0).all()
    assert sorted(seen) == list(range(len(whole)))
    with pytest.raises(ValueError):
        next(pa.packed_batches(lengths, 2, 1024, 4, 0, rank=world, world=world))


def test_packer_is_reentrant_across_threads(L):
    """Concurrent calls from several threads (ctypes releases the GIL) return
    the same results as serial calls: the packer keeps no shared state."""
    import concurrent.futures as cf
    rng = np.random.default_rng(31)
    jobs = []
    for j in range(16):
        lengths, offsets = _random_dataset(rng, 400, 1, 300, 1024)
        jobs.append((lengths, offsets, 1000 + j))
    serial = [_lib_pack(l, 60, 1024, s, 1, o) for l, o, s in jobs]
    with cf.ThreadPoolExecutor(8) as ex:
        threaded = list(ex.map(lambda a: _lib_pack(a[0], 60, 1024, a[2], 1, a[1]), jobs))
    for a, b in zip(serial, threaded):
        np.testing.assert_array_equal(a["seg"], b["seg"])
        np.testing.assert_array_equal(a["placement"], b["placement"])


def test_packed_loss_equals_unpacked_loss(L):
    """The supervised set is that of an unpacked run (0.5.1 README, "Sequence
    packing"), at the level of the loss: given each token's final hidden
    state, the masked mean NLL over the packed rows -- targets from
    row_targets, -1 ignored -- equals the mean over every sequence run alone
    under the unpacked rule (the fp64 cross-entropy oracle on both sides)."""
    from oracle import linear_ce as lce
    rng = np.random.default_rng(41)
    V, D, N, rows = 97, 12, 256, 6
    lengths, offsets = _random_dataset(rng, 25, 1, 120, N)
    tokens = [int(t) for t in rng.integers(0, V, size=sum(lengths))]
    W = rng.standard_normal((V, D))
    hid = rng.standard_normal((sum(lengths), D))  # each token's hidden state, unpacked order
    r = _lib_pack(lengths, rows, N, 8, 0, offsets, tokens, pad_token=0)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)

    packed_h = rng.standard_normal((rows * N, D))  # padding rows: anything
    for s, at in enumerate(r["placement"]):
        if at >= 0:
            packed_h[at:at + lengths[s]] = hid[starts[s]:starts[s] + lengths[s]]
    tg = r["row_targets"].reshape(-1)
    keep = tg >= 0
    nll_p, _, _ = lce.forward(packed_h[keep], W, tg[keep])

    nll_u = []
    for s, at in enumerate(r["placement"]):
        if at < 0:
            continue
        L_, o = lengths[s], offsets[s]
        seq_t = tokens[starts[s]:starts[s] + L_]
        pos = [p for p in range(L_ - 1) if p + 1 >= o]
        if pos:
            nll_u.append(lce.forward(hid[starts[s] + np.array(pos)], W, [seq_t[p + 1] for p in pos])[0])
    nll_u = np.concatenate(nll_u)
    assert len(nll_p) == len(nll_u) == int(r["loss_mask"].sum())
    assert nll_p.mean() == pytest.approx(nll_u.mean(), rel=1e-12)
    np.testing.assert_allclose(np.sort(nll_p), np.sort(nll_u), rtol=1e-12)
