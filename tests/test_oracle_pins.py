"""Pins of the fp64 oracle to things other than itself (CPU only).

The oracle follows the definition of block-diagonal causal attention
(mlx-train-perf 0.5.1 README, "Sequence packing"; changelog entry adding
`flash_attention(segments=...)` and the PACKED kernels). These tests tie it to:
  * a hand-worked example (tests/golden/hand_worked_two_segments.json),
  * torch's scaled_dot_product_attention + autograd in float64 with an explicit
    boolean block-diagonal mask (a library routine, forward and gradients),
  * central finite differences of L = sum(dO * O) (gradients vs forward),
  * the two invariants the changelog states: a packed row equals each
    sequence run alone, and a single segment equals plain causal attention,
  * closed forms (length-1 segments, Q = 0, constant V, per-segment sums),
  * the negative control the README describes (dropping the segment mask
    must move the result far past the tolerance).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(B, Hq, Hkv, N, D, seed=11):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    do = rng.standard_normal((B, Hq, N, D))
    return q, k, v, do


def sdpa_reference(q, k, v, seg, scale, do):
    """Library pin: torch SDPA (float64, CPU) with a dense boolean mask that
    encodes 'same segment and not in the future', GQA by repeat_interleave."""
    B, Hq, N, D = q.shape
    G = Hq // k.shape[1]
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    idx = torch.arange(N)
    causal = idx[None, :] <= idx[:, None]
    if seg is None:
        mask = causal[None, None].expand(B, 1, N, N)
    else:
        s = torch.tensor(seg)
        mask = (causal[None] & (s[:, :, None] == s[:, None, :]))[:, None]
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=mask, scale=scale)
    scores = torch.einsum("bhic,bhjc->bhij", tq, kk) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    o.backward(torch.tensor(do))
    return {"o": o.detach().numpy(), "lse": lse.detach().numpy(), "dq": tq.grad.numpy(),
            "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}


# ---------------------------------------------------------------- hand-worked
def test_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_two_segments.json")))
    q, k, v, do = (np.array(g[x]) for x in ("q", "k", "v", "do"))
    seg = np.array(g["seg"], dtype=np.int32)
    r = oracle.attention(q, k, v, seg, g["scale"], do)
    for name, val in g["expect"].items():
        np.testing.assert_allclose(r[name], np.array(val), rtol=0, atol=1e-14, err_msg=name)
    # plain causal sees across the boundary: row 2 changes
    o_c, _, _ = oracle.forward(q, k, v, None, g["scale"])
    assert abs(o_c[0, 0, 2] - np.array(g["expect"]["o"])[0, 0, 2]).max() > 0.5


# ---------------------------------------------------------------- library pin
@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, N, D, lengths per row)
    (1, 2, 2, 40, 16, [[40]]),
    (1, 4, 2, 40, 8, [[1, 12, 27]]),
    (2, 4, 1, 33, 8, [[5, 1, 1, 26], [33]]),
    (2, 6, 3, 48, 16, [[16, 16, 16], [7, 30, 11]]),
])
def test_matches_torch_sdpa_float64(case):
    B, Hq, Hkv, N, D, lens = case
    q, k, v, do = rand_inputs(B, Hq, Hkv, N, D, seed=B * 100 + N)
    seg = np.stack([synth.lengths_to_ids(l) for l in lens]).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    r = oracle.attention(q, k, v, seg, scale, do)
    ref = sdpa_reference(q, k, v, seg, scale, do)
    for name in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[name], ref[name], rtol=0, atol=1e-12, err_msg=name)
    # delta definition: rowsum(dO * O)
    np.testing.assert_allclose(r["delta"], (do * ref["o"]).sum(-1), rtol=0, atol=1e-12)


def test_causal_none_matches_sdpa_is_causal():
    q, k, v, do = rand_inputs(1, 4, 2, 37, 8, seed=3)
    scale = 0.3
    o, lse, _ = oracle.forward(q, k, v, None, scale)
    tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(2, 1), tv.repeat_interleave(2, 1), is_causal=True, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- finite differences
def test_finite_differences():
    B, Hq, Hkv, N, D = 1, 4, 2, 24, 8
    q, k, v, do = rand_inputs(B, Hq, Hkv, N, D, seed=5)
    seg = synth.lengths_to_ids([9, 1, 14])[None].astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    r = oracle.attention(q, k, v, seg, scale, do)

    def loss(qq, kk, vv):
        o, _, _ = oracle.forward(qq, kk, vv, seg, scale)
        return float((o * do).sum())

    h = 1e-6
    for name, arr, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        fd = np.empty_like(arr)
        flat, fdf = arr.reshape(-1), fd.reshape(-1)
        for t in range(flat.size):
            keep = flat[t]
            flat[t] = keep + h
            lp = loss(q, k, v)
            flat[t] = keep - h
            lm = loss(q, k, v)
            flat[t] = keep
            fdf[t] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max()
        assert err <= 1e-6 * max(1.0, np.abs(grad).max()), (name, err)


# ---------------------------------------------------------------- invariants
def test_packed_row_equals_segments_alone():
    lens = [7, 1, 20, 3, 17]
    N = sum(lens)
    q, k, v, do = rand_inputs(1, 4, 2, N, 8, seed=21)
    seg = synth.lengths_to_ids(lens)[None].astype(np.int32)
    scale = 0.35
    r = oracle.attention(q, k, v, seg, scale, do)
    start = 0
    for L in lens:
        sl = slice(start, start + L)
        part = oracle.attention(q[:, :, sl], k[:, :, sl], v[:, :, sl],
                                np.zeros((1, L), np.int32), scale, do[:, :, sl])
        for name in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[name][:, :, sl], part[name], rtol=0, atol=1e-13, err_msg=name)
        start += L


def _dense_causal_textbook(q, k, v, scale):
    """Independent dense causal softmax attention (numpy, one head)."""
    N = q.shape[0]
    s = (q @ k.T) * scale
    s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=1, keepdims=True)
    return w @ v


def test_single_segment_equals_textbook_causal():
    q, k, v, do = rand_inputs(1, 2, 1, 50, 16, seed=9)
    scale = 0.25
    o1, _, _ = oracle.forward(q, k, v, np.full((1, 50), 3, np.int32), scale)
    o2, _, _ = oracle.forward(q, k, v, None, scale)
    assert np.array_equal(o1, o2)
    for h in range(2):
        np.testing.assert_allclose(o1[0, h], _dense_causal_textbook(q[0, h], k[0, 0], v[0, 0], scale),
                                   rtol=0, atol=1e-12)


def test_segment_ids_need_not_be_contiguous_values():
    """Ids are compared for equality only: relabelling them changes nothing."""
    lens = [5, 9, 4]
    q, k, v, do = rand_inputs(1, 2, 2, 18, 8, seed=2)
    a = synth.lengths_to_ids(lens)[None].astype(np.int32)
    b = np.array([[-7] * 5 + [100] * 9 + [3] * 4], np.int32)
    ra = oracle.attention(q, k, v, a, 0.4, do)
    rb = oracle.attention(q, k, v, b, 0.4, do)
    for name in ra:
        assert np.array_equal(ra[name], rb[name]), name


# ---------------------------------------------------------------- closed forms
def test_all_length_one_segments():
    B, Hq, Hkv, N, D = 1, 4, 2, 12, 8
    q, k, v, do = rand_inputs(B, Hq, Hkv, N, D, seed=4)
    seg = np.arange(N, dtype=np.int32)[None]
    r = oracle.attention(q, k, v, seg, 0.5, do)
    G = Hq // Hkv
    np.testing.assert_allclose(r["o"], np.repeat(v, G, axis=1), atol=1e-15, rtol=0)
    assert np.abs(r["dq"]).max() < 1e-15 and np.abs(r["dk"]).max() < 1e-15
    np.testing.assert_allclose(r["dv"], do.reshape(B, Hkv, G, N, D).sum(2), atol=1e-14, rtol=0)
    np.testing.assert_allclose(r["lse"], 0.5 * np.einsum("bhnc,bhnc->bhn", q, np.repeat(k, G, 1)),
                               atol=1e-14, rtol=0)


def test_zero_query_gives_prefix_mean():
    lens = [6, 10]
    N = 16
    _, k, v, do = rand_inputs(1, 2, 1, N, 8, seed=8)
    q = np.zeros((1, 2, N, 8))
    seg = synth.lengths_to_ids(lens)[None].astype(np.int32)
    o, lse, _ = oracle.forward(q, k, v, seg, 1.0)
    start = 0
    for L in lens:
        for t in range(L):
            i = start + t
            np.testing.assert_allclose(o[0, :, i], np.broadcast_to(v[0, 0, start:i + 1].mean(0), (2, 8)),
                                       atol=1e-14, rtol=0)
            np.testing.assert_allclose(lse[0, :, i], math.log(t + 1), atol=1e-14, rtol=0)
        start += L


def test_constant_value_within_segment():
    lens = [9, 7]
    q, k, _, do = rand_inputs(1, 2, 1, 16, 4, seed=12)
    v = np.empty((1, 1, 16, 4))
    v[0, 0, :9] = [1.5, -2.0, 0.25, 3.0]
    v[0, 0, 9:] = [-1.0, 0.5, 2.0, 0.0]
    seg = synth.lengths_to_ids(lens)[None].astype(np.int32)
    o, _, _ = oracle.forward(q, k, v, seg, 0.5)
    np.testing.assert_allclose(o[0, :, :9], np.broadcast_to(v[0, 0, 0], (2, 9, 4)), atol=1e-14, rtol=0)
    np.testing.assert_allclose(o[0, :, 9:], np.broadcast_to(v[0, 0, 9], (2, 7, 4)), atol=1e-14, rtol=0)


def test_per_segment_gradient_sums():
    """Rows of P sum to 1 and rows of dS sum to 0, so per segment
    sum_j dk_j = 0 and sum_j dv_j = sum over the group's heads of sum_i dO_i."""
    lens = [13, 2, 21]
    N = sum(lens)
    B, Hq, Hkv, D = 1, 6, 2, 8
    q, k, v, do = rand_inputs(B, Hq, Hkv, N, D, seed=31)
    seg = synth.lengths_to_ids(lens)[None].astype(np.int32)
    r = oracle.attention(q, k, v, seg, 0.3, do)
    G = Hq // Hkv
    start = 0
    for L in lens:
        sl = slice(start, start + L)
        assert np.abs(r["dk"][:, :, sl].sum(2)).max() < 1e-12
        np.testing.assert_allclose(r["dv"][:, :, sl].sum(2),
                                   do[:, :, sl].sum(2).reshape(B, Hkv, G, D).sum(2), atol=1e-12, rtol=0)
        start += L


# ---------------------------------------------------------------- negative control
def test_dropping_segment_mask_moves_result():
    w = synth.workload("tiny_3seg")
    t = w.tensors()
    q, k, v, do = (synth.bf16_bits_to_f64(t[x]) for x in ("q", "k", "v", "do"))
    packed, _, _ = oracle.forward(q, k, v, w.seg, w.scale)
    causal, _, _ = oracle.forward(q, k, v, None, w.scale)
    assert np.abs(packed - causal).max() > 0.1  # O tolerance is 1e-2


# ---------------------------------------------------------------- row API
def test_row_subsets_match_full():
    B, Hq, Hkv, N, D = 2, 4, 2, 30, 8
    q, k, v, do = rand_inputs(B, Hq, Hkv, N, D, seed=17)
    seg = np.stack([synth.lengths_to_ids([10, 20]), synth.lengths_to_ids([3, 27])]).astype(np.int32)
    r = oracle.attention(q, k, v, seg, 0.4, do)
    rows = np.array([0, 5, 29, 77, 200, B * Hq * N - 1])
    o, lse, delta = oracle.forward(q, k, v, seg, 0.4, do, rows=rows)
    assert np.array_equal(o, r["o"].reshape(-1, D)[rows])
    assert np.array_equal(lse, r["lse"].reshape(-1)[rows])
    dq = oracle.dq(q, k, v, seg, 0.4, do, r["lse"], r["delta"], rows=rows)
    assert np.array_equal(dq, r["dq"].reshape(-1, D)[rows])
    krows = np.array([0, 9, 10, 31, B * Hkv * N - 1])
    dk, dv = oracle.dkv(q, k, v, seg, 0.4, do, r["lse"], r["delta"], rows=krows)
    assert np.array_equal(dk, r["dk"].reshape(-1, D)[krows])
    assert np.array_equal(dv, r["dv"].reshape(-1, D)[krows])
