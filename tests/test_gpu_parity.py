"""GPU results against the fp64 oracle (through the C ABI).

Tolerances (the target's): O max-abs <= 1e-2 over every compared element;
dQ/dK/dV relative L2 <= 2e-2 over every compared element; lse max-abs 1e-3.
Small cases compare every element; the full-size workloads compare rows the
oracle computes one by one (segment starts/ends, tile edges, random rows) and
check per-segment gradient sums, which hold at any size. The packed kernels
with a single segment must be bit-identical to the causal kernels (changelog
entry adding the PACKED kernels). Dropping the segment mask must fail the
tolerance (mlx-train-perf 0.5.1 README, "Sequence packing": contamination
test).
"""
import time

import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa
import synth
from _gpu_common import (Case, assert_full_parity, assert_group_parity, assert_sampled_parity,
                         assert_segment_sums, f64, O_MAXABS)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


SMALL = [
    ("tiny_3seg", synth.workload("tiny_3seg")),
    ("tiny_fixed_1_100_155", synth.workload("tiny_fixed_1_100_155")),
    ("ragged_gqa_d128", synth.custom(2, 4, 2, 512, 128, [[1, 130, 5, 120, 256], [512]], seed=21)),
    ("many_len3_d64", synth.custom(1, 2, 1, 384, 64, [[3] * 128], seed=22)),
    ("len1_runs_d128", synth.custom(1, 2, 2, 256, 128, [[1] * 40 + [88, 128]], seed=23)),
    ("gqa8_d64", synth.custom(1, 8, 1, 640, 64, [[300, 213, 127]], seed=24)),
    # odd group size and odd tile count: the forward pairs consecutive query
    # tiles and the last pair has one tile only
    ("g3_odd_tiles_d64", synth.custom(2, 3, 1, 384, 64, [[200, 184], [384]], seed=27)),
    # head dim 96: the 128-wide kernels with tiles whose columns 96..127 the
    # loads fill with zeros and the stores leave out
    ("ragged_gqa_d96", synth.custom(2, 4, 2, 512, 96, [[1, 130, 5, 120, 256], [512]], seed=29)),
    ("len1_runs_g3_d96", synth.custom(1, 3, 1, 384, 96, [[1] * 30 + [3] * 20 + [294]], seed=30)),
    # N not a multiple of 128: whole tiles with a tail that TMA reads as zeros
    ("ragged_n200_d64", synth.custom(1, 2, 2, 200, 64, [[1, 100, 99]], seed=31)),
    ("ragged_n300_gqa_d128", synth.custom(2, 4, 2, 300, 128, [[150, 150], [1, 298, 1]], seed=32)),
    ("ragged_n129_d96", synth.custom(1, 3, 1, 129, 96, [[129]], seed=33)),
    ("ragged_n1_d64", synth.custom(1, 2, 1, 1, 64, [[1]], seed=34)),
    ("ragged_n127_d128", synth.custom(1, 2, 1, 127, 128, [[60, 67]], seed=35)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[n for n, _ in SMALL])
def test_small_full_parity(name, w, cuda_dev):
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run(), c.oracle_full(), name))


def test_causal_entry_points_full_parity(cuda_dev):
    w = synth.custom(1, 4, 1, 384, 128, [[384]], seed=25)
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run(causal=True), c.oracle_full(causal=True), "causal"))


def test_causal_ragged_n_full_parity(cuda_dev):
    w = synth.custom(1, 4, 2, 333, 64, [[333]], seed=36)
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run(causal=True), c.oracle_full(causal=True), "causal ragged"))


STRIDED = [
    ("bnhd_gqa_d128", synth.custom(2, 4, 2, 512, 128, [[1, 130, 5, 120, 256], [512]], seed=37)),
    ("bnhd_ragged_n300_d64", synth.custom(1, 4, 1, 300, 64, [[100, 200]], seed=38)),
    ("bnhd_ragged_n200_d96", synth.custom(2, 2, 2, 200, 96, [[200], [7, 193]], seed=39)),
]


@pytest.mark.parametrize("name,w", STRIDED, ids=[n for n, _ in STRIDED])
def test_strided_bnhd_full_parity(name, w, cuda_dev):
    """(B, N, H, D) memory through the strided entry points: oracle parity,
    and bit-identical to the contiguous call on the same values."""
    c = Case(w, cuda_dev)
    g = c.run_strided()
    print(assert_full_parity(g, c.oracle_full(), name))
    ref = c.run()
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(g[n], ref[n]), n


def test_strided_bnhd_causal(cuda_dev):
    w = synth.custom(1, 4, 2, 256, 128, [[256]], seed=40)
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run_strided(causal=True), c.oracle_full(causal=True), "bnhd causal"))


def _run_f32(c, q, k, v, do, causal=False):
    seg = None if causal else c.seg
    ws = pa.workspace(q, k, strided=True)
    out, lse = pa.forward(q, k, v, seg, ws=ws)
    assert pa.pa_device_status(ws) == 0  # read before the backward's tile-table step clears it
    dq, dk, dv = pa.backward(q, k, v, out, do, lse, seg, ws=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(ws) == 0
    assert out.dtype == dq.dtype == dk.dtype == torch.float32
    return {"o": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


FP32 = [
    ("f32_gqa_d128", synth.custom(2, 4, 2, 512, 128, [[1, 130, 5, 120, 256], [512]], seed=42), False),
    ("f32_ragged_n300_d96_bnhd", synth.custom(1, 4, 2, 300, 96, [[100, 200]], seed=43), True),
]


@pytest.mark.parametrize("name,w,bnhd", FP32, ids=[n for n, _, _ in FP32])
def test_fp32_io(name, w, bnhd, cuda_dev):
    """fp32 tensors are rounded to bf16 on the way in and results widened on
    the way out: on bf16-representable inputs the fp32 call returns the bf16
    call's results exactly, and it meets the oracle's bars."""
    c = Case(w, cuda_dev)
    lay = (lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)) if bnhd else (lambda t: t)
    g32 = _run_f32(c, *(lay(t.float()) for t in (c.q, c.k, c.v, c.do)))
    print(assert_full_parity(g32, c.oracle_full(), name))
    ref = c.run()
    for n in ("o", "dq", "dk", "dv"):
        assert torch.equal(g32[n], ref[n].float()), n
    assert torch.equal(g32["lse"], ref["lse"])


def test_fp32_io_rounds_to_nearest_even(cuda_dev):
    """Inputs that bf16 cannot hold: the fp32 call equals the bf16 call on
    the inputs rounded by torch (round to nearest even)."""
    w = synth.custom(1, 2, 2, 256, 64, [[100, 156]], seed=44)
    c = Case(w, cuda_dev)
    gen = torch.Generator(device="cpu").manual_seed(44)
    q, k, v, do = (torch.randn(t.shape, generator=gen).to(cuda_dev) for t in (c.q, c.k, c.v, c.do))
    g32 = _run_f32(c, q, k, v, do)
    out, lse = pa.forward(q.bfloat16(), k.bfloat16(), v.bfloat16(), c.seg)
    dq, dk, dv = pa.backward(q.bfloat16(), k.bfloat16(), v.bfloat16(), out, do.bfloat16(), lse, c.seg)
    for n, ref in (("o", out), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(g32[n], ref.float()), n


def test_ragged_n_5000_sampled(cuda_dev):
    w = synth.custom(1, 16, 4, 5000, 128, [[1000, 2999, 1, 1000]], seed=41)
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag="ragged_5000"))
    assert_segment_sums(c, g)


def test_non_contiguous_ids_full_parity(cuda_dev):
    """Ids are compared for equality only: a sequence id may reappear later
    in the row and its tokens still see each other."""
    w = synth.custom(1, 2, 2, 512, 128, [[100, 100, 100, 212]], seed=26)
    w.seg[0] = np.array([5] * 100 + [9] * 100 + [5] * 100 + [-3] * 212, np.int32)
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run(), c.oracle_full(), "noncontig"))


def test_skipped_key_tiles_full_parity(cuda_dev):
    """Ids alternate between two values in blocks, so a query tile's walk
    skips every other key tile: row 0 in tile-aligned blocks of 128 (skipped
    tiles only), row 1 in blocks of 96 (skips plus tiles that span two ids)."""
    w = synth.custom(2, 4, 2, 1024, 128, [[1024], [1024]], seed=28)
    w.seg[0] = np.array([(i // 128) % 2 for i in range(1024)], np.int32)
    w.seg[1] = np.array([7 + (i // 96) % 2 for i in range(1024)], np.int32)
    c = Case(w, cuda_dev)
    print(assert_full_parity(c.run(), c.oracle_full(), "skipped"))


def test_causal_2k_gqa(cuda_dev):
    w = synth.workload("causal_2k_gqa")
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag=w.name))
    assert_segment_sums(c, g)


def test_packed_4x4096_short(cuda_dev):
    w = synth.workload("packed_4x4096_short")
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag=w.name))
    # every element of every kv group (short segments make this cheap)
    errors = []
    for hk in range(w.Hkv):
        try:
            print(assert_group_parity(c, g, hk, tag=f"{w.name} group {hk}"))
        except AssertionError as e:
            errors.append(str(e).splitlines()[0])
    try:
        assert_segment_sums(c, g)
    except AssertionError as e:
        errors.append(str(e).splitlines()[0])
    assert not errors, "\n".join(errors)


def test_8k_packed_group_full(cuda_dev):
    w = synth.workload("8k_packed")
    c = Case(w, cuda_dev)
    print(assert_group_parity(c, c.run(), 3, tag="8k_packed group 3"))


def test_8k_one_segment_group_full(cuda_dev):
    """The headline row: every element of one kv group (4 query heads x 8192
    rows of O, lse and dQ; the kv head's dK and dV) against the oracle."""
    w = synth.workload("8k_one_segment")
    c = Case(w, cuda_dev)
    print(assert_group_parity(c, c.run(), 5, tag="8k_one_segment group 5"))


@pytest.mark.parametrize("name", ["8k_one_segment", "8k_packed"])
def test_8k(name, cuda_dev):
    w = synth.workload(name)
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag=name))
    assert_segment_sums(c, g)


@pytest.mark.parametrize("name", ["long_32k_one_segment", "long_32k_packed", "long_64k_one_segment",
                                  "long_64k_packed"])
def test_long_context(name, cuda_dev):
    w = synth.workload(name)
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag=name))
    assert_segment_sums(c, g)


@pytest.mark.parametrize("name", ["8k_one_segment_d96", "packed_2x4096_short_d96"])
def test_head_dim_96(name, cuda_dev):
    w = synth.workload(name)
    c = Case(w, cuda_dev)
    g = c.run()
    print(assert_sampled_parity(c, g, tag=name))
    assert_segment_sums(c, g)


def test_head_dim_96_full_group(cuda_dev):
    w = synth.workload("packed_2x4096_short_d96")
    c = Case(w, cuda_dev)
    print(assert_group_parity(c, c.run(), 1, tag="packed_2x4096_short_d96 group 1"))


@pytest.mark.parametrize("name", ["causal_2k_gqa", "8k_one_segment", "long_32k_one_segment", "8k_one_segment_d96"])
def test_single_segment_bit_identical_to_causal(name, cuda_dev):
    w = synth.workload(name)
    c = Case(w, cuda_dev)
    packed = c.run()
    causal = c.run(causal=True)
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(bits(packed[n]), bits(causal[n])), n


def test_bounded_wait_gives_up_and_context_survives(cuda_dev):
    """A wait that nothing completes runs out after its limit, reports
    PA_DEVERR_TIMEOUT with its site in the status word, and the next calls
    on the same context still compute correct results."""
    w = synth.workload("tiny_3seg")
    c = Case(w, cuda_dev)
    t0 = time.time()
    pa.pa_selftest_wait_timeout(c.ws)
    st = pa.pa_device_status(c.ws)
    took = time.time() - t0
    assert st == (0x1 | (99 << 8)), hex(st)  # PA_DEVERR_TIMEOUT, site 99
    assert 1.0 < took < 30.0, took
    assert pa.pa_device_status(c.ws) == 0  # reading cleared it
    print(assert_full_parity(c.run(), c.oracle_full(), "after-timeout"))


@pytest.mark.parametrize("name", ["tiny_3seg", "long_32k_packed", "8k_packed", "packed_4x4096_short"])
def test_forward_alone_is_healthy_and_prompt(name, cuda_dev):
    """The forward on its own leaves a clean status word (every bounded wait
    completed) and takes well under the 2 s wait limit: a pipeline that
    waits for work that never comes would show up here even when its
    outputs are right."""
    w = synth.workload(name)
    c = Case(w, cuda_dev, host64=False)
    pa.forward(c.q, c.k, c.v, c.seg, ws=c.ws)  # warm-up
    torch.cuda.synchronize()
    assert pa.pa_device_status(c.ws) == 0
    t0 = time.time()
    for _ in range(3):
        pa.forward(c.q, c.k, c.v, c.seg, ws=c.ws)
    torch.cuda.synchronize()
    took = time.time() - t0
    assert pa.pa_device_status(c.ws) == 0
    assert took < 0.5, took


def test_runs_are_deterministic(cuda_dev):
    c = Case(synth.workload("packed_4x4096_short"), cuda_dev)
    a, b = c.run(), c.run()
    for n in a:
        assert torch.equal(a[n], b[n]), n


def test_dropping_the_mask_fails_parity(cuda_dev):
    """Negative control: the causal kernel on a packed row must miss the
    packed oracle by far more than the tolerance."""
    w = synth.workload("tiny_3seg")
    c = Case(w, cuda_dev)
    ref = c.oracle_full()
    wrong = c.run(causal=True)
    err = np.abs(f64(wrong["o"]) - ref["o"]).max()
    assert err > 10 * O_MAXABS, err
