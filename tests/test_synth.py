"""The seeded input generator: determinism, bf16 rounding, segment layouts."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    x = np.concatenate([synth.normals(3, 0, 20000) * 7.0,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 65504.0, 1e-30])])
    x = x.astype(np.float32)
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_generator_is_deterministic_and_streams_differ():
    a = synth.bf16_normal(1004, 1, (4, 64))
    b = synth.bf16_normal(1004, 1, (4, 64))
    c = synth.bf16_normal(1004, 2, (4, 64))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_normals_moments():
    z = synth.normals(42, 0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def test_uniforms_range():
    u = synth.uniforms(1, 1, 100000)
    assert u.min() > 0.0 and u.max() <= 1.0


def test_workload_segment_layouts():
    for name in synth.WORKLOADS:
        w = synth.workload(name)
        assert w.seg.shape == (w.B, w.N) and w.seg.dtype == np.int32
        for b in range(w.B):
            assert sum(w.lengths[b]) == w.N
            assert np.array_equal(w.seg[b], synth.lengths_to_ids(w.lengths[b]))
    t = synth.workload("tiny_3seg")
    assert len(t.lengths[0]) == 3 and min(t.lengths[0]) >= 1
    f = synth.workload("tiny_fixed_1_100_155")
    assert f.lengths[0] == [1, 100, 155]
    for name, lo, hi in (("8k_packed", 256, 2048), ("long_64k_packed", 512, 8192)):
        lens = synth.workload(name).lengths[0]
        assert all(lo <= L <= hi for L in lens[:-1]) and 1 <= lens[-1] <= hi


def test_packed_short_rows_match_the_described_shape():
    w = synth.workload("packed_4x4096_short")
    real = [l[:-1] if p else l for l, p in zip(w.lengths, w.pad)]
    allreal = np.concatenate(real)
    assert 8 <= allreal.min() and allreal.max() <= 1024
    assert 70 <= np.median(allreal) <= 100          # lognormal median 84
    per_row = [len(r) for r in real]
    assert all(25 <= n <= 60 for n in per_row)       # tens of sequences per 4,096 row
    for l, p in zip(w.lengths, w.pad):
        assert p == (l[-1] if p else 0)


def test_first_fit_places_in_first_row_with_room():
    rows = synth.first_fit([5, 4, 3, 2, 6], B=2, N=8)
    assert rows == [[5, 3], [4, 2]]  # 6 fits nowhere and is dropped
