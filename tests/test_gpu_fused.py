"""The single-pass backward (pa_bwd_fused) against the fp64 oracle and
against the split backward.

The operation is pa_bwd's, so the bars are the path's: dQ/dK/dV relative L2
<= 2e-2 against the oracle on every compared element. dK and dV are summed
inside one CTA in the split kernel's order from the same bf16 operands, so
they must equal pa_bwd's bit for bit. dQ is the sum of fp32 shares added in
no fixed order, and its dS comes from the dK/dV side's products (V dO^T
rather than dO V^T, each rounded to bf16), so against the split kernel's dQ
it agrees to the rounding of dS, not bitwise: relative L2 <= 1e-2 over the
tensor and no row off by more than 5% of its norm plus the tensor's mean
row magnitude (a row whose terms cancel has no relative bound).
"""
import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa
import synth
from _gpu_common import Case, assert_full_parity, assert_group_parity, assert_sampled_parity, assert_segment_sums, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


def run_fused(c: Case, causal: bool = False, split: dict | None = None):
    """Forward through pa_fwd (or the split run's outputs), then pa_bwd_fused."""
    seg = None if causal else c.seg
    if split is None:
        out, lse = pa.forward(c.q, c.k, c.v, seg, ws=c.ws)
        assert pa.pa_device_status(c.ws) == 0
    else:
        out, lse = split["o"], split["lse"]
    w = c.w
    ws = torch.empty(pa.pa_bwd_fused_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.D), dtype=torch.uint8,
                     device=c.q.device)
    dq, dk, dv = pa.backward_fused(c.q, c.k, c.v, out, c.do, lse, seg, ws=ws)
    torch.cuda.synchronize()
    st = pa.pa_device_status(ws)
    assert st == 0, f"device status after the single-pass backward {st:#x}"
    return {"o": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def assert_matches_split(fused: dict, split: dict, tag: str):
    assert torch.equal(fused["dk"], split["dk"]), f"{tag}: dK differs from the split kernel"
    assert torch.equal(fused["dv"], split["dv"]), f"{tag}: dV differs from the split kernel"
    a, b = f64(fused["dq"]), f64(split["dq"])
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    D = a.shape[-1]
    a2, b2 = a.reshape(-1, D), b.reshape(-1, D)
    floor = np.sqrt(D) * np.abs(b2).mean()
    row = float((np.linalg.norm(a2 - b2, axis=1) / (np.linalg.norm(b2, axis=1) + floor)).max())
    print(f"{tag}: dQ vs split relL2 {rel:.2e}, worst row {row:.2e}")
    assert rel <= 1e-2 and row <= 0.05, tag


SMALL = [
    ("tiny_3seg", synth.workload("tiny_3seg")),
    ("ragged_gqa_d128", synth.custom(2, 4, 2, 512, 128, [[1, 130, 5, 120, 256], [512]], seed=21)),
    ("many_len3_d64", synth.custom(1, 2, 1, 384, 64, [[3] * 128], seed=22)),
    ("len1_runs_d128", synth.custom(1, 2, 2, 256, 128, [[1] * 40 + [88, 128]], seed=23)),
    ("gqa8_d64", synth.custom(1, 8, 1, 640, 64, [[300, 213, 127]], seed=24)),
    ("g3_odd_tiles_d64", synth.custom(2, 3, 1, 384, 64, [[200, 184], [384]], seed=27)),
    ("ragged_gqa_d96", synth.custom(2, 4, 2, 512, 96, [[1, 130, 5, 120, 256], [512]], seed=29)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[n for n, _ in SMALL])
def test_fused_small_full_parity(name, w, cuda_dev):
    c = Case(w, cuda_dev)
    split = c.run()
    fused = run_fused(c, split=split)
    print(assert_full_parity(fused, c.oracle_full(), f"fused {name}"))
    assert_matches_split(fused, split, name)


def test_fused_causal_full_parity(cuda_dev):
    w = synth.custom(1, 4, 1, 384, 128, [[384]], seed=25)
    c = Case(w, cuda_dev)
    split = c.run(causal=True)
    fused = run_fused(c, causal=True, split=split)
    print(assert_full_parity(fused, c.oracle_full(causal=True), "fused causal"))
    assert_matches_split(fused, split, "causal")


def test_fused_packed_4x4096_short(cuda_dev):
    w = synth.workload("packed_4x4096_short")
    c = Case(w, cuda_dev)
    split = c.run()
    fused = run_fused(c, split=split)
    assert_matches_split(fused, split, w.name)
    print(assert_group_parity(c, fused, 2, tag=f"fused {w.name} group 2"))
    assert_segment_sums(c, fused)


@pytest.mark.parametrize("name", ["8k_one_segment", "8k_packed"])
def test_fused_8k(name, cuda_dev):
    w = synth.workload(name)
    c = Case(w, cuda_dev)
    split = c.run()
    fused = run_fused(c, split=split)
    assert_matches_split(fused, split, name)
    print(assert_sampled_parity(c, fused, tag=f"fused {name}"))


def test_fused_8k_one_segment_group_full(cuda_dev):
    w = synth.workload("8k_one_segment")
    c = Case(w, cuda_dev)
    print(assert_group_parity(c, run_fused(c), 5, tag="fused 8k_one_segment group 5"))


def test_fused_long_32k_packed_d64(cuda_dev):
    w = synth.workload("long_32k_packed")
    c = Case(w, cuda_dev)
    split = c.run()
    fused = run_fused(c, split=split)
    assert_matches_split(fused, split, w.name)
    print(assert_sampled_parity(c, fused, tag=f"fused {w.name}"))
    assert_segment_sums(c, fused)


def test_fused_refuses_ragged_n(cuda_dev):
    q = torch.zeros((1, 2, 300, 64), dtype=torch.bfloat16, device=cuda_dev)
    assert pa.pa_bwd_fused_workspace_bytes(1, 2, 2, 300, 64) == 0
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_dev)
    lse = torch.zeros((1, 2, 300), dtype=torch.float32, device=cuda_dev)
    with pytest.raises(pa.PAError) as e:
        pa.pa_bwd_fused(q, q, q, q, q, lse, None, q, q, q, ws)
    assert e.value.code == 4  # PA_ERR_SHAPE
