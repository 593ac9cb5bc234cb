"""Fused linear cross-entropy forward and backward on the GPU against the
fp64 oracle (mlx-train-perf 0.5.1 README, "The fused cross-entropy loss": the
per-token NLL, log-sum-exp and target logit of H W^T, with no (N, V) logits
stored, and the gradients into the hidden states and the head).

Inputs are bf16 normals from the seeded generator; the oracle takes the same
bf16 values in fp64. The kernel accumulates the D products of each logit in
fp32, so the bar is max |err| <= 1e-3 + 1e-5 |exact| on each output."""
import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa
import synth
from oracle import linear_ce as lce

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


def _inputs(N, V, D, seed, dev, ignored=()):
    hb = synth.bf16_normal(seed, 50, (N, D))
    wb = synth.bf16_normal(seed, 51, (V, D))
    t = (synth.uint64s(seed, 52, N) % np.uint64(V)).astype(np.int32)
    for i, val in ignored:
        t[i] = val
    to = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    return hb, wb, t, to(hb), to(wb), torch.from_numpy(t).to(dev)


def _run(H, W, T):
    N, D = H.shape
    ws = torch.empty(pa.pa_lce_workspace_bytes(N, W.shape[0], D), dtype=torch.uint8, device=H.device)
    nll, lse, tgt = pa.linear_cross_entropy_forward(H, W, T, ws=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(ws) == 0
    return nll, lse, tgt


CASES = [
    # name, N, V, D: ragged vocabulary; ragged tokens over many splits; a
    # 4-stage ring that wraps (8 K slices) with 3 vocabulary tiles per CTA
    ("ragged_v", 256, 1000, 128),
    ("ragged_n", 300, 4096, 256),
    ("ring_wraps", 2048, 5000, 512),
    ("d64_small_v", 128, 130, 64),
]


@pytest.mark.parametrize("name,N,V,D", CASES, ids=[c[0] for c in CASES])
def test_lce_forward_matches_oracle(name, N, V, D, cuda_dev):
    hb, wb, t, H, W, T = _inputs(N, V, D, 60 + len(name), cuda_dev, ignored=[(3, -1), (N - 1, V)])
    nll, lse, tgt = _run(H, W, T)
    h64, w64 = synth.bf16_bits_to_f64(hb), synth.bf16_bits_to_f64(wb)
    valid = (t >= 0) & (t < V)
    t_safe = np.where(valid, t, 0)
    e_nll, e_lse, e_tgt = lce.forward(h64, w64, t_safe)
    e_nll, e_tgt = np.where(valid, e_nll, 0.0), np.where(valid, e_tgt, 0.0)
    for got, exp, n in ((lse, e_lse, "lse"), (tgt, e_tgt, "target_logit"), (nll, e_nll, "nll")):
        g = got.cpu().numpy().astype(np.float64)
        err = np.abs(g - exp)
        bar = ATOL + RTOL * np.abs(exp)
        print(f"{name} {n}: max err {err.max():.3e} (|exact| up to {np.abs(exp).max():.1f})")
        assert (err <= bar).all(), (n, float(err.max()), int(err.argmax()))
    assert float(nll[3]) == 0.0 and float(tgt[N - 1]) == 0.0  # ignored targets


def test_lce_forward_is_deterministic(cuda_dev):
    _, _, _, H, W, T = _inputs(512, 3000, 256, 70, cuda_dev)
    a, b = _run(H, W, T), _run(H, W, T)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ------------------------------------------------------------------ backward
# dH and dW of L = sum_i g_i nll_i against the oracle's fp64 backward, on the
# forward's shapes plus one whose vocabulary spans three chunks (the fp32 dH
# accumulator starts, adds and finishes) and one of 36 token tiles, whose
# last group is partial in both the dz kernel's pair order (groups of 32
# token tiles) and the GEMM's tile order (groups of 16 row blocks). dz is
# rounded to bf16 and the
# results are stored in bf16, so the bar is the attention gradients': relative
# L2 <= 2e-2 over each tensor, and no row off by more than 10% of its norm.
BWD_CASES = CASES + [("three_chunks", 384, 17000, 128), ("partial_groups", 4500, 3000, 128)]
GRAD_RELL2, ROW_REL = 2e-2, 0.1


def _bwd_inputs(N, V, D, seed, dev):
    hb, wb, t, H, W, T = _inputs(N, V, D, seed, dev, ignored=[(3, -1), (N - 1, V)])
    mask = (synth.uint64s(seed, 53, N) % np.uint64(5) != 0).astype(np.float64)  # a loss mask, ~80% ones
    valid = (t >= 0) & (t < V)
    g = lce.upstream(mask * valid, "mean")
    return hb, wb, t, valid, g, H, W, T


def _bwd(H, W, T, g_np, train_head=True):
    N, D = H.shape
    _, lse, _ = _run(H, W, T)
    g = torch.from_numpy(g_np.astype(np.float32)).to(H.device)
    ws = torch.empty(pa.pa_lce_bwd_workspace_bytes(N, W.shape[0], D), dtype=torch.uint8, device=H.device)
    dh, dw = pa.linear_cross_entropy_backward(H, W, T, lse, g, train_head=train_head, ws=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(ws) == 0
    return dh, dw


def _check_grad(got, exp, name, zero_rows=None):
    """Relative L2 over the tensor; per row, the error against the row's norm
    plus a floor of the tensor's mean magnitude (rows of vocabulary entries
    with negligible probability are ~1e-40 in fp64 and 0 after fp32 exp);
    rows whose exact value is 0 by construction must be exactly 0."""
    g = got.float().cpu().numpy().astype(np.float64)
    D = exp.shape[1]
    rel = np.linalg.norm(g - exp) / np.linalg.norm(exp)
    row = np.linalg.norm(g - exp, axis=1) / (np.linalg.norm(exp, axis=1) + np.sqrt(D) * np.abs(exp).mean())
    print(f"{name}: relL2 {rel:.3e}, worst row {row.max():.3e}")
    assert rel <= GRAD_RELL2, (name, rel)
    assert row.max() <= ROW_REL, (name, float(row.max()), int(row.argmax()))
    if zero_rows is not None:
        assert np.all(g[zero_rows] == 0.0), name


@pytest.mark.parametrize("name,N,V,D", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_lce_backward_matches_oracle(name, N, V, D, cuda_dev):
    hb, wb, t, valid, g, H, W, T = _bwd_inputs(N, V, D, 80 + len(name), cuda_dev)
    dh, dw = _bwd(H, W, T, g)
    h64, w64 = synth.bf16_bits_to_f64(hb), synth.bf16_bits_to_f64(wb)
    e_dh, e_dw = lce.backward(h64, w64, np.where(valid, t, 0), g)
    _check_grad(dh, e_dh, f"{name} dH", zero_rows=(g == 0))  # masked and ignored tokens
    _check_grad(dw, e_dw, f"{name} dW")


def test_lce_backward_frozen_head_and_determinism(cuda_dev):
    """Without dhead the call computes the same dhidden, bit for bit, and two
    calls give the same bits."""
    _, _, _, _, g, H, W, T = _bwd_inputs(256, 17000, 128, 90, cuda_dev)
    dh1, dw1 = _bwd(H, W, T, g)
    dh2, dw2 = _bwd(H, W, T, g)
    dh3, dw3 = _bwd(H, W, T, g, train_head=False)
    assert dw3 is None
    assert torch.equal(dh1, dh2) and torch.equal(dw1, dw2) and torch.equal(dh1, dh3)
