"""Pins of the fp64 linear cross-entropy oracle against things other than
itself (mlx-train-perf 0.5.1 README, "The fused cross-entropy loss": per-token
NLL, log-sum-exp and target logit of H W^T, and the gradients, without the
(N, V) logits in the fused kernel; the oracle builds them)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import linear_ce as lce

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _case(seed, N=7, D=5, V=11, scale=1.0):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D)) * scale
    W = rng.standard_normal((V, D)) * scale
    t = rng.integers(0, V, N)
    g = rng.standard_normal(N)
    return H, W, t, g


def test_hand_worked_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "linear_ce_hand_worked.json")))
    nll, lse, tgt = lce.forward(fx["H"], fx["W"], fx["targets"])
    np.testing.assert_allclose(nll, fx["nll"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, fx["lse"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(tgt, fx["target_logit"], rtol=0, atol=1e-15)
    dH, dW = lce.backward(fx["H"], fx["W"], fx["targets"], fx["g"])
    np.testing.assert_allclose(dH, fx["dH"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dW, fx["dW"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_torch_cross_entropy_float64(seed):
    H, W, t, g = _case(seed, scale=2.0)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = Ht @ Wt.T
    nll_t = torch.nn.functional.cross_entropy(z, torch.tensor(t), reduction="none")
    (nll_t * torch.tensor(g)).sum().backward()
    nll, lse, tgt = lce.forward(H, W, t)
    np.testing.assert_allclose(nll, nll_t.detach().numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(z, 1).detach().numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(tgt, z[torch.arange(len(t)), torch.tensor(t)].detach().numpy(), rtol=1e-13,
                               atol=1e-13)
    dH, dW = lce.backward(H, W, t, g)
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_finite_differences():
    H, W, t, g = _case(3, N=4, D=3, V=6)
    dH, dW = lce.backward(H, W, t, g)
    L = lambda H_, W_: float((g * lce.forward(H_, W_, t)[0]).sum())
    eps = 1e-6
    for (A, grad, which) in ((H, dH, 0), (W, dW, 1)):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            Ap, Am = A.copy(), A.copy()
            Ap[idx] += eps
            Am[idx] -= eps
            args_p = (Ap, W) if which == 0 else (H, Ap)
            args_m = (Am, W) if which == 0 else (H, Am)
            num[idx] = (L(*args_p) - L(*args_m)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_vocabulary_sum_of_dW_is_zero():
    """Each token's dz sums to zero over the vocabulary (softmax minus a
    one-hot), so the rows of dW sum to the zero vector."""
    H, W, t, g = _case(4, N=9, D=6, V=13)
    _, dW = lce.backward(H, W, t, g)
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-13)


def test_common_shift_of_head_rows():
    """Adding c to every row of W adds <H_i, c> to all of token i's logits:
    lse and the target logit move by it, the NLL does not."""
    H, W, t, _ = _case(5)
    c = np.random.default_rng(6).standard_normal(W.shape[1])
    nll0, lse0, tgt0 = lce.forward(H, W, t)
    nll1, lse1, tgt1 = lce.forward(H, W + c, t)
    np.testing.assert_allclose(nll1, nll0, atol=1e-12)
    np.testing.assert_allclose(lse1 - lse0, H @ c, atol=1e-12)
    np.testing.assert_allclose(tgt1 - tgt0, H @ c, atol=1e-12)


def test_uniform_logits():
    """Equal head rows: every logit of a token is the same, so the NLL is
    ln V, and dH = g (mean row - target row) = 0."""
    rng = np.random.default_rng(7)
    V, D = 17, 4
    H = rng.standard_normal((5, D))
    W = np.tile(rng.standard_normal(D), (V, 1))
    t = rng.integers(0, V, 5)
    nll, lse, tgt = lce.forward(H, W, t)
    np.testing.assert_allclose(nll, np.log(V), atol=1e-13)
    dH, _ = lce.backward(H, W, t, np.ones(5))
    np.testing.assert_allclose(dH, 0.0, atol=1e-13)


def test_chunked_logsumexp_combination():
    """The fused kernel's vocabulary tiling: per-chunk (max, sum of exp)
    merged with the running maximum gives the full log-sum-exp."""
    H, W, t, _ = _case(8, N=6, D=4, V=37, scale=3.0)
    _, lse, _ = lce.forward(H, W, t)
    z = lce.logits(H, W)
    m = np.full(z.shape[0], -np.inf)
    s = np.zeros(z.shape[0])
    for v0 in range(0, z.shape[1], 8):
        zc = z[:, v0:v0 + 8]
        mc = zc.max(axis=1)
        m_new = np.maximum(m, mc)
        s = s * np.exp(m - m_new) + np.exp(zc - m_new[:, None]).sum(axis=1)
        m = m_new
    np.testing.assert_allclose(m + np.log(s), lse, atol=1e-13)


def test_masked_mean_reduction():
    H, W, t, _ = _case(9)
    mask = np.array([1, 0, 1, 1, 0, 1, 0], dtype=np.float64)
    nll, _, _ = lce.forward(H, W, t)
    assert lce.loss(H, W, t, mask, "mean") == pytest.approx((nll * mask).sum() / mask.sum(), abs=1e-14)
    assert lce.loss(H, W, t, mask, "sum") == pytest.approx((nll * mask).sum(), abs=1e-14)
    dH, _ = lce.backward(H, W, t, lce.upstream(mask, "mean"))
    assert np.abs(dH[mask == 0]).max() == 0.0
