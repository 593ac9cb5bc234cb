"""fp64 restatement of the fused linear cross-entropy loss (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the tests may import this module; the library
never calls it and shares no code with it.

What it computes (mlx-train-perf 0.5.1 README, "The fused cross-entropy loss"
and "If you maintain a trainer"): the cross-entropy of next-token targets
under logits z = H W^T, where H (N, D) holds the final hidden states and the
head W (V, D) one row per vocabulary entry. The fused kernel returns three
length-N arrays -- the per-token NLL, the log-sum-exp and the target logit --
and a gradient back into the hidden states; it never stores the (N, V)
logits. This oracle is the plain definition and does build them (in fp64),
which is what makes it obviously correct:

    z_iv      = <H_i, W_v>
    lse_i     = log sum_v exp(z_iv)
    tgt_i     = z_{i, t_i}
    nll_i     = lse_i - tgt_i
    dz_iv     = g_i (softmax(z_i)_v - [v == t_i])      for an upstream g_i = dL/dnll_i
    dH_i      = sum_v dz_iv W_v
    dW_v      = sum_i dz_iv H_i

Readings: the head has no bias (a dense or tied head); a loss mask (the
packer's supervision mask) enters only through g, as g_i = mask_i / count for
reduction "mean" and g_i = mask_i for "sum".

Pins: tests/test_linear_ce_oracle.py (a hand-worked fixture, torch float64
cross_entropy with autograd, central finite differences, the zero vocabulary
sum of dW, invariance of the NLL under a common shift of the head's rows,
uniform logits, and the chunked log-sum-exp combination).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def logits(H, W) -> np.ndarray:
    return _f64(H) @ _f64(W).T


def forward(H, W, targets):
    """(nll, lse, target_logit), each (N,) fp64."""
    z = logits(H, W)
    m = z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
    t = np.asarray(targets, dtype=np.int64)
    tgt = z[np.arange(z.shape[0]), t]
    return lse - tgt, lse, tgt


def upstream(mask, reduction: str = "mean") -> np.ndarray:
    """g_i = dL/dnll_i for a masked reduction of the per-token NLL."""
    m = _f64(mask)
    if reduction == "mean":
        return m / max(m.sum(), 1.0)
    if reduction == "sum":
        return m
    raise ValueError(reduction)


def loss(H, W, targets, mask, reduction: str = "mean") -> float:
    nll, _, _ = forward(H, W, targets)
    return float((upstream(mask, reduction) * nll).sum())


def backward(H, W, targets, g):
    """(dH (N, D), dW (V, D)) of L = sum_i g_i nll_i."""
    z = logits(H, W)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    t = np.asarray(targets, dtype=np.int64)
    dz = p
    dz[np.arange(z.shape[0]), t] -= 1.0
    dz *= _f64(g)[:, None]
    return dz @ _f64(W), dz.T @ _f64(H)
