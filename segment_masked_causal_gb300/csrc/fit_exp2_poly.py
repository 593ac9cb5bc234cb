"""Fit the cubic behind the FMA-pipe exp2 in sm103.cuh (ex2_fma2).

    python segment_masked_causal_gb300/csrc/fit_exp2_poly.py

Method. Cody and Waite's range reduction for base 2: x = n + f with
n = round(x) (an integer) and f in [-1/2, 1/2], so 2^x = 2^n * 2^f, and
2^n is an integer added to the exponent field. 2^f is approximated by
p(f) = 1 + c1 f + c2 f^2 + c3 f^3. The constant term is fixed at 1 so that
p(0) is exactly 1.0 and a clamped input of -127 gives exactly +0.0.

The coefficients minimise the largest relative error max |p(f) / 2^f - 1|
over a dense grid of [-1/2, 1/2]: the discrete Chebyshev (minimax)
approximation problem, solved as a linear program in (c1, c2, c3, delta):
minimise delta subject to |p(f_i) - 2^f_i| <= delta * 2^f_i at every grid
point. The coefficients are then rounded to fp32 and the whole fp32 recipe
(the kernel's steps, one rounding per operation) is evaluated over a grid of
inputs to bound its error.
"""
from __future__ import annotations

import numpy as np

GRID = 4097
MAGIC = np.float32(12582912.0)  # 1.5 * 2^23: adding it rounds to an integer


def fit(grid: int = GRID) -> tuple[np.ndarray, float]:
    """The minimax coefficients (c1, c2, c3) in fp64 and their error bound."""
    from scipy.optimize import linprog

    f = np.linspace(-0.5, 0.5, grid)
    e = np.exp2(f)
    A = np.stack([f, f * f, f ** 3], axis=1)
    # p - e <= d e and e - p <= d e, with p = 1 + A c
    a_ub = np.vstack([np.hstack([A, -e[:, None]]), np.hstack([-A, -e[:, None]])])
    b_ub = np.concatenate([e - 1.0, 1.0 - e])
    res = linprog(c=[0, 0, 0, 1], A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * 3 + [(0, None)],
                  method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:3], float(res.x[3])


def coefficients_f32() -> np.ndarray:
    """(c1, c2, c3) rounded to fp32, as the kernel holds them."""
    c, _ = fit()
    return c.astype(np.float32)


def _fma32(a: np.ndarray, b: np.ndarray, c: np.ndarray) -> np.ndarray:
    """a*b + c for fp32 operands: the product is exact in fp64, the sum is
    rounded to fp64 and then to fp32 (a fused multiply-add up to that rare
    double rounding)."""
    return (np.float64(1.0) * a * b + c).astype(np.float32)


def exp2_fp32(t: np.ndarray, c: np.ndarray) -> np.ndarray:
    """The kernel's fp32 recipe, step by step, on the host (float32 numpy)."""
    t = np.maximum(np.asarray(t, np.float32), np.float32(-127.0))
    u = (t + MAGIC).astype(np.float32)
    mn = (MAGIC - u).astype(np.float32)  # -n, exact
    f = (t + mn).astype(np.float32)
    c1, c2, c3 = (np.float32(v) for v in c)
    p = _fma32(np.full_like(f, c3), f, c2)
    p = _fma32(p, f, c1)
    p = _fma32(p, f, np.float32(1.0))
    bits = (p.view(np.uint32) + (u.view(np.uint32) << np.uint32(23))).astype(np.uint32)
    return bits.view(np.float32)


def max_rel_error(c: np.ndarray, lo: float = -126.0, hi: float = 8.0, n: int = 1 << 20) -> float:
    t = np.linspace(lo, hi, n).astype(np.float32)
    y = exp2_fp32(t, c).astype(np.float64)
    ref = np.exp2(t.astype(np.float64))
    return float(np.max(np.abs(y / ref - 1.0)))


if __name__ == "__main__":
    c64, delta = fit()
    c = c64.astype(np.float32)
    print("minimax relative error of the cubic (fp64 coefficients): %.3e" % delta)
    for i, v in enumerate(c, 1):
        print("c%d = %s  (%.9g)" % (i, float(v).hex(), v))
    print("fp32 recipe, max relative error on [-126, 8]: %.3e" % max_rel_error(c))
