"""The FMA-pipe exponential the forward can use for part of its keys
(ex2_fma2 in segment_masked_causal_gb300/csrc/sm103.cuh; the build option
PA_FWD_FMA_EX2_PAIRS, none by default), checked on the
host against the mathematics: the softmax weight exp(s - m) of the 0.5.1
README's "Packed attention" is 2^t with t = (s - m) log2 e, and the routine
must give 2^t to well within the bf16 rounding that P then takes (relative
2^-9).

The kernel's constants must be the fp32 rounding of the minimax fit that
fit_exp2_poly.py performs, and the kernel's fp32 steps, replayed in numpy,
must stay within the fit's error bound against fp64 exp2 over every input
the forward can pass (t in [-126, 8]), give exact powers of two at
integers, and give exactly +0.0 from -127 down to -inf."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "segment_masked_causal_gb300", "csrc")
sys.path.insert(0, CSRC)
import fit_exp2_poly as fit  # noqa: E402

pytest.importorskip("scipy")


def kernel_constants() -> np.ndarray:
    src = open(os.path.join(CSRC, "sm103.cuh")).read()
    vals = {k: float.fromhex(v) for k, v in re.findall(r"\b(kC[123]) = (0x[0-9a-fA-F.]+p[-+]?\d+)f", src)}
    assert sorted(vals) == ["kC1", "kC2", "kC3"], vals
    return np.array([vals["kC1"], vals["kC2"], vals["kC3"]], dtype=np.float32)


def test_constants_are_the_fit():
    c = kernel_constants()
    ref = fit.coefficients_f32()
    # the linear program's optimum, rounded to fp32; one ulp of slack for
    # solver round-off on another machine
    ulps = np.abs(c.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1, (c, ref)


def test_fit_is_near_taylor_and_beats_it():
    """The cubic is close to the Taylor coefficients ln2, ln2^2/2, ln2^3/6,
    and its worst relative error on [-1/2, 1/2] is several times smaller
    than the truncated Taylor series' (about 6e-4 at |f| = 1/2)."""
    c64, delta = fit.fit()
    l2 = np.log(2.0)
    taylor = np.array([l2, l2 ** 2 / 2, l2 ** 3 / 6])
    assert np.allclose(c64, taylor, rtol=0.05)
    f = np.linspace(-0.5, 0.5, 10001)
    e = np.exp2(f)
    err = lambda cc: np.max(np.abs((1 + cc[0] * f + cc[1] * f * f + cc[2] * f ** 3) / e - 1))
    assert err(c64) <= 1.02 * delta
    assert err(taylor) > 4 * delta
    assert 5e-5 < delta < 1.2e-4


def test_recipe_error_bound():
    c = kernel_constants()
    assert fit.max_rel_error(c) <= 1.05e-4
    # well inside bf16's relative rounding step, which P takes next
    assert fit.max_rel_error(c) < 2.0 ** -9 / 10


def test_integers_are_exact_powers_of_two():
    c = kernel_constants()
    n = np.arange(-126, 9, dtype=np.float32)
    y = fit.exp2_fp32(n, c).astype(np.float64)
    assert np.array_equal(y, np.exp2(n.astype(np.float64)))


def test_clamp_gives_exact_zero():
    c = kernel_constants()
    x = np.array([-np.inf, -1e30, -300.0, -128.0, -127.5, -127.0], dtype=np.float32)
    y = fit.exp2_fp32(x, c)
    assert np.all(y.view(np.uint32) == 0), y


def test_below_the_normal_range_is_tiny_and_non_negative():
    c = kernel_constants()
    x = np.linspace(-127.0, -126.0, 4097, dtype=np.float32)
    y = fit.exp2_fp32(x, c).astype(np.float64)
    assert np.all(y >= 0) and np.all(y < 2.0 ** -125)


def test_monotone_on_a_fine_grid():
    """Softmax weights must keep the scores' order: checked over one binade
    step by step and across integer boundaries."""
    c = kernel_constants()
    x = np.linspace(-20.0, 8.0, 1 << 18, dtype=np.float32)
    y = fit.exp2_fp32(x, c)
    assert np.all(np.diff(y.astype(np.float64)) >= 0)
