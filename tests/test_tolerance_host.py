"""The O bar used by the GPU parity tests (CPU): 1e-2 below |O| = 4 and
widened by the excess of bf16's half spacing above that."""
import numpy as np
import torch

from _gpu_common import O_MAXABS, check_o, o_tolerance


def test_bar_is_1e2_below_four():
    x = np.array([0.3, -1.5, 2.5, 3.99])
    assert np.all(o_tolerance(x) == O_MAXABS)


def test_bar_on_four_to_eight_adds_the_extra_half_spacing():
    # bf16 spacing on [4, 8) is 2^-5; half of it minus half the [2, 4) spacing is 2^-6 - 2^-7 = 2^-7
    x = np.array([4.0, 4.0172, 5.7, -4.171939, 7.99])
    assert np.allclose(o_tolerance(x), O_MAXABS + 2.0 ** -7)


def test_exactly_rounded_outputs_pass_and_one_step_off_fails():
    exact = np.random.default_rng(0).standard_normal(200000) * 2.5
    rounded = torch.tensor(exact, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert check_o(rounded, exact)[2]
    assert check_o(np.array([-4.03125]), np.array([-4.017232]))[2]   # the nearest bf16 of the exact value
    assert not check_o(np.array([4.0625]), np.array([4.0172]))[2]    # one more step away
    assert not check_o(np.array([1.0101]), np.array([1.0]))[2]
