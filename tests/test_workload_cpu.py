"""The stack workload's selection bias: the stored beta reproduces its
calibration target with the oracle's routing (experts 0..25 take 50 +- 1 % of
the top-6 picks), and without the bias those experts get about their share."""
import os
import sys

import pytest

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))

import make_stack_bias as msb  # noqa: E402


@pytest.fixture(scope="module")
def cal():
    return msb.calibration_inputs()


def test_stored_beta_gives_half_the_picks(cal):
    x, router = cal
    beta = msb.read_beta()
    assert 0.0 < beta < 1.0
    assert abs(msb.biased_fraction(x, router, beta) - 0.5) <= 0.01


def test_without_bias_the_26_experts_get_about_their_share(cal):
    x, router = cal
    frac = msb.biased_fraction(x, router, 0.0)
    assert abs(frac - 26 / 256) < 0.03
