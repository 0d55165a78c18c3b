"""The pre-norm routing check of the GPU tests (tests/_common.py), on the CPU:
it accepts the oracle's routing, and a routing that another bf16 rounding of
an undecided normalised element gives; it rejects one that no such rounding
explains. The window NORM_REL is widened here so that a small case has
undecided elements."""
import numpy as np
import pytest

import synth
from oracle import moe

import _common
from _common import TINY, oracle_config, oracle_inputs


@pytest.fixture
def case(monkeypatch):
    monkeypatch.setattr(_common, "NORM_REL", 2.0 ** -14)
    d, seed, B = TINY, 3, 4
    x, router = oracle_inputs(d, seed, 0, B)
    r = x * 4.0
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(seed, 0, d["hidden"]))
    return d, r, gamma, router, oracle_config(d)


def test_undecided_elements_are_the_rounding_neighbours(case):
    d, r, gamma, router, cfg = case
    xn, alt = _common.prenorm_undecided(r, gamma, 1e-6)
    assert np.array_equal(xn, moe.rmsnorm(r, gamma, 1e-6))
    und = alt != xn
    assert 0 < und.sum() < und.size // 4
    # the alternative is the adjacent bf16 value on the other side of the boundary
    step = np.abs(alt[und] - xn[und])
    assert np.all(step > 0) and np.all(step <= np.abs(xn[und]) * 2.0 ** -7 + 1e-300)


def test_oracle_routing_passes_without_rerounding(case):
    d, r, gamma, router, cfg = case
    rt = moe.route(moe.rmsnorm(r, gamma, 1e-6), router, cfg)
    excluded, rerounded = _common.check_routing_prenorm(r, gamma, 1e-6, router, cfg, None, rt.idx, rt.w)
    assert rerounded == []


def _flipped_routing(case, decided):
    """A routing of token t with one element rounded the other way, chosen so
    that the weights move by more than W_TOL: an undecided element
    (decided=False) or a decided one moved by one bf16 step (decided=True)."""
    d, r, gamma, router, cfg = case
    xn, alt = _common.prenorm_undecided(r, gamma, 1e-6)
    base = moe.route(xn, router, cfg)
    for t in range(xn.shape[0]):
        cand = np.nonzero(alt[t] != xn[t])[0] if not decided else np.nonzero(alt[t] == xn[t])[0]
        for h in cand:
            row = xn[t].copy()
            # decided: the next bf16 value up, which no rounding of this element gives
            row[h] = alt[t, h] if not decided else moe.bf16_round(xn[t, h] * (1 + 2.0 ** -7))
            rt = moe.route(row[None, :], router, cfg)
            if rt.idx[0].tolist() == base.idx[t].tolist() and np.abs(rt.w[0] - base.w[t]).max() > 4 * _common.W_TOL:
                idx, w = base.idx.copy(), base.w.copy()
                idx[t], w[t] = rt.idx[0], rt.w[0]
                return t, idx, w
    pytest.skip("no element moves the weights by more than the tolerance")


def test_a_routing_from_the_other_rounding_passes(case):
    d, r, gamma, router, cfg = case
    t, idx, w = _flipped_routing(case, decided=False)
    excluded, rerounded = _common.check_routing_prenorm(r, gamma, 1e-6, router, cfg, None, idx, w)
    assert rerounded == [t]


def test_a_routing_no_rounding_explains_fails(case):
    d, r, gamma, router, cfg = case
    t, idx, w = _flipped_routing(case, decided=True)
    with pytest.raises(AssertionError):
        _common.check_routing_prenorm(r, gamma, 1e-6, router, cfg, None, idx, w)
    rt = moe.route(moe.rmsnorm(r, gamma, 1e-6), router, cfg)
    w2 = rt.w.copy()
    w2[0, 0] += np.float32(1e-5)  # a weight off by 1e-5 with the oracle's indices
    with pytest.raises(AssertionError):
        _common.check_routing_prenorm(r, gamma, 1e-6, router, cfg, None, rt.idx, w2)
