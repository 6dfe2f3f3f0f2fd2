"""Pins of the oracle's confidence monitor and adaptive budget (ActKV §6.1,
§6.2 Algorithm 2) against closed forms, library routines and the rules the
page states: uniform logits give log V; a single high logit gives its closed
form; k = 1 is −log P_max; confidence is invariant to a logit shift; min
pooling on a hand example; the percentile equals numpy.percentile; the slope
equals numpy.polyfit on the kept windows; the budget rises only on a falling
trend and never falls."""
from __future__ import annotations

import math

import numpy as np
import pytest


def test_uniform_logits_give_log_v(orc):
    for V in (7, 1000, 151936):
        assert orc.token_confidence(np.full(V, 1.25, np.float32), k=20 if V >= 20 else 3) == \
            pytest.approx(math.log(V), rel=1e-13)


def test_single_high_logit_closed_form(orc):
    """logits (a, 0, …, 0): LSE = log(e^a + V − 1); the top k are a and k−1
    zeros, so C = LSE − a/k."""
    V, a, k = 5000, 9.0, 20
    lg = np.zeros(V, np.float32)
    lg[1234] = a
    lse = math.log(math.exp(a) + V - 1)
    assert orc.token_confidence(lg, k) == pytest.approx(lse - a / k, rel=1e-13)


def test_k_one_is_minus_log_pmax(orc):
    rng = np.random.default_rng(0)
    lg = rng.normal(0, 2, 4096).astype(np.float32)
    x = lg.astype(np.float64)
    lse = x.max() + math.log(np.exp(x - x.max()).sum())
    assert orc.token_confidence(lg, 1) == pytest.approx(lse - x.max(), rel=1e-12)


def test_confidence_is_shift_invariant_and_rises_with_a_dominant_token(orc):
    rng = np.random.default_rng(1)
    lg = (rng.integers(-40, 41, 2048) / 8).astype(np.float32)  # the shift below is exact
    c0 = orc.token_confidence(lg, 20)
    assert orc.token_confidence(lg + np.float32(64.0), 20) == pytest.approx(c0, rel=1e-12)
    # one token pulling away from the rest (the page's "peaked" case) raises
    # it: d/da [log(e^a + V − 1) − a/k] > 0 once e^a/(e^a + V − 1) > 1/k
    V, k = 2048, 20
    cs = []
    for a in (12.0, 16.0, 20.0):
        x = np.zeros(V, np.float32)
        x[7] = a
        cs.append(orc.token_confidence(x, k))
    assert cs[0] < cs[1] < cs[2]


def test_min_pooling_hand_example(orc):
    """w = 3, s = 2 over 8 values: windows [0,3) [2,5) [4,7); with b = 100
    every window is kept, so the slope is polyfit's over the three minima."""
    c = np.array([5, 4, 6, 3, 7, 2, 8, 9], np.float64)
    slope, nw, nk = orc.conf_trend(c, w=3, s=2, b=100.0)
    assert (nw, nk) == (3, 3)
    mins = [4.0, 3.0, 2.0]
    assert slope == pytest.approx(np.polyfit([0, 1, 2], mins, 1)[0], rel=1e-12)
    assert orc.conf_trend(c[:2], w=3, s=2, b=50.0) == (0.0, 0, 0)  # shorter than a window


@pytest.mark.parametrize("seed", range(20))
def test_percentile_and_slope_match_numpy(orc, seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(50, 600))
    w, s = int(rng.integers(1, 20)), int(rng.integers(1, 10))
    b = float(rng.choice([10.0, 25.0, 50.0, 90.0]))
    c = rng.normal(10, 1, L) - np.linspace(0, rng.normal(0, 2), L)
    slope, nw, nk = orc.conf_trend(c, w, s, b)
    if L < w:
        assert nw == 0
        return
    n = (L - w) // s + 1
    rp = np.array([c[m * s:m * s + w].min() for m in range(n)])
    q = np.percentile(rp, b)
    keep = np.nonzero(rp <= q)[0]
    assert (nw, nk) == (n, len(keep))
    if len(keep) >= 2:
        assert slope == pytest.approx(np.polyfit(keep, rp[keep], 1)[0], rel=1e-9, abs=1e-12)


def test_exact_line_and_constant(orc):
    c = 3.0 - 0.5 * np.arange(40, dtype=np.float64)
    assert orc.conf_trend(c, w=1, s=1, b=100.0)[0] == pytest.approx(-0.5, rel=1e-14)
    assert orc.conf_trend(np.full(40, 2.5), w=4, s=3, b=50.0)[0] == 0.0


def test_budget_rises_only_on_a_falling_trend(orc):
    assert orc.adapt_budget(-1e-6, 1024, 256, 8192) == 1280
    assert orc.adapt_budget(0.0, 1024, 256, 8192) == 1024     # flat: kept
    assert orc.adapt_budget(0.3, 1024, 256, 8192) == 1024     # recovering: never lowered
    assert orc.adapt_budget(-2.0, 8000, 256, 8192) == 8192    # capped
    # a budget already above the cap (the cap lowered between steps) is not cut
    assert orc.adapt_budget(-2.0, 9000, 256, 8192) == 9000
    b = 512
    for slope in (-1, 1, -1, -1, 0, 2, -1):
        nb = orc.adapt_budget(slope, b, 128, 4096)
        assert nb >= b and (nb > b) == (slope < 0)
        b = nb
