"""Pins of the oracle's LRFU keep score (ActKV §5.2, attention-aware LRFU,
Algorithm 1) against what the page states and what mathematics fixes:
the λ = 0 (recency) and λ = 1 (frequency) limits the page describes, the
hit set as the top-p mass set (closed forms: equal scores, one dominant
entry, geometric scores), brute force over every subset on tiny inputs, and
the decay of a score over steps.  Nothing here restates the oracle's loop."""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest


def test_equal_scores_take_the_first_p_fraction(orc):
    """n equal scores: the top-p set is the first ⌈p·n⌉ entries by index
    (ties rank by index); p·n = 6 exactly here."""
    ks, hits = orc.lrfu_update(np.ones(8, np.float32), np.zeros(8), p=0.75, lam=0.0)
    assert hits.tolist() == [True] * 6 + [False] * 2
    assert ks.tolist() == [1.0] * 6 + [0.0] * 2


def test_one_dominant_entry_is_the_only_hit(orc):
    s = np.array([0.2, 10.0, 0.3, 0.1, 0.4], np.float32)   # 10/11 > 0.9
    _, hits = orc.lrfu_update(s, np.zeros(5), p=0.9, lam=0.5)
    assert hits.tolist() == [False, True, False, False, False]


def test_geometric_scores_closed_form(orc):
    """s_i = 2^-i: the first m entries hold 2 − 2^(1−m) of the total
    2 − 2^(1−n); the hit count is the least m reaching p of it."""
    n, p = 20, 0.9
    s = np.array([2.0 ** -i for i in range(n)], np.float32)
    rng = np.random.default_rng(0)
    perm = rng.permutation(n)
    _, hits = orc.lrfu_update(s[perm], np.zeros(n), p=p, lam=0.0)
    total = 2.0 - 2.0 ** (1 - n)
    m = next(k for k in range(1, n + 1) if 2.0 - 2.0 ** (1 - k) >= p * total)
    assert int(hits.sum()) == m
    assert set(perm[hits].tolist()) == set(range(m))  # the m largest


def test_lambda_zero_is_recency(orc):
    """λ = 0: the keep score is the latest step's hit-gated score alone."""
    s = np.array([3.0, 1.0, 0.5, 0.25], np.float32)
    ks = np.array([100.0, 100.0, 100.0, 100.0], np.float32)
    ks, hits = orc.lrfu_update(s, ks, p=0.9, lam=0.0)
    # mass 4.75, target 4.275: 3 + 1 + 0.5 is the shortest prefix reaching it
    assert hits.tolist() == [True, True, True, False]
    assert ks.tolist() == [3.0, 1.0, 0.5, 0.0]


def test_lambda_one_is_frequency(orc):
    """λ = 1: the keep score sums every step's hit-gated scores (no decay)."""
    rng = np.random.default_rng(1)
    ks = np.zeros(12, np.float32)
    want = np.zeros(12)
    for _ in range(5):
        s = rng.integers(1, 9, 12).astype(np.float32)
        ks, hits = orc.lrfu_update(s, ks, p=0.9, lam=1.0)
        want += np.where(hits, s, 0.0)
    np.testing.assert_allclose(ks, want, rtol=0, atol=0)


def test_decay_over_two_steps(orc):
    """An entry hit at step 1 and missed at step 2 keeps λ·s₁; one hit at
    both keeps λ·s₁ + s₂ (scores chosen exactly representable)."""
    lam = 0.5
    s1 = np.array([4.0, 4.0, 0.0, 0.0], np.float32)
    s2 = np.array([0.0, 4.0, 4.0, 0.0], np.float32)
    ks, _ = orc.lrfu_update(s1, np.zeros(4), p=0.9, lam=lam)
    ks, _ = orc.lrfu_update(s2, ks, p=0.9, lam=lam)
    assert ks.tolist() == [2.0, 6.0, 4.0, 0.0]


def test_zero_mass_and_nan_are_never_hits(orc):
    s = np.array([0.0, -1.0, np.nan, 2.0, 0.0, np.inf], np.float32)
    ks, hits = orc.lrfu_update(s, np.ones(6), p=1.0, lam=0.25)
    assert hits.tolist() == [False, False, False, True, False, False]
    assert ks.tolist() == [0.25, 0.25, 0.25, 2.25, 0.25, 0.25]
    _, hits = orc.lrfu_update(np.zeros(4, np.float32), np.zeros(4), p=0.9, lam=0.5)
    assert not hits.any()


@pytest.mark.parametrize("seed", range(60))
def test_hit_set_is_the_smallest_mass_set_brute_force(orc, seed):
    """Over every subset: the hit set has the least size among subsets whose
    mass reaches p·total; among those of that size it has the largest mass,
    and equal scores rank by index."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 11))
    s = rng.choice(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 7.0], np.float32), n)
    p = float(rng.choice([0.5, 0.75, 0.9, 1.0]))
    _, hits = orc.lrfu_update(s, np.zeros(n), p=p, lam=0.5)
    total = float(s.astype(np.float64).sum())
    target = p * total
    best = None
    for size in range(0, n + 1):
        cands = [c for c in itertools.combinations(range(n), size)
                 if sum(float(s[i]) for i in c) >= target]
        if cands:
            best = size
            break
    if total == 0.0:
        assert not hits.any()
        return
    assert int(hits.sum()) == best
    got = tuple(np.nonzero(hits)[0].tolist())
    mass = sum(float(s[i]) for i in got)
    assert mass >= target - 1e-12
    top = sorted(range(n), key=lambda i: (-float(s[i]), i))[:best]
    assert sorted(top) == list(got)
    assert all(float(s[i]) > 0 for i in got)
    assert math.isclose(mass, sum(float(s[i]) for i in top))
