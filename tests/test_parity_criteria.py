"""The parity criteria of the GPU tests, checked on the CPU: each accepts a
result at its bound and rejects one just past it, so a loose criterion cannot
hide a wrong kernel.  The "GPU" arrays here are the oracle-side values with a
planted error."""
from __future__ import annotations

import numpy as np
import pytest

from helpers import (assert_scores_close, bf16_ulp, check_rerope_k, f64, kth_gap,
                     mask_bits)


def _bits(x) -> np.ndarray:
    a = np.asarray(x, np.float32)
    b = a.view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def test_scores_accept_within_and_reject_past_the_relative_bound():
    rng = np.random.default_rng(0)
    ref = rng.uniform(1e-6, 1.0, 1000)
    assert_scores_close(ref * (1 + 0.9e-3), ref)
    assert_scores_close(ref * (1 - 0.9e-3), ref)
    bad = ref.copy()
    bad[417] *= 1 + 1.1e-3
    with pytest.raises(AssertionError):
        assert_scores_close(bad, ref)
    # an exact zero must come back as (essentially) zero
    z = np.zeros(4)
    assert_scores_close(z, z)
    with pytest.raises(AssertionError):
        assert_scores_close(np.array([0.0, 1e-20, 0.0, 0.0]), z)
    # two-dimensional outputs are checked element by element too
    with pytest.raises(AssertionError):
        assert_scores_close(bad.reshape(10, 100), ref.reshape(10, 100))


def test_bf16_ulp_is_the_spacing_at_the_value():
    for v, ulp in ((1.0, 2.0 ** -7), (1.5, 2.0 ** -7), (0.75, 2.0 ** -8), (-3.0, 2.0 ** -6),
                   (1024.0, 8.0)):
        assert bf16_ulp(np.array([v]))[0] == ulp
        # the next bf16 value above |v| is exactly one spacing away
        b = int(_bits([abs(v)])[0])
        assert f64(np.array([b + 1], np.uint16))[0] - abs(v) == ulp


def _rotated_case():
    # raw pairs (x_j, x_{j+D/2}) with D = 8: well-conditioned values, and in
    # column 1 a pair whose rotation nearly cancels
    raw = np.array([[1.0, 3.0, 0.5, -2.0, 2.0, 3.0, 0.25, 1.0]], np.float32)
    ref = np.array([[1.5, 1.0 / 64.0, -0.75, 2.5, -1.25, 4.0, 0.5, 3.0]], np.float32)
    return _bits(raw), _bits(ref)


def test_rerope_accepts_one_ulp_and_rejects_two():
    raw, ref = _rotated_case()
    one = ref.copy()
    one[0, 0] += 1  # 1.5 → next bf16: one ulp
    n_cancel, n_ulp1 = check_rerope_k(one, ref, raw)
    assert n_ulp1 == 1
    two = ref.copy()
    two[0, 0] += 2
    with pytest.raises(AssertionError):
        check_rerope_k(two, ref, raw)
    # a sign flip is far past any bound
    flip = ref.copy()
    flip[0, 2] ^= 0x8000
    with pytest.raises(AssertionError):
        check_rerope_k(flip, ref, raw)


def test_rerope_cancellation_clause():
    raw, ref = _rotated_case()
    # column 1: |ref| = 2^-6 < 2^-8 · (|3| + |3|), a cancelled value; its
    # bound is the larger of its ulp (2^-13) and 2^-16 · 6: one ulp passes,
    # two do not
    g = ref.copy()
    g[0, 1] += 1
    n_cancel, _ = check_rerope_k(g, ref, raw)
    assert n_cancel == 1
    g[0, 1] += 1
    with pytest.raises(AssertionError):
        check_rerope_k(g, ref, raw)
    # a cancelled value of zero: the bound is 2^-16 · (|x_j| + |x_{j+D/2}|)
    ref0 = ref.copy()
    ref0[0, 1] = 0
    small = ref0.copy()
    small[0, 1] = _bits([2.0 ** -16 * 4])[0]  # 2^-14 ≤ 2^-16 · 6
    check_rerope_k(small, ref0, raw)
    big = ref0.copy()
    big[0, 1] = _bits([2.0 ** -16 * 8])[0]  # 2^-13 > 2^-16 · 6
    with pytest.raises(AssertionError):
        check_rerope_k(big, ref0, raw)


def test_kth_gap_and_mask_bits():
    e = 2.0 ** -19
    s = np.array([9.0, 5.0, 4.0, 4.0 + e, 1.0, 7.0], np.float32)
    # budget 4, one sink, one recent: the free items are 5, 4, 4 + e, 1 and
    # k = 2, so the boundary lies between 4 + e and 4
    assert kth_gap(s, 4, 1, 1) == e / (4.0 + e)
    assert kth_gap(s, 6, 1, 1) is None
    m = np.array([0b1011, 1 << 31], np.uint32)
    got = mask_bits(m, 64)
    assert got[:4].tolist() == [True, True, False, True]
    assert got[63] and got.sum() == 4
