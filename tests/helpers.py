"""Shared test helpers: bf16 bit handling and the parity criteria.

Tolerances (the floating-point bar of the build):
  * scores, rule scores: |gpu − oracle| ≤ 1e-3·|oracle| (+1e-30 for values
    that underflow fp32);
  * re-RoPEd K: within 1 bf16 ulp of the oracle's once-rounded fp64
    rotation; where the rotated value cancels (|ref| < 2^-8·(|x_j| +
    |x_{j+D/2}|)) the bound is 2^-16·(|x_j| + |x_{j+D/2}|), and such cases
    are counted;
  * V, indices, counts, keep masks, slot maps, refcounts, free lists:
    bit-exact.
"""
from __future__ import annotations

import numpy as np

SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-30
NEAR_TIE_REL = 1e-5


def f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 at |v| (normal range)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 8)


def assert_scores_close(gpu, ref, what="scores"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    bound = SCORE_RTOL * np.abs(ref) + SCORE_ATOL
    bad = np.nonzero(err > bound)[0] if err.ndim == 1 else np.argwhere(err > bound)
    assert len(bad) == 0, (
        f"{what}: {len(bad)} of {err.size} outside 1e-3 rel; worst rel "
        f"{float(np.max(err / (np.abs(ref) + 1e-300))):.3e}")
    return float(np.max(err / (np.abs(ref) + 1e-300))) if err.size else 0.0


def check_rerope_k(gpu_bits, ref_bits, raw_bits):
    """K view vs oracle within 1 ulp; raw_bits are the gathered pre-RoPE
    rows aligned with the view ([..., D]).  Returns (n_cancel, n_ulp1)."""
    g = f64(gpu_bits)
    r = f64(ref_bits)
    x = f64(raw_bits)
    D = x.shape[-1]
    h = D // 2
    mag_half = np.abs(x[..., :h]) + np.abs(x[..., h:])
    mag = np.concatenate([mag_half, mag_half], axis=-1)
    err = np.abs(g - r)
    cancel = np.abs(r) < np.ldexp(mag, -8)
    bound = np.where(r != 0, bf16_ulp(r), 0.0)
    bound = np.where(cancel, np.maximum(bound, np.ldexp(mag, -16)), bound)
    bad = err > bound
    assert not np.any(bad), (
        f"re-RoPE K: {int(bad.sum())} elements beyond 1 ulp; first at "
        f"{np.argwhere(bad)[0].tolist()} gpu={g[bad][0]} ref={r[bad][0]}")
    return int(cancel.sum()), int(np.sum(err > 0))


def kth_gap(scores: np.ndarray, budget: int, n_sink: int, n_recent: int):
    """Relative gap between the k-th and (k+1)-th non-forced scores (the
    selection boundary); None when nothing is dropped."""
    n = len(scores)
    if n <= budget:
        return None
    k = budget - n_sink - n_recent
    idx = np.arange(n)
    free = scores[(idx >= n_sink) & (idx < n - n_recent)].astype(np.float64)
    if k <= 0 or k >= len(free):
        return None
    s = np.sort(free)[::-1]
    a, b = s[k - 1], s[k]
    return float(abs(a - b) / max(abs(a), 1e-300))


def mask_bits(mask_row: np.ndarray, n: int) -> np.ndarray:
    m = np.asarray(mask_row).view(np.uint32)
    i = np.arange(n)
    return ((m[i // 32] >> (i % 32).astype(np.uint32)) & 1).astype(bool)


# ---------------------------------------------------------------- Mean-K
# Hand-built 32-token columns for the Mean-K rounding cases, laid out so that
# each 8-column (16-byte) chunk is either entirely inside the fp32
# error-free-sum guards (columns 0..7: magnitudes within 2^-29 of each
# other, no zero next to a non-zero value; columns 16..23: all zeros) or
# entirely outside them (columns 8..15).  `MEANK_CLOSED_FORM` maps column →
# the bf16 bits of the exact mean.

def _bf16_bits_of(x: float) -> int:
    """bf16 bits of a value that bf16 represents exactly."""
    b = int(np.array([x], np.float32).view(np.uint32)[0])
    assert b & 0xFFFF == 0, f"{x} is not a bf16 value"
    return b >> 16


def _pairs(v: float, n: int):
    return [v, -v] * n


_T = 2.0 ** -26   # below half an fp32 ulp at 1 + 2^-8: fp32 drops it

MEANK_COLUMNS = {
    0: [0.75] * 32,
    # exact sum 1 + 2^-8 + 2^-25: fp32 rounds it onto the bf16 midpoint of
    # [1, 1 + 2^-7]; the exact value is above it → rounds up
    1: [1.0, 2.0 ** -8, _T, _T] + _pairs(2.0 ** -20, 14),
    # exact tie 1 + 2^-8 → round to even (1.0)
    2: [1.0, 2.0 ** -8] + _pairs(2.0 ** -20, 15),
    # exact sum 1 + 2^-8 − 2^-25: just below the midpoint → rounds down
    3: [1.0, 2.0 ** -8, -_T, -_T] + _pairs(2.0 ** -20, 14),
    # negated trap: −(1 + 2^-8 + 2^-25) → magnitude rounds up
    4: [-1.0, -(2.0 ** -8), -_T, -_T] + _pairs(2.0 ** -20, 14),
    5: [0.5] * 32,
    6: [-0.25] * 32,
    # exact cancellation to zero without a zero input: +0
    7: _pairs(1.0, 16),
    # a zero among non-zero values
    8: [1.5, 0.0] + [0.25] * 30,
    # a subnormal among normal values
    9: [1.0, float(np.float32(2.0 ** -130))] + [0.5] * 30,
    # huge magnitudes: the exact mean is 2^120
    10: [2.0 ** 120] * 32,
    # magnitudes spanning more than 34 binades: exact sum 1 + 2^-40
    11: [1.0, 2.0 ** -40] + _pairs(2.0 ** -20, 15),
    12: [1.0, float("nan")] + [0.5] * 30,
    13: [float("inf"), float("-inf")] + [0.5] * 30,
    14: [float("inf")] + [0.5] * 31,
    # sums beyond the fp32 range: mean of 32 × (2 − 2^-7)·2^127
    15: [(2.0 - 2.0 ** -7) * 2.0 ** 127] * 32,
}
for _c in range(16, 20):
    MEANK_COLUMNS[_c] = [0.0] * 32
for _c in range(20, 24):
    MEANK_COLUMNS[_c] = [-0.0] * 32

MEANK_CLOSED_FORM = {
    0: _bf16_bits_of(0.75),
    1: _bf16_bits_of((1.0 + 2.0 ** -7) / 32),
    2: _bf16_bits_of(1.0 / 32),
    3: _bf16_bits_of(1.0 / 32),
    4: _bf16_bits_of(-(1.0 + 2.0 ** -7) / 32),
    5: _bf16_bits_of(0.5),
    6: _bf16_bits_of(-0.25),
    7: 0x0000,
    8: _bf16_bits_of((1.5 + 30 * 0.25) / 32),
    9: _bf16_bits_of(0.5),   # (16 + 2^-130) / 32 rounds to 0.5
    10: _bf16_bits_of(2.0 ** 120),
    11: _bf16_bits_of(1.0 / 32),
    12: 0x7FC0,
    13: 0x7FC0,
    14: 0x7F80,
    15: _bf16_bits_of((2.0 - 2.0 ** -7) * 2.0 ** 127),
    16: 0x0000,
    20: 0x0000,   # +0 + (−0) = +0: the sum starts from +0
}


def meank_adversarial_kraw(n_blocks: int = 3, D: int = 128, seed: int = 0) -> np.ndarray:
    """bf16 bits [2][32·n_blocks][D]: row 0 block 0 holds MEANK_COLUMNS in
    columns 0..23; everything else is N(0,1)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, 32 * n_blocks, D)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)   # truncated to bf16
    for col, vals in MEANK_COLUMNS.items():
        assert len(vals) == 32, col
        for t, v in enumerate(vals):
            b = int(np.array([v], np.float32).view(np.uint32)[0])
            assert b & 0xFFFF == 0 or np.isnan(v), (col, t, v)
            bits[0, t, col] = b >> 16
    return bits
