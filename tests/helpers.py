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
