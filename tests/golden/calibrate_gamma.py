"""Calibrate the planted query strength gamma of the 3 %-planted configs.

KVMem ("Query-conditioned retrieval") reports that the top-8 blocks of an
analysed window capture 66.5 % of the historical attention mass.  The
synthetic configs plant a direction u in 3 % of the blocks (alpha ~ U(2,4))
and add gamma·u to the query; this script bisects gamma, on the oracle's
Mean-K score of a fixed sample of (layer, KV head) units of the 8B-class
config, so that the mean top-8 share of the score mass is 0.65.

Run:  python tests/golden/calibrate_gamma.py
It prints the gamma that ``workloads.GAMMA_PLANTED`` holds (rounded to 0.5);
``tests/test_oracle_pins.py::test_gamma_calibration`` re-checks the share.
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as W  # noqa: E402

SAMPLE = [(0, 0), (1, 3), (5, 7), (9, 2), (17, 5), (22, 1), (30, 6), (35, 4)]
TARGET = 0.65


def top8_share(gamma: float, sample=SAMPLE) -> float:
    cfg = W.scaled(W.config_8b(), gamma=float(gamma))
    shares = []
    for l, h in sample:
        k = W.bf16_bits(cfg.kraw_unit(l, h, 0))
        mk = oracle.meank(k[None])[0]
        q = np.stack([W.bf16_bits(cfg.q_unit(0, l, h * cfg.G + g))
                      for g in range(cfg.G)])
        s = oracle.score_unit(q, mk).astype(np.float64)
        shares.append(np.sort(s)[::-1][:8].sum() / s.sum())
    return float(np.mean(shares))


def main() -> None:
    lo, hi = 20.0, 160.0
    for _ in range(12):
        mid = 0.5 * (lo + hi)
        if top8_share(mid) < TARGET:
            lo = mid
        else:
            hi = mid
    gamma = round(0.5 * (lo + hi) * 2) / 2
    print(f"gamma={gamma} share={top8_share(gamma):.4f}")


if __name__ == "__main__":
    main()
