"""The oracle's Mean-K rounding on hand-built columns whose exact mean is
known in closed form: midpoint ties, values just off a midpoint, signed
zeros, NaN, infinities and fp32-overflowing sums.  The oracle reads the
mean as the exact sum ÷ 32 rounded once to bf16 (KVMem, "Query-conditioned
retrieval")."""
from __future__ import annotations

import numpy as np

from helpers import MEANK_CLOSED_FORM, meank_adversarial_kraw


def test_oracle_meank_closed_forms(orc):
    kraw = meank_adversarial_kraw()
    mk = orc.meank(kraw)
    for col, want in MEANK_CLOSED_FORM.items():
        assert int(mk[0, 0, col]) == want, (col, hex(int(mk[0, 0, col])), hex(want))
