"""GPU Mean-K build on hand-built columns: the fp32 error-free sum and its
midpoint correction (columns 0..7), the fp64 fallback for columns outside
its guards (8..15), all bit-exact against the oracle and the closed forms."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402
from helpers import MEANK_CLOSED_FORM, meank_adversarial_kraw  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


@pytest.mark.parametrize("D", [128, 64])
def test_meank_rounding_cases_bit_exact(kvc, orc, D):
    kraw = meank_adversarial_kraw(n_blocks=5, D=D, seed=D)
    rows, n_tok = kraw.shape[0], kraw.shape[1]
    kr = W.from_bits(kraw, DEV)
    mk = torch.empty(rows, n_tok // 32, D, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_build_meank(kr, mk, 1, rows, D, n_tok, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    got = W.bf16_bits(mk)
    ref = orc.meank(kraw)
    bad = np.argwhere(got != ref)
    assert len(bad) == 0, f"{len(bad)} Mean-K elements differ; first {bad[:4].tolist()}"
    for col, want in MEANK_CLOSED_FORM.items():
        assert int(got[0, 0, col]) == want, col
