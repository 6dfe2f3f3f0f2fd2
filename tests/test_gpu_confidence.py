"""ActKV's confidence monitor and adaptive budget on the GPU against the
oracle: token confidence over vocabularies from 7 to 151936 logits, top-k
from 1 to 64, ties at the k-th logit, a dominant logit (within 1e-5
relative: fp32 LSE); trace trend over ragged traces, short traces and
several window/stride/percentile settings (window counts and kept counts
exact, slope within fp64 rounding, budgets exact except slopes within
1e-12 of zero, which are counted)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def _rows(rng, V):
    rows = [rng.normal(0, 2, V), rng.normal(0, 0.1, V),
            rng.integers(-3, 4, V).astype(np.float64),          # ties everywhere
            np.where(np.arange(V) == V // 3, 30.0, rng.normal(0, 1, V)),
            np.full(V, -7.5)]
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("V,k", [(7, 1), (7, 7), (1000, 20), (151936, 20), (151936, 64),
                                 (50000, 1)])
def test_token_confidence_matches_oracle(kvc, orc, V, k):
    rng = np.random.default_rng(V + k)
    lg = _rows(rng, V)
    conf = torch.empty(len(lg), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_token_confidence(torch.from_numpy(lg).to(DEV), len(lg), V, k, conf, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    got = conf.cpu().numpy()
    for t in range(len(lg)):
        ref = orc.token_confidence(lg[t], k)
        assert abs(got[t] - ref) <= 1e-5 * max(abs(ref), 1.0), (t, got[t], ref)


@pytest.mark.parametrize("w,s,b", [(16, 4, 10.0), (1, 1, 50.0), (128, 32, 25.0),
                                   (64, 64, 100.0)])
def test_trend_and_budget_match_oracle(kvc, orc, w, s, b):
    rng = np.random.default_rng(w * 7 + s)
    lens = [0, 5, w, w + 1, 300, 2048, 5000, 777]
    traces = []
    for j, L in enumerate(lens):
        drift = rng.normal(0, 1.5)
        traces.append((rng.normal(10, 0.5, L) - drift * np.linspace(0, 1, L)).astype(np.float32))
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    conf = torch.from_numpy(np.concatenate(traces)).to(DEV)
    n = len(lens)
    slope = torch.empty(n, dtype=torch.float64, device=DEV)
    budget0 = np.array([512, 1024, 8000, 256, 4096, 128, 2048, 8192], np.int32)
    budget = torch.from_numpy(budget0.copy()).to(DEV)
    kept = torch.empty(n, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    b32 = float(np.float32(b))
    kvc.kvc_conf_trend_budget(conf, torch.from_numpy(off).to(DEV), n, max(lens), w, s, b32, 256,
                              8192, slope, budget, kept, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    got_s, got_b, got_k = slope.cpu().numpy(), budget.cpu().numpy(), kept.cpu().numpy()
    near = 0
    for t in range(n):
        ref_s, nw, nk = orc.conf_trend(traces[t].astype(np.float64), w, s, b32)
        assert got_k[t] == nk
        assert abs(got_s[t] - ref_s) <= 1e-9 * max(abs(ref_s), 1e-3), (t, got_s[t], ref_s)
        if abs(ref_s) < 1e-12 and ref_s != 0.0:
            near += 1
            continue
        assert got_b[t] == orc.adapt_budget(ref_s, int(budget0[t]), 256, 8192)
    print(f"near-zero slopes: {near}")
