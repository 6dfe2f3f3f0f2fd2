"""KVMem's tiered execution view on the GPU: the Mean-K index and the raw
history in pinned host memory, scoring in bounded layer tiles, and a pack
that reuses the blocks the previous step kept and reads the rest from host
memory.  Two consecutive agent steps (new query windows over the same
history) against the device-resident event (scores, kept lists and views
bit for bit) and the oracle (views of every packed unit: V bit-exact, K
within 1 bf16 ulp); the raw-K cache holds the kept blocks' raw keys; the
hit count equals the overlap of consecutive kept lists."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402
from helpers import check_rerope_k  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("stage_layers", [1, 3])
def test_tiered_steps_match_resident_and_oracle(kvc, orc, stage_layers):
    from query_conditioned_kv_gb300.event import MeanKEvent, TieredMeanKEvent
    cfg = W.scaled(W.config_8b(), L=5, L_pack=3, hist=[16384, 9216, 32768], budget=48)
    kraw, vraw = cfg.kv_raw(DEV)
    meank = cfg.meank_direct(DEV)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h = meank.cpu().pin_memory()
    kraw_h, vraw_h = kraw.cpu().pin_memory(), vraw.cpu().pin_memory()
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
            cfg.n_recent)
    kw = dict(L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0, device=DEV)
    res = MeanKEvent(*args, **kw)
    tie = TieredMeanKEvent(*args, stage_layers=stage_layers, **kw)
    toff = cfg.tok_off()
    kraw_b, vraw_b = _bits(kraw), _bits(vraw)
    prev = None
    for step in range(2):
        q = cfg.q(DEV, step=step)
        res.run_serial(q, meank, kraw, vraw)
        cur = tie.cur
        tie.n_hits.zero_()
        tie.step(q, meank_h, kraw_h, vraw_h)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(tie.dev_status) == 0
        assert torch.equal(tie.scores, res.scores)
        assert torch.equal(tie.kept_sets[cur], res.kept)
        assert torch.equal(tie.count_sets[cur], res.kept_count)
        assert torch.equal(tie.kview, res.kview)
        assert torch.equal(tie.vviews[cur], res.vview)
        kept = res.kept.cpu().numpy()[:cfg.lp].reshape(-1, cfg.budget)
        cnt = res.kept_count.cpu().numpy()[:cfg.lp].reshape(-1)
        # the oracle's views, and the raw keys the cache must hold
        kv_ref = np.zeros((cfg.lp, cfg.H, cfg.n_sess, cfg.view_tokens, cfg.D), np.uint16)
        vv_ref, raw = np.zeros_like(kv_ref), np.zeros_like(kv_ref)
        hits = 0
        for l in range(cfg.lp):
            for h in range(cfg.H):
                for r in range(cfg.n_sess):
                    s = (l * cfg.H + h) * cfg.n_sess + r
                    ku = kraw_b[l, h, toff[r]:toff[r + 1]]
                    vu = vraw_b[l, h, toff[r]:toff[r + 1]]
                    kv_ref[l, h, r], vv_ref[l, h, r] = orc.pack_unit(
                        ku, vu, kept[s], cnt[s], cfg.budget, cfg.pos0, cfg.theta)
                    for i in range(cnt[s]):
                        raw[l, h, r, 32 * i:32 * i + 32] = ku[32 * kept[s, i]:32 * kept[s, i] + 32]
                    if prev is not None:
                        hits += len(set(kept[s, :cnt[s]]) & set(prev[0][s, :prev[1][s]]))
        assert np.array_equal(_bits(tie.vviews[cur]), vv_ref)
        check_rerope_k(_bits(tie.kview), kv_ref, raw)
        assert np.array_equal(_bits(tie.kcaches[cur]), raw)
        assert int(tie.n_hits.item()) == hits
        if prev is not None:
            assert hits > 0  # consecutive steps share the planted blocks
        prev = (kept.copy(), cnt.copy())
