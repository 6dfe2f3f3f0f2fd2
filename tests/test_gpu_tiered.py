"""KVMem's tiered execution view on the GPU: the Mean-K index and the raw
history in pinned host memory, scoring in bounded layer tiles, and a pack
that reuses the blocks the previous step kept and reads the rest from host
memory.  Two consecutive agent steps (new query windows over the same
history):
* scores bit for bit equal to the device-resident event's (the same
  kernel, and a unit's partial sums merge in one order whatever else the
  launch holds);
* kept lists bit for bit against the oracle's selection on the tiered
  scores;
* views bit for bit against the resident pack of the same kept lists, and
  against the oracle (V bit-exact, K within 1 bf16 ulp);
* the raw-K cache holds the kept blocks' raw keys, and the hit count equals
  the overlap of consecutive kept lists."""
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
        cur = tie.cur
        tie.n_hits.zero_()
        tie.step(q, meank_h, kraw_h, vraw_h)
        res.score(q, meank)
        # the resident pack of the tiered kept lists: the same views bit for bit
        res.pack(kraw, vraw, kept=tie.kept_sets[cur], kept_count=tie.count_sets[cur])
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(tie.dev_status) == 0
        assert kvc.kvc_device_status(res.dev_status) == 0
        assert torch.equal(tie.scores, res.scores)  # a unit's sums merge in one order
        assert torch.equal(tie.kview, res.kview)
        assert torch.equal(tie.vviews[cur], res.vview)
        # kept lists: the oracle's selection on the tiered scores
        sc = tie.scores.cpu().numpy().reshape(-1)
        kref, cref, _ = orc.select_segments(sc, cfg.seg_off(), cfg.budget, cfg.n_sink,
                                            cfg.n_recent)
        assert np.array_equal(tie.kept_sets[cur].cpu().numpy().reshape(-1, cfg.budget), kref)
        assert np.array_equal(tie.count_sets[cur].cpu().numpy().reshape(-1), cref)
        kept = kref[:cfg.lp * cfg.H * cfg.n_sess]
        cnt = cref[:cfg.lp * cfg.H * cfg.n_sess]
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


def test_tiered_full_size_8b(kvc, orc):
    """The 8B-class 128K workload as bench.py times it (4-layer tiles, two
    steps with consecutive query windows): scores, kept lists and views bit
    for bit against the device-resident event; sampled units' views against
    the oracle; the raw-K cache of those units."""
    from query_conditioned_kv_gb300.event import MeanKEvent, TieredMeanKEvent
    cfg = W.config_8b()
    kraw, vraw = cfg.kv_raw(DEV)
    meank = cfg.meank_direct(DEV)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h = meank.cpu().pin_memory()
    kraw_h, vraw_h = kraw.cpu().pin_memory(), vraw.cpu().pin_memory()
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
            cfg.n_recent)
    kw = dict(L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0, device=DEV)
    res = MeanKEvent(*args, **kw)
    tie = TieredMeanKEvent(*args, stage_layers=4, **kw)
    for step in range(2):
        q = cfg.q(DEV, step=step)
        cur = tie.cur
        tie.step(q, meank_h, kraw_h, vraw_h)
        res.score(q, meank)
        res.pack(kraw, vraw, kept=tie.kept_sets[cur], kept_count=tie.count_sets[cur])
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(tie.dev_status) == 0
        assert kvc.kvc_device_status(res.dev_status) == 0
        assert torch.equal(tie.scores, res.scores)  # a unit's sums merge in one order
        assert torch.equal(tie.kview, res.kview)
        assert torch.equal(tie.vviews[cur], res.vview)
        kept = tie.kept_sets[cur].cpu().numpy()
        cnt = tie.count_sets[cur].cpu().numpy()
        sc = tie.scores.cpu().numpy()
        for (l, h) in ((0, 0), (cfg.lp - 1, cfg.H - 1)):
            kref, cref, _ = orc.select(sc[l, h], cfg.budget, cfg.n_sink, cfg.n_recent)
            assert cref == cnt[l, h, 0] and np.array_equal(kept[l, h, 0], kref)
            ku = _bits(kraw[l, h])
            vu = _bits(vraw[l, h])
            kv_ref, vv_ref = orc.pack_unit(ku, vu, kept[l, h, 0], cnt[l, h, 0], cfg.budget,
                                           cfg.pos0, cfg.theta)
            raw = np.zeros_like(kv_ref)
            for i in range(cnt[l, h, 0]):
                b = kept[l, h, 0, i]
                raw[32 * i:32 * i + 32] = ku[32 * b:32 * b + 32]
            assert np.array_equal(_bits(tie.vviews[cur][l, h, 0]), vv_ref)
            check_rerope_k(_bits(tie.kview[l, h, 0]), kv_ref, raw)
            assert np.array_equal(_bits(tie.kcaches[cur][l, h, 0]), raw)


def test_repository_view_matches_tiered(kvc, tmp_path):
    """KVMem's repository view: the packed layers' raw history in a backing
    file, one unit per (layer, head, block), with 64 fewer host slots than
    units (the last layer and head's recent blocks, kept by every step, start
    out on file only), so units move between the file and host RAM.  Three steps' views, raw-K caches and hit
    counts bit for bit equal to TieredMeanKEvent's (whole history pinned in
    host memory); the repository's counters agree with its plans."""
    from query_conditioned_kv_gb300.event import RepoTieredEvent, TieredMeanKEvent
    cfg = W.scaled(W.config_8b(), L=4, L_pack=2, hist=[16384, 9216, 32768], budget=48)
    kraw, vraw = cfg.kv_raw(DEV)
    meank = cfg.meank_direct(DEV)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h = meank.cpu().pin_memory()
    kraw_h, vraw_h = kraw.cpu().pin_memory(), vraw.cpu().pin_memory()
    n_blocks = cfg.n_tok // 32
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
            cfg.n_recent)
    kw = dict(L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0, device=DEV)
    tie = TieredMeanKEvent(*args, stage_layers=2, **kw)
    n_units = cfg.lp * cfg.H * n_blocks
    repo = kvc.KvcRepo(tmp_path / "hist.bin", n_blocks, cfg.lp, cfg.H, cfg.D,
                       n_slots=n_units - 64, io_threads=4)
    repo.put(0, n_blocks, kraw_h, vraw_h, cfg.n_tok)
    assert repo.where(n_units - 1) == 2
    rep = RepoTieredEvent(*args, stage_layers=2, repo=repo, **kw)
    missed = 0
    for step in range(3):
        q = cfg.q(DEV, step=step)
        cur = tie.cur
        tie.n_hits.zero_()
        rep.n_hits.zero_()
        tie.step(q, meank_h, kraw_h, vraw_h)
        rep.step(q, meank_h)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(tie.dev_status) == 0
        assert kvc.kvc_device_status(rep.dev_status) == 0
        assert torch.equal(rep.kept_sets[cur], tie.kept_sets[cur])
        assert torch.equal(rep.kview, tie.kview)
        assert torch.equal(rep.vviews[cur], tie.vviews[cur])
        assert torch.equal(rep.kcaches[cur], tie.kcaches[cur])
        assert int(rep.n_hits.item()) == int(tie.n_hits.item())
        n_used, n_need = rep.last_plan
        assert 0 < n_need <= n_used
        missed += n_need
        assert repo.where(n_units - 1) == 1  # a recent block: kept, so in host RAM
    st = repo.stats()
    assert st["steps"] == 3 and st["needed"] == missed
    assert st["fetched"] > 0 and st["evictions"] > 0
    assert st["bytes_read"] == st["fetched"] * repo.slot_elems * 2
    repo.close()


def test_slots_pack_refuses_a_missing_slot(kvc, tmp_path):
    """A missed block without a host slot is recorded as KVC_ERR_BOUNDS on
    the device and packed as zeros, not read from a wrong address."""
    cfg = W.scaled(W.config_8b(), L=1, L_pack=1, hist=[4096], budget=16)
    from query_conditioned_kv_gb300.event import MeanKEvent
    kraw, vraw = cfg.kv_raw(DEV)
    meank = cfg.meank_direct(DEV)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
            cfg.n_recent)
    ev = MeanKEvent(*args, L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0, device=DEV)
    ev.score(cfg.q(DEV), meank)
    ev.select()
    n_blocks = cfg.n_tok // 32
    repo = kvc.KvcRepo(tmp_path / "m.bin", n_blocks, cfg.lp, cfg.H, cfg.D, n_slots=4)
    slots = torch.full((repo.n_units,), -1, dtype=torch.int32, device=DEV)
    kcache = torch.empty_like(ev.kview)
    ev.kview.fill_(1)
    ks, vs = repo.slots()
    kvc.kvc_pack_tiered_slots(ks, vs, repo.slot_elems, repo.n_slots, slots, None, None, None,
                              None, ev.kept, ev.kept_count, cfg.lp, cfg.H, cfg.D, ev.tok_off,
                              ev.n_sess, ev.n_tok, ev.budget, ev.rope_tab, kcache, ev.kview,
                              ev.vview, None, ev.dev_status)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 7
    assert int(ev.kview.abs().max().item()) == 0
    repo.close()
