"""Full-size parity: every workload at its benchmark size, run the way a user
runs the event (the launch configuration bench.py times for the 8B-class
event).  Outputs the oracle can compute unit by unit are checked on a sample
of units against the oracle; properties that hold at any size are checked on
every unit: kept counts, chronological order and the forced set, V views bit-
exact against a gather of the raw V, slot maps / refcounts / free list
bit-exact against the oracle's redirect of the same keep mask.

Memory: each test frees what it allocated (the 1M-token and ragged configs
hold 80–210 GB while they run)."""
from __future__ import annotations

import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402
from helpers import (NEAR_TIE_REL, assert_scores_close, check_rerope_k,  # noqa: E402
                     kth_gap)

DEV = "cuda"


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def _bits(t):
    return W.bf16_bits(t)


def _check_selection_properties(kept, cnt, nb, budget, n_sink, n_recent):
    """kept [n][budget] (device), cnt [n]; every segment has nb[s] items."""
    kept = kept.reshape(-1, budget)
    cnt = cnt.reshape(-1)
    nb = torch.as_tensor(nb, device=kept.device).reshape(-1)
    want = torch.minimum(nb, torch.full_like(nb, budget))
    assert torch.equal(cnt.to(torch.int64), want.to(torch.int64)), "kept counts"
    idx = torch.arange(budget, device=kept.device)[None, :]
    live = idx < cnt[:, None]
    k = kept.to(torch.int64)
    assert torch.all(k[~live] == -1)
    inc = (k[:, 1:] > k[:, :-1]) | ~live[:, 1:]
    assert torch.all(inc), "chronological order"
    assert torch.all((k >= 0)[live]) and torch.all((k < nb[:, None])[live])
    full = cnt == budget
    if n_sink:
        assert torch.all(k[full, 0] == 0), "sink block kept"
    if n_recent:
        last = (nb[full, None] - n_recent + torch.arange(n_recent, device=k.device)[None, :])
        assert torch.equal(k[full, budget - n_recent:], last), "recent blocks kept"


def _check_v_views(vview, vraw, kept, cnt, tok_off, budget):
    """Every V view equals the gather of the raw V rows of its kept blocks."""
    Lp, H, n_sess, V, D = vview.shape
    ar = torch.arange(32, device=vview.device)
    for l in range(Lp):
        for r in range(n_sess):
            k = kept[l, :, r].to(torch.int64)                       # [H][budget]
            c = cnt[l, :, r]
            src = (k[:, :, None] * 32 + ar[None, None, :]).reshape(H, -1) + int(tok_off[r])
            valid = (torch.arange(budget, device=k.device)[None, :] < c[:, None])
            valid = valid[:, :, None].expand(H, budget, 32).reshape(H, -1)
            src = torch.where(valid, src, torch.zeros_like(src))
            g = torch.gather(vraw[l], 1, src[:, :, None].expand(H, V, D))
            g = torch.where(valid[:, :, None], g, torch.zeros_like(g))
            assert torch.equal(g, vview[l, :, r]), f"V view layer {l} session {r}"


def _oracle_unit(orc, cfg, q, meank, kraw, vraw, ev, l, h, r, meank_bits=None):
    """Oracle score / select / pack of one unit vs the GPU's."""
    boff, toff = cfg.blk_off(), cfg.tok_off()
    b0, b1 = int(boff[r]), int(boff[r + 1])
    t0, t1 = int(toff[r]), int(toff[r + 1])
    qrows = _bits(q[l, r, h * cfg.G:(h + 1) * cfg.G])
    if l < cfg.lp:
        ku = _bits(kraw[l, h, t0:t1])
        mk = orc.meank(ku[None])[0]
        assert np.array_equal(_bits(meank[l, h, b0:b1]), mk), "Mean-K"
    else:
        mk = _bits(meank[l, h, b0:b1]) if meank_bits is None else meank_bits
    s_ref = orc.score_unit(qrows, mk)
    s_gpu = ev.scores[l, h, b0:b1].cpu().numpy()
    assert_scores_close(s_gpu, s_ref, f"scores l{l} h{h} r{r}")
    k_ref, c_ref, _ = orc.select(s_ref, cfg.budget, cfg.n_sink, cfg.n_recent)
    k_gpu = ev.kept[l, h, r].cpu().numpy()
    near = 0
    if not np.array_equal(k_gpu, k_ref):
        gap = kth_gap(s_ref, cfg.budget, cfg.n_sink, cfg.n_recent)
        assert gap is not None and gap < NEAR_TIE_REL, f"kept l{l} h{h} r{r} gap {gap}"
        near = 1
    if l < cfg.lp:
        vu = _bits(vraw[l, h, t0:t1])
        kv_ref, vv_ref = orc.pack_unit(ku, vu, k_gpu, int(ev.kept_count[l, h, r]), cfg.budget,
                                       cfg.pos0, cfg.theta)
        assert np.array_equal(_bits(ev.vview[l, h, r]), vv_ref)
        cnt = int(ev.kept_count[l, h, r])
        raw = np.zeros_like(kv_ref)
        for i in range(cnt):
            raw[32 * i:32 * i + 32] = ku[32 * k_gpu[i]:32 * k_gpu[i] + 32]
        check_rerope_k(_bits(ev.kview[l, h, r]), kv_ref, raw)
    return near


def _meank_event(kvc, cfg):
    from query_conditioned_kv_gb300.event import MeanKEvent
    q = cfg.q(DEV)
    kraw, vraw = cfg.kv_raw(DEV)
    meank = cfg.meank_direct(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_build_meank(kraw, meank[:cfg.lp], cfg.lp, cfg.H, cfg.D, cfg.n_tok, st)
    ev = MeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                    cfg.n_recent, cfg.lp, cfg.theta, cfg.pos0, device=DEV)
    ev.run(q, meank, kraw, vraw)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    assert kvc.kvc_device_status(ev.dev_status) == 0
    return q, kraw, vraw, meank, ev


def _nb_per_segment(cfg):
    nb = np.asarray(cfg.nb, dtype=np.int64)
    return np.broadcast_to(nb[None, None, :], (cfg.L, cfg.H, cfg.n_sess)).copy()


def test_fullsize_8b_128k_event(kvc, orc):
    """The benchmarked event: 36 layers × 8 KV heads × 131072 tokens."""
    cfg = W.config_8b()
    q, kraw, vraw, meank, ev = _meank_event(kvc, cfg)
    _check_selection_properties(ev.kept, ev.kept_count, _nb_per_segment(cfg), cfg.budget,
                                cfg.n_sink, cfg.n_recent)
    _check_v_views(ev.vview, vraw, ev.kept, ev.kept_count, cfg.tok_off(), cfg.budget)
    sample = [(0, 0), (5, 3), (11, 6), (17, 5), (22, 1), (28, 4), (31, 2), (35, 7)]
    near = sum(_oracle_unit(orc, cfg, q, meank, kraw, vraw, ev, l, h, 0) for l, h in sample)
    print(f"8b_128k: near-tie units {near} of {len(sample)} sampled")


def test_fullsize_27b_1m_event(kvc, orc):
    """1M-token workspace, 64 layers scored (Mean-K index device-resident),
    16 layers packed (2048-block views)."""
    cfg = W.config_27b()
    q, kraw, vraw, meank, ev = _meank_event(kvc, cfg)
    _check_selection_properties(ev.kept, ev.kept_count, _nb_per_segment(cfg), cfg.budget,
                                cfg.n_sink, cfg.n_recent)
    _check_v_views(ev.vview, vraw, ev.kept, ev.kept_count, cfg.tok_off(), cfg.budget)
    # 8 of the 512 units: packed layers (< 16) and scored-only ones, the
    # first and last layer, every KV head position of a cluster schedule
    sample = [(0, 0), (3, 2), (15, 7), (16, 1), (29, 4), (40, 6), (52, 3), (63, 5)]
    near = sum(_oracle_unit(orc, cfg, q, meank, kraw, vraw, ev, l, h, 0) for l, h in sample)
    print(f"27b_1m: near-tie units {near} of {len(sample)} sampled")


def test_fullsize_ragged_128_event(kvc, orc):
    """128 ragged sessions (16K–256K tokens), 36 layers scored, 2 packed."""
    cfg = W.config_ragged()
    q, kraw, vraw, meank, ev = _meank_event(kvc, cfg)
    _check_selection_properties(ev.kept, ev.kept_count, _nb_per_segment(cfg), cfg.budget,
                                cfg.n_sink, cfg.n_recent)
    _check_v_views(ev.vview, vraw, ev.kept, ev.kept_count, cfg.tok_off(), cfg.budget)
    shortest = int(np.argmin(cfg.hist))
    longest = int(np.argmax(cfg.hist))
    # 8 of the 128 sessions, the shortest and the longest among them; packed
    # units (layers 0 and 1) and scored-only ones
    sample = [(0, 1, shortest), (1, 6, longest), (20, 3, 57), (0, 4, 9), (35, 0, 100),
              (1, 2, 127), (12, 7, 33), (27, 5, 76)]
    near = sum(_oracle_unit(orc, cfg, q, meank, kraw, vraw, ev, l, h, r) for l, h, r in sample)
    print(f"ragged_128: sessions {cfg.n_sess}, tokens {cfg.n_tok}, near-tie units {near} "
          f"of {len(sample)} sampled")


def test_fullsize_slotmap_64x32k_event(kvc, orc):
    """64 sessions × 32768 positions over a refcounted shared prefix:
    QueryMemory over 4 turns, rule score, select, redirect + free."""
    from query_conditioned_kv_gb300.event import SlotMapEvent
    cfg = W.config_slotmap()
    sm = cfg.slot_maps()
    rc = cfg.refcounts(sm)
    kp = torch.empty(cfg.L, cfg.n_slots, cfg.H, cfg.D, dtype=torch.bfloat16, device=DEV)
    for l in range(cfg.L):
        kp[l] = cfg.kpool_layer(l, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = torch.zeros(cfg.n_sess, cfg.L, cfg.Hq, cfg.D, dtype=torch.float32, device=DEV)
    for t in range(cfg.turns):
        qt = cfg.q_turn(t, DEV)
        kvc.kvc_qmem_update(M, qt, cfg.n_sess, cfg.L, cfg.Hq, cfg.D, cfg.T, cfg.decay, cfg.gain, 1)
        del qt
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots, cfg.budget,
                      cfg.prefix, cfg.sentinel, device=DEV)
    sm_d = torch.from_numpy(sm).to(DEV)
    rc_d = torch.from_numpy(rc).to(DEV)
    ev.run(M, kp, sm_d, rc_d)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    rule = ev.rule
    # every live position's rule mass sums to L·Hq per session
    sums = rule.to(torch.float64).sum(dim=1)
    assert torch.allclose(sums, torch.full_like(sums, cfg.L * cfg.Hq), rtol=1e-3)
    # 4 of the 64 sessions against the oracle: two fixed ones, and two chosen
    # by their drop pattern — the session that drops the most shared-prefix
    # positions and the one that drops the fewest (its drops are all, or
    # nearly all, private positions)
    mask_np = ev.keepmask.cpu().numpy().view(np.uint32)
    kept_bits = np.unpackbits(mask_np.view(np.uint8), bitorder="little").reshape(cfg.n_sess, -1)
    prefix_drops = cfg.prefix - kept_bits[:, :cfg.prefix].sum(axis=1)
    heavy, light = int(prefix_drops.argmax()), int(prefix_drops.argmin())
    sample = list(dict.fromkeys([0, 37, heavy, light, 21, 63]))[:4]
    print(f"slotmap: shared-prefix positions dropped per session: max "
          f"{int(prefix_drops.max())} (session {heavy}), min {int(prefix_drops.min())} "
          f"(session {light}); sessions checked {sample}")
    # the oracle's memories of the sampled sessions, from the generator's turns
    M_ref = np.zeros((len(sample), cfg.L, cfg.Hq, cfg.D), np.float32)
    for t in range(cfg.turns):
        qt = cfg.q_turn(t, DEV)
        M_ref = orc.qmem_update(M_ref, _bits(qt[sample]), cfg.decay, cfg.gain)
        del qt
    np.testing.assert_allclose(M[sample].cpu().numpy(), M_ref, rtol=2e-5, atol=2e-7)
    near = 0
    for i, r in enumerate(sample):
        slots = torch.from_numpy(sm[r].astype(np.int64)).to(DEV)
        k_rows = _bits(kp[:, slots])                     # [L][N][H][D]: position → row
        ident = np.arange(cfg.N, dtype=np.int32)
        ref = orc.rule_session(M_ref[i], k_rows, ident, cfg.H, -1)
        assert_scores_close(rule[r].cpu().numpy(), ref, f"rule session {r}")
        del k_rows
        # the GPU's kept positions against the oracle's selection on its own
        # scores; a difference is allowed only at a near-tie boundary
        k_ref, _, _ = orc.select(ref, cfg.budget, 0, 0)
        if not np.array_equal(ev.kept[r].cpu().numpy(), k_ref):
            gap = kth_gap(ref, cfg.budget, 0, 0)
            assert gap is not None and gap < NEAR_TIE_REL, f"kept session {r} gap {gap}"
            near += 1
    print(f"slotmap: near-tie sessions {near} of {len(sample)} sampled")
    # select properties, then redirect/free bit-exact against the oracle on
    # the GPU's own keep mask (integer stage)
    nb = np.full((cfg.n_sess,), cfg.N, np.int64)
    _check_selection_properties(ev.kept, ev.kept_count, nb, cfg.budget, 0, 0)
    mask = ev.keepmask.cpu().numpy().view(np.uint32)
    sm_ref, rc_ref, freed_ref, code, nf = orc.redirect_free(sm, mask, rc, cfg.prefix, cfg.sentinel)
    assert code == 0
    assert np.array_equal(sm_d.cpu().numpy(), sm_ref)
    assert np.array_equal(rc_d.cpu().numpy(), rc_ref)
    assert int(ev.n_freed.item()) == nf
    assert np.array_equal(ev.freed[:nf].cpu().numpy(), freed_ref)
    print(f"slotmap: freed {nf} slots of {cfg.n_slots}")
