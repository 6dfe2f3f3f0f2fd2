"""GPU ↔ oracle parity of the QueryMemory event: memory update, rule score,
token select, redirect + alias-aware free (bit-exact slot maps, refcounts
and free lists), plus the dead-slot sentinel."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402
from helpers import NEAR_TIE_REL, assert_scores_close, kth_gap  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def small_cfg(H=8, D=128, Hq=None, **kw):
    base = dict(name="sm", n_sess=3, N=1008, prefix=256, page=16, L=2, H=H,
                Hq=4 * H if Hq is None else Hq, D=D, T=32, turns=4, budget=300, seed=31)
    base.update(kw)
    return W.SlotMapConfig(**base)


def kpool_of(cfg, device):
    return torch.stack([cfg.kpool_layer(l, device) for l in range(cfg.L)])


def memory_chain(orc, cfg):
    """Oracle QueryMemory after cfg.turns turns (an input of the score)."""
    M = np.zeros((cfg.n_sess, cfg.L, cfg.Hq, cfg.D), np.float32)
    for t in range(cfg.turns):
        M = orc.qmem_update(M, W.bf16_bits(cfg.q_turn(t)), cfg.decay, cfg.gain)
    return M


def with_prior_redirects(cfg, sm, rng, frac=0.05):
    """Positions already redirected by an earlier event (private part only)."""
    sm = sm.copy()
    dead = rng.random(sm.shape) < frac
    dead[:, :cfg.prefix] = False
    sm[dead] = cfg.sentinel
    return sm


def test_qmem_update_parity(kvc, orc):
    cfg = small_cfg()
    M = torch.zeros(cfg.n_sess, cfg.L, cfg.Hq, cfg.D, dtype=torch.float32, device=DEV)
    Mo = np.zeros(tuple(M.shape), np.float32)
    for t in range(cfg.turns):
        q = cfg.q_turn(t, DEV)
        kvc.kvc_qmem_update(M, q, cfg.n_sess, cfg.L, cfg.Hq, cfg.D, cfg.T,
                            cfg.decay, cfg.gain, 1)
        Mo = orc.qmem_update(Mo, W.bf16_bits(q), cfg.decay, cfg.gain)
        torch.cuda.synchronize()
        np.testing.assert_allclose(M.cpu().numpy(), Mo, rtol=2e-5, atol=2e-7)
    n = np.linalg.norm(M.cpu().numpy().astype(np.float64), axis=-1)
    np.testing.assert_allclose(n, 1.0, rtol=1e-5)
    # renorm off follows the plain EMA
    M2 = torch.zeros_like(M)
    q = cfg.q_turn(0, DEV)
    kvc.kvc_qmem_update(M2, q, cfg.n_sess, cfg.L, cfg.Hq, cfg.D, cfg.T, 0.9, 0.1, 0)
    ref = orc.qmem_update(np.zeros(tuple(M.shape), np.float32), W.bf16_bits(q),
                          renorm=False)
    torch.cuda.synchronize()
    np.testing.assert_allclose(M2.cpu().numpy(), ref, rtol=2e-5, atol=1e-8)


@pytest.mark.parametrize("H,Hq,D", [(8, 32, 128), (2, 8, 128), (4, 16, 64), (8, 48, 128),
                                    (4, 4, 128), (2, 16, 64), (1, 3, 64), (8, 16, 64),
                                    (8, 64, 128)])
def test_rule_score_parity(kvc, orc, H, Hq, D):
    """GQA groups of 1..8 query heads, both head sizes; 1008 positions (a
    ragged last tile) with 5% of the private positions already dead."""
    cfg = small_cfg(H=H, D=D, Hq=Hq)
    rng = np.random.default_rng(H * 1000 + D + Hq)
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng)
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    from query_conditioned_kv_gb300.event import SlotMapEvent
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                      cfg.budget, cfg.prefix, cfg.sentinel, device=DEV)
    ev.score(torch.from_numpy(M).to(DEV), kp, torch.from_numpy(sm).to(DEV))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    got = ev.rule.cpu().numpy()
    kpb = W.bf16_bits(kp)
    for r in range(cfg.n_sess):
        ref = orc.rule_session(M[r], kpb, sm[r], cfg.H, cfg.sentinel)
        dead = sm[r] == cfg.sentinel
        assert np.all(got[r][dead] == -1.0) and np.all(ref[dead] == -1.0)
        assert_scores_close(got[r][~dead], ref[~dead], "rule")
        live_sum = float(got[r][~dead].astype(np.float64).sum())
        assert abs(live_sum - cfg.L * cfg.Hq) < 1e-3 * cfg.L * cfg.Hq


def _rule_gpu(kvc, cfg, M, kp, sm, path=None):
    from query_conditioned_kv_gb300.event import SlotMapEvent
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                      cfg.budget, cfg.prefix, cfg.sentinel, device=DEV)
    ev.score(torch.from_numpy(M).to(DEV), kp, torch.from_numpy(sm).to(DEV),
             kernel="qmem_" + path if path else "auto")
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    return ev.rule.cpu().numpy()


@pytest.mark.parametrize("Hq", [16, 32, 64])
def test_rule_score_gathered_rows(kvc, orc, Hq):
    """Slot maps that are not page-contiguous: every position of the private
    part points at a random slot (the tensor-core kernel then gathers one
    row per position), plus blocks whose slots are contiguous but not
    page-aligned, dead positions inside a page, and a session whose first
    positions are all dead.  Against the oracle, and the two logits kernels
    against each other."""
    cfg = small_cfg(H=8, D=128, Hq=Hq)
    rng = np.random.default_rng(Hq)
    sm = cfg.slot_maps()
    priv = sm[:, cfg.prefix:]
    flat = priv.reshape(-1).copy()
    rng.shuffle(flat)                                  # scatter every private position
    sm[:, cfg.prefix:] = flat.reshape(priv.shape)
    sm[0, 300:316] = np.arange(16) + 1000              # contiguous, not page-aligned
    sm[1, cfg.prefix + 16: cfg.prefix + 32: 3] = cfg.sentinel  # dead inside a block
    sm[2, :64] = cfg.sentinel                          # a dead run
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    got = _rule_gpu(kvc, cfg, M, kp, sm)
    cc = _rule_gpu(kvc, cfg, M, kp, sm, "cc")
    spill = _rule_gpu(kvc, cfg, M, kp, sm, "tc_spill")
    kpb = W.bf16_bits(kp)
    for r in range(cfg.n_sess):
        ref = orc.rule_session(M[r], kpb, sm[r], cfg.H, cfg.sentinel)
        dead = sm[r] == cfg.sentinel
        assert np.all(got[r][dead] == -1.0) and np.all(cc[r][dead] == -1.0)
        assert np.all(spill[r][dead] == -1.0)
        assert_scores_close(got[r][~dead], ref[~dead], "rule (tensor cores)")
        assert_scores_close(cc[r][~dead], ref[~dead], "rule (CUDA cores)")
        assert_scores_close(spill[r][~dead], ref[~dead], "rule (tensor cores, spilled)")


@pytest.mark.parametrize("n_sess,L,N,Hq", [(4, 3, 8192, 32), (1, 2, 51200, 32),
                                           (2, 2, 4000, 16), (3, 2, 1008, 16),
                                           (2, 2, 4000, 64)])
def test_rule_score_every_finish(kvc, orc, n_sess, L, N, Hq):
    """The three ways to the rule score against the oracle: the tensor-core
    kernel that forms each layer's share from the logits still in L2 (rows of
    one (session, layer) counted and their LSEs published inside the kernel),
    the tensor-core kernel that spills the logits for a second kernel, and the
    CUDA-core kernel.  Cases: rows spread over several waves of the grid; a
    row of 200 tiles, more than one wave on a 152-SM part; N not a multiple
    of 32 (4000, 1008: partial L2 lines are kept, not dropped); 5% of the
    private positions already dead.  The in-kernel finish repeats bit for
    bit.  Groups of 8 query heads have no in-kernel finish: naming it is
    refused before any launch, and the library's own choice is the spilled
    one."""
    cfg = small_cfg(H=8, D=128, Hq=Hq, n_sess=n_sess, L=L, N=N,
                    prefix=256 if N > 2000 else 128)
    rng = np.random.default_rng(N + Hq)
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng)
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    auto = _rule_gpu(kvc, cfg, M, kp, sm)
    spill = _rule_gpu(kvc, cfg, M, kp, sm, "tc_spill")
    cc = _rule_gpu(kvc, cfg, M, kp, sm, "cc")
    runs = [("spilled", spill), ("CUDA cores", cc)]
    if Hq // 8 <= 4:
        fused = _rule_gpu(kvc, cfg, M, kp, sm, "tc")
        fused2 = _rule_gpu(kvc, cfg, M, kp, sm, "tc")
        assert np.array_equal(fused.view(np.uint32), fused2.view(np.uint32))
        assert np.array_equal(auto.view(np.uint32), fused.view(np.uint32))
        runs.append(("fused", fused))
    else:
        with pytest.raises(kvc.KvcError) as ei:
            _rule_gpu(kvc, cfg, M, kp, sm, "tc")
        assert ei.value.code == 2
        assert np.array_equal(auto.view(np.uint32), spill.view(np.uint32))
    kpb = W.bf16_bits(kp)
    for r in range(cfg.n_sess):
        ref = orc.rule_session(M[r], kpb, sm[r], cfg.H, cfg.sentinel)
        dead = sm[r] == cfg.sentinel
        for name, got in runs:
            assert np.all(got[r][dead] == -1.0), name
            assert_scores_close(got[r][~dead], ref[~dead], f"rule ({name})")


@pytest.mark.parametrize("n_sess,L,N,dead_sess", [(2, 1, 48, None), (1, 1, 256, None),
                                                  (3, 2, 256, 1), (2, 3, 1008, 0)])
def test_rule_score_fused_edges(kvc, orc, n_sess, L, N, dead_sess):
    """Edges of the in-kernel finish: a session shorter than one 256-position
    tile, exactly one tile (one item, one CTA doing every role), and a
    session whose every position is already dead (its rows have no live
    position, so their LSE is −inf and every rule is −1).  Against the
    oracle, and the spilled finish bit for bit on the dead session."""
    cfg = small_cfg(H=8, D=128, Hq=32, n_sess=n_sess, L=L, N=N, prefix=16, budget=8)
    rng = np.random.default_rng(N + L)
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng)
    if dead_sess is not None:
        sm[dead_sess, :] = cfg.sentinel
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    fused = _rule_gpu(kvc, cfg, M, kp, sm, "tc")
    spill = _rule_gpu(kvc, cfg, M, kp, sm, "tc_spill")
    kpb = W.bf16_bits(kp)
    for r in range(cfg.n_sess):
        ref = orc.rule_session(M[r], kpb, sm[r], cfg.H, cfg.sentinel)
        dead = sm[r] == cfg.sentinel
        assert np.all(fused[r][dead] == -1.0) and np.all(ref[dead] == -1.0)
        if (~dead).any():
            assert_scores_close(fused[r][~dead], ref[~dead], f"rule session {r}")
    if dead_sess is not None:
        assert np.all(fused[dead_sess] == -1.0)
        assert np.array_equal(fused[dead_sess], spill[dead_sess])


def test_rule_score_long_session(kvc, orc):
    """One session longer than two waves of 256-position tiles, one layer:
    a row whose items span three turns of every CTA.  The in-kernel finish
    (the library's choice) against the oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    N = (2 * n_sm + 1) * 256 + 16
    cfg = small_cfg(H=8, D=128, Hq=32, n_sess=1, L=1, N=N, prefix=256)
    rng = np.random.default_rng(7)
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng)
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    auto = _rule_gpu(kvc, cfg, M, kp, sm)
    fused = _rule_gpu(kvc, cfg, M, kp, sm, "tc")
    assert np.array_equal(auto.view(np.uint32), fused.view(np.uint32))
    ref = orc.rule_session(M[0], W.bf16_bits(kp), sm[0], cfg.H, cfg.sentinel)
    dead = sm[0] == cfg.sentinel
    assert np.all(fused[0][dead] == -1.0)
    assert_scores_close(fused[0][~dead], ref[~dead], "rule (long session)")


def _redirect_case(orc, cfg, rng):
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng)
    rc = cfg.refcounts(sm)
    rule = rng.random(sm.shape).astype(np.float32)
    rule[sm == cfg.sentinel] = -1.0
    off = (np.arange(cfg.n_sess + 1) * cfg.N).astype(np.int64)
    _, _, mask = orc.select_segments(rule.reshape(-1), off, cfg.budget, 0, 0)
    return sm, rc, mask


def test_redirect_free_bit_exact(kvc, orc):
    cfg = small_cfg()
    rng = np.random.default_rng(5)
    sm, rc, mask = _redirect_case(orc, cfg, rng)
    # the shared prefix is dropped by every session in places: counts reach
    # zero there, yet nothing in the prefix may be freed
    mask[:, :2] = 0
    from query_conditioned_kv_gb300.event import SlotMapEvent
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                      cfg.budget, cfg.prefix, cfg.sentinel, device=DEV)
    sm_d = torch.from_numpy(sm).to(DEV)
    rc_d = torch.from_numpy(rc).to(DEV)
    ev.redirect(sm_d, rc_d, keepmask=torch.from_numpy(mask.view(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    sm_ref, rc_ref, freed_ref, code, nf = orc.redirect_free(sm, mask, rc, cfg.prefix,
                                                            cfg.sentinel)
    assert code == 0
    assert np.array_equal(sm_d.cpu().numpy(), sm_ref)
    assert np.array_equal(rc_d.cpu().numpy(), rc_ref)
    n = int(ev.n_freed.item())
    assert n == nf
    assert np.array_equal(ev.freed[:n].cpu().numpy(), freed_ref)
    # every freed slot is unreferenced, not the dead slot, not in the prefix
    live = set(sm_ref.reshape(-1).tolist())
    pref = set(sm[:, :cfg.prefix].reshape(-1).tolist())
    for u in freed_ref.tolist():
        assert u not in live and u != cfg.sentinel and u not in pref


def test_redirect_capacity_and_bounds(kvc, orc):
    cfg = small_cfg()
    rng = np.random.default_rng(6)
    sm, rc, mask = _redirect_case(orc, cfg, rng)
    from query_conditioned_kv_gb300.event import SlotMapEvent
    cap = 7
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                      cfg.budget, cfg.prefix, cfg.sentinel, freed_cap=cap, device=DEV)
    ev.redirect(torch.from_numpy(sm).to(DEV), torch.from_numpy(rc).to(DEV),
                keepmask=torch.from_numpy(mask.view(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 10  # KVC_ERR_CAPACITY
    _, _, freed_ref, _, nf = orc.redirect_free(sm, mask, rc, cfg.prefix, cfg.sentinel)
    assert int(ev.n_freed.item()) == nf > cap
    assert np.array_equal(ev.freed[:cap].cpu().numpy(), freed_ref[:cap])
    # a slot outside the pool: recorded, left in place, nothing dereferenced
    sm2 = sm.copy()
    j = int(np.nonzero(~np.asarray([(mask[0, i // 32] >> (i % 32)) & 1
                                    for i in range(cfg.N)], bool))[0][-1])
    sm2[0, j] = cfg.n_slots + 5
    ev2 = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                       cfg.budget, cfg.prefix, cfg.sentinel, device=DEV)
    sm2_d = torch.from_numpy(sm2).to(DEV)
    ev2.redirect(sm2_d, torch.from_numpy(rc).to(DEV),
                 keepmask=torch.from_numpy(mask.view(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev2.dev_status) == 7  # KVC_ERR_BOUNDS
    assert int(sm2_d[0, j].item()) == cfg.n_slots + 5


def test_sentinel_rows(kvc):
    L, H, D, n_slots = 3, 8, 128, 40
    kp = torch.randn(L, n_slots, H, D, device=DEV).to(torch.bfloat16)
    vp = torch.randn(L, n_slots, H, D, device=DEV).to(torch.bfloat16)
    before_k, before_v = kp.clone(), vp.clone()
    kvc.kvc_init_sentinel(kp, vp, L, H, D, n_slots, 0)
    torch.cuda.synchronize()
    kb = kp.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = vp.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(kb[:, 0] == 0xC61C) and np.all(vb[:, 0] == 0)
    assert float(kp[0, 0, 0, 0].float()) == -9984.0
    assert torch.equal(kp[:, 1:], before_k[:, 1:]) and torch.equal(vp[:, 1:], before_v[:, 1:])


def test_slotmap_event_end_to_end(kvc, orc):
    cfg = small_cfg(n_sess=4, N=2048 + 16 * 5, prefix=512, budget=700)
    rng = np.random.default_rng(8)
    sm = with_prior_redirects(cfg, cfg.slot_maps(), rng, frac=0.03)
    rc = cfg.refcounts(sm)
    kp = kpool_of(cfg, DEV)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    M = memory_chain(orc, cfg)
    from query_conditioned_kv_gb300.event import SlotMapEvent
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                      cfg.budget, cfg.prefix, cfg.sentinel, device=DEV)
    sm_d = torch.from_numpy(sm).to(DEV)
    rc_d = torch.from_numpy(rc).to(DEV)
    ev.run(torch.from_numpy(M).to(DEV), kp, sm_d, rc_d)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    kpb = W.bf16_bits(kp)
    rule_ref = np.stack([orc.rule_session(M[r], kpb, sm[r], cfg.H, cfg.sentinel)
                         for r in range(cfg.n_sess)])
    off = (np.arange(cfg.n_sess + 1) * cfg.N).astype(np.int64)
    kept_ref, cnt_ref, mask_ref = orc.select_segments(rule_ref.reshape(-1), off,
                                                      cfg.budget, 0, 0)
    kept = ev.kept.cpu().numpy()
    assert np.array_equal(ev.kept_count.cpu().numpy(), cnt_ref)
    near = 0
    for r in range(cfg.n_sess):
        if not np.array_equal(kept[r], kept_ref[r]):
            gap = kth_gap(rule_ref[r], cfg.budget, 0, 0)
            assert gap is not None and gap < NEAR_TIE_REL, (r, gap)
            near += 1
    # redirect/free of the GPU's own keep mask equals the oracle's on it
    mask = ev.keepmask.cpu().numpy().view(np.uint32)
    sm_ref, rc_ref, freed_ref, code, nf = orc.redirect_free(sm, mask, rc, cfg.prefix,
                                                            cfg.sentinel)
    assert code == 0
    assert np.array_equal(sm_d.cpu().numpy(), sm_ref)
    assert np.array_equal(rc_d.cpu().numpy(), rc_ref)
    assert int(ev.n_freed.item()) == nf
    assert np.array_equal(ev.freed[:nf].cpu().numpy(), freed_ref)
    print(f"slot-map event: near-tie sessions {near} of {cfg.n_sess}")
