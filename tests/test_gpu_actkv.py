"""ActKV paged primitives on the GPU against the oracle.

* LSE-recovery score (ActKV §7.1, Algorithm 3): both kernels (tensor-core
  page tiles and the CUDA-core path) on shapes that cover each, ragged
  sequence lengths with partial last pages, inactive requests, restart and
  running-mean steps; within 1e-3 relative of the fp64 oracle fed the same
  bf16 inputs and the same fp32 LSE.
* Tail plan (§7.2, Algorithm 4): bit-exact against the oracle on masks of
  every density, empty and full requests, lengths off the block grid.
* Compaction: the pools after the copies equal the oracle's plan applied to
  the pools on the host, bit for bit.
* The whole operation at the Table 1 shapes (block size 16, 8 KV heads,
  head dim 128, 6K → 4K tokens), at 4 and 64 requests: sampled requests'
  scores against the oracle, select and plan bit-exact stage-wise, the
  copies checked on the device.
"""
from __future__ import annotations


import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from helpers import assert_scores_close  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _mk_inputs(orc, rng, n_req, L, H, Hq, D, BS, max_blocks, seq, spare=3):
    n_blocks = n_req * max_blocks + spare
    n_slots = n_blocks * BS
    kp = torch.randn(L, n_slots, H, D, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30))))
    kp = kp.to(torch.bfloat16)
    q = (torch.randn(n_req, L, Hq, D, generator=torch.Generator().manual_seed(7)) * 1.5
         ).to(torch.bfloat16)
    bt = rng.permutation(n_blocks)[:n_req * max_blocks].reshape(n_req, max_blocks).astype(np.int32)
    kp_bits, q_bits = _bits(kp), _bits(q)
    lse = np.zeros((n_req, L, Hq), np.float32)
    for r in range(n_req):
        if seq[r] > 0:
            lse[r] = orc.attention_lse(q_bits[r], kp_bits, bt[r], BS, seq[r], H).astype(np.float32)
    return kp, q, bt, lse, kp_bits, q_bits, n_slots


def _gpu_recover(kvc, q, lse, kp, bt, seq, cnt, state, n_slots, L, H, Hq, D, BS, path=None,
                 ws=True):
    n_req, max_blocks = bt.shape
    st = torch.from_numpy(state.astype(np.float32)).to(DEV)
    wsb = kvc.kvc_recover_score_workspace_size(n_req, max_blocks, L, H, Hq, D, BS)
    wst = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV) if ws else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_recover_score_ex(q.to(DEV), torch.from_numpy(lse).to(DEV), kp.to(DEV), n_slots,
                             torch.from_numpy(bt).to(DEV), max_blocks,
                             torch.from_numpy(np.asarray(seq, np.int32)).to(DEV),
                             torch.from_numpy(np.asarray(cnt, np.int32)).to(DEV), n_req, L, H,
                             Hq, D, BS, st, wst, ("recover_" + path) if path else "auto",
                             status)
    torch.cuda.synchronize()
    return st.cpu().numpy(), kvc.kvc_device_status(status)


SHAPES = [  # H, Hq, D, BS
    (8, 32, 128, 16),   # tensor cores, G 4 (the Table 1 tile)
    (8, 16, 64, 16),    # tensor cores, G 2, one 64-column K block
    (8, 64, 128, 16),   # tensor cores, G 8
    (4, 16, 128, 16),   # CUDA cores: 4 KV heads
    (8, 24, 64, 8),     # CUDA cores: page of 8, G 3
]


@pytest.mark.parametrize("H,Hq,D,BS", SHAPES)
@pytest.mark.parametrize("path", [None, "cc", "one_group"])
def test_recover_matches_oracle(kvc, orc, H, Hq, D, BS, path):
    """Both kernels; on the tensor cores both with layer groups (few pages:
    partial sums in the workspace, then the finalize) and without (no
    workspace: one kernel)."""
    if path in ("cc", "one_group") and not kvc.kvc_recover_tensor_core(H, Hq, D, BS):
        pytest.skip("already the CUDA-core path")
    ws = path != "one_group"
    path = None if path == "one_group" else path
    rng = np.random.default_rng(H * 1000 + Hq * 10 + D + BS)
    n_req, L, max_blocks = 5, 3, 7
    seq = [max_blocks * BS, max_blocks * BS - BS - 3, 1, 3 * BS + 2, 0]
    kp, q, bt, lse, kp_bits, q_bits, n_slots = _mk_inputs(orc, rng, n_req, L, H, Hq, D, BS,
                                                          max_blocks, seq)
    cap = max_blocks * BS
    state = rng.random((n_req, cap)).astype(np.float32)
    ref = state.astype(np.float64).copy()
    # step 1: restart (count 1); step 2: running-mean steps and an inactive request
    for cnt in ([1, 1, 1, 1, 1], [2, 3, 2, 0, 2]):
        prev = state
        state, status = _gpu_recover(kvc, q, lse, kp, bt, seq, cnt, state, n_slots, L, H, Hq,
                                     D, BS, path, ws)
        assert status == 0
        for r in range(n_req):
            if cnt[r] < 1:  # not generating an action: untouched
                assert np.array_equal(state[r], prev[r])
                continue
            ref[r] = orc.recover_step(q_bits[r], lse[r].astype(np.float64), kp_bits, bt[r],
                                      BS, seq[r], cnt[r], H, ref[r])
            assert_scores_close(state[r], ref[r], f"request {r} count {cnt[r]}")
        assert np.all(np.isfinite(state))
    # positions past each sequence were restarted to exactly 0, then kept at 0
    for r in range(n_req):
        assert np.all(state[r, seq[r]:] == 0.0)


def test_recover_tensor_core_and_cuda_core_agree(kvc, orc):
    """The two kernels compute the same sums in the same order per
    (slot, head) over layers; they agree far inside the oracle tolerance."""
    rng = np.random.default_rng(11)
    H, Hq, D, BS, L, n_req, max_blocks = 8, 32, 128, 16, 4, 3, 9
    seq = [144, 131, 77]
    kp, q, bt, lse, *_ , n_slots = _mk_inputs(orc, rng, n_req, L, H, Hq, D, BS, max_blocks, seq)
    z = np.zeros((n_req, max_blocks * BS), np.float32)
    a, _ = _gpu_recover(kvc, q, lse, kp, bt, seq, [1] * n_req, z, n_slots, L, H, Hq, D, BS)
    b, _ = _gpu_recover(kvc, q, lse, kp, bt, seq, [1] * n_req, z, n_slots, L, H, Hq, D, BS, "cc")
    assert_scores_close(a.ravel(), b.ravel().astype(np.float64), "tc vs cc")


def test_recover_bad_block_id_is_recorded(kvc, orc):
    rng = np.random.default_rng(5)
    H, Hq, D, BS, L, n_req, max_blocks = 8, 32, 128, 16, 2, 2, 4
    seq = [64, 64]
    kp, q, bt, lse, kp_bits, q_bits, n_slots = _mk_inputs(orc, rng, n_req, L, H, Hq, D, BS,
                                                          max_blocks, seq)
    bt = bt.copy()
    bt[1, 2] = n_slots // BS + 5  # outside the pool
    z = np.ones((n_req, max_blocks * BS), np.float32)
    for path in (None, "cc"):
        st, status = _gpu_recover(kvc, q, lse, kp, bt, seq, [1, 1], z, n_slots, L, H, Hq, D, BS,
                                  path)
        assert status == 7  # KVC_ERR_BOUNDS
        assert np.all(st[1, 2 * BS:3 * BS] == 0.0)  # the bad page scores 0
        ref = orc.recover_step(q_bits[0], lse[0].astype(np.float64), kp_bits, bt[0], BS, 64, 1,
                               H, np.zeros(max_blocks * BS))
        assert_scores_close(st[0], ref, "good request beside a bad one")


# ----------------------------------------------------------------- plan

def _plan_gpu(kvc, km, seq, bt, BS, n_slots):
    n_req, max_blocks = bt.shape
    cap = max_blocks * BS
    words = km.shape[1]
    i32 = dict(dtype=torch.int32, device=DEV)
    out = {k: torch.full((n_req, cap), -7, **i32) for k in ("src", "dst")}
    out.update({k: torch.full((n_req,), -7, **i32) for k in ("n_pairs", "X", "n_freed")})
    out.update({k: torch.full((n_req, max_blocks), -7, **i32) for k in ("freed", "new_table")})
    out["tail"] = torch.full((n_req, (cap + 31) // 32), -7, **i32)
    status = torch.zeros(1, **i32)
    kvc.kvc_tail_plan(torch.from_numpy(km.view(np.int32)).to(DEV), words,
                      torch.from_numpy(np.asarray(seq, np.int32)).to(DEV),
                      torch.from_numpy(bt).to(DEV), max_blocks, n_req, BS, n_slots,
                      out["src"], out["dst"], out["n_pairs"], out["X"], out["freed"],
                      out["n_freed"], out["new_table"], out["tail"], status)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["tail"] = res["tail"].view(np.uint32)
    return res, kvc.kvc_device_status(status)


def _mask_words(keep: np.ndarray, words: int) -> np.ndarray:
    km = np.zeros(words, np.uint32)
    for p in np.nonzero(keep)[0]:
        km[p // 32] |= np.uint32(1 << (p % 32))
    return km


def _check_plan(orc, res, r, km_row, n, bt_row, BS):
    p = orc.tail_plan(km_row, n, bt_row, BS)
    npairs = len(p["src"])
    assert res["n_pairs"][r] == npairs and res["X"][r] == p["X"]
    assert np.array_equal(res["src"][r, :npairs], p["src"])
    assert np.array_equal(res["dst"][r, :npairs], p["dst"])
    assert np.all(res["src"][r, npairs:] == -1) and np.all(res["dst"][r, npairs:] == -1)
    nf = len(p["freed"])
    assert res["n_freed"][r] == nf
    assert np.array_equal(res["freed"][r, :nf], p["freed"])
    assert np.all(res["freed"][r, nf:] == -1)
    assert np.array_equal(res["new_table"][r, :p["X"]], p["new_table"])
    assert np.all(res["new_table"][r, p["X"]:] == -1)
    tw = len(p["tail_mask"])
    assert np.array_equal(res["tail"][r, :tw], p["tail_mask"])
    assert np.all(res["tail"][r, tw:] == 0)
    return p


@pytest.mark.parametrize("BS", [4, 16])
def test_tail_plan_bit_exact(kvc, orc, BS):
    rng = np.random.default_rng(BS)
    max_blocks = 40
    cap = max_blocks * BS
    dens = [0.0, 1.0, 0.1, 0.5, 0.9, 0.66, 0.3, 0.5, 1.0, 0.97]
    seq = [cap, cap, cap - 3, cap // 2 + 1, 1, 0, cap - BS, 37, BS * 3, cap]
    n_req = len(seq)
    words = (cap + 31) // 32 + 1   # a row stride wider than needed
    clean = np.zeros((n_req, words), np.uint32)
    for r in range(n_req):
        clean[r] = _mask_words(rng.random(seq[r]) < dens[r], words)
    # set bits past each sequence: the plan must ignore them
    noisy = clean.copy()
    for r in range(n_req):
        junk = np.zeros(words * 32, bool)
        junk[seq[r]:] = rng.random(words * 32 - seq[r]) < 0.5
        noisy[r] |= _mask_words(junk, words)
    n_blocks = n_req * max_blocks + 9
    bt = rng.permutation(n_blocks)[:n_req * max_blocks].reshape(n_req, max_blocks).astype(np.int32)
    res, status = _plan_gpu(kvc, noisy, seq, bt, BS, n_blocks * BS)
    assert status == 0
    for r in range(n_req):
        _check_plan(orc, res, r, clean[r], seq[r], bt[r], BS)


def test_tail_plan_bad_length_gives_empty_plan(kvc, orc):
    BS, max_blocks = 16, 4
    km = np.full((2, 2), 0xFFFFFFFF, np.uint32)
    bt = np.arange(8, dtype=np.int32).reshape(2, 4)
    res, status = _plan_gpu(kvc, km, [65, 64], bt, BS, 8 * BS)
    assert status == 7
    assert res["n_pairs"][0] == 0 and res["X"][0] == 0 and res["n_freed"][0] == 0
    assert np.all(res["freed"][0] == -1) and np.all(res["new_table"][0] == -1)
    assert res["X"][1] == 4 and res["n_pairs"][1] == 0


# ------------------------------------------------------------ compaction

def test_compaction_applies_the_plan_bit_exact(kvc, orc):
    rng = np.random.default_rng(21)
    L, H, D, BS, max_blocks, n_req = 3, 8, 64, 16, 12, 4
    cap = max_blocks * BS
    seq = [cap, cap - 5, 70, 0]
    n_blocks = n_req * max_blocks + 6
    n_slots = n_blocks * BS
    bt = rng.permutation(n_blocks)[:n_req * max_blocks].reshape(n_req, max_blocks).astype(np.int32)
    words = (cap + 31) // 32
    km = np.stack([_mask_words(rng.random(seq[r]) < 0.6, words) for r in range(n_req)])
    res, status = _plan_gpu(kvc, km, seq, bt, BS, n_slots)
    assert status == 0
    kp = rng.integers(0, 1 << 16, (L, n_slots, H, D), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, (L, n_slots, H, D), dtype=np.uint16)
    kd = torch.from_numpy(kp.view(np.int16)).to(DEV)
    vd = torch.from_numpy(vp.view(np.int16)).to(DEV)
    status_t = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_tail_compact(kd, vd, n_slots, L, H, D, torch.from_numpy(res["src"]).to(DEV),
                         torch.from_numpy(res["dst"]).to(DEV),
                         torch.from_numpy(res["n_pairs"]).to(DEV), cap, n_req, status_t)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(status_t) == 0
    kref, vref = kp.copy(), vp.copy()
    moved = 0
    for r in range(n_req):
        p = _check_plan(orc, res, r, km[r], seq[r], bt[r], BS)
        for s_, d_ in zip(p["src"], p["dst"]):
            kref[:, d_] = kp[:, s_]
            vref[:, d_] = vp[:, s_]
            moved += 1
    assert moved > 0
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), kref)
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), vref)


# ------------------------------------------- whole op at Table 1 shapes

@pytest.mark.parametrize("n_req", [4, 64])
def test_paged_event_table1_shapes(kvc, orc, n_req):
    import workloads as wl
    from query_conditioned_kv_gb300.event import PagedEvent
    cfg = wl.config_paged(n_req)
    assert kvc.kvc_recover_tensor_core(cfg.H, cfg.Hq, cfg.D, cfg.BS)
    kp, vp = cfg.pools(DEV)
    q = cfg.q(DEV)
    lse = cfg.lse(q)
    bt_np = cfg.block_tables()
    bt = torch.from_numpy(bt_np).to(DEV)
    seq = torch.from_numpy(cfg.seqused()).to(DEV)
    cnt = torch.full((n_req,), 1, dtype=torch.int32, device=DEV)
    ev = PagedEvent(n_req, cfg.max_blocks, cfg.BS, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                    cfg.keep, device=DEV)
    ev.score(q, lse, kp, bt, seq, cnt)
    ev.select()
    ev.plan(seq, bt)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    state = ev.state.cpu().numpy()
    # sampled requests: recovery score against the oracle on the request's own pages
    BS, cap = cfg.BS, cfg.cap
    for r in sorted({0, n_req - 1}):
        slots = (bt[r][:, None].long() * BS + torch.arange(BS, device=DEV)).reshape(-1)
        sub = _bits(kp[:, slots])                       # [L][cap][H][D]
        ref = orc.recover_step(_bits(q[r]), lse[r].double().cpu().numpy(), sub,
                               np.arange(cfg.max_blocks, dtype=np.int32), BS, cfg.seq, 1,
                               cfg.H, np.zeros(cap))
        assert_scores_close(state[r], ref, f"request {r}")
    # select and plan, stage-wise bit-exact on the GPU's own scores
    off = np.arange(n_req + 1, dtype=np.int64) * cap
    kref, cref, mref = orc.select_segments(state.reshape(-1), off, cfg.keep, 0, 0,
                                           mask_words=ev.words)
    assert np.array_equal(ev.kept_count.cpu().numpy(), cref)
    assert np.array_equal(ev.kept.cpu().numpy(), kref)
    km = ev.keepmask.cpu().numpy().view(np.uint32)
    assert np.array_equal(km, mref)
    res = {"src": ev.src, "dst": ev.dst, "n_pairs": ev.n_pairs, "X": ev.n_tail,
           "freed": ev.freed, "n_freed": ev.n_freed, "new_table": ev.new_table,
           "tail": ev.tail_mask}
    res = {k: v.cpu().numpy() for k, v in res.items()}
    res["tail"] = res["tail"].view(np.uint32)
    for r in range(n_req):
        _check_plan(orc, res, r, km[r], cfg.seq, bt_np[r], BS)
    # compaction: destinations receive the sources' rows; nothing else moves
    r = n_req // 2
    npairs = int(res["n_pairs"][r])
    src = torch.from_numpy(res["src"][r, :npairs]).to(DEV).long()
    dst = torch.from_numpy(res["dst"][r, :npairs]).to(DEV).long()
    k_src, v_src = kp[:, src].clone(), vp[:, src].clone()
    probe = torch.from_numpy(np.setdiff1d(
        (bt_np[r][:, None] * BS + np.arange(BS)).reshape(-1), res["dst"][r, :npairs])).to(DEV)
    k_probe = kp[:, probe].clone()
    ev.compact(kp, vp)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(ev.dev_status) == 0
    assert torch.equal(kp[:, dst], k_src) and torch.equal(vp[:, dst], v_src)
    assert torch.equal(kp[:, probe], k_probe)
