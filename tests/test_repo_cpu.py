"""The repository view (KVMem, "Tiered movement"), host side, no GPU: units
(layer, KV head, 32-token block) of raw K/V in a backing file, the most-used
ones in host slots.

* every unit's record in its host slot equals the gather of its tokens from
  the [L][H][n_tok][D] history, step after step;
* which blocks hold host slots follows the documented policy, checked against
  a plain model of it (free slots first, then the blocks with the fewest uses,
  ties by last use, then by index, never a block the step needs);
* a step's file reads come in one vectored read per run of consecutive blocks;
* the plan (used / needed blocks from kept lists) against brute force;
* errors: more needed blocks than slots, a block never put, an unwritable
  path."""
from __future__ import annotations

import numpy as np
import pytest

import query_conditioned_kv_gb300 as kvc

L, H, D = 2, 3, 64
TOK = 32


def _history(n_blocks, seed):
    rng = np.random.default_rng(seed)
    n_tok = n_blocks * TOK
    k = rng.integers(0, 1 << 16, size=(L, H, n_tok, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(L, H, n_tok, D), dtype=np.uint16)
    return k, v, n_tok


def _record(k, v, u, n_blocks):
    """[2][32][D] record of unit u = (l·H + h)·n_blocks + g."""
    lh, g = divmod(u, n_blocks)
    l, h = divmod(lh, H)
    return np.concatenate([k[l, h, g * TOK:(g + 1) * TOK].reshape(-1),
                           v[l, h, g * TOK:(g + 1) * TOK].reshape(-1)])


def _put_model(model, b0, nb, n_blocks):
    for lh in range(L * H):
        for g in range(b0, b0 + nb):
            model.put(lh * n_blocks + g)


class Model:
    """The placement policy as the header states it."""

    def __init__(self, n_blocks, n_slots):
        self.slot_of = [-1] * n_blocks
        self.block_in = [-1] * n_slots
        self.free = list(range(n_slots))[::-1]  # slot 0 handed out first
        self.uses = [0] * n_blocks
        self.last = [0] * n_blocks
        self.stored = [False] * n_blocks
        self.step_no = 0
        self.runs = 0
        self.fetched = 0

    def put(self, g):
        if self.slot_of[g] < 0 and self.free:
            s = self.free.pop()
            self.slot_of[g], self.block_in[s] = s, g
        self.stored[g] = True

    def step(self, used, need):
        want = list(dict.fromkeys(need))
        self.step_no += 1
        for g in used:
            self.uses[g] += 1
            self.last[g] = self.step_no
        fetch = sorted(g for g in want if self.slot_of[g] < 0)
        dest = []
        while len(dest) < len(fetch) and self.free:
            dest.append(self.free.pop())
        if len(dest) < len(fetch):
            cand = [s for s, b in enumerate(self.block_in) if b >= 0 and b not in want]
            cand.sort(key=lambda s: (self.uses[self.block_in[s]], self.last[self.block_in[s]],
                                     self.block_in[s]))
            for s in cand[:len(fetch) - len(dest)]:
                self.slot_of[self.block_in[s]] = -1
                self.block_in[s] = -1
                dest.append(s)
        for g, s in zip(fetch, dest):
            self.slot_of[g], self.block_in[s] = s, g
        self.fetched += len(fetch)
        self.runs += sum(1 for i, g in enumerate(fetch) if i == 0 or g != fetch[i - 1] + 1)

    def resident(self):
        return {g for g, s in enumerate(self.slot_of) if s >= 0}


def _arena_bits(repo):
    """The arena as uint16 (a pinned bf16 tensor when a GPU is present)."""
    a = repo.arena
    if hasattr(a, "view") and not isinstance(a, np.ndarray):
        import torch
        return a.view(torch.int16).numpy().view(np.uint16)
    return a


def _check_slots(repo, k, v, n_blocks):
    arena = _arena_bits(repo)
    for u in range(L * H * n_blocks):
        s = repo.host_slot[u]
        if s >= 0:
            got = arena[s * repo.slot_elems:(s + 1) * repo.slot_elems]
            assert np.array_equal(got, _record(k, v, u, n_blocks)), f"unit {u}"


def test_repo_records_and_placement_follow_the_policy(tmp_path):
    n_blocks, n_slots = 40, 9
    n_units = L * H * n_blocks
    k, v, n_tok = _history(n_blocks, 1)
    repo = kvc.KvcRepo(tmp_path / "hist.bin", n_blocks, L, H, D, n_slots, io_threads=3)
    model = Model(n_units, n_slots)
    repo.put(0, 25, k, v, n_tok)
    repo.put(25, n_blocks - 25, k, v, n_tok)
    _put_model(model, 0, 25, n_blocks)
    _put_model(model, 25, n_blocks - 25, n_blocks)
    # the first n_slots units put (layer 0, head 0, blocks 0 …) hold the slots
    assert [repo.where(u) for u in range(n_units)] == [1] * n_slots + [2] * (n_units - n_slots)
    rng = np.random.default_rng(2)
    hot = [3, 17, 30, 100, 200]  # kept in most steps: they should end up holding slots
    table = repo.slot_table().copy()  # a copy kept up to date from the changes alone
    for step in range(40):
        used = set(rng.choice(n_units, size=6, replace=False).tolist())
        if step % 4:
            used |= set(hot)
        need = sorted(rng.choice(sorted(used), size=min(len(used), n_slots - 1),
                                 replace=False).tolist())
        used = sorted(used)
        repo.step(used, need)
        model.step(used, need)
        units, slots = repo.changes()
        table[units] = slots
        assert np.array_equal(table, repo.host_slot), f"step {step}: changes"
        res = {u for u in range(n_units) if repo.where(u) == 1}
        assert res == model.resident(), f"step {step}"
        assert all(repo.host_slot[g] >= 0 for g in need)
        assert sorted(np.flatnonzero(repo.host_slot >= 0).tolist()) == sorted(res)
        _check_slots(repo, k, v, n_blocks)
    st = repo.stats()
    assert st["steps"] == 40
    assert st["fetched"] == model.fetched and st["read_calls"] == model.runs
    assert st["bytes_read"] == model.fetched * repo.slot_elems * 2
    assert st["bytes_written"] == n_units * repo.slot_elems * 2
    assert st["needed"] == st["host_hits"] + st["fetched"]
    assert set(hot) <= model.resident() or st["fetched"] > 0
    repo.close()


def test_repo_reads_runs_in_one_call_each(tmp_path):
    n_blocks, n_slots = 64, 40
    k, v, n_tok = _history(n_blocks, 3)
    repo = kvc.KvcRepo(tmp_path / "h.bin", n_blocks, L, H, D, n_slots, io_threads=4)
    repo.put(0, n_blocks, k, v, n_tok)  # units 0..39 (layer 0, head 0) take the slots
    need = list(range(44, 52)) + list(range(55, 60)) + [62] + [2 * n_blocks + 5]  # 4 runs
    need = sorted(need)
    repo.step(need, need)
    st = repo.stats()
    assert st["fetched"] == len(need) and st["read_calls"] == 4
    _check_slots(repo, k, v, n_blocks)
    # blocks re-put after a change read back as changed
    k2 = k.copy()
    k2[:, :, 50 * TOK:51 * TOK] ^= 0x5555
    repo.put(50, 1, k2, v, n_tok)
    repo.step([50], [50])
    _check_slots(repo, k2, v, n_blocks)
    repo.close()


@pytest.mark.parametrize("io_threads", [1, 4, 7])
def test_repo_put_writes_every_record(tmp_path, io_threads):
    """Rows longer than one vectored write (150 blocks: writes of 64, 64, 22
    records), more rows than some thread counts divide evenly, most units
    without a host slot (written from staging records): every unit read back
    from the file, a slot's worth at a time, equals its gather."""
    n_blocks, n_slots = 150, 16
    k, v, n_tok = _history(n_blocks, 11)
    repo = kvc.KvcRepo(tmp_path / "w.bin", n_blocks, L, H, D, n_slots, io_threads=io_threads)
    repo.put(0, 100, k, v, n_tok)
    repo.put(100, n_blocks - 100, k, v, n_tok)
    n_units = L * H * n_blocks
    assert repo.stats()["bytes_written"] == n_units * 2 * TOK * D * 2
    assert all(repo.where(u) in (1, 2) for u in range(n_units))
    for u0 in range(0, n_units, n_slots):
        need = list(range(u0, min(u0 + n_slots, n_units)))
        repo.step(need, need)
        _check_slots(repo, k, v, n_blocks)
    repo.close()


def test_repo_errors(tmp_path):
    n_blocks = 12
    k, v, n_tok = _history(n_blocks, 4)
    repo = kvc.KvcRepo(tmp_path / "e.bin", n_blocks, L, H, D, 4)
    repo.put(0, 8, k, v, n_tok)
    with pytest.raises(kvc.KvcError) as e:  # more blocks needed at once than slots
        repo.step([0, 1, 2, 3, 4], [0, 1, 2, 3, 4])
    assert e.value.code == 10
    with pytest.raises(kvc.KvcError) as e:  # block 9 (of layer 0, head 0) was never put
        repo.step([9], [9])
    assert e.value.code == 1
    with pytest.raises(kvc.KvcError) as e:  # outside the history
        repo.put(10, 3, k, v, n_tok)
    assert e.value.code == 1
    with pytest.raises(ValueError):  # a history array shorter than n_tok says
        repo.put(0, 1, k[:, :, :TOK], v, n_tok)
    with pytest.raises(ValueError):  # 4-byte elements where bf16 is expected
        repo.put(0, 1, k.astype(np.float32), v, n_tok)
    with pytest.raises(ValueError):  # kept lists shorter than L·H·n_sess·budget
        kvc.kvc_repo_plan(np.zeros(5, np.int32), np.zeros(L * H, np.int32), None, None, L, H,
                          1, 4, np.array([0, n_tok], np.int64), n_blocks)
    n_units = L * H * n_blocks
    assert repo.where(-1) == -1 and repo.where(n_units) == -1 and repo.where(9) == 0
    repo.step([0, 5], [5])  # the repository still works after refused calls
    assert repo.where(5) == 1
    repo.close()
    with pytest.raises(kvc.KvcError) as e:
        kvc.KvcRepo(tmp_path / "no_such_dir" / "x.bin", n_blocks, L, H, D, 4)
    assert e.value.code == 11


def test_repo_direct_io(tmp_path):
    n_blocks = 10
    k, v, n_tok = _history(n_blocks, 5)
    try:
        repo = kvc.KvcRepo(tmp_path / "d.bin", n_blocks, L, H, D, 3, direct=True)
    except kvc.KvcError as e:
        assert e.code == 11
        pytest.skip("this file system refuses direct I/O")
    repo.put(0, n_blocks, k, v, n_tok)
    repo.step([7, 8, 9], [7, 8, 9])
    _check_slots(repo, k, v, n_blocks)
    repo.close()


def _plan_brute(kept, cnt, kept_prev, cnt_prev, n_seg, n_sess, tok_off, budget, n_blocks):
    used, need = set(), set()
    for s in range(n_seg):
        r = s % n_sess
        g0 = (s // n_sess) * n_blocks + tok_off[r] // TOK
        cur = kept[s * budget:s * budget + cnt[s]]
        prev = set() if kept_prev is None else set(
            kept_prev[s * budget:s * budget + min(max(cnt_prev[s], 0), budget)].tolist())
        for kb in cur.tolist():
            used.add(g0 + kb)
            if kb not in prev:
                need.add(g0 + kb)
    return sorted(used), sorted(need)


@pytest.mark.parametrize("first", [True, False])
def test_repo_plan_matches_brute_force(first):
    rng = np.random.default_rng(6 + first)
    Lp, Hp, n_sess, budget = 3, 2, 2, 12
    nbs = [20, 33]
    tok_off = np.array([0, nbs[0] * TOK, (nbs[0] + nbs[1]) * TOK], np.int64)
    n_seg = Lp * Hp * n_sess

    def lists():
        kept = np.full(n_seg * budget, -1, np.int32)
        cnt = np.zeros(n_seg, np.int32)
        for s in range(n_seg):
            nb = nbs[s % n_sess]
            c = int(rng.integers(0, budget + 1))
            kept[s * budget:s * budget + c] = np.sort(rng.choice(nb, size=c, replace=False))
            cnt[s] = c
        return kept, cnt

    kept, cnt = lists()
    kp, cp = (None, None) if first else lists()
    n_blocks = sum(nbs)
    used, need = kvc.kvc_repo_plan(kept, cnt, kp, cp, Lp, Hp, n_sess, budget, tok_off,
                                   n_blocks)
    ru, rn = _plan_brute(kept, cnt, kp, cp, n_seg, n_sess, tok_off, budget, n_blocks)
    assert used.tolist() == ru and need.tolist() == rn
    if first:
        assert need.tolist() == used.tolist()
    # a kept index outside its session is refused
    bad = kept.copy()
    bad[0] = nbs[0]
    cnt2 = cnt.copy()
    cnt2[0] = max(cnt2[0], 1)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_repo_plan(bad, cnt2, None, None, Lp, Hp, n_sess, budget, tok_off, n_blocks)
    assert e.value.code == 7


def test_repo_io_error_leaves_a_consistent_table(tmp_path):
    """A failed file read (the backing file cut short after the put): the
    step reports KVC_ERR_IO, its evictions stand, its fetched units end up
    without a slot, changes() lists both, and the repository keeps working
    for units still in host RAM."""
    import os
    n_blocks, n_slots = 16, 8
    k, v, n_tok = _history(n_blocks, 9)
    path = tmp_path / "io.bin"
    repo = kvc.KvcRepo(path, n_blocks, L, H, D, n_slots)
    repo.put(0, n_blocks, k, v, n_tok)  # units 0..7 hold the slots
    before = repo.slot_table().copy()
    os.truncate(path, 0)
    with pytest.raises(kvc.KvcError) as e:
        repo.step([20, 21], [20, 21])  # both on file only: reads hit end of file
    assert e.value.code == 11
    units, slots = repo.changes()
    table = before.copy()
    table[units] = slots
    assert np.array_equal(table, repo.slot_table())
    assert repo.where(20) == 2 and repo.where(21) == 2  # still on file, no slot
    # the two evicted units and the two that failed to arrive, all slotless
    assert (slots == -1).all() and sorted(units.tolist()) == [0, 1, 20, 21]
    assert int((repo.slot_table() >= 0).sum()) == n_slots - 2
    repo.step([3], [3] if repo.where(3) == 1 else [])  # a resident unit still works
    repo.close()
