"""Pins of the oracle's LSE-recovery scorer and tail-compaction plan (ActKV
§7.1 Algorithm 3, §7.2 Algorithm 4) against closed forms, invariants and
brute force: nothing here restates the oracle's own loops."""
from __future__ import annotations

import math

import numpy as np
import pytest


def _bits(x) -> np.ndarray:
    """float → bf16 bits (the values used are bf16-exact)."""
    a = np.asarray(x, np.float32)
    b = a.view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def _pool(vecs):
    """kpool [L=1][n_slots][H=1][D] from a list of D-vectors."""
    v = np.asarray(vecs, np.float32)
    return _bits(v)[None, :, None, :]


def test_lse_is_log_of_n_for_a_zero_query(orc):
    D, n = 8, 12
    k = np.random.default_rng(0).integers(-4, 5, (n, D)).astype(np.float32)
    q = np.zeros((1, 1, D), np.float32)
    lse = orc.attention_lse(_bits(q), _pool(k), np.arange(1, dtype=np.int32), 16, n, 1)
    assert lse[0, 0] == pytest.approx(math.log(n), rel=1e-14)


def test_lse_maps_query_heads_to_their_kv_head(orc):
    """H = 2 KV heads, Hq = 4: every key of KV head 0 is zero and every key of
    KV head 1 is 3·e0, every query row is 2·e0.  Query heads 0, 1 read KV head
    0 (LSE = ln n) and heads 2, 3 read KV head 1 (LSE = ln n + 6/√4)."""
    D, n, H, Hq = 4, 5, 2, 4
    kp = np.zeros((1, n, H, D), np.float32)
    kp[0, :, 1, 0] = 3.0
    q = np.zeros((1, Hq, D), np.float32)
    q[0, :, 0] = 2.0
    lse = orc.attention_lse(_bits(q), _bits(kp), np.array([0], np.int32), 16, n, H)
    want = [math.log(n), math.log(n), math.log(n) + 3.0, math.log(n) + 3.0]
    np.testing.assert_allclose(lse[0], want, rtol=1e-14)


def test_one_aligned_key_closed_form(orc):
    """q·k = c for key 0 and 0 for the other n−1 keys: p_0 = e^{c/√D}/(e^{c/√D}+n−1)."""
    D, n, c = 16, 9, 8.0
    keys = np.zeros((n, D), np.float32)
    keys[0, 0] = 2.0
    for j in range(1, n):
        keys[j, 1 + (j % (D - 1))] = 1.0
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = c / 2.0
    bt = np.array([0], np.int32)
    lse = orc.attention_lse(_bits(q), _pool(keys), bt, 16, n, 1)
    e = math.exp(c / math.sqrt(D))
    assert lse[0, 0] == pytest.approx(math.log(e + n - 1), rel=1e-14)
    st = orc.recover_step(_bits(q), lse, _pool(keys), bt, 16, n, 1, 1, np.zeros(16))
    assert st[0] == pytest.approx(e / (e + n - 1), rel=1e-13)
    assert st[1] == pytest.approx(1.0 / (e + n - 1), rel=1e-13)
    assert np.all(st[n:] == 0.0)  # past the sequence: not visible


def test_recovered_probabilities_sum_to_one(orc):
    rng = np.random.default_rng(1)
    D, n, BS = 32, 45, 16
    k = (rng.integers(-8, 9, (n, D)) / 8).astype(np.float32)
    q = (rng.integers(-8, 9, (1, 1, D)) / 4).astype(np.float32)
    bt = np.arange(3, dtype=np.int32)
    lse = orc.attention_lse(_bits(q), _pool(k), bt, BS, n, 1)
    st = orc.recover_step(_bits(q), lse, _pool(k), bt, BS, n, 1, 1, np.zeros(48))
    assert st.sum() == pytest.approx(1.0, rel=1e-12)


def test_group_max_and_sum_over_heads_and_layers(orc):
    """G = 2 query heads per KV head, H = 2, L = 2: token 0's key is e0 in KV
    head 0 and e1 in KV head 1, so query head hq scores a[hq] against head 0
    and b[hq] against head 1; the score is Σ_l Σ_h max over h's group, which
    fails for any other head-to-group mapping."""
    D, n = 4, 2
    L, H, Hq = 2, 2, 4
    kp = np.zeros((L, n, H, D), np.float32)  # token 1 stays zero
    kp[:, 0, 0, 0] = 1.0
    kp[:, 0, 1, 1] = 1.0
    a = np.array([[2.0, 4.0, 6.0, 0.0], [1.0, 3.0, 5.0, 7.0]], np.float32)  # [l][hq] on e0
    b = np.array([[8.0, 2.0, 0.0, 10.0], [9.0, 1.0, 3.0, 11.0]], np.float32)  # [l][hq] on e1
    q = np.zeros((L, Hq, D), np.float32)
    q[:, :, 0] = a
    q[:, :, 1] = b
    lse = np.zeros((L, Hq))  # p = exp(q·k/√D) directly
    st = orc.recover_step(_bits(q), lse, _bits(kp), np.array([0], np.int32), 16, n, 1, H,
                          np.zeros(16))
    rt = math.sqrt(D)
    want0 = sum(max(math.exp(a[l, 0] / rt), math.exp(a[l, 1] / rt)) +
                max(math.exp(b[l, 2] / rt), math.exp(b[l, 3] / rt)) for l in range(L))
    assert st[0] == pytest.approx(want0, rel=1e-13)
    assert st[1] == pytest.approx(L * H * 1.0, rel=1e-13)  # q·0 = 0: exp(0) = 1


def test_running_mean_reset_and_visibility(orc):
    """Three steps with known x give their mean; count = 1 restarts; a key
    not yet visible contributes 0 to the steps before it appears."""
    D = 4
    keys = np.zeros((3, D), np.float32)
    q = np.zeros((1, 1, D), np.float32)
    bt = np.array([0], np.int32)
    st = np.full(16, 123.0)
    xs = []
    for t, lse0 in enumerate([0.0, -math.log(2.0), -math.log(4.0)]):
        # q = 0: p = exp(0 − lse) = 1, 2, 4 on every visible key
        st = orc.recover_step(_bits(q), np.array([[lse0]]), _pool(keys), bt, 16, 2 + (t == 2),
                              t + 1, 1, st)
        xs.append(math.exp(-lse0))
    assert st[0] == pytest.approx(sum(xs) / 3, rel=1e-14)
    assert st[2] == pytest.approx(4.0 / 3, rel=1e-14)  # visible only to the third step
    st = orc.recover_step(_bits(q), np.array([[0.0]]), _pool(keys), bt, 16, 3, 1, 1, st)
    assert st[0] == 1.0 and st[2] == 1.0
    # the restart ignores whatever the state held (not a number included)
    st = orc.recover_step(_bits(q), np.array([[0.0]]), _pool(keys), bt, 16, 3, 1, 1,
                          np.full(16, np.nan))
    assert st[0] == 1.0 and st[3] == 0.0


def test_block_table_indirection(orc):
    """A permuted block table over a permuted pool scores like the identity."""
    rng = np.random.default_rng(3)
    D, BS, nb = 8, 4, 5
    n = nb * BS - 2
    k = (rng.integers(-4, 5, (nb * BS, D)) / 4).astype(np.float32)
    q = (rng.integers(-4, 5, (1, 2, D)) / 2).astype(np.float32)
    perm = rng.permutation(nb).astype(np.int32)
    kperm = np.empty_like(k)
    for b in range(nb):
        kperm[perm[b] * BS:(perm[b] + 1) * BS] = k[b * BS:(b + 1) * BS]
    lse = np.array([[0.5, -0.25]])
    a = orc.recover_step(_bits(q), lse, _pool(k), np.arange(nb, dtype=np.int32), BS, n, 1,
                         1, np.zeros(nb * BS))
    b = orc.recover_step(_bits(q), lse, _pool(kperm), perm, BS, n, 1, 1, np.zeros(nb * BS))
    assert np.array_equal(a, b)


def test_tail_plan_worked_example(orc):
    """21 tokens in blocks [7, 3] of 16 slots; tokens 0, 4, 16, 17, 19 kept."""
    km = np.array([(1 << 0) | (1 << 4) | (1 << 16) | (1 << 17) | (1 << 19)], np.uint32)
    p = orc.tail_plan(km, 21, np.array([7, 3], np.int32), 16)
    assert p["X"] == 1
    assert p["src"].tolist() == [7 * 16 + 0, 7 * 16 + 4]
    assert p["dst"].tolist() == [3 * 16 + 2, 3 * 16 + 4]
    assert p["freed"].tolist() == [7] and p["new_table"].tolist() == [3]
    assert p["tail_mask"].tolist() == [0b11111]


@pytest.mark.parametrize("seed", range(40))
def test_tail_plan_invariants_brute_force(orc, seed):
    """Applying the planned copies to a token array leaves exactly the
    retained tokens in the last X = ⌈m/BS⌉ blocks, moves nothing into a
    retained slot, reads no slot it writes, and frees the other blocks."""
    rng = np.random.default_rng(seed)
    BS = int(rng.choice([4, 16]))
    n = int(rng.integers(1, 120))
    Y = (n + BS - 1) // BS
    keep = rng.random(n) < rng.choice([0.1, 0.5, 0.9, 1.0])
    words = (n + 31) // 32
    km = np.zeros(words, np.uint32)
    for p in np.nonzero(keep)[0]:
        km[p // 32] |= np.uint32(1 << (p % 32))
    bt = rng.permutation(Y + 7)[:Y].astype(np.int32)
    p = orc.tail_plan(km, n, bt, BS)
    m = int(keep.sum())
    X = (m + BS - 1) // BS
    assert p["X"] == X
    assert p["freed"].tolist() == bt[:Y - X].tolist()
    assert p["new_table"].tolist() == bt[Y - X:].tolist()
    # physical slot → token id (−1: empty), then the copies
    slots = {}
    for pos in range(Y * BS):
        slots[int(bt[pos // BS]) * BS + pos % BS] = pos if pos < n else -1
    src, dst = p["src"].tolist(), p["dst"].tolist()
    assert len(set(src) & set(dst)) == 0 and len(set(dst)) == len(dst)
    for s_, d_ in zip(src, dst):
        assert slots[d_] == -1 or not keep[slots[d_]]  # never overwrite a retained token
        slots[d_] = slots[s_]
    region = [int(b) * BS + i for b in bt[Y - X:] for i in range(BS)]
    held = [slots[s_] for s_ in region]
    kept_ids = sorted(np.nonzero(keep)[0].tolist())
    mask = p["tail_mask"]
    live = [slot_i for slot_i in range(X * BS) if (int(mask[slot_i // 32]) >> (slot_i % 32)) & 1]
    assert sorted(held[i] for i in live) == kept_ids
    assert len(live) == m
