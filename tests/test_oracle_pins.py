"""Pins of the CPU oracle against what the pages and mathematics fix.

None of these re-types the oracle's formula: each checks a closed form, a
brute-force enumeration, a library routine, an invariant or the pages'
worked example, chosen so that a plausible mistake (a dropped term, a wrong
sign or index, a transposed operand, a sum where a max belongs) fails.
CPU only.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def bf16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def nearest_bf16(x: Fraction) -> int:
    """Independent RNE: search the bf16 neighbours of fp32(x) exactly."""
    if x == 0:
        return 0
    f = np.float32(float(x))
    c = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
    best = None
    for b in (c - 1, c, c + 1, c + 2):
        b &= 0xFFFF
        if (b & 0x7F80) == 0x7F80:
            continue
        v = bf16_value(b)
        if (v < 0) != (x < 0) and v != 0:
            continue
        d = abs(v - x)
        key = (d, b & 1)  # smaller error, then even mantissa
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def bits(arr_f32) -> np.ndarray:
    """fp32 values that are exact in bf16 → bf16 bit patterns."""
    a = np.asarray(arr_f32, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def sigmoid1() -> float:
    return math.e / (math.e + 1.0)


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_exact_nearest_even(orc):
    rng = np.random.default_rng(7)
    xs = list(rng.standard_normal(400) * 10.0 ** rng.integers(-6, 6, 400))
    # exact midpoints between bf16 neighbours: ties must go to even
    for b in (0x3F80, 0x3F81, 0x4123, 0xC61C, 0x0081):
        lo, hi = bf16_value(b), bf16_value(b + 1)
        xs.append(float((lo + hi) / 2))
    for x in xs:
        assert orc.f64_to_bf16(x) == nearest_bf16(Fraction(x)), x


def test_bf16_rounding_of_subnormals(orc):
    # below 2^-126 bf16 values are multiples of 2^-133: random values across
    # that range, and the exact midpoints between subnormal neighbours
    # (including the step from the largest subnormal to the smallest normal)
    rng = np.random.default_rng(11)
    xs = list(rng.uniform(-1.0, 1.0, 300) * 2.0 ** -126)
    xs += list(rng.uniform(0.0, 1.0, 100) * 2.0 ** -130)
    for b in (0x0001, 0x0002, 0x0040, 0x0055, 0x007F, 0x8003, 0x807F):
        lo, hi = bf16_value(b), bf16_value(b + 1)
        xs.append(float((lo + hi) / 2))
    for x in xs:
        assert orc.f64_to_bf16(x) == nearest_bf16(Fraction(x)), x


def test_sentinel_key_bits(orc):
    # IntentKV §2 "Layout": the dead slot's K is -1e4; in bf16 that is -9984
    assert orc.f64_to_bf16(-1e4) == 0xC61C
    assert float(orc.bf16_to_f64(np.array([0xC61C], np.uint16))[0]) == -9984.0


# ---------------------------------------------------------------- Mean-K

def test_meank_constant_block_is_constant(orc):
    k = np.full((1, 64, 8), 0x3FC0, dtype=np.uint16)  # 1.5 everywhere
    mk = orc.meank(k)
    assert mk.shape == (1, 2, 8) and np.all(mk == 0x3FC0)


def test_meank_every_row_of_a_layered_index(orc):
    # kraw [L=2][H=3][64][8]: every token of (l, h, block b) holds
    # 4l + h + b/2, exact in bf16, so each block mean is that value
    L, H = 2, 3
    v = np.zeros((L, H, 64, 8), np.float32)
    for l in range(L):
        for h in range(H):
            for b in range(2):
                v[l, h, 32 * b:32 * (b + 1)] = 4 * l + h + b / 2
    mk = orc.meank(bits(v))
    want = np.array([[[4 * l + h + b / 2] * 8 for b in range(2)]
                     for l in range(L) for h in range(H)], np.float32).reshape(L, H, 2, 8)
    assert np.array_equal(mk, bits(want))


def test_meank_is_exact_block_mean_rounded_once(orc):
    rng = np.random.default_rng(1)
    D = 16
    vals = rng.standard_normal((3, 96, D)).astype(np.float32)
    kb = (vals.view(np.uint32) >> 16).astype(np.uint16)  # truncation → bf16
    mk = orc.meank(kb)
    for r in range(3):
        for b in range(3):
            for d in range(D):
                s = sum(bf16_value(int(kb[r, b * 32 + t, d])) for t in range(32))
                assert mk[r, b, d] == nearest_bf16(s / 32), (r, b, d)


def test_meank_block_boundaries(orc):
    # token t holds value t: block b's mean is 32b + 15.5
    k = bits(np.repeat(np.arange(128, dtype=np.float32)[:, None], 4, 1))[None]
    mk = orc.meank(k)
    for b in range(4):
        assert mk[0, b, 0] == nearest_bf16(Fraction(32 * b) + Fraction(31, 2))


# ----------------------------------------------------------------- score

def _unit(qrows, mkrows):
    return bits(qrows), bits(mkrows)


def test_score_uniform_meank_gives_one_over_nb(orc):
    rng = np.random.default_rng(2)
    G, Wn, D, nb = 3, 5, 64, 37
    q = (rng.standard_normal((G, Wn, D)).astype(np.float32).view(np.uint32)
         >> 16).astype(np.uint16)
    mk = np.tile(bits(np.full(D, 0.25, np.float32)), (nb, 1))
    s = orc.score_unit(q, mk)
    assert np.all(s == np.float32(1.0 / nb))


def test_score_single_query_is_textbook_softmax(orc):
    rng = np.random.default_rng(3)
    D, nb = 128, 300
    qf = rng.standard_normal(D).astype(np.float32)
    mf = (rng.standard_normal((nb, D)) * 0.3).astype(np.float32)
    q = (qf.view(np.uint32) >> 16).astype(np.uint16)[None, None]
    mk = (mf.view(np.uint32) >> 16).astype(np.uint16)
    z = (orc.bf16_to_f64(mk) @ orc.bf16_to_f64(q[0, 0])) / math.sqrt(D)
    ref = scipy.special.softmax(z)
    s = orc.score_unit(q, mk)
    np.testing.assert_allclose(s, ref, rtol=1e-6)
    assert abs(float(s.astype(np.float64).sum()) - 1.0) < 1e-5


def test_score_takes_max_over_gqa_group(orc):
    # G=2, W=1, Nb=2, D=64: head g sees logit 8·1/sqrt(64) = 1 on block g, 0
    # on the other, so each head's softmax is (σ, 1-σ) / (1-σ, σ) with
    # σ = e/(e+1); the max over the group is σ on both blocks (a sum over
    # the group would give 1, a mean 1/2).
    D = 64
    q = np.zeros((2, 1, D), np.float32)
    q[0, 0, 0] = 8.0
    q[1, 0, 1] = 8.0
    mk = np.zeros((2, D), np.float32)
    mk[0, 0] = 1.0
    mk[1, 1] = 1.0
    qb, mb = _unit(q, mk)
    s = orc.score_unit(qb, mb)
    np.testing.assert_allclose(s, [sigmoid1(), sigmoid1()], rtol=1e-7)


def test_score_takes_mean_over_window(orc):
    # G=1, W=2, Nb=2, D=16: token 0 sees logits (1, 0) (4·1/sqrt(16)),
    # token 1 sees (0, 0) → scores ((σ + 1/2)/2, (1 - σ + 1/2)/2)
    D = 16
    q = np.zeros((1, 2, D), np.float32)
    q[0, 0, 0] = 4.0
    mk = np.zeros((2, D), np.float32)
    mk[0, 0] = 1.0
    qb, mb = _unit(q, mk)
    s = orc.score_unit(qb, mb)
    sg = sigmoid1()
    np.testing.assert_allclose(s, [(sg + 0.5) / 2, (1 - sg + 0.5) / 2],
                               rtol=1e-7)


def test_score_reads_query_heads_major(orc):
    # q is [G][W][D]: G = 2 heads × W = 3 window tokens, D = 16, Nb = 3 unit
    # Mean-K rows.  Row i of q (i = g·W + w) is 4·e_t[i], a logit of 1 on
    # block t[i] and 0 on the other two, so its softmax is A = e/(e+2) there
    # and B = 1/(e+2) elsewhere.  With t = (0, 0, 1, 2, 2, 1) the group of
    # token w is rows {w, W + w}: blocks {0,2}, {0,2}, {1,1}, giving scores
    # ((2A+B)/3, (A+2B)/3, (2A+B)/3); reading q as [W][G] pairs rows
    # {0,1}, {2,3}, {4,5} instead and gives ((A+2B)/3, (2A+B)/3, (2A+B)/3).
    D, G, Wn = 16, 2, 3
    t = (0, 0, 1, 2, 2, 1)
    q = np.zeros((G, Wn, D), np.float32)
    for i, blk in enumerate(t):
        q[i // Wn, i % Wn, blk] = 4.0
    mk = np.eye(3, D, dtype=np.float32)
    s = orc.score_unit(*_unit(q, mk))
    A, B = math.e / (math.e + 2.0), 1.0 / (math.e + 2.0)
    np.testing.assert_allclose(s, [(2 * A + B) / 3, (A + 2 * B) / 3, (2 * A + B) / 3],
                               rtol=1e-7)


def test_score_meank_slices_units_by_layer_head_and_session(orc):
    # L = 2, H = 2 KV heads with G = 2 query heads each, W = 1, D = 16, two
    # sessions owning blocks [0, 2) and [2, 5).  Layer 0's Mean-K row of block
    # b is e_b in both KV heads; query head hq of session r is 4·e_t[r][hq], a
    # logit of 1 on block t (0 elsewhere; 0 everywhere when t lies outside the
    # session).  A softmax over n blocks with one logit of 1 is A_n = e/(e+n-1)
    # there and B_n = 1/(e+n-1) elsewhere.  Layer 1's Mean-K is zero: uniform
    # 1/n per session.  Query heads 2h and 2h+1 belong to KV head h.
    L, n_sess, H, Hq, D = 2, 2, 2, 4, 16
    t = [(0, 0, 1, 1), (2, 3, 4, 7)]
    q = np.zeros((L, n_sess, Hq, 1, D), np.float32)
    for r in range(n_sess):
        for hq in range(Hq):
            q[:, r, hq, 0, t[r][hq]] = 4.0
    mk = np.zeros((L, H, 5, D), np.float32)
    mk[0, :, :, :5] = np.eye(5, dtype=np.float32)
    s = orc.score_meank(bits(q), bits(mk), H, np.array([0, 2, 5]))
    e = math.e
    A2, B2, A3, B3 = e / (e + 1), 1 / (e + 1), e / (e + 2), 1 / (e + 2)
    want = np.array([[[A2, B2, A3, A3, B3],
                      [B2, A2, 1 / 3, 1 / 3, A3]],
                     [[1 / 2, 1 / 2, 1 / 3, 1 / 3, 1 / 3]] * 2])
    np.testing.assert_allclose(s, want, rtol=1e-7)


def test_score_mass_bounds(orc):
    rng = np.random.default_rng(4)
    for G in (1, 2, 4):
        q = (rng.standard_normal((G, 6, 64)).astype(np.float32).view(np.uint32)
             >> 16).astype(np.uint16)
        mk = (rng.standard_normal((50, 64)).astype(np.float32).view(np.uint32)
              >> 16).astype(np.uint16)
        tot = float(orc.score_unit(q, mk).astype(np.float64).sum())
        if G == 1:
            assert abs(tot - 1.0) < 1e-5
        else:
            assert 1.0 - 1e-6 <= tot <= G + 1e-6


def test_tiny_config_planted_blocks_are_selected(orc):
    # the tiny config plants +3u in 4 blocks and adds 3u to the query: every
    # planted block must survive the 16-block budget in both KV heads
    cfg = W.config_tiny()
    blocks, _ = cfg.planted(0, 0, 0)
    for h in range(cfg.H):
        k = W.bf16_bits(cfg.kraw_unit(0, h, 0))
        mk = orc.meank(k[None])[0]
        q = np.stack([W.bf16_bits(cfg.q_unit(0, 0, h * cfg.G + g))
                      for g in range(cfg.G)])
        s = orc.score_unit(q, mk)
        kept, cnt, _ = orc.select(s, cfg.budget, cfg.n_sink, cfg.n_recent)
        assert cnt == cfg.budget
        assert set(blocks.tolist()) <= set(kept[:cnt].tolist())


def test_gamma_calibration_top8_share():
    # KVMem reports 66.5 % of the mass in the top-8 blocks; the frozen gamma
    # reproduces about 65 % on the 8B-class recipe (two sampled units)
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "calib", os.path.join(GOLDEN, "calibrate_gamma.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    share = mod.top8_share(W.GAMMA_PLANTED, sample=[(0, 0), (9, 2)])
    assert 0.55 < share < 0.75


# ---------------------------------------------------------------- select

def _brute_select(scores, budget, n_sink, n_recent):
    n = len(scores)
    if n <= budget:
        return list(range(n))
    forced = sorted(set(range(min(n_sink, n))) |
                    set(range(max(0, n - n_recent), n)))
    rest = [i for i in range(n) if i not in forced]
    k = budget - len(forced)
    best = None
    for comb in itertools.combinations(rest, k):
        tot = sum(Fraction(float(scores[i])) for i in comb)
        key = (-tot, tuple(sorted(comb)))
        if best is None or key < best[0]:
            best = (key, comb)
    return sorted(forced + list(best[1]))


def test_select_equals_brute_force(orc):
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 15))
        budget = int(rng.integers(1, 12))
        n_sink = int(rng.integers(0, 3))
        n_recent = int(rng.integers(0, 3))
        if n_sink + n_recent > budget:
            continue
        if trial % 2:
            s = (rng.integers(0, 5, n) / 8.0).astype(np.float32)  # many ties
        else:
            s = rng.standard_normal(n).astype(np.float32)
        kept, cnt, mask = orc.select(s, budget, n_sink, n_recent)
        want = _brute_select(s, budget, n_sink, n_recent)
        assert kept[:cnt].tolist() == want, (s, budget, n_sink, n_recent)
        assert np.all(kept[cnt:] == -1)
        got_mask = [i for i in range(n) if (mask[i // 32] >> (i % 32)) & 1]
        assert got_mask == want


def test_select_invariants_large(orc):
    rng = np.random.default_rng(6)
    n, budget, n_sink, n_recent = 4096, 256, 1, 4
    s = rng.random(n).astype(np.float32)
    kept, cnt, mask = orc.select(s, budget, n_sink, n_recent)
    k = kept[:cnt]
    assert cnt == budget
    assert np.all(np.diff(k) > 0)
    forced = {0, n - 4, n - 3, n - 2, n - 1}
    assert forced <= set(k.tolist())
    free_kept = [i for i in k if i not in forced]
    dropped = [i for i in range(n) if i not in set(k.tolist())]
    assert min(s[free_kept]) >= max(s[dropped])


def test_select_segments_closed_form(orc):
    # three segments of 5, 40 and 33 items, scores −i (the earliest item is
    # the best); budget 6 with 1 sink and 2 recent: a segment that fits is
    # kept whole, the others keep items 0–3 and their last two items
    off = np.array([0, 5, 45, 78])
    sc = np.concatenate([-np.arange(n, dtype=np.float32) for n in (5, 40, 33)])
    kept, cnt, mask = orc.select_segments(sc, off, 6, 1, 2)
    assert cnt.tolist() == [5, 6, 6]
    assert kept.tolist() == [[0, 1, 2, 3, 4, -1], [0, 1, 2, 3, 38, 39],
                             [0, 1, 2, 3, 31, 32]]
    assert mask.tolist() == [[0x1F, 0], [0xF, 0xC0], [0x8000000F, 0x1]]


def test_select_negative_zero_ties_positive_zero(orc):
    s = np.array([-0.0, 0.0, -0.0, 0.0, 1.0], np.float32)
    kept, cnt, _ = orc.select(s, 3, 0, 0)
    assert kept[:cnt].tolist() == [0, 1, 4]


def test_select_short_segment_keeps_all(orc):
    kept, cnt, _ = orc.select(np.array([3, 1, 2], np.float32), 8, 1, 4)
    assert cnt == 3 and kept[:3].tolist() == [0, 1, 2]
    assert np.all(kept[3:] == -1)


# ------------------------------------------------------------------ RoPE

@pytest.mark.parametrize("D", [64, 128])
def test_rope_closed_forms(orc, D):
    theta = 1e6
    half = D // 2
    for p in (0.0, 1.0, 7.0, 511.0, 65535.0):
        for j in (0, 1, 5, half - 1):
            f = theta ** (-2.0 * j / D)
            x = np.zeros(D)
            x[j] = 1.0
            y = orc.rope_f64(x, p, theta)
            assert abs(y[j] - math.cos(p * f)) < 1e-12
            assert abs(y[j + half] - math.sin(p * f)) < 1e-12
            x = np.zeros(D)
            x[j + half] = 1.0
            y = orc.rope_f64(x, p, theta)
            assert abs(y[j] + math.sin(p * f)) < 1e-12
            assert abs(y[j + half] - math.cos(p * f)) < 1e-12
            assert np.count_nonzero(np.abs(y) > 1e-15) <= 2


def test_rope_identity_norm_and_relative_offset(orc):
    rng = np.random.default_rng(8)
    D, theta = 128, 1e6
    x = rng.standard_normal(D)
    assert np.array_equal(orc.rope_f64(x, 0.0, theta), x)
    y = orc.rope_f64(x, 12345.0, theta)
    half = D // 2
    np.testing.assert_allclose(x[:half] ** 2 + x[half:] ** 2,
                               y[:half] ** 2 + y[half:] ** 2, rtol=1e-12)
    q = rng.standard_normal(D)
    for _ in range(20):
        P, p, dlt = rng.integers(0, 70000, 3).astype(float)
        a = orc.rope_f64(q, P, theta) @ orc.rope_f64(x, p, theta)
        b = orc.rope_f64(q, P + dlt, theta) @ orc.rope_f64(x, p + dlt, theta)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_pack_gathers_kept_blocks_in_order(orc):
    D, n_tok, budget = 64, 256, 4
    # V row t holds value t in every element: the view must list tokens of
    # blocks 1, 3, 6 in chronological order, then zeros
    v = bits(np.repeat(np.arange(n_tok, dtype=np.float32)[:, None], D, 1))
    k = v.copy()
    kept = np.array([1, 3, 6, -1], np.int32)
    kv, vv = orc.pack_unit(k, v, kept, 3, budget, 0, 1e6)
    src = np.concatenate([np.arange(32) + 32 * b for b in (1, 3, 6)])
    assert np.array_equal(vv[:96], v[src])
    assert np.all(vv[96:] == 0) and np.all(kv[96:] == 0)
    # position 0 of the view is the identity rotation: K bit-identical there
    assert np.array_equal(kv[0], k[32])


def test_pack_rerope_closed_form(orc):
    # raw K = e_0 at every token: view token i holds cos(i) at 0 and sin(i)
    # at D/2 (frequency θ^0 = 1), each rounded once to bf16
    D, n_tok, budget, pos0 = 64, 128, 2, 1000
    k = np.zeros((n_tok, D), np.uint16)
    k[:, 0] = 0x3F80
    kept = np.array([3, 0], np.int32)
    kv, _ = orc.pack_unit(k, k, kept, 2, budget, pos0, 1e6)
    for i in range(64):
        p = pos0 + i
        assert kv[i, 0] == nearest_bf16(Fraction(math.cos(p)))
        assert kv[i, D // 2] == nearest_bf16(Fraction(math.sin(p)))
        others = np.delete(kv[i], [0, D // 2])
        assert np.all((others & 0x7FFF) == 0)


# ------------------------------------------------------ paged addressing

def test_slot_map_worked_example(orc):
    with open(os.path.join(GOLDEN, "slot_map_example.json")) as f:
        ex = json.load(f)
    got = orc.slot_map(ex["block_table"], ex["BS"], ex["seqused_k"])
    assert got.tolist() == ex["slot_map"]


def test_workload_slot_maps_follow_page_tables(orc):
    cfg = W.SlotMapConfig(name="t", n_sess=3, N=256, prefix=64, page=16, L=1,
                          H=2, Hq=4, D=64, T=4, turns=1, budget=64)
    bt = cfg.block_tables()
    sm = cfg.slot_maps(bt)
    for r in range(cfg.n_sess):
        assert np.array_equal(sm[r], orc.slot_map(bt[r], cfg.page, cfg.N))
    rc = cfg.refcounts(sm)
    assert np.all(rc[sm[0, :64]] == 3)           # shared prefix
    assert np.all(rc[sm[:, 64:].reshape(-1)] == 1)  # private slots
    assert rc[cfg.sentinel] == 0 and cfg.sentinel not in set(sm.reshape(-1))


# ------------------------------------------------------------ QueryMemory

def test_qmem_closed_forms(orc):
    D, T = 64, 4
    M = np.zeros((1, D), np.float32)
    q1 = np.zeros((1, T, D), np.float32)
    q1[0, :, 0] = 2.0
    M1 = orc.qmem_update(M, bits(q1))
    e0 = np.zeros(D, np.float32)
    e0[0] = 1
    assert np.array_equal(M1[0], e0)
    q2 = np.zeros((1, T, D), np.float32)
    q2[0, :, 1] = 1.0
    M2 = orc.qmem_update(M1, bits(q2))
    want = np.zeros(D)
    want[0], want[1] = 0.9 / math.sqrt(0.82), 0.1 / math.sqrt(0.82)
    np.testing.assert_allclose(M2[0], want, rtol=1e-7, atol=1e-9)
    # without renormalisation the EMA is 0.9·e0 + 0.1·e1
    M2n = orc.qmem_update(M1, bits(q2), renorm=False)
    assert M2n[0, 0] == np.float32(0.9) and M2n[0, 1] == np.float32(0.1)
    # the mean is over the turn's tokens: tokens (4, 0, 0, 0) → mean 1
    q3 = np.zeros((1, T, D), np.float32)
    q3[0, 0, 2] = 4.0
    M3 = orc.qmem_update(np.zeros((1, D), np.float32), bits(q3), renorm=False)
    assert M3[0, 2] == np.float32(0.1)


def test_qmem_updates_every_memory_row(orc):
    # M [n_sess=2][L=3][Hq=2][D] from zero, every token of row i equal to
    # (i + 1)·e_(i mod D): without renormalisation each row becomes
    # 0.1·(i + 1)·e_(i mod D)
    D, T = 16, 3
    q = np.zeros((2, 3, 2, T, D), np.float32)
    for i in range(12):
        q.reshape(12, T, D)[i, :, i % D] = i + 1
    M = orc.qmem_update(np.zeros((2, 3, 2, D), np.float32), bits(q), renorm=False)
    want = np.zeros((12, D), np.float32)
    for i in range(12):
        want[i, i % D] = np.float32(0.1 * (i + 1))
    assert np.array_equal(M.reshape(12, D), want)


def test_qmem_unit_norm_after_every_update(orc):
    rng = np.random.default_rng(9)
    M = np.zeros((6, 128), np.float32)
    for _ in range(5):
        q = (rng.standard_normal((6, 32, 128)).astype(np.float32).view(np.uint32)
             >> 16).astype(np.uint16)
        M = orc.qmem_update(M, q)
        np.testing.assert_allclose(np.linalg.norm(M.astype(np.float64), axis=1),
                                   1.0, rtol=1e-6)


# ------------------------------------------------------------ rule score

def _pool(L, n_slots, H, D, fill=0.0):
    return np.full((L, n_slots, H, D), bits(np.float32(fill)).item(),
                   dtype=np.uint16)


def test_rule_mass_sums_to_layers_times_heads(orc):
    rng = np.random.default_rng(10)
    L, H, Hq, D, N = 2, 2, 4, 64, 50
    kp = (rng.standard_normal((L, N + 1, H, D)).astype(np.float32)
          .view(np.uint32) >> 16).astype(np.uint16)
    M = rng.standard_normal((L, Hq, D)).astype(np.float32)
    sm = np.arange(1, N + 1, dtype=np.int32)
    r = orc.rule_session(M, kp, sm, H, 0)
    assert abs(float(r.astype(np.float64).sum()) - L * Hq) < 1e-4
    # dead positions: −1, and the live mass is still L·Hq
    sm2 = sm.copy()
    sm2[[3, 17, 40]] = 0
    r2 = orc.rule_session(M, kp, sm2, H, 0)
    assert np.all(r2[[3, 17, 40]] == -1.0)
    live = np.delete(r2, [3, 17, 40]).astype(np.float64)
    assert abs(live.sum() - L * Hq) < 1e-4
    # the dead slot's K does not matter
    kp3 = kp.copy()
    kp3[:, 0] = 0xC61C
    assert np.array_equal(orc.rule_session(M, kp3, sm2, H, 0), r2)


def test_rule_uniform_keys(orc):
    L, H, Hq, D, N = 1, 2, 6, 64, 40
    kp = _pool(L, N + 1, H, D, 0.5)
    rng = np.random.default_rng(11)
    M = rng.standard_normal((L, Hq, D)).astype(np.float32)
    r = orc.rule_session(M, kp, np.arange(1, N + 1, dtype=np.int32), H, 0)
    np.testing.assert_allclose(r, L * Hq / N, rtol=1e-6)


def test_rule_gqa_expansion_closed_form(orc):
    # H=2, Hq=4 (G=2): query heads 0,1 read KV head 0, heads 2,3 read KV
    # head 1.  KV head 0 holds 8·e0 at position 0, KV head 1 holds 8·e1 at
    # position 1, zeros elsewhere; M = e0 for heads 0,1 and e1 for heads 2,3.
    # Heads 0,1 peak on position 0 with logit 8/8 = 1, heads 2,3 on
    # position 1; rule_0 = rule_1 = 2p + 2q with p = e/(e+N-1),
    # q = 1/(e+N-1).
    L, H, Hq, D, N = 1, 2, 4, 64, 10
    kp = _pool(L, N + 1, H, D, 0.0)
    kp[0, 1, 0, 0] = bits(np.float32(8.0)).item()  # position 0 → slot 1
    kp[0, 2, 1, 1] = bits(np.float32(8.0)).item()  # position 1 → slot 2
    M = np.zeros((L, Hq, D), np.float32)
    M[0, 0, 0] = M[0, 1, 0] = 1.0
    M[0, 2, 1] = M[0, 3, 1] = 1.0
    r = orc.rule_session(M, kp, np.arange(1, N + 1, dtype=np.int32), H, 0)
    e = math.e
    p, q = e / (e + N - 1), 1 / (e + N - 1)
    np.testing.assert_allclose(r[:2], [2 * p + 2 * q] * 2, rtol=1e-7)
    np.testing.assert_allclose(r[2:], [4 * q] * (N - 2), rtol=1e-7)


# ------------------------------------------------------- redirect / free

def _mask_from_keep(keep_bool):
    n_sess, N = keep_bool.shape
    words = (N + 31) // 32
    m = np.zeros((n_sess, words), np.uint32)
    for r in range(n_sess):
        for j in range(N):
            if keep_bool[r, j]:
                m[r, j // 32] |= np.uint32(1 << (j % 32))
    return m


def test_redirect_free_against_set_formula(orc):
    # IntentKV §4 check 6 / §7: u = S_r[j] is freed iff (a) j ≥ prefix,
    # (b) u ≠ s†, (c) u is not referenced by any remaining entry.  Pools with
    # a shared prefix (siblings), earlier redirects and intra-session aliases.
    rng = np.random.default_rng(12)
    sentinel = 0
    for trial in range(200):
        n_sess = int(rng.integers(1, 4))
        N = int(rng.integers(4, 40))
        prefix = int(rng.integers(0, N // 2 + 1))
        pref_slots = np.arange(1, prefix + 1)
        nxt = prefix + 1
        sm = np.zeros((n_sess, N), np.int32)
        for r in range(n_sess):
            sm[r, :prefix] = pref_slots
            priv = np.arange(nxt, nxt + N - prefix)
            nxt += N - prefix
            # a few aliases inside the private part, a few prior redirects
            if N - prefix > 2 and trial % 3 == 0:
                priv[-1] = priv[0]
            sm[r, prefix:] = priv
            dead = rng.random(N) < 0.1
            sm[r, dead] = sentinel
        n_slots = nxt
        rc = np.bincount(sm.reshape(-1), minlength=n_slots).astype(np.int32)
        rc[sentinel] = 0
        keep = rng.random((n_sess, N)) < 0.4
        km = _mask_from_keep(keep)
        new_sm, new_rc, freed, code, nf = orc.redirect_free(
            sm, km, rc, prefix, sentinel)
        assert code == 0
        dropped = ~keep
        # every dropped position reads the dead slot; kept ones unchanged
        assert np.all(new_sm[dropped] == sentinel)
        assert np.array_equal(new_sm[keep], sm[keep])
        # refcount conservation
        n_drop_refs = int(np.sum(dropped & (sm != sentinel)))
        assert int(rc.sum()) - int(new_rc.sum()) == n_drop_refs
        # the set formula (prefix slots only ever sit at prefix positions)
        remaining = set(new_sm.reshape(-1).tolist())
        want = set()
        for r in range(n_sess):
            for j in range(N):
                u = int(sm[r, j])
                if dropped[r, j] and j >= prefix and u != sentinel \
                        and u not in remaining:
                    want.add(u)
        assert set(freed.tolist()) == want
        assert len(freed) == len(want)  # no slot freed twice
        # order: by (session, position) of each slot's last dropping reference
        last = {}
        for r in range(n_sess):
            for j in range(N):
                if dropped[r, j] and sm[r, j] != sentinel:
                    last[int(sm[r, j])] = r * N + j
        assert freed.tolist() == sorted(want, key=lambda u: last[u])


def test_redirect_prefix_slots_never_freed(orc):
    # two sessions share prefix slots 1..4; both drop them: counts reach zero
    # but the radix-protected prefix is never returned to the allocator
    sm = np.array([[1, 2, 3, 4, 5, 6], [1, 2, 3, 4, 7, 8]], np.int32)
    rc = np.array([0, 2, 2, 2, 2, 1, 1, 1, 1], np.int32)
    keep = np.zeros((2, 6), bool)
    new_sm, new_rc, freed, code, nf = orc.redirect_free(
        sm, _mask_from_keep(keep), rc, 4, 0)
    assert code == 0
    assert freed.tolist() == [5, 6, 7, 8]
    assert np.all(new_rc[1:5] == 0)


def test_redirect_sibling_keeps_slot_alive(orc):
    # session 0 drops slot 5 which session 1 still keeps: not freed
    sm = np.array([[5, 6], [5, 7]], np.int32)
    rc = np.array([0, 0, 0, 0, 0, 2, 1, 1], np.int32)
    keep = np.array([[False, False], [True, True]])
    new_sm, new_rc, freed, code, _ = orc.redirect_free(
        sm, _mask_from_keep(keep), rc, 0, 0)
    assert freed.tolist() == [6] and new_rc[5] == 1
    assert new_sm.tolist() == [[0, 0], [5, 7]]
