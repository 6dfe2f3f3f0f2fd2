"""CPU oracle of the query-conditioned KV compression event.

TEST INFRASTRUCTURE ONLY: the product library never imports, links or calls
this package.  Only ``tests/``, the package smoke check and the benchmark's
CPU-baseline leg use it.

The arithmetic lives in ``oracle.c`` (plain scalar C, fp64); this module only
marshals numpy arrays into it and loops over the independent units
(session, layer, KV head) in the order of the definitions.  bf16 tensors are
numpy ``uint16`` arrays holding the bit patterns.

Every function in this file is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (closed forms, brute force, the pages' worked
example, invariants); nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")

BLOCK = 32


def lib():
    """Load (building if needed) liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c = ctypes
        L.orc_bf16_to_f64.argtypes = [c.c_uint16]
        L.orc_bf16_to_f64.restype = c.c_double
        L.orc_f64_to_bf16.argtypes = [c.c_double]
        L.orc_f64_to_bf16.restype = c.c_uint16
        L.orc_meank.argtypes = [_u16p, _u16p, c.c_int64, c.c_int64, c.c_int]
        L.orc_score_unit.argtypes = [_u16p, _u16p, c.c_int, c.c_int, c.c_int,
                                     c.c_int64, _f32p]
        L.orc_qmem_update.argtypes = [_f32p, _u16p, c.c_int64, c.c_int,
                                      c.c_int, c.c_double, c.c_double, c.c_int]
        L.orc_rule_session.argtypes = [_f32p, _u16p, c.c_int64, _i32p, c.c_int,
                                       c.c_int, c.c_int, c.c_int, c.c_int,
                                       c.c_int32, _f32p]
        L.orc_select.argtypes = [_f32p, c.c_int, c.c_int, c.c_int, c.c_int,
                                 _i32p, _i32p, c.c_void_p]
        L.orc_rope_f64.argtypes = [_f64p, _f64p, c.c_int, c.c_double,
                                   c.c_double]
        L.orc_pack_unit.argtypes = [_u16p, _u16p, c.c_int64, c.c_int, _i32p,
                                    c.c_int, c.c_int, c.c_int64, c.c_double,
                                    _u16p, _u16p]
        L.orc_slot_map.argtypes = [_i32p, c.c_int, c.c_int, c.c_int, _i32p]
        L.orc_redirect_free.argtypes = [_i32p, _u32p, c.c_int, c.c_int, _i32p,
                                        c.c_int64, c.c_int, c.c_int32, _i32p,
                                        c.c_int, _i32p]
        L.orc_attention_lse.argtypes = [_u16p, _u16p, c.c_int64, _i32p, c.c_int, c.c_int,
                                        c.c_int, c.c_int, c.c_int, c.c_int, _f64p]
        L.orc_recover_step.argtypes = [_u16p, _f64p, _u16p, c.c_int64, _i32p, c.c_int,
                                       c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                       c.c_int, _f64p]
        L.orc_tail_plan.argtypes = [_u32p, c.c_int, _i32p, c.c_int, _i32p, _i32p,
                                    c.POINTER(c.c_int), c.POINTER(c.c_int), _i32p,
                                    c.POINTER(c.c_int), _i32p, _u32p]
        L.orc_lrfu_update.argtypes = [_f32p, c.c_int, c.c_double, c.c_double, _f32p,
                                      np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")]
        L.orc_token_confidence.argtypes = [_f32p, c.c_int, c.c_int, c.POINTER(c.c_double)]
        L.orc_conf_trend.argtypes = [_f64p, c.c_int, c.c_int, c.c_int, c.c_double,
                                     c.POINTER(c.c_double), c.POINTER(c.c_int),
                                     c.POINTER(c.c_int)]
        L.orc_adapt_budget.argtypes = [c.c_double, c.c_int, c.c_int, c.c_int]
        for name in ("orc_meank", "orc_score_unit", "orc_qmem_update",
                     "orc_rule_session", "orc_select", "orc_rope_f64",
                     "orc_pack_unit", "orc_slot_map", "orc_redirect_free",
                     "orc_attention_lse", "orc_recover_step", "orc_tail_plan",
                     "orc_lrfu_update", "orc_token_confidence", "orc_conf_trend",
                     "orc_adapt_budget"):
            getattr(L, name).restype = c.c_int
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16

def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) → exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x: float) -> int:
    """One fp64 → bf16 round-to-nearest-even step (scalar)."""
    return int(lib().orc_f64_to_bf16(float(x)))


# ---------------------------------------------------------------- Mean-K

def meank(kraw: np.ndarray) -> np.ndarray:
    """Mean-K index: kraw [..., n_tok, D] uint16 → [..., n_tok/32, D] uint16."""
    kraw = _c(kraw, np.uint16)
    *lead, n_tok, D = kraw.shape
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty((*lead, n_tok // BLOCK, D), dtype=np.uint16)
    _check(lib().orc_meank(kraw, out, rows, n_tok, D), "orc_meank")
    return out


# ----------------------------------------------------------------- score

def score_unit(q_unit: np.ndarray, meank_unit: np.ndarray) -> np.ndarray:
    """One (session, layer, KV head): q [G][W][D], meank [Nb][D] → fp32 [Nb]."""
    q_unit = _c(q_unit, np.uint16)
    meank_unit = _c(meank_unit, np.uint16)
    G, W, D = q_unit.shape
    nb = meank_unit.shape[0]
    out = np.empty(nb, dtype=np.float32)
    _check(lib().orc_score_unit(q_unit, meank_unit, G, W, D, nb, out),
           "orc_score_unit")
    return out


def score_meank(q: np.ndarray, meank_all: np.ndarray, H: int,
                blk_off) -> np.ndarray:
    """Mean-K score of every unit.

    q [L][n_sess][Hq][W][D], meank_all [L][H][nb_total][D] → fp32
    [L][H][nb_total]; session r owns blocks [blk_off[r], blk_off[r+1]).
    """
    L, n_sess, Hq, W, D = q.shape
    G = Hq // H
    nb_total = meank_all.shape[2]
    out = np.zeros((L, H, nb_total), dtype=np.float32)
    for l in range(L):
        for h in range(H):
            for r in range(n_sess):
                b0, b1 = int(blk_off[r]), int(blk_off[r + 1])
                out[l, h, b0:b1] = score_unit(q[l, r, h * G:(h + 1) * G],
                                              meank_all[l, h, b0:b1])
    return out


# ------------------------------------------------------------ QueryMemory

def qmem_update(M: np.ndarray, q_turn: np.ndarray, decay=0.9, gain=0.1,
                renorm=True) -> np.ndarray:
    """M [..., D] fp32, q_turn [..., T, D] uint16 → updated copy of M."""
    M = np.array(M, dtype=np.float32, order="C", copy=True)
    q_turn = _c(q_turn, np.uint16)
    *lead, T, D = q_turn.shape
    rows = int(np.prod(lead)) if lead else 1
    _check(lib().orc_qmem_update(M, q_turn, rows, T, D, float(decay),
                                 float(gain), int(bool(renorm))),
           "orc_qmem_update")
    return M


def rule_session(M_sess: np.ndarray, kpool: np.ndarray, slot_map_row,
                 H: int, sentinel: int) -> np.ndarray:
    """Rule score of one session: M [L][Hq][D], kpool [L][n_slots][H][D]."""
    M_sess = _c(M_sess, np.float32)
    kpool = _c(kpool, np.uint16)
    sm = _c(slot_map_row, np.int32)
    L, Hq, D = M_sess.shape
    n_slots = kpool.shape[1]
    out = np.empty(sm.shape[0], dtype=np.float32)
    _check(lib().orc_rule_session(M_sess, kpool, n_slots, sm, sm.shape[0], L,
                                  H, Hq, D, int(sentinel), out),
           "orc_rule_session")
    return out


# ---------------------------------------------------------------- select

def select(scores, budget: int, n_sink: int, n_recent: int):
    """One segment → (kept [budget] int32 with -1 padding, count, mask)."""
    s = _c(scores, np.float32)
    n = s.shape[0]
    kept = np.empty(budget, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    mask = np.zeros((n + 31) // 32, dtype=np.uint32)
    _check(lib().orc_select(s, n, budget, n_sink, n_recent, kept, cnt,
                            mask.ctypes.data), "orc_select")
    return kept, int(cnt[0]), mask


def select_segments(scores_flat, seg_off, budget, n_sink, n_recent,
                    mask_words=None):
    """All segments: kept [n_seg][budget], count [n_seg], mask [n_seg][words]."""
    n_seg = len(seg_off) - 1
    lens = [int(seg_off[s + 1]) - int(seg_off[s]) for s in range(n_seg)]
    words = mask_words if mask_words is not None else (max(lens) + 31) // 32
    kept = np.full((n_seg, budget), -1, dtype=np.int32)
    cnt = np.zeros(n_seg, dtype=np.int32)
    mask = np.zeros((n_seg, words), dtype=np.uint32)
    for s in range(n_seg):
        a, b = int(seg_off[s]), int(seg_off[s + 1])
        k, c, m = select(scores_flat[a:b], budget, n_sink, n_recent)
        kept[s], cnt[s] = k, c
        mask[s, :m.shape[0]] = m
    return kept, cnt, mask


# ------------------------------------------------------------------ RoPE

def rope_f64(x, pos: float, theta: float) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty_like(x)
    _check(lib().orc_rope_f64(x, out, x.shape[0], float(pos), float(theta)),
           "orc_rope_f64")
    return out


def pack_unit(kraw_unit, vraw_unit, kept_row, count: int, budget: int,
              pos0: int, theta: float):
    """One unit: kraw/vraw [n_tok][D] uint16 → kview, vview [32·budget][D]."""
    kraw_unit = _c(kraw_unit, np.uint16)
    vraw_unit = _c(vraw_unit, np.uint16)
    kept_row = _c(kept_row, np.int32)
    n_tok, D = kraw_unit.shape
    kv = np.empty((BLOCK * budget, D), dtype=np.uint16)
    vv = np.empty((BLOCK * budget, D), dtype=np.uint16)
    _check(lib().orc_pack_unit(kraw_unit, vraw_unit, n_tok, D, kept_row,
                               int(count), int(budget), int(pos0),
                               float(theta), kv, vv), "orc_pack_unit")
    return kv, vv


# ------------------------------------------------------ paged addressing

def slot_map(block_table, BS: int, seqused: int) -> np.ndarray:
    bt = _c(block_table, np.int32)
    out = np.empty(seqused, dtype=np.int32)
    _check(lib().orc_slot_map(bt, bt.shape[0], BS, seqused, out),
           "orc_slot_map")
    return out


# ------------------------------------------------------ redirect and free

def redirect_free(slot_map_all, keepmask, refcnt, prefix_len: int,
                  sentinel: int, cap=None):
    """Returns (new slot_map, new refcnt, freed list, rc).

    slot_map_all [n_sess][N] int32, keepmask [n_sess][ceil(N/32)] uint32,
    refcnt [n_slots] int32.  rc is the oracle's return code (0, 4 or 6).
    """
    sm = np.array(slot_map_all, dtype=np.int32, order="C", copy=True)
    rc_arr = np.array(refcnt, dtype=np.int32, order="C", copy=True)
    km = _c(keepmask, np.uint32)
    n_sess, N = sm.shape
    cap = rc_arr.shape[0] if cap is None else cap
    freed = np.empty(max(cap, 1), dtype=np.int32)
    nf = np.zeros(1, dtype=np.int32)
    rc = lib().orc_redirect_free(sm, km, n_sess, N, rc_arr, rc_arr.shape[0],
                                 int(prefix_len), int(sentinel), freed,
                                 int(cap), nf)
    if rc not in (0, 4, 6):
        raise OracleError(f"orc_redirect_free returned {rc}")
    return sm, rc_arr, freed[:min(int(nf[0]), cap)].copy(), int(rc), int(nf[0])


# ----------------------------------------------- LSE recovery, compaction

def attention_lse(q, kpool, block_table, BS: int, seq_len: int, H: int) -> np.ndarray:
    """The attention backend's LSE of one request's step: q [L][Hq][D] and
    kpool [L][n_slots][H][D] bf16 bits → lse [L][Hq] (natural log)."""
    q = _c(q, np.uint16)
    kpool = _c(kpool, np.uint16)
    bt = _c(block_table, np.int32)
    L, Hq, D = q.shape
    out = np.empty((L, Hq), dtype=np.float64)
    _check(lib().orc_attention_lse(q, kpool, kpool.shape[1], bt, BS, seq_len, L, H, Hq, D,
                                   out), "orc_attention_lse")
    return out


def recover_step(q, lse, kpool, block_table, BS: int, seq_len: int, count: int, H: int,
                 state) -> np.ndarray:
    """One decode step of one request's action score (state [n_blocks·BS]
    float64, updated copy returned)."""
    q = _c(q, np.uint16)
    kpool = _c(kpool, np.uint16)
    bt = _c(block_table, np.int32)
    L, Hq, D = q.shape
    st = np.array(state, dtype=np.float64, copy=True)
    _check(lib().orc_recover_step(q, _c(lse, np.float64), kpool, kpool.shape[1], bt,
                                  bt.shape[0], BS, seq_len, count, L, H, Hq, D, st),
           "orc_recover_step")
    return st


def tail_plan(keepmask, n: int, block_table, BS: int) -> dict:
    """Compaction plan of one request (see orc_tail_plan)."""
    import ctypes as c
    km = _c(keepmask, np.uint32)
    bt = _c(block_table, np.int32)
    Y = (n + BS - 1) // BS
    src = np.zeros(max(n, 1), np.int32)
    dst = np.zeros(max(n, 1), np.int32)
    freed = np.zeros(max(Y, 1), np.int32)
    new_table = np.zeros(max(Y, 1), np.int32)
    tail = np.zeros(max((Y * BS + 31) // 32, 1), np.uint32)
    npairs, X, nfreed = c.c_int(0), c.c_int(0), c.c_int(0)
    _check(lib().orc_tail_plan(km, n, bt, BS, src, dst, c.byref(npairs), c.byref(X), freed,
                               c.byref(nfreed), new_table, tail), "orc_tail_plan")
    x = X.value
    return {"src": src[:npairs.value], "dst": dst[:npairs.value], "X": x,
            "freed": freed[:nfreed.value], "new_table": new_table[:x],
            "tail_mask": tail[:(x * BS + 31) // 32]}


# ------------------------------------------------------ LRFU keep score

def lrfu_update(scores, ks, p: float = 0.9, lam: float = 0.5):
    """One LRFU step of one segment: returns (new keep scores fp32, hits bool)."""
    sc = _c(scores, np.float32)
    k = np.array(ks, dtype=np.float32, copy=True)
    hits = np.zeros(len(sc), np.uint8)
    _check(lib().orc_lrfu_update(sc, len(sc), float(p), float(lam), k, hits),
           "orc_lrfu_update")
    return k, hits.astype(bool)


# --------------------------------------------------- confidence monitor

def token_confidence(logits, k: int = 20) -> float:
    """−mean log-probability of the top-k tokens of one row of logits."""
    import ctypes as c
    lg = _c(logits, np.float32)
    out = c.c_double(0.0)
    _check(lib().orc_token_confidence(lg, len(lg), k, c.byref(out)), "orc_token_confidence")
    return out.value


def conf_trend(conf, w: int, s: int, b: float):
    """(slope, n_windows, n_kept) of one trace's confidence sequence."""
    import ctypes as c
    cf = _c(conf, np.float64)
    sl, nw, nk = c.c_double(0.0), c.c_int(0), c.c_int(0)
    _check(lib().orc_conf_trend(cf, len(cf), w, s, float(b), c.byref(sl), c.byref(nw),
                                c.byref(nk)), "orc_conf_trend")
    return sl.value, nw.value, nk.value


def adapt_budget(slope: float, budget: int, step: int, max_budget: int) -> int:
    return int(lib().orc_adapt_budget(float(slope), int(budget), int(step), int(max_budget)))
