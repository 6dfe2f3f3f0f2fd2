"""Seeded synthetic inputs for the KV compression event.

This module holds NONE of the method's arithmetic (no scoring, selection,
RoPE or redirection): only random draws and the structure of the inputs —
shapes, the planted-direction blocks, the ragged history lengths, the paged
block tables.  Both the CUDA path's tests/benchmark and the oracle's tests
take their inputs from here.

Determinism: every unit tensor (one (session, layer, head) slice) is drawn
from its own ``torch.Generator`` seeded from (config seed, tensor tag, unit
index), so any unit can be regenerated alone, on the same device type,
without materialising the rest of the config.

Input recipe (the pages' workloads are agent traces on Qwen-class models;
none are available, so these stand in for them):
  * raw pre-RoPE K and V: bf16 of N(0,1) fp32 draws;
  * a seeded unit direction u per (layer, KV head) (one shared u in the tiny
    config); a seeded subset of blocks (3 % of them, or 4 fixed-count blocks
    in the tiny config) gets +alpha·u added to all 32 token keys before the
    bf16 rounding, alpha ~ U(lo, hi) per block;
  * the query window: bf16 of N(0,1) + gamma·u, with u the direction of the
    query head's KV head;
  * Mean-K of layers whose raw K is not resident is drawn directly as bf16
    of N(0, 1/32) + alpha·u (the distribution of a 32-token mean);
  * slot-map config: page size 16, a shared refcounted prefix, private pages
    in a seeded shuffled order, slot 0 the dead slot;
  * paged (ActKV) config: K/V pools of N(0,1) rows drawn for a window of
    pages and repeated periodically over the pool (the values are data, the
    periodicity changes no arithmetic and keeps generation of tens of GB
    quick), 3 % of the slots of each (layer, KV head) planted with +alpha·u,
    each request's pages a seeded shuffled subset of the pool, the current
    query token N(0,1) + gamma·u, and the attention LSE of the step stood in
    by its value for Gaussian keys, ln(n) + |q|²/(2D).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

BLOCK = 32


def _mix(*parts: int) -> int:
    """splitmix64 fold of integers → a 63-bit seed (deterministic, portable)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x + (int(p) & 0xFFFFFFFFFFFFFFFF) + 0x9E3779B97F4A7C15) \
            & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


_TAGS = {"u": 1, "plant": 2, "k": 3, "v": 4, "q": 5, "mk": 6, "hist": 7,
         "qturn": 8, "pages": 9, "kpool": 10, "vpool": 11, "lse": 12, "keep": 13,
         "logits": 14, "conftrace": 15}


def _gen(device, seed: int, tag: str, *idx: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(seed, _TAGS[tag], *idx))
    return g


def _np_rng(seed: int, tag: str, *idx: int) -> np.random.Generator:
    return np.random.default_rng(_mix(seed, _TAGS[tag], *idx))


# ----------------------------------------------------------------- Mean-K

@dataclasses.dataclass
class MeanKConfig:
    """A Mean-K-mode event: score + select + pack."""
    name: str
    L: int                    # layers scored and selected
    H: int                    # KV heads
    Hq: int                   # query heads
    D: int                    # head dim
    W: int                    # query-window tokens
    hist: List[int]           # history tokens per session (multiples of 32)
    budget: int               # kept blocks per (layer, KV head, session)
    n_sink: int
    n_recent: int
    plant_frac: float = 0.03  # fraction of blocks with a planted direction
    plant_count: int = 0      # if > 0: exactly this many planted blocks
    alpha: tuple = (2.0, 4.0)  # planted key strength range (fixed if lo==hi)
    gamma: float = 3.0        # planted query strength
    shared_u: bool = False    # one direction and one planted set for all units
    theta: float = 1e6
    pos0: int = 0
    L_pack: Optional[int] = None  # layers with raw K/V resident (packed)
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.H

    @property
    def n_sess(self) -> int:
        return len(self.hist)

    @property
    def lp(self) -> int:
        return self.L if self.L_pack is None else self.L_pack

    @property
    def n_tok(self) -> int:
        return int(sum(self.hist))

    @property
    def nb(self) -> List[int]:
        return [n // BLOCK for n in self.hist]

    @property
    def nb_total(self) -> int:
        return self.n_tok // BLOCK

    @property
    def view_tokens(self) -> int:
        return BLOCK * self.budget

    def tok_off(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.hist)]).astype(np.int64)

    def blk_off(self) -> np.ndarray:
        return self.tok_off() // BLOCK

    # --- per-unit structure (CPU, small) ---------------------------------
    def direction(self, l: int, h: int) -> np.ndarray:
        """Seeded unit vector u (fp32) of KV head h in layer l."""
        key = (0, 0) if self.shared_u else (l, h)
        g = _np_rng(self.seed, "u", *key).standard_normal(self.D)
        return (g / math.sqrt(float(np.dot(g, g)))).astype(np.float32)

    def planted(self, l: int, h: int, r: int):
        """(block indices, alpha per block) planted in unit (l, h, r)."""
        nb = self.nb[r]
        key = (0, 0, r) if self.shared_u else (l, h, r)
        rng = _np_rng(self.seed, "plant", *key)
        cnt = self.plant_count if self.plant_count > 0 else \
            int(round(self.plant_frac * nb))
        cnt = min(cnt, nb)
        blocks = np.sort(rng.choice(nb, size=cnt, replace=False))
        lo, hi = self.alpha
        alpha = rng.uniform(lo, hi, size=cnt) if hi > lo else \
            np.full(cnt, lo)
        return blocks.astype(np.int64), alpha.astype(np.float32)

    # --- unit tensors -------------------------------------------------------
    def kraw_unit(self, l: int, h: int, r: int, device="cpu") -> torch.Tensor:
        n = self.hist[r]
        x = torch.randn(n, self.D, generator=_gen(device, self.seed, "k", l, h, r),
                        device=device, dtype=torch.float32)
        blocks, alpha = self.planted(l, h, r)
        if len(blocks):
            u = torch.from_numpy(self.direction(l, h)).to(device)
            bt = torch.from_numpy(blocks).to(device)
            a = torch.from_numpy(alpha).to(device)
            xv = x.view(n // BLOCK, BLOCK, self.D)
            xv[bt] += a[:, None, None] * u[None, None, :]
        return x.to(torch.bfloat16)

    def vraw_unit(self, l: int, h: int, r: int, device="cpu") -> torch.Tensor:
        x = torch.randn(self.hist[r], self.D,
                        generator=_gen(device, self.seed, "v", l, h, r),
                        device=device, dtype=torch.float32)
        return x.to(torch.bfloat16)

    def meank_direct_unit(self, l: int, h: int, r: int,
                          device="cpu") -> torch.Tensor:
        """Mean-K drawn directly (layers without resident raw K)."""
        nb = self.nb[r]
        x = torch.randn(nb, self.D,
                        generator=_gen(device, self.seed, "mk", l, h, r),
                        device=device, dtype=torch.float32) / math.sqrt(BLOCK)
        blocks, alpha = self.planted(l, h, r)
        if len(blocks):
            u = torch.from_numpy(self.direction(l, h)).to(device)
            x[torch.from_numpy(blocks).to(device)] += \
                torch.from_numpy(alpha).to(device)[:, None] * u[None, :]
        return x.to(torch.bfloat16)

    def q_unit(self, r: int, l: int, hq: int, device="cpu", step: int = 0) -> torch.Tensor:
        """Query window of agent step `step` (0: the event's window; later
        steps draw new noise around the same planted directions)."""
        key = (r, l, hq) if step == 0 else (r, l, hq, step)
        x = torch.randn(self.W, self.D,
                        generator=_gen(device, self.seed, "q", *key),
                        device=device, dtype=torch.float32)
        u = torch.from_numpy(self.direction(l, hq // self.G)).to(device)
        return (x + self.gamma * u[None, :]).to(torch.bfloat16)

    # --- whole tensors --------------------------------------------------
    def q(self, device="cpu", step: int = 0) -> torch.Tensor:
        """bf16 [L][n_sess][Hq][W][D] query windows (layer-major)."""
        out = torch.empty(self.L, self.n_sess, self.Hq, self.W, self.D,
                          dtype=torch.bfloat16, device=device)
        for l in range(self.L):
            for r in range(self.n_sess):
                for hq in range(self.Hq):
                    out[l, r, hq] = self.q_unit(r, l, hq, device, step)
        return out

    def kv_raw(self, device="cpu"):
        """(kraw, vraw) bf16 [lp][H][n_tok][D] for the resident layers."""
        shape = (self.lp, self.H, self.n_tok, self.D)
        kraw = torch.empty(shape, dtype=torch.bfloat16, device=device)
        vraw = torch.empty(shape, dtype=torch.bfloat16, device=device)
        off = self.tok_off()
        for l in range(self.lp):
            for h in range(self.H):
                for r in range(self.n_sess):
                    kraw[l, h, off[r]:off[r + 1]] = self.kraw_unit(l, h, r, device)
                    vraw[l, h, off[r]:off[r + 1]] = self.vraw_unit(l, h, r, device)
        return kraw, vraw

    def meank_direct(self, device="cpu") -> torch.Tensor:
        """bf16 [L][H][nb_total][D]; rows of layers < lp are left zero (the
        caller builds them from raw K)."""
        out = torch.zeros(self.L, self.H, self.nb_total, self.D,
                          dtype=torch.bfloat16, device=device)
        boff = self.blk_off()
        for l in range(self.lp, self.L):
            for h in range(self.H):
                for r in range(self.n_sess):
                    out[l, h, boff[r]:boff[r + 1]] = \
                        self.meank_direct_unit(l, h, r, device)
        return out

    def seg_off(self) -> np.ndarray:
        """Select segments ordered (l, h, r), r fastest, over [L][H][nb_total]."""
        boff = self.blk_off()
        offs = [0]
        for l in range(self.L):
            for h in range(self.H):
                base = (l * self.H + h) * self.nb_total
                for r in range(self.n_sess):
                    offs.append(base + int(boff[r + 1]))
        return np.asarray(offs, dtype=np.int64)


def _ragged_hist(seed: int, n_sess: int, lo: int, hi: int) -> List[int]:
    rng = _np_rng(seed, "hist")
    raw = rng.integers(lo, hi + 1, size=n_sess)
    return [int(BLOCK * (int(x) // BLOCK)) for x in raw]


# Planted query strength for the 3 %-planted configs, chosen (on the oracle)
# so that the top-8 blocks of a (layer, KV head) hold about 65 % of the
# score mass, the concentration KVMem reports for real traces.
GAMMA_PLANTED = 67.5


def config_tiny() -> MeanKConfig:
    """1 layer, 2 KV / 4 query heads, D 64, 4096-token history, 16-query
    window, q = N(0,1) + 3u, 4 blocks planted with +3u; 16 kept blocks
    (1 sink, 2 recent); view at positions 0..511."""
    return MeanKConfig(name="tiny", L=1, H=2, Hq=4, D=64, W=16, hist=[4096],
                       budget=16, n_sink=1, n_recent=2, plant_count=4,
                       alpha=(3.0, 3.0), gamma=3.0, shared_u=True, seed=0)


def config_8b() -> MeanKConfig:
    """8B-class single session: 36 layers, 8 KV / 32 query heads, D 128,
    131072-token history, 32-query window, 256 kept blocks (1 sink, 4
    recent), view at positions 0..8191."""
    return MeanKConfig(name="8b_128k", L=36, H=8, Hq=32, D=128, W=32,
                       hist=[131072], budget=256, n_sink=1, n_recent=4,
                       gamma=GAMMA_PLANTED, seed=1)


def config_27b() -> MeanKConfig:
    """27B-class 1M-token workspace: 64 layers scored, 8 KV / 48 query heads,
    D 128, 1048576 tokens, 2048 kept blocks (1 sink, 8 recent); raw K/V
    resident and packed for 16 layers."""
    return MeanKConfig(name="27b_1m", L=64, H=8, Hq=48, D=128, W=32,
                       hist=[1048576], budget=2048, n_sink=1, n_recent=8,
                       gamma=GAMMA_PLANTED, L_pack=16, seed=2)


def config_ragged(n_sess: int = 128, L_pack: int = 2) -> MeanKConfig:
    """Batched ragged step: 128 sessions of U[16384, 262144] tokens (rounded
    down to 32), 8B-class heads, 512 kept blocks (1 sink, 4 recent); all 36
    layers scored and selected, raw K/V packed for L_pack layers."""
    return MeanKConfig(name="ragged_128", L=36, H=8, Hq=32, D=128, W=32,
                       hist=_ragged_hist(4, n_sess, 16384, 262144),
                       budget=512, n_sink=1, n_recent=4, gamma=GAMMA_PLANTED,
                       L_pack=L_pack, seed=4)


def scaled(cfg: MeanKConfig, **kw) -> MeanKConfig:
    """Same recipe, smaller sizes (for oracle-speed parity cases)."""
    return dataclasses.replace(cfg, **kw)


# -------------------------------------------------------------- slot map

@dataclasses.dataclass
class SlotMapConfig:
    """A QueryMemory-mode event: score + select + redirect/free."""
    name: str
    n_sess: int
    N: int            # logical positions per session (prefix included)
    prefix: int       # shared, refcounted prefix positions
    page: int         # slots per page
    L: int
    H: int
    Hq: int
    D: int
    T: int            # query tokens per turn
    turns: int
    budget: int       # kept positions per session
    decay: float = 0.9
    gain: float = 0.1
    seed: int = 3
    sentinel: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.H

    @property
    def private_pages(self) -> int:
        return (self.N - self.prefix) // self.page

    @property
    def n_pages(self) -> int:
        # page 0 holds the dead slot; then the prefix pages; then private pages
        return 1 + self.prefix // self.page + self.n_sess * self.private_pages

    @property
    def n_slots(self) -> int:
        return self.n_pages * self.page

    def block_tables(self) -> np.ndarray:
        """[n_sess][N/page] int32 physical page ids (seeded shuffled private
        pages, shared prefix pages)."""
        pp = self.prefix // self.page
        first_private = 1 + pp
        perm = _np_rng(self.seed, "pages").permutation(
            self.n_sess * self.private_pages) + first_private
        bt = np.empty((self.n_sess, self.N // self.page), dtype=np.int32)
        for r in range(self.n_sess):
            bt[r, :pp] = np.arange(1, 1 + pp)
            bt[r, pp:] = perm[r * self.private_pages:(r + 1) * self.private_pages]
        return bt

    def slot_maps(self, block_tables: Optional[np.ndarray] = None) -> np.ndarray:
        """[n_sess][N] int32: page-table expansion (position p → slot
        bt[p / page]·page + p % page)."""
        bt = self.block_tables() if block_tables is None else block_tables
        p = np.arange(self.N)
        # the fancy index leaves a column-major array: hand out row-major
        return np.ascontiguousarray(
            (bt[:, p // self.page] * self.page + p % self.page).astype(np.int32))

    def refcounts(self, slot_maps: np.ndarray) -> np.ndarray:
        """One count per slot-map reference; the dead slot holds none."""
        rc = np.bincount(slot_maps.reshape(-1), minlength=self.n_slots)
        rc = rc.astype(np.int32)
        rc[self.sentinel] = 0
        return rc

    def kpool_layer(self, l: int, device="cpu", slots=None) -> torch.Tensor:
        """bf16 [n_slots][H][D] N(0,1) K rows of layer l (drawn per page
        chunk so any slice can be regenerated alone)."""
        out = torch.empty(self.n_slots, self.H, self.D, dtype=torch.bfloat16,
                          device=device)
        chunk = 1 << 16
        for c0 in range(0, self.n_slots, chunk):
            c1 = min(self.n_slots, c0 + chunk)
            out[c0:c1] = torch.randn(
                c1 - c0, self.H, self.D, dtype=torch.float32, device=device,
                generator=_gen(device, self.seed, "kpool", l, c0 // chunk)
            ).to(torch.bfloat16)
        return out

    def q_turn(self, t: int, device="cpu") -> torch.Tensor:
        """bf16 [n_sess][L][Hq][T][D] pre-RoPE queries of turn t."""
        return torch.randn(self.n_sess, self.L, self.Hq, self.T, self.D,
                           generator=_gen(device, self.seed, "qturn", t),
                           device=device, dtype=torch.float32
                           ).to(torch.bfloat16)


def config_slotmap() -> SlotMapConfig:
    """64 sessions sharing a refcounted 4096-token prefix, 32768 positions
    each (prefix included), page size 16, 8B-class heads, 4 turns of 32
    query tokens, 8192 kept positions per session."""
    return SlotMapConfig(name="slotmap_64x32k", n_sess=64, N=32768,
                         prefix=4096, page=16, L=36, H=8, Hq=32, D=128, T=32,
                         turns=4, budget=8192)


# ------------------------------------------------------------ paged (ActKV)

@dataclasses.dataclass
class PagedConfig:
    """An ActKV compression operation on a paged KV cache: one LSE-recovery
    step, keep the top `keep` tokens of each request, tail compaction."""
    name: str
    n_req: int
    seq: int               # tokens per request before compression
    keep: int              # tokens kept per request
    BS: int = 16           # slots per block
    L: int = 36
    H: int = 8
    Hq: int = 32
    D: int = 128
    spare_blocks: int = 64  # free blocks of the pool (not owned by a request)
    count: int = 1         # action-token index of the timed step
    plant_frac: float = 0.03
    alpha: tuple = (2.0, 4.0)
    gamma: float = 3.0
    window_blocks: int = 4096  # distinct pages drawn per layer (then repeated)
    seed: int = 5

    @property
    def G(self) -> int:
        return self.Hq // self.H

    @property
    def max_blocks(self) -> int:
        return (self.seq + self.BS - 1) // self.BS

    @property
    def cap(self) -> int:
        return self.max_blocks * self.BS

    @property
    def n_blocks(self) -> int:
        return self.n_req * self.max_blocks + self.spare_blocks

    @property
    def n_slots(self) -> int:
        return self.n_blocks * self.BS

    def block_tables(self) -> np.ndarray:
        """[n_req][max_blocks] int32: a seeded shuffled assignment of the
        pool's blocks (row-major)."""
        perm = _np_rng(self.seed, "pages").permutation(self.n_blocks)
        bt = perm[:self.n_req * self.max_blocks].reshape(self.n_req, self.max_blocks)
        return np.ascontiguousarray(bt.astype(np.int32))

    def seqused(self) -> np.ndarray:
        return np.full(self.n_req, self.seq, dtype=np.int32)

    def direction(self, l: int, h: int) -> np.ndarray:
        g = _np_rng(self.seed, "u", l, h).standard_normal(self.D)
        return (g / math.sqrt(float(np.dot(g, g)))).astype(np.float32)

    def _pool_layer(self, tag: str, l: int, device, plant: bool) -> torch.Tensor:
        n_win = min(self.window_blocks, self.n_blocks) * self.BS
        base = torch.randn(n_win, self.H, self.D, dtype=torch.float32, device=device,
                           generator=_gen(device, self.seed, tag, l))
        if plant:
            rng = _np_rng(self.seed, "plant", l)
            for h in range(self.H):
                cnt = int(round(self.plant_frac * n_win))
                idx = torch.from_numpy(rng.choice(n_win, size=cnt, replace=False)).to(device)
                a = torch.from_numpy(rng.uniform(*self.alpha, size=cnt).astype(np.float32))
                u = torch.from_numpy(self.direction(l, h)).to(device)
                base[idx, h] += a.to(device)[:, None] * u[None, :]
        base = base.to(torch.bfloat16)
        out = torch.empty(self.n_slots, self.H, self.D, dtype=torch.bfloat16, device=device)
        for c0 in range(0, self.n_slots, n_win):
            c1 = min(self.n_slots, c0 + n_win)
            out[c0:c1] = base[:c1 - c0]
        return out

    def pools(self, device="cpu"):
        """(kpool, vpool) bf16 [L][n_slots][H][D]."""
        shape = (self.L, self.n_slots, self.H, self.D)
        kp = torch.empty(shape, dtype=torch.bfloat16, device=device)
        vp = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for l in range(self.L):
            kp[l] = self._pool_layer("kpool", l, device, True)
            vp[l] = self._pool_layer("vpool", l, device, False)
        return kp, vp

    def q(self, device="cpu") -> torch.Tensor:
        """bf16 [n_req][L][Hq][D]: the current (action) query token."""
        x = torch.randn(self.n_req, self.L, self.Hq, self.D, dtype=torch.float32,
                        device=device, generator=_gen(device, self.seed, "q"))
        u = torch.stack([torch.stack([torch.from_numpy(self.direction(l, hq // self.G))
                                      for hq in range(self.Hq)]) for l in range(self.L)])
        return (x + self.gamma * u.to(device)[None]).to(torch.bfloat16)

    def lse(self, q: torch.Tensor) -> torch.Tensor:
        """fp32 [n_req][L][Hq] stand-in for the backend's LSE of the step:
        ln(seq) + |q|²/(2D), the log-partition of Gaussian keys."""
        qf = q.float()
        return (math.log(self.seq) + (qf * qf).sum(-1) / (2.0 * self.D)).contiguous()


def config_paged(n_req: int = 64) -> PagedConfig:
    """ActKV Table 1 shapes: block size 16, 8 KV heads, head dim 128; n_req
    concurrent requests, each compressed from 6K to 4K entries; 8B-class
    depth (36 layers, 32 query heads)."""
    return PagedConfig(name=f"paged_r{n_req}_6k_to_4k", n_req=n_req, seq=6144, keep=4096)


# ------------------------------------------------- confidence monitor

@dataclasses.dataclass
class ConfidenceConfig:
    """ActKV's confidence monitor on one decode step of n_req requests (one
    row of logits each, Qwen-class vocabulary), and the trend over each
    request's trace of token confidences."""
    name: str = "conf_64x151936"
    n_req: int = 64
    vocab: int = 151936
    top_k: int = 20
    trace_len: int = 8192
    window: int = 128
    stride: int = 32
    bottom_pct: float = 10.0
    budget0: int = 1024
    budget_step: int = 256
    max_budget: int = 8192
    seed: int = 6

    def logits(self, device="cpu") -> torch.Tensor:
        """fp32 [n_req][vocab]: N(0, 2²) logits, plus per row a few tokens
        lifted by U(4, 12) (a peaked head, as sampled text has)."""
        g = _gen(device, self.seed, "logits")
        x = torch.randn(self.n_req, self.vocab, generator=g, device=device) * 2.0
        rng = _np_rng(self.seed, "logits", 1)
        for r in range(self.n_req):
            idx = torch.from_numpy(rng.choice(self.vocab, 8, replace=False)).to(device)
            x[r, idx] += torch.from_numpy(rng.uniform(4, 12, 8).astype(np.float32)).to(device)
        return x.contiguous()

    def traces(self, device="cpu") -> torch.Tensor:
        """fp32 [n_req][trace_len] token confidences: noise around a level
        with a seeded drift per request (half of them falling)."""
        rng = _np_rng(self.seed, "conftrace")
        t = np.linspace(0.0, 1.0, self.trace_len)
        rows = [rng.normal(12.0, 0.6, self.trace_len) - rng.normal(0.0, 1.0) * t
                for _ in range(self.n_req)]
        return torch.from_numpy(np.stack(rows).astype(np.float32)).to(device)


# ---------------------------------------------------------------- helpers

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor → numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns → bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).to(device)
