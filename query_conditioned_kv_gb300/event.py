"""One compression event as a user runs it: buffers plus the C-ABI calls.

``MeanKEvent``   score (Mean-K) → select → pack + re-RoPE
``SlotMapEvent`` score (QueryMemory) → select → redirect + free
``PagedEvent``   LSE-recovery score → LRFU keep score → select → tail plan →
                 in-place compaction
``TieredMeanKEvent`` the Mean-K event with the index and the raw history in
                 host memory: score in bounded layer tiles, select, tiered pack

Both only allocate caller-side buffers with torch and call the library's
entry points; an event can be captured in a CUDA graph (``capture()``) so
that its launches replay without host overhead.

``MeanKEvent.run`` pipelines over groups of layers: the score of group g+1
(tensor-core and exponential heavy) runs on the caller's stream while the
select and pack of group g (latency-bound, then HBM-bound streaming) run on a
second stream, so the two kinds of work share the SMs instead of taking
turns.  Every call
covers whole layers, which is possible because every tensor is laid out
layer-major.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import (BLOCK_TOKENS, kvc_pack_rerope, kvc_pack_tiered, kvc_pack_tiered_slots,
               kvc_repo_plan, kvc_recover_score_ex,
               kvc_recover_score_workspace_size, kvc_score_ex, kvc_score_qmem_ex,
               kvc_redirect_free,
               kvc_redirect_free_workspace_size, kvc_rope_table, kvc_score,
               kvc_lrfu_update, kvc_score_qmem, kvc_score_qmem_workspace_size,
               kvc_score_workspace_size, kvc_select, kvc_tail_compact, kvc_tail_plan)


def _dev_i64(x, device) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.int64), device=device)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def groups_hint(L: int) -> int:
    """Layer groups of the event.  One group (score all layers, then select,
    then pack) measures fastest on GB300 for the 8B-class event: the
    tensor-core scorer fills every SM's registers, so a concurrent pack could
    not share the SMs anyway, and a single persistent score launch balances
    its units best.  More groups remain available for experiments."""
    return 1


class MeanKEvent:
    """Buffers and calls of a Mean-K-mode event over ragged sessions.

    Layouts (see include/kvc.h): q [L][n_sess][Hq][W][D], meank
    [L][H][nb_total][D], kraw/vraw [L_pack][H][n_tok][D]; outputs scores
    [L][H][nb_total], kept [L][H][n_sess][budget], kview/vview
    [L_pack][H][n_sess][32·budget][D].  Pack runs on the first L_pack layers.
    """

    def __init__(self, L: int, H: int, Hq: int, D: int, W: int,
                 hist: Sequence[int], budget: int, n_sink: int, n_recent: int,
                 L_pack: Optional[int] = None, theta: float = 1e6,
                 pos0: int = 0, keepmask: bool = False, device="cuda",
                 groups: Optional[int] = None):
        self.L, self.H, self.Hq, self.D, self.W = L, H, Hq, D, W
        self.hist = [int(n) for n in hist]
        if any(n % BLOCK_TOKENS for n in self.hist):
            raise ValueError("history lengths must be multiples of 32 tokens")
        self.n_sess = len(self.hist)
        self.budget, self.n_sink, self.n_recent = budget, n_sink, n_recent
        self.L_pack = L if L_pack is None else L_pack
        self.device = torch.device(device)
        tok_off = np.concatenate([[0], np.cumsum(self.hist)]).astype(np.int64)
        blk_off = tok_off // BLOCK_TOKENS
        self.n_tok = int(tok_off[-1])
        self.nb_total = int(blk_off[-1])
        self.nb_max = max(n // BLOCK_TOKENS for n in self.hist)
        seg = [0]
        for l in range(L):
            for h in range(H):
                base = (l * H + h) * self.nb_total
                for r in range(self.n_sess):
                    seg.append(base + int(blk_off[r + 1]))
        self.n_seg = L * H * self.n_sess
        dev = self.device
        self.tok_off = _dev_i64(tok_off, dev)
        self.blk_off = _dev_i64(blk_off, dev)
        self.seg_off = _dev_i64(seg, dev)
        self.scores = torch.empty(L, H, self.nb_total, dtype=torch.float32, device=dev)
        self.kept = torch.empty(L, H, self.n_sess, budget, dtype=torch.int32, device=dev)
        self.kept_count = torch.empty(L, H, self.n_sess, dtype=torch.int32, device=dev)
        words = (self.nb_max + 31) // 32
        self.keepmask = (torch.empty(self.n_seg, words, dtype=torch.int32, device=dev)
                         if keepmask else None)
        self.ws = _ws(kvc_score_workspace_size(L, H, Hq, W, self.n_sess, self.nb_max,
                                               self.nb_total), dev)
        self.view_tokens = BLOCK_TOKENS * budget
        self.rope_tab = torch.empty(self.view_tokens, D // 2, 2, dtype=torch.float32,
                                    device=dev)
        kvc_rope_table(self.rope_tab, self.view_tokens, pos0, D, theta)
        shape = (self.L_pack, H, self.n_sess, self.view_tokens, D)
        self.kview = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        self.vview = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None
        self.side = torch.cuda.Stream(device=dev)
        self.groups = self._layer_groups(groups_hint(L) if groups is None else groups)
        self.score_kernel = "auto"  # the scorer run() uses (a kvc_kernel name)

    @staticmethod
    def _split(L: int, n: int):
        n = max(1, min(n, L))
        edges = [round(i * L / n) for i in range(n + 1)]
        return [(edges[i], edges[i + 1]) for i in range(n) if edges[i + 1] > edges[i]]

    def _layer_groups(self, n: int):
        return self._split(self.L, n)

    # -- the three steps, on a range of layers [l0, l1) ------------------
    def score(self, q, meank, stream=None, l0=0, l1=None, kernel=None):
        """Scores of layers [l0, l1); `kernel` names one scorer (kvc_score_ex);
        by default the event's `score_kernel` ("auto": the library's choice)."""
        l1 = self.L if l1 is None else l1
        kernel = self.score_kernel if kernel is None else kernel
        kvc_score_ex(q[l0:l1], meank[l0:l1], self.scores[l0:l1], l1 - l0, self.H, self.Hq,
                     self.D, self.W, self.blk_off, self.n_sess, self.nb_total, self.nb_max,
                     self.ws, kernel, self.dev_status, stream)

    def select(self, scores=None, stream=None, l0=0, l1=None):
        l1 = self.L if l1 is None else l1
        per = self.H * self.n_sess
        kvc_select(self.scores if scores is None else scores,
                   self.seg_off[l0 * per:l1 * per + 1], (l1 - l0) * per, self.nb_max,
                   self.budget, self.n_sink, self.n_recent, self.kept[l0:l1],
                   self.kept_count[l0:l1],
                   None if self.keepmask is None else self.keepmask[l0 * per:l1 * per],
                   self.dev_status, stream)

    def pack(self, kraw, vraw, kept=None, kept_count=None, stream=None, l0=0, l1=None):
        l1 = self.L_pack if l1 is None else min(l1, self.L_pack)
        if l1 <= l0:
            return
        kept = self.kept if kept is None else kept
        kept_count = self.kept_count if kept_count is None else kept_count
        kvc_pack_rerope(kraw[l0:l1], vraw[l0:l1], kept[l0:l1], kept_count[l0:l1],
                        l1 - l0, self.H, self.D, self.tok_off, self.n_sess, self.n_tok,
                        self.budget, self.rope_tab, self.kview[l0:l1], self.vview[l0:l1],
                        self.dev_status, stream)

    def run_serial(self, q, meank, kraw, vraw, stream=None):
        """score → select → pack over all layers, one stream."""
        self.score(q, meank, stream)
        self.select(stream=stream)
        self.pack(kraw, vraw, stream=stream)

    def run(self, q, meank, kraw, vraw, timers=None):
        """The event, layer groups pipelined over two streams (asynchronous
        with respect to the host; ordered after prior work on the current
        stream, and the current stream waits for all of it).  With one layer
        group every launch stays on the current stream.  `timers`, if
        given, is a list that receives (stage, start, end) CUDA events around
        every launch, recorded on the launching stream."""
        main = torch.cuda.current_stream(self.device)
        side = self.side if len(self.groups) > 1 else main
        if side is not main:
            side.wait_stream(main)

        def timed(stage, stream, fn):
            if timers is None:
                fn()
                return
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            timers.append((stage, a, b))

        for (l0, l1) in self.groups:
            timed("score", main, lambda: self.score(q, meank, main, l0, l1))
            if side is not main:
                done = torch.cuda.Event()
                done.record(main)
                side.wait_event(done)
            with torch.cuda.stream(side):
                timed("select", side, lambda: self.select(None, side, l0, l1))
                if l0 < self.L_pack:
                    timed("pack", side, lambda: self.pack(kraw, vraw, stream=side, l0=l0, l1=l1))
        if side is not main:
            main.wait_stream(side)

    # -- CUDA graph ----------------------------------------------------
    def capture(self, q, meank, kraw, vraw):
        """Capture run() on these input tensors; replay() re-runs it."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.run(q, meank, kraw, vraw)  # warm-up (sets kernel attributes)
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(q, meank, kraw, vraw)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()


class TieredMeanKEvent(MeanKEvent):
    """KVMem's tiered execution view ("Tiered movement"): the Mean-K index and
    the raw K/V history stay in pinned host memory; only the execution view,
    the scores and this event's scratch live on the GPU.

    score   the index is scored in bounded tiles of `stage_layers` layers:
            each tile is copied host → device into one of two staging
            buffers on a copy stream while the previous tile is scored on
            the current stream (the scorer is the device-resident one, and
            a unit's partial sums merge in one order whatever else a launch
            holds, so the scores are the same bit for bit);
    select  as MeanKEvent;
    pack    kvc_pack_tiered: blocks that the previous step also kept come
            from the previous view (raw K from a raw-K cache, V from the V
            view), the others are read by the kernel from host memory.
    Two sets of (kept lists, raw-K cache, V view) alternate between steps.
    """

    def __init__(self, *args, stage_layers: int = 4, **kw):
        super().__init__(*args, **kw)
        dev = self.device
        self.stage_layers = max(1, min(stage_layers, self.L))
        self.stage = [torch.empty(self.stage_layers, self.H, self.nb_total, self.D,
                                  dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.kept_sets = [self.kept, torch.empty_like(self.kept)]
        self.count_sets = [self.kept_count, torch.empty_like(self.kept_count)]
        self.kcaches = [torch.empty_like(self.kview), torch.empty_like(self.kview)]
        self.vviews = [self.vview, torch.empty_like(self.vview)]
        self.n_hits = torch.zeros(1, dtype=torch.int32, device=dev)
        self.cur, self.steps = 0, 0
        # per staging buffer: an event after the last score that read it
        # (kept across calls, so the next step's first copies need wait only
        # for that, not for the previous step's select and pack)
        self.stage_free = [None, None]

    def score_tiered(self, q, meank_host, after_tile=None):
        """Scores of every layer from the host-resident index [L][H][nb][D].
        `after_tile(l0, l1)`, if given, is called after each tile's score is
        queued (on the current stream, while the copy stream brings in the
        next tiles)."""
        main = torch.cuda.current_stream(self.device)
        cs = self.copy_stream
        free = self.stage_free
        for gi, (l0, l1) in enumerate(self._split(self.L, -(-self.L // self.stage_layers))):
            b = gi % 2
            n = l1 - l0
            with torch.cuda.stream(cs):
                if free[b] is not None:
                    cs.wait_event(free[b])
                self.stage[b][:n].copy_(meank_host[l0:l1], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(cs)
            main.wait_event(ready)
            kvc_score(q[l0:l1], self.stage[b][:n], self.scores[l0:l1], n, self.H, self.Hq,
                      self.D, self.W, self.blk_off, self.n_sess, self.nb_total, self.nb_max,
                      self.ws, self.dev_status, main)
            free[b] = torch.cuda.Event()
            free[b].record(main)
            if after_tile is not None:
                after_tile(l0, l1)

    def pack_tiered(self, kraw_host, vraw_host, l0=0, l1=None):
        """The tiered pack of packed layers [l0, l1) (all of them by default)."""
        l1 = self.L_pack if l1 is None else min(l1, self.L_pack)
        if l1 <= l0:
            return
        cur, prev = self.cur, 1 - self.cur
        first = self.steps == 0
        sl = slice(l0, l1)
        kvc_pack_tiered(kraw_host[sl], vraw_host[sl],
                        None if first else self.kept_sets[prev][sl],
                        None if first else self.count_sets[prev][sl],
                        None if first else self.kcaches[prev][sl],
                        None if first else self.vviews[prev][sl],
                        self.kept_sets[cur][sl], self.count_sets[cur][sl],
                        l1 - l0, self.H, self.D, self.tok_off, self.n_sess, self.n_tok,
                        self.budget, self.rope_tab, self.kcaches[cur][sl], self.kview[sl],
                        self.vviews[cur][sl], self.n_hits, self.dev_status)

    def step(self, q, meank_host, kraw_host, vraw_host, pipelined=True):
        """One agent step; afterwards kview / vview hold this step's view.
        Pipelined (the default): each index tile's select and pack are queued
        right after its score, so they run while the copy stream brings in
        the next tiles (layers are independent: the same outputs bit for bit
        as score, select, pack one after another)."""
        cur = self.cur
        self.kept, self.kept_count = self.kept_sets[cur], self.count_sets[cur]
        self.vview = self.vviews[cur]
        if pipelined:
            main = torch.cuda.current_stream(self.device)

            def tile(l0, l1):
                self.select(stream=main, l0=l0, l1=l1)
                self.pack_tiered(kraw_host, vraw_host, l0, l1)

            self.score_tiered(q, meank_host, after_tile=tile)
        else:
            self.score_tiered(q, meank_host)
            self.select()
            self.pack_tiered(kraw_host, vraw_host)
        self.cur, self.steps = 1 - cur, self.steps + 1


class RepoTieredEvent(TieredMeanKEvent):
    """KVMem's tiered view with its repository view ("Tiered movement": the
    repository view tracks where each block lives, blocks recalled often
    prefer host RAM over NVMe).  The raw history lives in a KvcRepo: every
    block in its backing file, the most-used ones in host slots.  A step
    scores and selects as TieredMeanKEvent, copies the packed layers' kept
    lists to the host, plans the blocks the step uses and the ones it misses
    (kvc_repo_plan), brings the misses into host slots (kvc_repo_step: one
    vectored read per run of consecutive blocks), applies the slots that
    changed to the slot table it keeps on the GPU, and packs with
    kvc_pack_tiered_slots, which reuses the previous view on the GPU and reads
    only the misses from the slots.  The repository holds the L_pack packed
    layers: repo.L == L_pack, repo.n_blocks == n_tok / 32."""

    def __init__(self, *args, repo, **kw):
        super().__init__(*args, **kw)
        if repo.L != self.L_pack or repo.H != self.H or repo.D != self.D or \
                repo.n_blocks * BLOCK_TOKENS != self.n_tok:
            raise ValueError("the repository must hold the packed layers of this history")
        self.repo = repo
        # the slot table stays on the GPU; each step applies only its changes
        self.host_slot = torch.from_numpy(repo.slot_table().copy()).to(self.device)
        self.tok_off_host = self.tok_off.cpu().numpy()
        self.prev_host = None
        self.last_plan = (0, 0)  # (blocks used, blocks missed) of the last step

    def pack_repo(self):
        cur, prev = self.cur, 1 - self.cur
        first = self.steps == 0
        Lp = self.L_pack
        kept = self.kept_sets[cur][:Lp].cpu().numpy().reshape(-1)
        cnt = self.count_sets[cur][:Lp].cpu().numpy().reshape(-1)
        kp, cp = (None, None) if first else self.prev_host
        used, need = kvc_repo_plan(kept, cnt, kp, cp, Lp, self.H, self.n_sess, self.budget,
                                   self.tok_off_host, self.repo.n_blocks)
        self.repo.step(used, need, table=False)
        units, slots = self.repo.changes()
        if len(units):
            self.host_slot[torch.from_numpy(units).to(self.device)] = \
                torch.from_numpy(slots).to(self.device)
        ks, vs = self.repo.slots()
        kvc_pack_tiered_slots(ks, vs, self.repo.slot_elems, self.repo.n_slots, self.host_slot,
                              None if first else self.kept_sets[prev][:Lp],
                              None if first else self.count_sets[prev][:Lp],
                              None if first else self.kcaches[prev],
                              None if first else self.vviews[prev],
                              self.kept_sets[cur][:Lp], self.count_sets[cur][:Lp], Lp, self.H,
                              self.D, self.tok_off, self.n_sess, self.n_tok, self.budget,
                              self.rope_tab, self.kcaches[cur], self.kview, self.vviews[cur],
                              self.n_hits, self.dev_status)
        self.prev_host = (kept, cnt)
        self.last_plan = (len(used), len(need))

    def step(self, q, meank_host):
        """One agent step; afterwards kview / vview hold this step's view."""
        cur = self.cur
        self.kept, self.kept_count = self.kept_sets[cur], self.count_sets[cur]
        self.vview = self.vviews[cur]
        self.score_tiered(q, meank_host)
        self.select()
        self.pack_repo()
        self.cur, self.steps = 1 - cur, self.steps + 1


def event_bytes(L: int, H: int, Hq: int, D: int, W: int, nb_total: int, n_sess: int,
                L_pack: int, view_tokens: int, budget: int) -> dict:
    """Bytes a Mean-K event must move through HBM, by stage: the Mean-K index
    and the query windows read once (score); the kept K and V rows read once
    and the execution views written once, plus the kept indices (pack).
    Select reads only the scores, which the score stage has just written."""
    meank = L * H * nb_total * D * 2
    q = n_sess * L * Hq * W * D * 2
    view = L_pack * H * n_sess * view_tokens * D
    pack = 2 * 2 * view * 2 + L * H * n_sess * budget * 4
    return {"score": meank + q, "select": 0, "pack": pack, "event": meank + q + pack}


class SlotMapEvent:
    """Buffers and calls of a QueryMemory-mode event: rule score over the
    paged K pool, token-level select (no forced set), redirect + free."""

    def __init__(self, n_sess: int, N: int, L: int, H: int, Hq: int, D: int,
                 n_slots: int, budget: int, prefix_len: int, sentinel: int = 0,
                 freed_cap: Optional[int] = None, device="cuda"):
        self.n_sess, self.N, self.L, self.H, self.Hq, self.D = n_sess, N, L, H, Hq, D
        self.n_slots, self.budget = n_slots, budget
        self.prefix_len, self.sentinel = prefix_len, sentinel
        dev = self.device = torch.device(device)
        self.rule = torch.empty(n_sess, N, dtype=torch.float32, device=dev)
        self.seg_off = _dev_i64(np.arange(n_sess + 1) * N, dev)
        self.kept = torch.empty(n_sess, budget, dtype=torch.int32, device=dev)
        self.kept_count = torch.empty(n_sess, dtype=torch.int32, device=dev)
        self.words = (N + 31) // 32
        self.keepmask = torch.empty(n_sess, self.words, dtype=torch.int32, device=dev)
        self.ws_score = _ws(kvc_score_qmem_workspace_size(n_sess, L, Hq, N), dev)
        self.ws_free = _ws(kvc_redirect_free_workspace_size(n_sess, N, n_slots), dev)
        self.freed_cap = n_slots if freed_cap is None else freed_cap
        self.freed = torch.empty(max(self.freed_cap, 1), dtype=torch.int32, device=dev)
        self.n_freed = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def score(self, M, kpool, slot_map, stream=None, kernel="auto"):
        kvc_score_qmem_ex(M, kpool, slot_map, self.sentinel, self.rule, self.n_sess,
                          self.L, self.H, self.Hq, self.D, self.N, self.n_slots,
                          self.ws_score, kernel, self.dev_status, stream)

    def select(self, rule=None, stream=None):
        kvc_select(self.rule if rule is None else rule, self.seg_off, self.n_sess,
                   self.N, self.budget, 0, 0, self.kept, self.kept_count,
                   self.keepmask, self.dev_status, stream)

    def redirect(self, slot_map, refcnt, keepmask=None, stream=None):
        kvc_redirect_free(slot_map, self.keepmask if keepmask is None else keepmask,
                          self.n_sess, self.N, refcnt, self.n_slots, self.prefix_len,
                          self.sentinel, self.freed, self.freed_cap, self.n_freed,
                          self.ws_free, self.dev_status, stream)

    def run(self, M, kpool, slot_map, refcnt, stream=None):
        self.score(M, kpool, slot_map, stream)
        self.select(stream=stream)
        self.redirect(slot_map, refcnt, stream=stream)


class PagedEvent:
    """Buffers and calls of an ActKV compression operation on a paged KV
    cache (ActKV §3.3 on the §2 layout): LSE-recovery score of the current
    action token (§7.1), the LRFU keep score at the end of the action region
    (§5.2), token-level select of `keep` tokens per request by keep score (no
    forced set), conflict-free tail plan and one-shot in-place compaction
    (§7.2).  All requests have max_blocks·block_size positions; select takes
    each request's whole row as its segment."""

    def __init__(self, n_req: int, max_blocks: int, block_size: int, L: int, H: int,
                 Hq: int, D: int, n_slots: int, keep: int, device="cuda"):
        self.n_req, self.max_blocks, self.BS = n_req, max_blocks, block_size
        self.L, self.H, self.Hq, self.D = L, H, Hq, D
        self.n_slots, self.keep = n_slots, keep
        self.cap = max_blocks * block_size
        dev = self.device = torch.device(device)
        self.state = torch.zeros(n_req, self.cap, dtype=torch.float32, device=dev)
        self.keep_score = torch.zeros(n_req, self.cap, dtype=torch.float32, device=dev)
        wsb = kvc_recover_score_workspace_size(n_req, max_blocks, L, H, Hq, D, block_size)
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        self.seg_off = _dev_i64(np.arange(n_req + 1) * self.cap, dev)
        self.kept = torch.empty(n_req, keep, dtype=torch.int32, device=dev)
        self.kept_count = torch.empty(n_req, dtype=torch.int32, device=dev)
        self.words = (self.cap + 31) // 32
        self.keepmask = torch.empty(n_req, self.words, dtype=torch.int32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.src = torch.empty(n_req, self.cap, **i32)
        self.dst = torch.empty(n_req, self.cap, **i32)
        self.n_pairs = torch.empty(n_req, **i32)
        self.n_tail = torch.empty(n_req, **i32)
        self.freed = torch.empty(n_req, max_blocks, **i32)
        self.n_freed = torch.empty(n_req, **i32)
        self.new_table = torch.empty(n_req, max_blocks, **i32)
        self.tail_mask = torch.empty(n_req, self.words, **i32)
        self.dev_status = torch.zeros(1, **i32)

    def score(self, q, lse, kpool, block_table, seqused, count, stream=None, kernel="auto"):
        kvc_recover_score_ex(q, lse, kpool, self.n_slots, block_table, self.max_blocks,
                             seqused, count, self.n_req, self.L, self.H, self.Hq, self.D,
                             self.BS, self.state, self.ws, kernel, self.dev_status, stream)

    def lrfu(self, top_p: float = 0.9, lam: float = 0.5, stream=None):
        kvc_lrfu_update(self.state, self.seg_off, self.n_req, self.cap, top_p, lam,
                        self.keep_score, None, self.dev_status, stream)

    def select(self, stream=None, source=None):
        kvc_select(self.state if source is None else source, self.seg_off, self.n_req,
                   self.cap, self.keep, 0, 0, self.kept, self.kept_count, self.keepmask,
                   self.dev_status, stream)

    def plan(self, seqused, block_table, stream=None):
        kvc_tail_plan(self.keepmask, self.words, seqused, block_table, self.max_blocks,
                      self.n_req, self.BS, self.n_slots, self.src, self.dst, self.n_pairs,
                      self.n_tail, self.freed, self.n_freed, self.new_table, self.tail_mask,
                      self.dev_status, stream)

    def compact(self, kpool, vpool, stream=None):
        kvc_tail_compact(kpool, vpool, self.n_slots, self.L, self.H, self.D, self.src,
                         self.dst, self.n_pairs, self.cap, self.n_req, self.dev_status, stream)

    def run(self, q, lse, kpool, vpool, block_table, seqused, count, stream=None, lrfu=True):
        self.score(q, lse, kpool, block_table, seqused, count, stream)
        if lrfu:
            self.lrfu(stream=stream)
        self.select(stream, self.keep_score if lrfu else None)
        self.plan(seqused, block_table, stream)
        self.compact(kpool, vpool, stream)


def paged_bytes(n_req: int, seq: int, L: int, H: int, Hq: int, D: int, n_pairs: int) -> dict:
    """Bytes an ActKV operation must move through HBM, by stage: every
    visible key row read once, the query token, LSE and the state read and
    written (score); the state read and the keep score read and written
    (lrfu); the keep scores read (select); the keep mask and block table
    (plan); K and V rows of every planned pair read and written once per
    layer (compact)."""
    score = n_req * seq * L * H * D * 2 + n_req * L * Hq * (D * 2 + 4) + n_req * seq * 8
    lrfu = n_req * seq * 12
    select = n_req * seq * 4
    plan = n_req * (seq // 8 + seq // 4)
    compact = n_pairs * L * 2 * H * D * 2 * 2
    return {"score": score, "lrfu": lrfu, "select": select, "plan": plan, "compact": compact,
            "event": score + lrfu + select + plan + compact}
