"""Profiling cases: small, self-contained launches of one kernel family.

A measurement harness beside bench.py (not part of the library package).

Each case builds a reduced 8B-class workload (fewer layers, so a capture
holds a few GB at most while its inputs still exceed the 129 MB L2), runs the
event once to produce realistic inputs for the stage, then launches the stage
`--iters` times.

  python profile_cases.py score --layers 16 --iters 3
  python profile_cases.py score --config 27b --layers 2 --iters 3
  python profile_cases.py pack  --layers 4  --iters 3
  python profile_cases.py select --layers 16 --iters 3
  python profile_cases.py meank  --layers 2  --iters 3
  python profile_cases.py qmem   --layers 4  --sessions 8 --iters 2
  python profile_cases.py event_timing --config 27b --iters 10
  python profile_cases.py paged  --sessions 4 --iters 3
  python profile_cases.py tiered --layers 8 --iters 2
  python profile_cases.py confidence --iters 3
  python profile_cases.py repo   --layers 8 --slots 1024 --iters 3 --path /tmp/kvc_repo.bin
  python profile_cases.py select_long --seg-len 312500 --segments 288 --budget 2048 --iters 10

event_timing times a whole Mean-K event (score → select → pack, one CUDA
graph) on a full workload — tiny, 8b, 27b or ragged — with L2 flushed
between replays, and prints one JSON line: time, tokens/s and the fraction
of the measured HBM peak.  The qmem case is the QueryMemory rule score on the 64 x 32768 slot-map
workload's shapes (shared 4096-position prefix, page 16), reduced to
`--sessions` sessions and `--layers` layers.  The paged case is ActKV's
compression operation at the Table 1 shapes (6K → 4K tokens per request,
36 layers) on `--sessions` requests: score → LRFU → select → plan →
compaction, `--iters` times.  The tiered case runs `--iters` pairs of agent
steps of the host-resident 8B-class event reduced to `--layers` layers; the
confidence case runs the confidence monitor on its bench workload.  The repo
case runs `--iters` pairs of steps of the same event with the raw history of
the packed layers in a repository (a backing file at `--path`, direct I/O
where the file system allows it, `--slots` blocks in host RAM) and prints
one JSON line per step: time, units (layer, head, block) used and missed,
units read from the file and their rate.  The select_long case times
kvc_select on `--segments` segments of `--seg-len` items each (longer than
shared memory stages: the streaming kernel), seeded uniform scores with a run
of equal values per segment, and prints one JSON line: the median time per
launch and per segment.
"""
from __future__ import annotations

import argparse
import os
import sys


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["score", "select", "pack", "event", "meank", "qmem",
                                     "event_timing", "paged", "tiered", "confidence", "repo",
                                     "select_long"])
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--sessions", type=int, default=8)
    ap.add_argument("--config", choices=["tiny", "8b", "27b", "ragged"], default="8b")
    ap.add_argument("--slots", type=int, default=1024)
    ap.add_argument("--path", default="/tmp/kvc_repo.bin")
    ap.add_argument("--seg-len", type=int, default=312_500)
    ap.add_argument("--segments", type=int, default=288)
    ap.add_argument("--budget", type=int, default=2048)
    ap.add_argument("--kernel", default="auto",
                    help="scorer to run (a kvc_kernel name: score_fused, score_ring, "
                         "qmem_cc, recover_cc, ...); default: the library's choice")
    args = ap.parse_args(argv)

    root = os.path.dirname(os.path.abspath(__file__))
    sys.path.insert(0, root)
    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import MeanKEvent

    dev = torch.device("cuda", 0)
    if args.case == "qmem":
        _qmem_case(args, dev)
        return
    if args.case == "event_timing":
        _event_timing(args, dev, root)
        return
    if args.case == "paged":
        _paged_case(args, dev)
        return
    if args.case == "tiered":
        _tiered_case(args, dev)
        return
    if args.case == "confidence":
        _confidence_case(args, dev)
        return
    if args.case == "repo":
        _repo_case(args, dev)
        return
    if args.case == "select_long":
        _select_long_case(args, dev)
        return
    base = {"8b": W.config_8b, "27b": W.config_27b, "tiny": W.config_tiny,
            "ragged": W.config_ragged}[args.config]()
    if args.config in ("27b", "ragged") and args.case not in ("score", "select"):
        raise SystemExit("the 27b and ragged configs profile the score and select cases only")
    cfg = W.scaled(base, L=args.layers, L_pack=None)
    q = cfg.q(dev)
    meank = torch.empty(cfg.L, cfg.H, cfg.nb_total, cfg.D, dtype=torch.bfloat16, device=dev)
    if args.case == "meank":
        kraw, _ = cfg.kv_raw(dev)
        for _ in range(args.iters):
            kvc.kvc_build_meank(kraw, meank, cfg.L, cfg.H, cfg.D, cfg.n_tok)
        torch.cuda.synchronize()
        print(f"profile case meank: {args.iters} launches on {args.layers} layers ok")
        return
    if args.case in ("pack", "event"):
        kraw, vraw = cfg.kv_raw(dev)
        kvc.kvc_build_meank(kraw, meank, cfg.L, cfg.H, cfg.D, cfg.n_tok)
    else:
        # score/select only need the index: draw it directly (same distribution)
        boff = cfg.blk_off()
        for l in range(cfg.L):
            for h in range(cfg.H):
                for r in range(cfg.n_sess):
                    meank[l, h, boff[r]:boff[r + 1]] = cfg.meank_direct_unit(l, h, r, dev)
        kraw = vraw = None
    ev = MeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                    cfg.n_recent, theta=cfg.theta, device=dev)
    ev.score(q, meank, kernel=args.kernel)
    ev.select()
    torch.cuda.synchronize()
    for _ in range(args.iters):
        if args.case == "score":
            ev.score(q, meank, kernel=args.kernel)
        elif args.case == "select":
            ev.select()
        elif args.case == "pack":
            ev.pack(kraw, vraw)
        else:
            ev.run(q, meank, kraw, vraw)
    torch.cuda.synchronize()
    st = kvc.kvc_device_status(ev.dev_status)
    if st != 0:
        raise SystemExit(f"device status {st}: {kvc.kvc_status_string(st)}")
    print(f"profile case {args.case}: {args.iters} launches on {args.layers} layers ok")


def _event_timing(args, dev, root):
    import json
    import statistics

    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import MeanKEvent, event_bytes

    cfg = {"tiny": W.config_tiny, "8b": W.config_8b, "27b": W.config_27b,
           "ragged": W.config_ragged}[args.config]()
    q = cfg.q(dev)
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)  # layers without raw K keep the drawn index
    kvc.kvc_build_meank(kraw, meank[:cfg.lp], cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    ev = MeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                    cfg.n_recent, cfg.lp, cfg.theta, cfg.pos0, device=dev)
    ev.score_kernel = args.kernel
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        ev.run(q, meank, kraw, vraw)
    ev.capture(q, meank, kraw, vraw)
    ev.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ms = []
    for k in range(args.iters):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ev.replay()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    # per-stage kernel time from an eager pass with an event pair per launch
    stages = {}
    for k in range(3):
        flush.fill_(k & 0xFF)
        timers = []
        ev.run(q, meank, kraw, vraw, timers=timers)
        torch.cuda.synchronize()
        for stage, a, b in timers:
            stages.setdefault(stage, []).append(a.elapsed_time(b))
    st = kvc.kvc_device_status(ev.dev_status)
    if st != 0:
        raise SystemExit(f"device status {st}: {kvc.kvc_status_string(st)}")
    peak = 6800.0
    peaks = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(peaks):
        with open(peaks) as f:
            peak = float(json.load(f)["hbm_gbs"])
    nbytes = event_bytes(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.nb_total, cfg.n_sess, cfg.lp,
                         cfg.view_tokens, cfg.budget)["event"]
    med = statistics.median(ms)
    print(json.dumps({"config": cfg.name, "sessions": cfg.n_sess, "history_tokens": cfg.n_tok,
                      "layers_scored": cfg.L, "layers_packed": cfg.lp,
                      "ms_median": med, "ms_min": min(ms), "ms_max": max(ms),
                      "tokens_per_s": cfg.n_tok / (med * 1e-3),
                      "stages_ms": {k: round(statistics.median(v), 4) for k, v in stages.items()},
                      "algorithmic_bytes": nbytes,
                      "achieved_gbs": nbytes / (med * 1e-3) / 1e9,
                      "frac_of_measured_hbm": nbytes / (med * 1e-3) / 1e9 / peak}))


def _qmem_case(args, dev):
    import dataclasses

    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import SlotMapEvent

    cfg = dataclasses.replace(W.config_slotmap(), n_sess=args.sessions, L=args.layers)
    kp = torch.empty(cfg.L, cfg.n_slots, cfg.H, cfg.D, dtype=torch.bfloat16, device=dev)
    for l in range(cfg.L):
        kp[l] = cfg.kpool_layer(l, dev)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    sm = torch.from_numpy(cfg.slot_maps()).to(dev)
    M = torch.zeros(cfg.n_sess, cfg.L, cfg.Hq, cfg.D, dtype=torch.float32, device=dev)
    for t in range(cfg.turns):
        kvc.kvc_qmem_update(M, cfg.q_turn(t, dev), cfg.n_sess, cfg.L, cfg.Hq, cfg.D, cfg.T,
                            cfg.decay, cfg.gain, 1)
    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots, cfg.budget,
                      cfg.prefix, cfg.sentinel, device=dev)
    times = []
    for _ in range(args.iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ev.score(M, kp, sm, kernel=args.kernel)
        b.record()
        times.append((a, b))
    torch.cuda.synchronize()
    st = kvc.kvc_device_status(ev.dev_status)
    if st != 0:
        raise SystemExit(f"device status {st}: {kvc.kvc_status_string(st)}")
    ms = sorted(a.elapsed_time(b) for a, b in times)
    print(f"profile case qmem: {args.iters} launches, {cfg.n_sess} sessions x {cfg.N} "
          f"positions, {cfg.L} layers ok; score median {ms[len(ms) // 2]:.3f} ms")



def _paged_case(args, dev):
    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import PagedEvent

    cfg = W.config_paged(args.sessions)
    kp, vp = cfg.pools(dev)
    q = cfg.q(dev)
    lse = cfg.lse(q)
    bt = torch.from_numpy(cfg.block_tables()).to(dev)
    seq = torch.from_numpy(cfg.seqused()).to(dev)
    cnt = torch.ones(cfg.n_req, dtype=torch.int32, device=dev)
    ev = PagedEvent(cfg.n_req, cfg.max_blocks, cfg.BS, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                    cfg.keep, device=dev)
    for _ in range(args.iters):
        ev.run(q, lse, kp, vp, bt, seq, cnt)
    torch.cuda.synchronize(dev)
    st = kvc.kvc_device_status(ev.dev_status)
    print(f"paged: {cfg.n_req} requests, pairs {int(ev.n_pairs.sum().item())}, status {st}")
    if st != 0:
        raise SystemExit(1)



def _tiered_case(args, dev):
    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import TieredMeanKEvent

    cfg = W.scaled(W.config_8b(), L=args.layers)
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h, kraw_h, vraw_h = (t.cpu().pin_memory() for t in (meank, kraw, vraw))
    del kraw, vraw, meank
    qs = [cfg.q(dev, step=0), cfg.q(dev, step=1)]
    ev = TieredMeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                          cfg.n_recent, theta=cfg.theta, device=dev, stage_layers=4)
    for i in range(2 * args.iters):
        ev.step(qs[i % 2], meank_h, kraw_h, vraw_h)
    torch.cuda.synchronize(dev)
    st = kvc.kvc_device_status(ev.dev_status)
    print(f"tiered: {2 * args.iters} steps on {cfg.L} layers, status {st}")
    if st != 0:
        raise SystemExit(1)


def _repo_case(args, dev):
    import json
    import time

    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import RepoTieredEvent

    cfg = W.scaled(W.config_8b(), L=args.layers)
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h, kraw_h, vraw_h = (t.cpu().pin_memory() for t in (meank, kraw, vraw))
    del kraw, vraw, meank
    n_blocks = cfg.n_tok // 32
    direct = True
    try:
        repo = kvc.KvcRepo(args.path, n_blocks, cfg.lp, cfg.H, cfg.D, args.slots,
                           io_threads=8, direct=True)
    except kvc.KvcError:
        direct = False
        repo = kvc.KvcRepo(args.path, n_blocks, cfg.lp, cfg.H, cfg.D, args.slots, io_threads=8)
    t0 = time.time()
    repo.put(0, n_blocks, kraw_h, vraw_h, cfg.n_tok)
    put_s = time.time() - t0
    del kraw_h, vraw_h
    qs = [cfg.q(dev, step=0), cfg.q(dev, step=1)]
    ev = RepoTieredEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                         cfg.n_recent, theta=cfg.theta, device=dev, stage_layers=4, repo=repo)
    rec = repo.slot_elems * 2
    print(json.dumps({"repo": {"blocks": n_blocks, "record_bytes": rec, "slots": args.slots,
                               "units": repo.n_units, "file_bytes": repo.n_units * rec,
                               "direct_io": direct,
                               "put_s": round(put_s, 2)}}))
    for i in range(2 * args.iters):
        before = repo.stats()
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        ev.step(qs[i % 2], meank_h)
        torch.cuda.synchronize(dev)
        ms = (time.perf_counter() - t) * 1e3
        after = repo.stats()
        fetched = after["fetched"] - before["fetched"]
        read = after["bytes_read"] - before["bytes_read"]
        print(json.dumps({"step": i, "ms": round(ms, 2), "used": ev.last_plan[0],
                          "missed": ev.last_plan[1], "read_from_file": fetched,
                          "read_calls": after["read_calls"] - before["read_calls"],
                          "file_GBps": round(read / (ms * 1e-3) / 1e9, 2) if read else 0.0}))
    st = kvc.kvc_device_status(ev.dev_status)
    repo.close()
    os.remove(args.path)
    if st != 0:
        raise SystemExit(f"device status {st}")


def _select_long_case(args, dev):
    import json

    import torch

    import query_conditioned_kv_gb300 as kvc

    n, S, budget = args.seg_len, args.segments, args.budget
    if n <= kvc.SELECT_STAGED_SEG:
        raise SystemExit(f"--seg-len must exceed {kvc.SELECT_STAGED_SEG} (the staged kernel's limit)")
    g = torch.Generator(device=dev)
    g.manual_seed(n + S)
    scores = torch.rand(S, n, generator=g, device=dev)
    scores[:, 1000:1700] = scores[:, 5:6]  # a run of equal scores in every segment
    scores = scores.reshape(-1).contiguous()
    off = torch.arange(S + 1, dtype=torch.int64, device=dev) * n
    words = (n + 31) // 32
    kept = torch.empty(S, budget, dtype=torch.int32, device=dev)
    cnt = torch.empty(S, dtype=torch.int32, device=dev)
    mask = torch.empty(S, words, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ms = []
    for k in range(args.iters + 2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kvc.kvc_select(scores, off, S, n, budget, 1, 8, kept, cnt, mask, st)
        b.record(stream)
        b.synchronize()
        if k >= 2:
            ms.append(a.elapsed_time(b))
    code = kvc.kvc_device_status(st)
    if code != 0:
        raise SystemExit(f"device status {code}: {kvc.kvc_status_string(code)}")
    if not bool((cnt == budget).all()):
        raise SystemExit("a segment did not keep exactly the budget")
    med = sorted(ms)[len(ms) // 2]
    print(json.dumps({"case": "select_long", "segments": S, "seg_len": n, "budget": budget,
                      "n_sink": 1, "n_recent": 8, "launches": len(ms),
                      "ms_per_launch_median": round(med, 4),
                      "us_per_segment": round(1e3 * med / S, 3),
                      "scores_gb": round(S * n * 4 / 1e9, 3),
                      "l2": "scores exceed the 129 MB L2" if S * n * 4 > (129 << 20)
                      else "scores fit in L2 (launches back to back)"}))


def _confidence_case(args, dev):
    import torch

    import query_conditioned_kv_gb300 as kvc
    import workloads as W

    cfg = W.ConfidenceConfig()
    lg, tr = cfg.logits(dev), cfg.traces(dev)
    conf = torch.empty(cfg.n_req, dtype=torch.float32, device=dev)
    off = torch.arange(cfg.n_req + 1, dtype=torch.int64, device=dev) * cfg.trace_len
    slope = torch.empty(cfg.n_req, dtype=torch.float64, device=dev)
    budget = torch.full((cfg.n_req,), cfg.budget0, dtype=torch.int32, device=dev)
    kept = torch.empty(cfg.n_req, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.iters):
        kvc.kvc_token_confidence(lg, cfg.n_req, cfg.vocab, cfg.top_k, conf, st)
        kvc.kvc_conf_trend_budget(tr, off, cfg.n_req, cfg.trace_len, cfg.window, cfg.stride,
                                  cfg.bottom_pct, cfg.budget_step, cfg.max_budget, slope, budget,
                                  kept, st)
    torch.cuda.synchronize(dev)
    s = kvc.kvc_device_status(st)
    print(f"confidence: {args.iters} iterations, status {s}")
    if s != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
