"""Benchmark of the query-conditioned KV compression event on GB300.

Workload: the 8B-class single-session event — 36 layers, 8 KV / 32 query
heads, head dim 128, a 131072-token history (4096 blocks of 32), a 32-query
window, 256 kept blocks per (layer, KV head) with 1 sink and 4 recent
blocks, re-RoPE pack to positions 0..8191.  Inputs are seeded synthetic
bf16 tensors resident in HBM (see workloads/).

One step = one event: score (Mean-K) → select → pack, replayed as one CUDA
graph (a per-launch breakdown comes from an eager pass).  The metric is KV
history tokens compressed per second; the roofline is algorithmic bytes over
measured kernel time against the measured HBM copy bandwidth.  The Mean-K
index build and, on its own workload (64 sessions × 32768 positions over a
paged, refcounted K pool), the QueryMemory event (memory update; rule score
→ select → redirect + free) are measured after the timed steps and reported
beside them (`meank_build`, `slotmap_event`; `--no-slotmap` skips the latter),
and so is ActKV's paged compression operation (LSE-recovery score → select →
tail plan → in-place compaction) at 1, 4, 16 and 64 requests of 6K → 4K
tokens (`actkv_event`; `--no-paged` skips it), and KVMem's tiered view with the
index and raw history in host memory, cold and warm steps (`tiered_event`;
`--no-tiered` skips it), and its repository view with the raw history in a
backing file (`repo_event`; `--no-repo` skips it), and ActKV's confidence monitor (`confidence_monitor`;
`--no-confidence` skips it).  The 27B-class 1M-token event (64 layers scored, 16
packed) and the 128-session ragged event are measured the same way as the
headline, each with its own roofline and a scaled oracle baseline on a seeded
sample of its units (`event_27b_1m`, `event_ragged_128`; `--no-27b`,
`--no-ragged` skip them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the plain fp64 definition) on a
bounded sample of the same workload on the host cores.  Under torchrun
(N > 1) every rank runs its own event (independent sessions, weak scaling,
no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens compressed/s per event (score+select+pack); % of HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "8b_128k: 36 layers, 8 KV / 32 query heads, d 128, 131072-token history, " \
           "W 32, budget 256 blocks (1 sink, 4 recent), view 8192 tokens"
L2_NOTE = "L2 flushed between steps (256 MiB write outside the event's timed span); " \
          "the event also touches 2.7 GB > 129 MB L2"


def bench_config(cfg, world: int) -> dict:
    """The `config` of the JSON line; both arms print the same one."""
    return {"workload": WORKLOAD, "sessions": cfg.n_sess, "history_tokens": cfg.n_tok,
            "layers": cfg.L, "kv_heads": cfg.H, "q_heads": cfg.Hq, "head_dim": cfg.D,
            "window": cfg.W, "budget_blocks": cfg.budget, "parallelism": f"replicas{world}",
            "l2": L2_NOTE}


def algorithmic_bytes(cfg):
    """Bytes the method must move per event (HBM), by stage."""
    from query_conditioned_kv_gb300.event import event_bytes
    return event_bytes(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.nb_total, cfg.n_sess, cfg.lp,
                       cfg.view_tokens, cfg.budget)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if its source
    fingerprint still matches the kernel source; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    rows = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or "=" not in line:
                continue
            k, v = line.strip().split("=", 1)
            rows[k.strip()] = v.strip()
    parts = sorted(k for k in rows if k.startswith(f"{kernel}.part"))
    if parts:
        # the kernel's own source: "path :: start marker :: end marker" per
        # part (an empty marker: the start or end of the file), concatenated
        text = ""
        for k in parts:
            path_, start, end = (x.strip() for x in rows[k].split("::"))
            with open(os.path.join(ROOT, path_), encoding="utf-8") as f:
                body = f.read()
            i = body.find(start) if start else 0
            j = body.find(end, i) if end else len(body)
            if i < 0 or j < 0:  # a marker is gone: the source has changed
                return None
            text += body[i:j]
        sha = hashlib.sha256(text.encode("utf-8")).hexdigest()[:16]
    else:
        src = rows.get(f"{kernel}.source")
        if not src:
            return None
        with open(os.path.join(ROOT, src), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if sha != rows.get(f"{kernel}.sha"):
        return None
    scale = float(rows.get(f"{kernel}.scale", "1"))
    return float(rows[f"{kernel}.bytes_per_launch"]) * scale


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed span."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def reduce_max_ms(ms: float, world: int, device) -> float:
    """Max over ranks of a per-rank time (the job is as slow as its slowest
    rank); identity at world size 1."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_meank_build(kvc, cfg, kraw, meank, dev, reps: int = 3):
    """The Mean-K index build (kept out of the event: the index is maintained
    as blocks fill), timed on its own with CUDA events after the first build.
    Algorithmic bytes: every raw K element read once, every mean written once."""
    import torch
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms = []
    for r in range(reps):
        flush.fill_(r)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kvc.kvc_build_meank(kraw, meank, cfg.L, cfg.H, cfg.D, cfg.n_tok)
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    del flush
    nbytes = kraw.numel() * 2 + meank.numel() * 2
    m = sorted(ms)[len(ms) // 2]
    return {"kernel": "k_build_meank", "ms": m, "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / (m * 1e-3) / 1e9,
            "note": "index maintenance, not part of the event; median of "
                    f"{reps} launches, L2 flushed before each"}


def whole_job_value(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank's history tokens over the slowest
    rank's event time."""
    return tokens_per_rank * world / (ms_max * 1e-3)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import MeanKEvent

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = W.config_8b()
    # inputs resident in HBM before the timed region
    q = cfg.q(dev)
    kraw, vraw = cfg.kv_raw(dev)
    meank = torch.empty(cfg.L, cfg.H, cfg.nb_total, cfg.D, dtype=torch.bfloat16, device=dev)
    kvc.kvc_build_meank(kraw, meank, cfg.L, cfg.H, cfg.D, cfg.n_tok)
    meank_build = time_meank_build(kvc, cfg, kraw, meank, dev)
    ev = MeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                    cfg.n_recent, theta=cfg.theta, pos0=cfg.pos0, device=dev,
                    groups=args.groups)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        flush.fill_(1)
        ev.run(q, meank, kraw, vraw)
    torch.cuda.synchronize(dev)
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError("device status error during warm-up")

    # stage breakdown: the event run eagerly, a CUDA event pair around every
    # launch (not the headline: the events themselves add launch gaps)
    timers = [[] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        ev.run(q, meank, kraw, vraw, timers=timers[k])
    torch.cuda.synchronize(dev)
    mean = {"score": 0.0, "select": 0.0, "pack": 0.0}
    n_launch = {"score": 0, "select": 0, "pack": 0}
    for tk in timers:
        for stage, a, b in tk:
            mean[stage] += a.elapsed_time(b) / args.steps
            n_launch[stage] += 1

    # the timed region: the event as one CUDA graph, replayed K times; the
    # L2 flush runs between replays, outside the event span
    ev.capture(q, meank, kraw, vraw)
    ev.replay()
    torch.cuda.synchronize(dev)
    bounds = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)  # L2 flush, outside the event span
        bounds[k][0].record(stream)
        ev.replay()
        bounds[k][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError("device status error in the timed region")
    step_ms = sorted(a.elapsed_time(b) for a, b in bounds)
    mean["event"] = sum(step_ms) / args.steps
    ms_event = mean["event"]
    ms_event = reduce_max_ms(ms_event, world, dev)
    value = whole_job_value(cfg.n_tok, world, ms_event)

    # e2e through the public API with host buffers (pinned), copies timed
    e2e = None
    if args.e2e_steps > 0:
        h_q = q.cpu().pin_memory()
        h_mk = meank.cpu().pin_memory()
        h_k = kraw.cpu().pin_memory()
        h_v = vraw.cpu().pin_memory()
        o_k = torch.empty(ev.kview.shape, dtype=torch.bfloat16).pin_memory()
        o_v = torch.empty(ev.vview.shape, dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_mk, h_k, h_v))
        d2h = 2 * ev.kview.numel() * 2
        for i in range(args.e2e_steps + 1):
            if i == 1:
                torch.cuda.synchronize(dev)
                te = time.perf_counter()
            q.copy_(h_q, non_blocking=True)
            meank.copy_(h_mk, non_blocking=True)
            kraw.copy_(h_k, non_blocking=True)
            vraw.copy_(h_v, non_blocking=True)
            ev.run(q, meank, kraw, vraw)
            o_k.copy_(ev.kview, non_blocking=True)
            o_v.copy_(ev.vview, non_blocking=True)
            torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - te) / args.e2e_steps
        e2e_copy_all = {"value": cfg.n_tok / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                        "note": "resident event on pinned host buffers: H2D of q, Mean-K and "
                                "raw K/V every step; D2H of the K/V execution view"}
        e2e = tiered_e2e(args, cfg, dev, h_q, h_mk, h_k, h_v)
        e2e["copy_all"] = e2e_copy_all
        del o_k, o_v

    ab = algorithmic_bytes(cfg)
    peak, peak_src = peaks()
    dom = max(("score", "select", "pack"), key=lambda s: mean[s])
    kern = {"score": "k_score_fused", "select": "k_select", "pack": "k_pack_rerope"}[dom]
    score_kernels = kvc.kvc_score_launches(max(1, cfg.L // len(ev.groups)), cfg.H, cfg.Hq,
                                           cfg.D, cfg.W, cfg.n_sess, cfg.nb_total)
    achieved = ab[dom] / (mean[dom] * 1e-3) / 1e9 if ab[dom] else 0.0
    pack_gbs = ab["pack"] / (mean["pack"] * 1e-3) / 1e9
    score_gbs = ab["score"] / (mean["score"] * 1e-3) / 1e9 if mean["score"] > 0 else 0.0
    event_gbs = ab["event"] / (ms_event * 1e-3) / 1e9
    traffic = ncu_traffic(dom)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_event,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded, workloads/)",
        "config": bench_config(cfg, world),
        "hbm_roofline_event": {"achieved_gbs": event_gbs, "peak_gbs": peak,
                               "frac": event_gbs / peak,
                               "algorithmic_bytes": ab["event"]},
        "stages_ms": {k: round(v, 4) for k, v in mean.items()},
        "stages_note": "per-launch kernel time of an eager run with a CUDA event pair "
                       f"around each launch ({len(ev.groups)} layer group(s)); the event "
                       "time is the CUDA-graph replay",
        "ms_p10_p50_p90": [round(step_ms[int(0.1 * (len(step_ms) - 1))], 4),
                           round(step_ms[(len(step_ms) - 1) // 2], 4),
                           round(step_ms[int(0.9 * (len(step_ms) - 1))], 4)],
        "roofline": {"bound": "hbm", "kernel": kern, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": ab[dom], "peak_source": peak_src},
        "pack_roofline": {"achieved": pack_gbs, "frac": pack_gbs / peak},
        "score_roofline": {"kernel": "k_score_fused", "algorithmic_bytes": ab["score"],
                           "achieved": score_gbs, "frac": score_gbs / peak},
        "meank_build": dict(meank_build, frac=meank_build["achieved_gbs"] / peak),
        "gpu_launches": n_launch["select"] + n_launch["pack"] + n_launch["score"] * score_kernels,
        "clocks": clk,
        "e2e": e2e,
        "wall_s_timed": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, dev)
    return line


# ------------------------------------------- the other Mean-K workloads

EVENT_WORKLOADS = {
    "27b_1m": ("27b_1m: 64 layers scored (Mean-K index of 4.3 GB device-resident), 16 "
               "layers packed (raw K/V 68.7 GB resident), 8 KV / 48 query heads, d 128, "
               "1048576-token workspace, W 32, budget 2048 blocks (1 sink, 8 recent), "
               "view 65536 tokens"),
    "ragged_128": ("ragged_128: 128 sessions of U[16384, 262144] tokens (rounded to 32), "
                   "36 layers scored, 2 packed, 8 KV / 32 query heads, d 128, W 32, budget "
                   "512 blocks (1 sink, 4 recent), view 16384 tokens per session"),
}


def _oracle_config_sample(cfg, name, dev, seed=7):
    """A seeded sample of the workload's units for the oracle baseline and the
    share of the event's tokens it stands for.  27b_1m: 8 of the 512 (layer,
    KV head) units, 2 of them in packed layers and 6 in scored-only layers
    (the event's 1:3 mix).  ragged_128: every unit of 8 of the 128 sessions,
    the shortest and the longest among them."""
    import numpy as np
    rng = np.random.default_rng(seed)
    if name == "27b_1m":
        packed = rng.choice(cfg.lp * cfg.H, size=2, replace=False)
        scored = rng.choice((cfg.L - cfg.lp) * cfg.H, size=6, replace=False) + cfg.lp * cfg.H
        picks = [(int(u) // cfg.H, int(u) % cfg.H, 0) for u in list(packed) + list(scored)]
        frac = len(picks) / (cfg.L * cfg.H * cfg.n_sess)
        what = (f"8 of {cfg.L * cfg.H} (layer, KV head) units (2 of them packed), "
                f"tokens scaled by {frac:.5f}")
    else:
        hist = np.asarray(cfg.hist)
        rest = [r for r in range(cfg.n_sess) if r not in (int(hist.argmin()), int(hist.argmax()))]
        sess = [int(hist.argmin()), int(hist.argmax())] + \
            [int(x) for x in rng.choice(rest, size=6, replace=False)]
        picks = [(l, h, r) for r in sess for l in range(cfg.L) for h in range(cfg.H)]
        frac = float(hist[sess].sum()) / cfg.n_tok
        what = (f"all {cfg.L * cfg.H} (layer, KV head) units of 8 of {cfg.n_sess} sessions "
                f"(shortest and longest included), {int(hist[sess].sum())} of "
                f"{cfg.n_tok} tokens: scaled by {frac:.5f}")
    return _oracle_units(cfg, picks, dev), frac, what


def config_event(args, dev, peak, name: str, reps: int = 20):
    """One Mean-K event of the 27b_1m or ragged_128 workload, measured like the
    headline: score → select → pack replayed as one CUDA graph, the L2 flushed
    (256 MiB write) between replays outside the event span, CUDA events on the
    stream; stages from an eager pass with an event pair per launch; the
    oracle baseline on a seeded sample of the same workload."""
    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import MeanKEvent, event_bytes

    cfg = {"27b_1m": W.config_27b, "ragged_128": W.config_ragged}[name]()
    q = cfg.q(dev)
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)  # layers without raw K keep the drawn index
    kvc.kvc_build_meank(kraw, meank[:cfg.lp], cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    ev = MeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                    cfg.n_recent, cfg.lp, cfg.theta, cfg.pos0, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        ev.run(q, meank, kraw, vraw)
    ev.capture(q, meank, kraw, vraw)
    ev.replay()
    torch.cuda.synchronize(dev)
    ms = []
    for k in range(reps):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ev.replay()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    stages = {}
    n_launch = {}
    for k in range(5):
        flush.fill_(k & 0xFF)
        timers = []
        ev.run(q, meank, kraw, vraw, timers=timers)
        torch.cuda.synchronize(dev)
        for stage, a, b in timers:
            stages.setdefault(stage, []).append(a.elapsed_time(b))
            if k == 0:
                n_launch[stage] = n_launch.get(stage, 0) + 1
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError(f"device status error in the {name} event")
    ab = event_bytes(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.nb_total, cfg.n_sess, cfg.lp,
                     cfg.view_tokens, cfg.budget)
    ms_sorted = sorted(ms)
    med = statistics.median(ms)
    st = {k: statistics.median(v) for k, v in stages.items()}
    score_kernels = kvc.kvc_score_launches(cfg.L // len(ev.groups), cfg.H, cfg.Hq, cfg.D, cfg.W,
                                           cfg.n_sess, ev.nb_max)
    out = {
        "workload": EVENT_WORKLOADS[name], "sessions": cfg.n_sess, "history_tokens": cfg.n_tok,
        "layers_scored": cfg.L, "layers_packed": cfg.lp,
        "value": cfg.n_tok / (med * 1e-3), "unit": UNIT, "ms_per_event": round(med, 4),
        "ms_p10_p50_p90": [round(ms_sorted[int(0.1 * (reps - 1))], 4), round(med, 4),
                           round(ms_sorted[int(0.9 * (reps - 1))], 4)],
        "reps": reps,
        "hbm_roofline_event": {"achieved_gbs": ab["event"] / (med * 1e-3) / 1e9,
                               "peak_gbs": peak,
                               "frac": ab["event"] / (med * 1e-3) / 1e9 / peak,
                               "algorithmic_bytes": ab["event"]},
        "stages_ms": {k: round(v, 4) for k, v in st.items()},
        "score_roofline": {"algorithmic_bytes": ab["score"],
                           "achieved": ab["score"] / (st["score"] * 1e-3) / 1e9,
                           "frac": ab["score"] / (st["score"] * 1e-3) / 1e9 / peak},
        "pack_roofline": {"kernel": "k_pack_rerope", "algorithmic_bytes": ab["pack"],
                          "achieved": ab["pack"] / (st["pack"] * 1e-3) / 1e9,
                          "frac": ab["pack"] / (st["pack"] * 1e-3) / 1e9 / peak},
        "gpu_launches": n_launch.get("select", 0) + n_launch.get("pack", 0)
        + n_launch.get("score", 0) * score_kernels,
        "l2": "L2 flushed between replays (256 MiB write outside the event span); the "
              "event moves " f"{ab['event'] / 1e9:.1f} GB",
    }
    del q, kraw, vraw, meank, ev, flush
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        units, frac, what = _oracle_config_sample(cfg, name, dev)
        secs = _oracle_event(cfg, units, cores)
        out["cpu_baseline"] = {"value": cfg.n_tok * frac / secs, "unit": UNIT, "cores": cores,
                               "kind": "oracle", "scaled": True,
                               "sample": f"{what}; score+select+pack (pack in packed layers), "
                                         f"fp64 C oracle, thread pool of {cores}, "
                                         f"{secs:.2f} s wall"}
    return out


# --------------------------------------------------- QueryMemory event

SLOTMAP_WORKLOAD = ("slotmap_64x32k: 64 sessions x 32768 positions (4096-position shared, "
                    "refcounted prefix; page 16), 36 layers, 8 KV / 32 query heads, d 128, "
                    "4 memory turns of 32 queries, 8192 kept positions per session")


def _oracle_slotmap(cfg, kp, sm_np, dev, n_sample: int = 4, seed: int = 11):
    """The oracle on 4 of the 64 sessions of the slot-map event: rule score
    over every layer and query head, then select, one thread per session.
    Inputs from the seeded generators only: the sessions' memories rebuilt
    with the oracle from the generator's query turns, their K rows gathered
    by position from the generated pool.  Redirect + free (integer work,
    negligible next to the score) is not timed."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch
    import oracle
    import workloads as W

    rng = np.random.default_rng(seed)
    sample = [0] + [int(x) for x in rng.choice(np.arange(1, cfg.n_sess), size=n_sample - 1,
                                               replace=False)]
    M_ref = np.zeros((len(sample), cfg.L, cfg.Hq, cfg.D), np.float32)
    for t in range(cfg.turns):
        qt = cfg.q_turn(t, dev)
        M_ref = oracle.qmem_update(M_ref, W.bf16_bits(qt[sample]), cfg.decay, cfg.gain)
        del qt
    rows = []
    for r in sample:
        slots = torch.from_numpy(sm_np[r].astype(np.int64)).to(dev)
        rows.append(W.bf16_bits(kp[:, slots]))  # [L][N][H][D], position → row
        del slots
    ident = np.arange(cfg.N, dtype=np.int32)

    def one(i):
        ref = oracle.rule_session(M_ref[i], rows[i], ident, cfg.H, -1)
        oracle.select(ref, cfg.budget, 0, 0)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(sample)) as ex:
        list(ex.map(one, range(len(sample))))
    secs = time.perf_counter() - t0
    frac = len(sample) / cfg.n_sess
    return {"value": cfg.n_sess * cfg.N * frac / secs, "unit": UNIT, "cores": len(sample),
            "kind": "oracle", "scaled": True,
            "sample": f"{len(sample)} of {cfg.n_sess} sessions (sessions {sample}): rule score "
                      f"over {cfg.L} layers x {cfg.Hq} query heads + select, fp64 C oracle, one "
                      f"thread per session; {secs:.1f} s wall; tokens scaled by {frac:.4f}; "
                      "redirect + free not timed"}


def slot_map_event(args, dev, peak, reps: int = 3):
    """The QueryMemory-mode event (rule score over the paged K pool → token
    select → redirect + free) on the full 64 x 32768 workload, each stage
    timed with CUDA events; the memory update is timed on its own.  The
    slot maps and refcounts are restored before every rep (outside the
    timed span); the inputs (135.6 GB of K) are far larger than L2."""
    import numpy as np
    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import SlotMapEvent

    cfg = W.config_slotmap()
    kp = torch.empty(cfg.L, cfg.n_slots, cfg.H, cfg.D, dtype=torch.bfloat16, device=dev)
    for l in range(cfg.L):
        kp[l] = cfg.kpool_layer(l, dev)
    kvc.kvc_init_sentinel(kp, None, cfg.L, cfg.H, cfg.D, cfg.n_slots, cfg.sentinel)
    sm_np = cfg.slot_maps()
    sm0 = torch.from_numpy(sm_np).to(dev)
    rc0 = torch.from_numpy(cfg.refcounts(sm_np)).to(dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        return a, b

    # memory recurrence: one update per turn
    M = torch.zeros(cfg.n_sess, cfg.L, cfg.Hq, cfg.D, dtype=torch.float32, device=dev)
    upd = []
    for t in range(cfg.turns):
        qt = cfg.q_turn(t, dev)
        upd.append(timed(lambda: kvc.kvc_qmem_update(M, qt, cfg.n_sess, cfg.L, cfg.Hq, cfg.D,
                                                      cfg.T, cfg.decay, cfg.gain, 1)))
        torch.cuda.synchronize(dev)
        q_bytes = qt.numel() * 2
        del qt
    upd_ms = statistics.median(a.elapsed_time(b) for a, b in upd)
    upd_bytes = q_bytes + 2 * M.numel() * 4

    ev = SlotMapEvent(cfg.n_sess, cfg.N, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots, cfg.budget,
                      cfg.prefix, cfg.sentinel, device=dev)
    sm = torch.empty_like(sm0)
    rc = torch.empty_like(rc0)
    stages = {"score": [], "select": [], "redirect": []}
    events = []
    for r in range(1 + reps):
        sm.copy_(sm0)
        rc.copy_(rc0)
        torch.cuda.synchronize(dev)
        t_all = timed(lambda: None)[0]
        st = {"score": timed(lambda: ev.score(M, kp, sm)),
              "select": timed(lambda: ev.select()),
              "redirect": timed(lambda: ev.redirect(sm, rc))}
        end = timed(lambda: None)[1]
        torch.cuda.synchronize(dev)
        if r == 0:
            continue  # warm-up
        for k, (a, b) in st.items():
            stages[k].append(a.elapsed_time(b))
        events.append(t_all.elapsed_time(end))
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError("device status error in the QueryMemory event")
    n_freed = int(ev.n_freed.item())

    n_unique = cfg.prefix + cfg.n_sess * (cfg.N - cfg.prefix)
    k_bytes = n_unique * cfg.L * cfg.H * cfg.D * 2
    sm_bytes = sm0.numel() * 4
    score_bytes = k_bytes + M.numel() * 4 + sm_bytes
    event_bytes = score_bytes + sm_bytes + rc0.numel() * 4
    ms = statistics.median(events)
    sc_ms = statistics.median(stages["score"])
    tokens = cfg.n_sess * cfg.N
    out = {
        "workload": SLOTMAP_WORKLOAD, "tokens_per_event": tokens,
        "value": tokens / (ms * 1e-3), "unit": UNIT, "ms_per_event": ms,
        "algorithmic_bytes": event_bytes,
        "hbm_roofline_event": {"achieved_gbs": event_bytes / (ms * 1e-3) / 1e9,
                               "frac": event_bytes / (ms * 1e-3) / 1e9 / peak},
        "stages_ms": {k: round(statistics.median(v), 4) for k, v in stages.items()},
        "score_roofline": {"kernels": "k_qmem_split + k_qmem_logits_tc (rule share formed "
                                      "in the same kernel) + k_qmem_rule_sum",
                           "algorithmic_bytes": score_bytes,
                           "achieved": score_bytes / (sc_ms * 1e-3) / 1e9,
                           "frac": score_bytes / (sc_ms * 1e-3) / 1e9 / peak,
                           "note": "unique K rows read once (shared prefix counted once); the "
                                   "logits stay in L2 and are dropped there; the per-layer "
                                   "shares (0.3 GB written + read) are overhead"},
        "qmem_update": {"ms": upd_ms, "algorithmic_bytes": upd_bytes,
                        "achieved_gbs": upd_bytes / (upd_ms * 1e-3) / 1e9,
                        "frac": upd_bytes / (upd_ms * 1e-3) / 1e9 / peak,
                        "note": "one turn: queries read once, M read and written once"},
        "freed_slots": n_freed, "reps": reps,
        "l2": "inputs (135.6 GB of K) far exceed the 129 MB L2; no flush",
    }
    if not args.no_cpu_baseline:
        del ev, M
        torch.cuda.empty_cache()
        out["cpu_baseline"] = _oracle_slotmap(cfg, kp, sm_np, dev)
        del kp
    else:
        del kp, ev, M
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------- ActKV paged operation

PAGED_WORKLOAD = ("paged_6k_to_4k: ActKV Table 1 shapes (block size 16, 8 KV heads, d 128), "
                  "36 layers, 32 query heads; r requests of 6144 tokens each compressed to "
                  "4096; LSE-recovery score of one action token (restart), LRFU keep score "
                  "(top-p 0.9, lambda 0.5), top-4096 select by keep score, tail plan, "
                  "in-place compaction of K and V")


def paged_event(args, dev, peak, reqs=(1, 4, 16, 64), reps: int = 5):
    """ActKV's compression operation on a paged KV cache, at the request
    counts of ActKV Table 1: each stage timed with CUDA events on the
    launching stream, the operation as their sum.  Every rep restarts the
    score (count 1); the compaction of a rep moves rows inside the pool, so
    the next rep's plan can differ slightly: each rep's compaction bytes use
    its own pair count (read after the rep).  The K and V pools (0.9–58 GB)
    exceed the 129 MB L2."""
    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import PagedEvent, paged_bytes

    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        return a, b

    rows = []
    for n_req in reqs:
        cfg = W.config_paged(n_req)
        kp, vp = cfg.pools(dev)
        q = cfg.q(dev)
        lse = cfg.lse(q)
        bt = torch.from_numpy(cfg.block_tables()).to(dev)
        seq = torch.from_numpy(cfg.seqused()).to(dev)
        cnt = torch.ones(n_req, dtype=torch.int32, device=dev)
        ev = PagedEvent(n_req, cfg.max_blocks, cfg.BS, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.n_slots,
                        cfg.keep, device=dev)
        stages = {"score": [], "lrfu": [], "select": [], "plan": [], "compact": []}
        events, fracs, pairs = [], [], []
        for r in range(args.warmup + reps):
            torch.cuda.synchronize(dev)
            st = {"score": timed(lambda: ev.score(q, lse, kp, bt, seq, cnt)),
                  "lrfu": timed(lambda: ev.lrfu()),
                  "select": timed(lambda: ev.select(source=ev.keep_score)),
                  "plan": timed(lambda: ev.plan(seq, bt)),
                  "compact": timed(lambda: ev.compact(kp, vp))}
            torch.cuda.synchronize(dev)
            if r < args.warmup:
                continue
            ms = {k: a.elapsed_time(b) for k, (a, b) in st.items()}
            for k, v in ms.items():
                stages[k].append(v)
            total = st["score"][0].elapsed_time(st["compact"][1])
            np_ = int(ev.n_pairs.sum().item())
            pairs.append(np_)
            events.append(total)
            b = paged_bytes(n_req, cfg.seq, cfg.L, cfg.H, cfg.Hq, cfg.D, np_)
            fracs.append(b["event"] / (total * 1e-3) / 1e9 / peak)
        if kvc.kvc_device_status(ev.dev_status) != 0:
            raise RuntimeError("device status error in the paged operation")
        ms = statistics.median(events)
        np_med = int(statistics.median(pairs))
        b = paged_bytes(n_req, cfg.seq, cfg.L, cfg.H, cfg.Hq, cfg.D, np_med)
        sc = statistics.median(stages["score"])
        cp = statistics.median(stages["compact"])
        tokens = n_req * cfg.seq
        rows.append({
            "n_req": n_req, "tokens_per_op": tokens, "ms_per_op": round(ms, 4),
            "value": tokens / (ms * 1e-3), "unit": UNIT,
            "pairs_moved": np_med, "algorithmic_bytes": b["event"],
            "hbm_frac_op": round(statistics.median(fracs), 4),
            "stages_ms": {k: round(statistics.median(v), 4) for k, v in stages.items()},
            "score_roofline": {"kernel": "k_recover_tc", "algorithmic_bytes": b["score"],
                               "achieved": b["score"] / (sc * 1e-3) / 1e9,
                               "frac": b["score"] / (sc * 1e-3) / 1e9 / peak},
            "compact_roofline": {"kernel": "k_tail_compact", "algorithmic_bytes": b["compact"],
                                 "achieved": b["compact"] / (cp * 1e-3) / 1e9,
                                 "frac": b["compact"] / (cp * 1e-3) / 1e9 / peak},
        })
        del kp, vp, q, ev
        torch.cuda.empty_cache()
    return {"workload": PAGED_WORKLOAD, "reps": reps, "rows": rows,
            "l2": "pools (0.9-58 GB) exceed the 129 MB L2; no flush"}


# ------------------------------------------------- tiered (host-resident)

TIERED_WORKLOAD = ("tiered_8b_128k: the 8b_128k event with the Mean-K index (302 MB) and "
                   "the raw K/V history (9.66 GB) in pinned host memory; score in 4-layer "
                   "tiles copied host->device, select, tiered pack (hits from the previous "
                   "view, misses read from host memory by the kernel); two agent steps")


def tiered_event(args, dev, peak, reps: int = 3):
    """KVMem's tiered view on the 8B-class workload.  Step 1 starts cold
    (every kept block comes from host memory); step 2 scores a new query
    window and reuses the blocks both steps keep.  Each rep replays the two
    steps; stages are timed with CUDA events on the current stream (the
    staging copies run on a side stream inside the score stage)."""
    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import TieredMeanKEvent

    cfg = W.config_8b()
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h = meank.cpu().pin_memory()
    kraw_h = kraw.cpu().pin_memory()
    vraw_h = vraw.cpu().pin_memory()
    del kraw, vraw, meank
    torch.cuda.empty_cache()
    # the host link's copy bandwidth, the denominator of the host-side stages
    src = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    link = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        link.append((1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9)
    link_gbs = max(link)
    del src, dst
    qs = [cfg.q(dev, step=0), cfg.q(dev, step=1)]
    ev = TieredMeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                          cfg.n_recent, L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0,
                          device=dev, stage_layers=4)
    stream = torch.cuda.current_stream(dev)

    def ev_pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    rows = {"cold": [], "warm": []}
    hits = {}
    for rep in range(args.warmup + reps):
        ev.steps = 0  # every rep starts cold
        for k, q in (("cold", qs[0]), ("warm", qs[1])):
            ev.n_hits.zero_()
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            cur = ev.cur
            ev.kept, ev.kept_count = ev.kept_sets[cur], ev.count_sets[cur]
            ev.vview = ev.vviews[cur]
            torch.cuda.synchronize(dev)
            marks[0].record(stream)
            ev.score_tiered(q, meank_h)
            marks[1].record(stream)
            ev.select()
            marks[2].record(stream)
            ev.pack_tiered(kraw_h, vraw_h)
            marks[3].record(stream)
            ev.cur, ev.steps = 1 - cur, ev.steps + 1
            torch.cuda.synchronize(dev)
            if rep >= args.warmup:
                rows[k].append([marks[i].elapsed_time(marks[i + 1]) for i in range(3)])
                hits[k] = int(ev.n_hits.item())
    # the same steps pipelined (each tile's select and pack under the next
    # tiles' copies), as TieredMeanKEvent.step runs them by default
    piped = {"cold": [], "warm": []}
    for rep in range(args.warmup + reps):
        ev.steps = 0
        for k, q in (("cold", qs[0]), ("warm", qs[1])):
            a, b = ev_pair()
            torch.cuda.synchronize(dev)
            a.record(stream)
            ev.step(q, meank_h, kraw_h, vraw_h)
            b.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= args.warmup:
                piped[k].append(a.elapsed_time(b))
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError("device status error in the tiered event")
    n_units = cfg.lp * cfg.H * cfg.n_sess
    kept_blocks = n_units * cfg.budget
    blk_bytes = 32 * cfg.D * 2
    meank_bytes = cfg.L * cfg.H * cfg.nb_total * cfg.D * 2
    out = {"workload": TIERED_WORKLOAD, "reps": reps, "tokens_per_step": cfg.n_tok,
           "h2d_copy_gbs": round(link_gbs, 1),
           "h2d_note": "best of 5 pinned host->device copies of 1 GiB (copy engine)"}
    for k, v in rows.items():
        sc, se, pk = (statistics.median(x[i] for x in v) for i in range(3))
        ms = sc + se + pk
        miss = kept_blocks - hits[k]
        host_bytes = meank_bytes + miss * 2 * blk_bytes
        out[k] = {
            "ms_per_step": round(ms, 4), "value": cfg.n_tok / (ms * 1e-3), "unit": UNIT,
            "stages_ms": {"score_tiered": round(sc, 4), "select": round(se, 4),
                          "pack_tiered": round(pk, 4)},
            "kept_blocks": kept_blocks, "hits": hits[k], "misses": miss,
            "host_to_gpu_bytes": host_bytes,
            "score_h2d_gbs": meank_bytes / (sc * 1e-3) / 1e9,
            "score_frac_of_h2d_copy": meank_bytes / (sc * 1e-3) / 1e9 / link_gbs,
            "pack_host_read_gbs": miss * 2 * blk_bytes / (pk * 1e-3) / 1e9,
            "ms_per_step_pipelined": round(statistics.median(piped[k]), 4),
            "note": "stages_ms from the stages run one after another; the pipelined "
                    "step (each index tile's select and pack under the next tiles' "
                    "copies) is what TieredMeanKEvent.step and e2e run",
        }
    del ev, meank_h, kraw_h, vraw_h
    torch.cuda.empty_cache()
    return out


def tiered_e2e(args, cfg, dev, h_q0, h_mk, h_k, h_v):
    """The event end to end with its inputs in pinned host memory, through the
    library's host-resident path (TieredMeanKEvent: the Mean-K index scored
    in tiles copied over the link, the view packed from blocks the previous
    step kept plus the misses read from host memory).  Consecutive steps
    alternate two query windows, as consecutive agent steps do.  Timed per
    step: H2D of the step's query window, the event, and D2H of the step's
    result (kept block lists and counts; the execution view stays on the
    GPU for the decode that follows)."""
    import torch
    from query_conditioned_kv_gb300.event import TieredMeanKEvent

    h_q = [h_q0, cfg.q(dev, step=1).cpu().pin_memory()]
    ev = TieredMeanKEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget, cfg.n_sink,
                          cfg.n_recent, L_pack=cfg.lp, theta=cfg.theta, pos0=cfg.pos0,
                          device=dev, stage_layers=4)
    q = torch.empty_like(h_q0, device=dev)
    o_kept = torch.empty(ev.kept.shape, dtype=torch.int32).pin_memory()
    o_cnt = torch.empty(ev.kept_count.shape, dtype=torch.int32).pin_memory()
    steps = max(args.e2e_steps, 2)
    hits = []
    for i in range(2 + steps):  # two untimed steps fill the previous view
        if i == 2:
            torch.cuda.synchronize(dev)
            te = time.perf_counter()
        ev.n_hits.zero_()
        q.copy_(h_q[i % 2], non_blocking=True)
        ev.step(q, h_mk, h_k, h_v)
        o_kept.copy_(ev.kept_sets[1 - ev.cur], non_blocking=True)
        o_cnt.copy_(ev.count_sets[1 - ev.cur], non_blocking=True)
        if i >= 2:
            hits.append(ev.n_hits)
            ev.n_hits = torch.zeros_like(ev.n_hits)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - te) / steps
    import query_conditioned_kv_gb300 as kvc
    if kvc.kvc_device_status(ev.dev_status) != 0:
        raise RuntimeError("device status error in the tiered e2e steps")
    kept_blocks = cfg.lp * cfg.H * cfg.n_sess * cfg.budget
    hit = sum(int(h.item()) for h in hits) / len(hits)
    blk = 32 * cfg.D * 2
    index_bytes = h_mk.numel() * 2
    h2d = int(h_q0.numel() * 2 + index_bytes + (kept_blocks - hit) * 2 * blk)
    d2h = int(o_kept.numel() * 4 + o_cnt.numel() * 4)
    out = {"value": cfg.n_tok / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
           "kept_blocks_reused": round(hit / kept_blocks, 4),
           "note": "C-ABI calls with the inputs in pinned host memory (host-resident path: "
                   "kvc_score on Mean-K tiles copied over the link, kvc_select, "
                   "kvc_pack_tiered reading missed blocks from host memory); consecutive "
                   "steps alternate two query windows; H2D counts the query window, the "
                   "index and the missed blocks' raw K/V; D2H is the kept lists"}
    del ev
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------- confidence monitor

REPO_WORKLOAD = ("repo_8b_8layers: the 8b_128k history reduced to 8 layers (scored and "
                 "packed), its raw K/V in a repository: 262,144 units (layer, KV head, "
                 "32-token block) of 16 KB in a backing file, 65,536 of them in host slots; "
                 "two alternating query windows")


def repo_event(args, dev, reps: int = 2):
    """KVMem's repository view: the tiered event with the packed layers' raw
    history in a backing file (direct I/O where the file system allows it)
    and only some units in host RAM.  Each step: tiled scoring of the host
    index, select, the kept lists to the host, the plan, the misses brought
    into host slots from the file, the tiered pack from the slots.  Wall time
    per step with a device synchronize on both sides; step 0 is cold."""
    import os
    import tempfile
    import time

    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W
    from query_conditioned_kv_gb300.event import RepoTieredEvent

    cfg = W.scaled(W.config_8b(), L=8)
    kraw, vraw = cfg.kv_raw(dev)
    meank = cfg.meank_direct(dev)
    kvc.kvc_build_meank(kraw, meank, cfg.lp, cfg.H, cfg.D, cfg.n_tok)
    meank_h, kraw_h, vraw_h = (t.cpu().pin_memory() for t in (meank, kraw, vraw))
    del kraw, vraw, meank
    torch.cuda.empty_cache()
    n_blocks, slots = cfg.n_tok // 32, 65536
    fd, path = tempfile.mkstemp(prefix="kvc_repo_", suffix=".bin")
    os.close(fd)
    try:
        direct = True
        try:
            repo = kvc.KvcRepo(path, n_blocks, cfg.lp, cfg.H, cfg.D, slots, io_threads=8,
                               direct=True)
        except kvc.KvcError:
            direct = False
            repo = kvc.KvcRepo(path, n_blocks, cfg.lp, cfg.H, cfg.D, slots, io_threads=8)
        t0 = time.time()
        repo.put(0, n_blocks, kraw_h, vraw_h, cfg.n_tok)
        put_s = time.time() - t0
        del kraw_h, vraw_h
        qs = [cfg.q(dev, step=0), cfg.q(dev, step=1)]
        ev = RepoTieredEvent(cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, cfg.hist, cfg.budget,
                             cfg.n_sink, cfg.n_recent, theta=cfg.theta, device=dev,
                             stage_layers=4, repo=repo)
        steps = []
        for i in range(2 * reps):
            before = repo.stats()
            torch.cuda.synchronize(dev)
            t = time.perf_counter()
            ev.step(qs[i % 2], meank_h)
            torch.cuda.synchronize(dev)
            ms = (time.perf_counter() - t) * 1e3
            after = repo.stats()
            read = after["bytes_read"] - before["bytes_read"]
            steps.append({"ms": round(ms, 3), "units_used": ev.last_plan[0],
                          "units_missed": ev.last_plan[1],
                          "units_from_file": after["fetched"] - before["fetched"],
                          "file_reads": after["read_calls"] - before["read_calls"],
                          "file_gbs": round(read / (ms * 1e-3) / 1e9, 2) if read else 0.0})
        if kvc.kvc_device_status(ev.dev_status) != 0:
            raise RuntimeError("device status error in the repository event")
        rec = repo.slot_elems * 2
        out = {"workload": REPO_WORKLOAD, "file_bytes": repo.n_units * rec,
               "record_bytes": rec, "host_slots": slots, "direct_io": direct,
               "put_s": round(put_s, 2), "tokens_per_step": cfg.n_tok, "steps": steps,
               "warm_ms": min(x["ms"] for x in steps[2:]) if len(steps) > 2 else None,
               "note": "wall time per step (host planning and file reads are part of it); "
                       "step 0 starts with layers 0-1 in host RAM and the rest on file"}
        repo.close()
        return out
    finally:
        os.remove(path)


def confidence_monitor(args, dev, peak, reps: int = 10):
    """ActKV's confidence monitor: token confidence of one decode step (64
    rows of 151936 fp32 logits, top-20) and the trace trend + budget update
    over 64 traces of 8192 token confidences (window 128, stride 32, bottom
    10%).  CUDA events on the current stream, median of `reps`, L2 flushed
    before each logits rep (the rows are 39 MB, under the L2 size)."""
    import torch
    import query_conditioned_kv_gb300 as kvc
    import workloads as W

    cfg = W.ConfidenceConfig()
    lg = cfg.logits(dev)
    tr = cfg.traces(dev)
    conf = torch.empty(cfg.n_req, dtype=torch.float32, device=dev)
    off = torch.arange(cfg.n_req + 1, dtype=torch.int64, device=dev) * cfg.trace_len
    slope = torch.empty(cfg.n_req, dtype=torch.float64, device=dev)
    budget = torch.empty(cfg.n_req, dtype=torch.int32, device=dev)
    kept = torch.empty(cfg.n_req, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    t_conf, t_trend = [], []
    for r in range(args.warmup + reps):
        flush.fill_(r & 255)
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        budget.fill_(cfg.budget0)
        a.record()
        kvc.kvc_token_confidence(lg, cfg.n_req, cfg.vocab, cfg.top_k, conf, st)
        b.record()
        kvc.kvc_conf_trend_budget(tr, off, cfg.n_req, cfg.trace_len, cfg.window, cfg.stride,
                                  cfg.bottom_pct, cfg.budget_step, cfg.max_budget, slope, budget,
                                  kept, st)
        c.record()
        torch.cuda.synchronize(dev)
        if r >= args.warmup:
            t_conf.append(a.elapsed_time(b))
            t_trend.append(b.elapsed_time(c))
    if kvc.kvc_device_status(st) != 0:
        raise RuntimeError("device status error in the confidence monitor")
    ms_c, ms_t = statistics.median(t_conf), statistics.median(t_trend)
    lg_bytes = lg.numel() * 4
    raised = int((budget > cfg.budget0).sum().item())
    del lg, tr, flush
    torch.cuda.empty_cache()
    return {"workload": f"{cfg.name}: {cfg.n_req} rows of {cfg.vocab} fp32 logits, top-{cfg.top_k}; "
                        f"{cfg.n_req} traces of {cfg.trace_len} confidences (w {cfg.window}, "
                        f"s {cfg.stride}, bottom {cfg.bottom_pct}%)",
            "token_confidence_ms": round(ms_c, 4),
            "token_confidence_rows_per_s": cfg.n_req / (ms_c * 1e-3),
            "logits_gbs": lg_bytes / (ms_c * 1e-3) / 1e9,
            "logits_frac_of_hbm": lg_bytes / (ms_c * 1e-3) / 1e9 / peak,
            "trend_budget_ms": round(ms_t, 4), "budgets_raised": raised}


# ------------------------------------------------------------ oracle arm

def _oracle_units(cfg, picks, dev):
    """Oracle inputs of the sampled (layer, KV head, session) units, from the
    seeded generators only: (l, h, r, q rows, raw K or None, raw V or None,
    Mean-K or None) as numpy bit patterns.  A layer with resident raw K gets
    its Mean-K from the oracle's own build; the others use the drawn index."""
    import numpy as np
    import torch
    import workloads as W
    units = []
    for l, h, r in picks:
        qg = np.stack([W.bf16_bits(cfg.q_unit(r, l, h * cfg.G + g, dev)) for g in range(cfg.G)])
        if l < cfg.lp:
            k = W.bf16_bits(cfg.kraw_unit(l, h, r, dev))
            v = W.bf16_bits(cfg.vraw_unit(l, h, r, dev))
            units.append((l, h, r, qg, k, v, None))
        else:
            mk = W.bf16_bits(cfg.meank_direct_unit(l, h, r, dev))
            units.append((l, h, r, qg, None, None, mk))
    if dev is not None and getattr(dev, "type", "cpu") == "cuda":
        torch.cuda.synchronize(dev)
    return units


def _oracle_sample(n_units, dev):
    """The first n_units (layer, KV head) units of the 8B-class event, spread
    over the layers (unit u → (l, h) of index 37·u mod 288)."""
    import workloads as W
    cfg = W.config_8b()
    picks = []
    for u in range(n_units):
        l, h = divmod(u * 37 % (cfg.L * cfg.H), cfg.H)
        picks.append((l, h, 0))
    return cfg, _oracle_units(cfg, picks, dev)


def _oracle_event(cfg, units, threads):
    """score → select → pack of the sampled units with the oracle (pack only
    where the unit's layer has resident raw K/V); returns seconds.  The Mean-K
    build (index maintenance) runs first and is not part of the timed event."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    mks = [u[6] if u[6] is not None else oracle.meank(u[4][None])[0] for u in units]

    def one(i):
        l, h, r, qg, k, v, _ = units[i]
        s = oracle.score_unit(qg, mks[i])
        kept, cnt, _ = oracle.select(s, cfg.budget, cfg.n_sink, cfg.n_recent)
        if k is not None:
            oracle.pack_unit(k, v, kept, cnt, cfg.budget, cfg.pos0, cfg.theta)
        return cnt

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(len(units))))
    return time.perf_counter() - t0


def cpu_baseline(args, dev=None):
    """The oracle on a sample of the 8B-class event's units: on every host
    core (a thread pool over the units), and on one thread."""
    cores = os.cpu_count() or 1
    n_units = args.cpu_units
    cfg, units = _oracle_sample(n_units, dev)
    secs = _oracle_event(cfg, units, cores)
    frac = n_units / (cfg.L * cfg.H)
    value = cfg.n_tok * frac / secs
    n1 = max(1, n_units // 4)
    secs1 = _oracle_event(cfg, units[:n1], 1)
    value1 = cfg.n_tok * (n1 / (cfg.L * cfg.H)) / secs1
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_units} of {cfg.L * cfg.H} (layer, KV head) units of the event "
                      f"(score+select+pack, fp64 C oracle, thread pool of {cores}); "
                      f"{secs:.2f} s wall, tokens scaled by {frac:.4f}",
            "single_thread": {"value": value1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} of the same units on one thread; "
                                        f"{secs1:.2f} s wall, tokens scaled by "
                                        f"{n1 / (cfg.L * cfg.H):.4f}"}}


def run_reference(args, rank, world):
    """The oracle arm: W untimed and K timed steps, each the whole event
    (score → select → pack) of a sample of (layer, KV head) units on the host
    cores.  The sample shrinks, from --cpu-units, only as far as keeps the
    K + W steps within about three minutes (measured on the first warm-up)."""
    import torch
    dev = None
    if torch.cuda.is_available():
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
    cores = os.cpu_count() or 1
    cfg, units = _oracle_sample(args.cpu_units, dev)
    n_steps, n_warm = max(1, args.steps), max(0, args.warmup)
    n = len(units)
    if n_warm > 0:
        est = _oracle_event(cfg, units, cores)
        n = max(1, min(n, int(n * 180.0 / (est * (n_steps + n_warm)))))
        for _ in range(n_warm - 1):
            _oracle_event(cfg, units[:n], cores)
    times = [_oracle_event(cfg, units[:n], cores) for _ in range(n_steps)]
    secs = sum(times) / len(times)
    frac = n / (cfg.L * cfg.H)
    value = cfg.n_tok * frac / secs
    sample = (f"each step: {n} of {cfg.L * cfg.H} (layer, KV head) units of the event "
              f"(score+select+pack, fp64 C oracle, thread pool of {cores}), i.e. "
              f"{frac:.4f} of its KV tokens; {n_steps} timed steps after {n_warm} warm-up")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": n_steps, "warmup": n_warm,
            "ms_per_step": secs * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, workloads/)",
            "config": bench_config(cfg, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-units", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-27b", action="store_true",
                    help="skip the 27B-class 1M-token event measurement")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the 128-session ragged event measurement")
    ap.add_argument("--no-slotmap", action="store_true",
                    help="skip the QueryMemory (slot-map) event measurement")
    ap.add_argument("--no-repo", action="store_true",
                    help="skip the repository-view measurement (repo_event)")
    ap.add_argument("--no-tiered", action="store_true",
                    help="skip the host-resident (tiered) event measurement")
    ap.add_argument("--no-confidence", action="store_true",
                    help="skip the confidence-monitor measurement")
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the ActKV paged-operation measurement")
    ap.add_argument("--groups", type=int, default=None,
                    help="layer groups of the pipelined event (default: the library's choice)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    import torch
    dev = torch.device("cuda", local_rank)

    def extra(key, fn):
        """One extra workload's measurement under `key`.  If it fails, the key
        holds the error and the line (the headline measured above) still
        prints."""
        torch.cuda.empty_cache()
        try:
            line[key] = fn()
        except Exception as e:
            line[key] = {"error": f"{type(e).__name__}: {e}"}
            print(f"bench: {key} failed: {type(e).__name__}: {e}", file=sys.stderr, flush=True)

    for name, flag in (("27b_1m", args.no_27b), ("ragged_128", args.no_ragged)):
        if not flag:
            extra("event_" + name,
                  lambda name=name: config_event(args, dev, name=name, peak=peaks()[0]))
    if not args.no_slotmap:
        extra("slotmap_event", lambda: slot_map_event(args, dev, peaks()[0]))
    if not args.no_tiered:
        extra("tiered_event", lambda: tiered_event(args, dev, peaks()[0]))
    if not args.no_repo:
        extra("repo_event", lambda: repo_event(args, dev))
    if not args.no_paged:
        extra("actkv_event", lambda: paged_event(args, dev, peaks()[0]))
    if not args.no_confidence:
        extra("confidence_monitor", lambda: confidence_monitor(args, dev, peaks()[0]))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
