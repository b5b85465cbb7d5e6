#!/usr/bin/env python
"""Benchmark of the KV residency path: selected KV rows resolved + gathered per second.

One step = one decode step of the workload = every layer group's ula_step_group
(dedup, translate, PB-LRU rotate/mark, victim selection, write-back + fill +
commit, gather of all layers) plus the step's appended-token alloc.

  value     : rows/s with the step inputs already in HBM (device-timed, CUDA events)
  e2e       : the same through the C ABI with host buffers: per step the selections are
              copied from pinned host memory, appended rows are read from pinned host
              memory by the alloc, and the per-request row offsets are read back
  roofline  : the gather kernel (dominant bytes), timed per launch with CUDA events on
              the stream each launch runs on, against the measured HBM copy peak
  host_link : the move kernel (write-back + fill over the host link) against the
              measured pinned copy bandwidth
  cpu_baseline : the CPU oracle on a bounded sample of the same workload (1 core)

--impl reference times the CPU oracle alone (the reference arm).
Multi-GPU (torchrun, N > 1): independent replicas, one per GPU; value = all ranks'
rows / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selected KV rows resolved+gathered/sec; HBM & host-link GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longdoc")
    ap.add_argument("--policy", choices=["pblru", "exact"], default="pblru",
                    help="replacement policy: PB-LRU, or exact LRU (timestamp scan)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of --steps steps each; value = their median")
    ap.add_argument("--hit-rates", action="store_true",
                    help="CPU only: the oracle over the workload's whole trace, PB-LRU against "
                         "exact LRU hit rates (one JSON line)")
    ap.add_argument("--one-stream", action="store_true",
                    help="issue every group's call on the one caller stream (each group's "
                         "step then waits for the previous group's); by default each group "
                         "has its own caller stream, so later groups' steps are issued ahead")
    ap.add_argument("--gather-beside", action="store_true",
                    help="run the hit gather beside the move (ULA_FLAG_GATHER_BESIDE_MOVE)")
    ap.add_argument("--profile-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layer-signal", action="store_true",
                    help="layer-major fill with a device flag per layer (reports how early "
                         "each layer is ready)")
    ap.add_argument("--latency-steps", type=int, default=20,
                    help="steps of the per-layer ready-time pass (synchronised per step)")
    ap.add_argument("--tp", type=int, default=1,
                    help="TP mode emulated with this many partitions (reports the local "
                         "buffers' hit rate and the fetched bytes)")
    ap.add_argument("--buffer-frac", type=float, default=2.0,
                    help="TP local buffer slots per rank and group, in steps' entries")
    ap.add_argument("--pool-frac", type=float, default=None,
                    help="GPU pool as a fraction of the history (policy comparisons)")
    ap.add_argument("--requests", type=int, default=None,
                    help="run the workload's recipe with fewer live requests (profiling cases)")
    ap.add_argument("--traffic-case", action="store_true",
                    help="after the warm-up steps, re-gather group 0's hit rows once (layer 0) "
                         "and print their number: the launch an ncu traffic capture takes")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed glue

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(values: dict, world: int, device=None) -> dict:
    """MAX of times and SUM of work over ranks (identity when world == 1)."""
    if world == 1:
        return dict(values)
    import torch
    import torch.distributed as dist
    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    mx, sm = t.clone(), t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    out = {}
    for i, k in enumerate(keys):
        out[k] = float(mx[i]) if k.endswith("_ms") else float(sm[i])
    return out


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------- peaks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def host_link_peaks(torch, nbytes=1 << 30):
    """Pinned copy-engine bandwidth, each direction alone and both at once (GB/s)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn, reps=4):
        b = 1e9
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            b = min(b, time.perf_counter() - t0)
        return b

    def h2d():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            h.copy_(d, non_blocking=True)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def both():
        ev[0].record(torch.cuda.current_stream())
        s1.wait_event(ev[0])
        s2.wait_event(ev[0])
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
            ev[1].record(s1)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
            ev[2].record(s2)

    h2d_beside = 0.0
    for _ in range(4):  # the H2D stream's own time while a D2H copy runs beside it
        both()
        torch.cuda.synchronize()
        h2d_beside = max(h2d_beside, nbytes / (ev[0].elapsed_time(ev[1]) / 1e3) / 1e9)
    out = {"h2d_gbs": nbytes / best(h2d) / 1e9, "d2h_gbs": nbytes / best(d2h) / 1e9,
           "bidir_gbs": 2 * nbytes / best(both) / 1e9, "h2d_beside_d2h_gbs": h2d_beside}
    del h, h2, d, d2
    return out


class LinkProbe:
    """The copy engines' bidirectional pinned-copy rate right now (both directions at
    once, `nbytes` each way, best of `reps`): taken beside each timed region, so that a
    region's move rate can be set against the link as it was at that moment (the host
    link is shared with other work on the machine)."""

    def __init__(self, torch, nbytes=256 << 20):
        self.torch, self.n = torch, nbytes
        self.h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        self.h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        self.d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.s1, self.s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def bidir_gbs(self, reps=3):
        """(both directions together, H2D's own rate while D2H runs beside it), GB/s."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        best, best_h2d = 0.0, 0.0
        for _ in range(reps):
            torch.cuda.synchronize()
            ev[0].record(torch.cuda.current_stream())
            self.s1.wait_event(ev[0])
            self.s2.wait_event(ev[0])
            with torch.cuda.stream(self.s1):
                self.d.copy_(self.h, non_blocking=True)
                ev[1].record(self.s1)
            with torch.cuda.stream(self.s2):
                self.h2.copy_(self.d2, non_blocking=True)
                ev[2].record(self.s2)
            torch.cuda.synchronize()
            t_h2d = ev[0].elapsed_time(ev[1]) / 1e3
            t_all = max(t_h2d, ev[0].elapsed_time(ev[2]) / 1e3)
            best = max(best, 2 * self.n / t_all / 1e9)
            best_h2d = max(best_h2d, self.n / t_h2d / 1e9)
        return best, best_h2d


# ------------------------------------------------------------------ GPU arm

def stage_initial(cache, w, synth, torch):
    """Initial contexts: rows generated into a pinned staging buffer, allocated chunk by chunk."""
    trace = synth.Trace(w)
    ctx, base, total = trace.initial()
    G, L, W = w.n_groups, w.layers_per_group, w.row_bytes
    chunk = 32768
    stage = torch.empty(chunk * G * L * W, dtype=torch.uint8, pin_memory=True)
    for b0, n0 in zip(base.tolist(), ctx.tolist()):
        off = 0
        while off < n0:
            m = min(chunk, n0 - off)
            buf = stage[: m * G * L * W]
            view = buf.numpy().reshape(G, m, L, W)
            for g in range(G):
                synth.content_range(w.seed, g, L, b0 + off, m, W, out=view[g])
            got = cache.alloc(m, buf)
            assert got == b0 + off, (got, b0 + off)
            cache.sync()
            off += m
    return trace


def gen_steps(trace, w, n, synth, np):
    """n steps of the trace: (selection, events, (rows of a joining request or None, rows of
    the appended tokens or None)), rows per group [G][n][L][W]."""
    G, L, W = w.n_groups, w.layers_per_group, w.row_bytes

    def rows_for(base, m):
        rows = np.empty((G, m, L, W), dtype=np.uint8)
        for g in range(G):
            synth.content_range(w.seed, g, L, base, m, W, out=rows[g])
        return rows

    steps = []
    for _ in range(n):
        sel, ev = trace.step()
        join = rows_for(ev["join_base"], ev["join_n"]) if ev["join_n"] else None
        app = rows_for(ev["append_base"], ev["append_n"]) if ev["append_n"] else None
        steps.append((sel, ev, (join, app)))
    return steps


def rows_to(rows, to):
    """A step's (join, append) rows as flat tensors made by `to` (device or pinned)."""
    return tuple(to(r) if r is not None else None for r in rows)


def apply_step_events(lib_cache, ev, rows_t):
    """The step's finishing request, joining request and appended tokens, in the order
    the trace assigned logical ranges."""
    if ev["free_n"]:
        lib_cache.free(ev["free_base"], ev["free_n"])
    if ev["join_n"]:
        assert lib_cache.alloc(ev["join_n"], rows_t[0]) == ev["join_base"]
    if ev["append_n"]:
        assert lib_cache.alloc(ev["append_n"], rows_t[1]) == ev["append_base"]


def run_tp(args, local):
    """TP mode emulated on one GPU: P partitions and per-rank local buffers, K timed steps."""
    import numpy as np
    import torch

    import synth
    from serving_step_sparse_gb300.cache import UlaTP

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_for(args)
    P = args.tp
    G, L, W, R = w.n_groups, w.layers_per_group, w.row_bytes, w.n_live
    E = w.entries_per_step
    S = -(-w.gpu_slots // P)
    H = -(-w.max_live_history // P) - S + E
    slots = int(args.buffer_frac * E)
    stream = torch.cuda.current_stream(dev)
    tp = UlaTP(row_bytes=W, layers_per_group=[L] * G, parts=P, gpu_slots=S, host_slots=H,
               ring_buckets=w.ring_buckets, max_logical=w.max_logical, max_entries=E,
               buffer_slots=slots, device=dev, stream=stream)
    trace = synth.Trace(w)
    ctx, base, total = trace.initial()
    chunk = 32768
    stage = torch.empty(chunk * G * L * W, dtype=torch.uint8, pin_memory=True)
    for b0, n0 in zip(base.tolist(), ctx.tolist()):
        off = 0
        while off < n0:
            m = min(chunk, n0 - off)
            view = stage[: m * G * L * W].numpy().reshape(G, m, L, W)
            for g in range(G):
                synth.content_range(w.seed, g, L, b0 + off, m, W, out=view[g])
            assert tp.alloc(m, stage[: m * G * L * W]) == b0 + off
            tp.sync()
            off += m
    n = args.warmup + args.steps
    steps = gen_steps(trace, w, n, synth, np)
    sel_dev = torch.from_numpy(np.stack([x[0] for x in steps]).view(np.int32)).to(dev)
    rows_dev = [rows_to(x[2], lambda r: torch.from_numpy(r.reshape(-1)).to(dev)) for x in steps]
    lo = [[tp.out_buffer(g, E) for _ in range(P)] for g in range(G)]
    ro = [[tp.out_buffer(g, E) for _ in range(P)] for g in range(G)]
    mk = lambda k: [torch.empty(k, dtype=torch.int32, device=dev) for _ in range(P)]
    ler, lrq, rer, rrq = mk(E), mk(R + 1), mk(E), mk(R + 1)

    def do_step(t):
        for g in range(G):
            tp.step_group(g, sel_dev[t][g], lo[g], ro[g], ler, lrq, rer, rrq)
        apply_step_events(tp, steps[t][1], rows_dev[t])

    for t in range(args.warmup):
        do_step(t)
    st0 = tp.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for t in range(args.warmup, n):
        do_step(t)
    e1.record(stream)
    st1 = tp.sync()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    d = [{k: st1[i][k] - st0[i][k] for k in st1[i]} for i in range(2 * P)]
    rows = sum(x["rows_gathered"] for x in d)
    rem_uniq = sum(x["uniq"] for x in d[P:])
    rem_hits = sum(x["hits"] for x in d[P:])
    fetched = sum(x["bytes_h2d"] for x in d[P:])
    host = sum(x["bytes_h2d"] for x in d[:P])
    tp.close()
    return {"metric": METRIC, "value": rows / (ms / 1e3), "unit": "rows/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic (seeded trace; rows are seeded random bytes)",
            "config": dict(w.summary(), parallelism=f"TP emulated: {P} partitions on one GPU",
                           partition_gpu_slots=S, partition_host_slots=H, buffer_slots=slots),
            "tp": {"parts": P, "buffer_hit_rate": rem_hits / max(1, rem_uniq),
                   "remote_rows_per_step": rem_uniq / args.steps,
                   "fetched_bytes_per_step": fetched / args.steps,
                   "host_fill_bytes_per_step": host / args.steps,
                   "note": "all P ranks' work runs on this one GPU; a fetch is a copy inside "
                           "HBM, standing in for the cross-GPU copy of TP mode"}}


def run_gpu(args, rank, world, local):
    import numpy as np
    import torch

    import synth
    from serving_step_sparse_gb300 import ula
    from serving_step_sparse_gb300.cache import UlaCache
    from synth.configs import WORKLOADS

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_for(args)
    G, L, W, R, Q, K = (w.n_groups, w.layers_per_group, w.row_bytes, w.n_live, w.q, w.k)
    E = w.entries_per_step
    stream = torch.cuda.current_stream(dev)

    t_setup = time.perf_counter()
    link = host_link_peaks(torch)
    cache = UlaCache(row_bytes=W, layers_per_group=[L] * G, gpu_slots=w.gpu_slots,
                     host_slots=w.host_slots, ring_buckets=w.ring_buckets,
                     max_logical=w.max_logical, max_entries=E, device=dev, stream=stream,
                     bypass_overflow=w.bypass, exact_lru=w.exact_lru,
                     layer_signal=args.layer_signal, gather_beside_move=args.gather_beside)
    trace = stage_initial(cache, w, synth, torch)
    NS, reps = args.steps, max(1, args.repeats)
    n_value, n_prof = NS * reps, min(args.profile_steps, NS)
    n_lat = min(args.latency_steps, NS)
    n_e2e = 0 if args.no_e2e else NS * reps
    # warm-up, timed, profiled, latency and e2e passes run consecutive steps of the trace
    # (past the recipe's trace length the generator continues the same recipe)
    need = args.warmup + n_value + n_prof + n_lat + n_e2e
    steps = gen_steps(trace, w, need, synth, np)
    outs = [cache.out_buffer(g, E) for g in range(G)]
    entry_row = [torch.empty(E, dtype=torch.int32, device=dev) for _ in range(G)]
    req_off = [torch.empty(R + 1, dtype=torch.int32, device=dev) for _ in range(G)]
    # device-resident inputs for the value, profiled and latency passes
    n_dev = args.warmup + n_value + n_prof + n_lat
    sel_dev = torch.from_numpy(np.stack([s[0] for s in steps[:n_dev]]).view(np.int32)).to(dev)
    rows_dev = [rows_to(s[2], lambda r: torch.from_numpy(r.reshape(-1)).to(dev))
                for s in steps[:n_dev]]
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    # Each group's calls go on a caller stream of their own, so later groups' (and the
    # next step's) calls are issued ahead: the library orders each group's step after that
    # group's previous step and alloc only, and runs a group's metadata while earlier
    # calls' copies run.  The step's appended tokens are allocated on the main stream (the
    # library places them in each group after that group's step).  `wait` makes the
    # group streams wait for the main stream first (inputs copied there).
    gstreams = [stream] * G if args.one_stream else [torch.cuda.Stream(dev) for _ in range(G)]
    step_evt = [torch.cuda.Event() for _ in range(4)]
    nstep = [0]

    def issue_groups(sel_t, wait=False):
        if args.one_stream:
            for g in range(G):
                cache.step_group(g, sel_t[g], outs[g], entry_row[g], req_off[g])
            return
        if wait:
            e = step_evt[nstep[0] % len(step_evt)]
            nstep[0] += 1
            e.record(stream)
            for g in range(G):
                gstreams[g].wait_event(e)
        for g in range(G):
            cache.step_group(g, sel_t[g], outs[g], entry_row[g], req_off[g], stream=gstreams[g])

    def join_groups():
        if not args.one_stream:
            for g in range(G):
                stream.wait_stream(gstreams[g])

    def do_step(sel_t, ev, rows_t):
        issue_groups(sel_t)
        apply_step_events(cache, ev, rows_t)

    # The clock sampler starts (and its start-up pause passes) before the warm-up steps,
    # so that the first timed region follows the warm-up without an idle gap.
    clocks = ClockSampler(local)
    clocks.start()
    for t in range(args.warmup):
        do_step(sel_dev[t], steps[t][1], rows_dev[t])
    st0 = cache.sync()
    if args.traffic_case:
        st = cache.export(0)
        out = cache.out_buffer(0, max(1, st["U"]))
        torch.empty(512 << 20, dtype=torch.uint8, device=dev).zero_()  # flush L2 (129 MB)
        torch.cuda.synchronize()
        # the step's gather launch: every layer of group 0's hit rows in one launch
        ula.ula_debug_regather(cache.ctx, 0, 0, out.data_ptr(), out.shape[1], stream.cuda_stream,
                               n_layers=L)
        torch.cuda.synchronize()
        print(json.dumps({"traffic_case": {"hit_rows": st["hits"], "unique_rows": st["U"],
                                           "gather_launches_before": args.warmup * G}}))
        clocks.stop()
        cache.close()
        sys.exit(0)
    ula.ula_profile_read(cache.ctx, reset=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()

    # ---- value: inputs resident in HBM; `reps` timed regions of NS steps each, with the
    # copy kernels' device spans recorded in the same pass
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe = LinkProbe(torch)
    repeats = []
    launches = 0
    t = args.warmup
    for rep in range(reps):
        sa = cache.sync()
        ula.ula_profile_spans(cache.ctx, True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        e0.record(stream)
        for _ in range(NS):
            do_step(sel_dev[t], steps[t][1], rows_dev[t])
            t += 1
        join_groups()
        e1.record(stream)
        torch.cuda.nvtx.range_pop()
        sb = cache.sync()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms = e0.elapsed_time(e1)
        spans = ula.ula_profile_spans_read(cache.ctx)
        ula.ula_profile_spans(cache.ctx, False)
        launches += sum(p["kernels"] for p in ula.ula_profile_read(cache.ctx, reset=True).values())
        d = {k: sb[k] - sa[k] for k in sb}
        ce, ce_h2d = probe.bidir_gbs()
        repeats.append({"ms": ms, "stats": d, "spans": span_summary(spans, d, L, W, G * NS),
                        "ce_bidir_gbs": ce, "ce_h2d_beside_d2h_gbs": ce_h2d})
    launches //= reps
    order = sorted(range(reps), key=lambda i: repeats[i]["ms"])
    med = repeats[order[reps // 2]]
    value_ms = med["ms"]
    rows_value = med["stats"]["rows_gathered"]
    st1 = cache.sync()

    # ---- profiled pass: per-phase CUDA-event durations (metadata phases included)
    ula.ula_profile_enable(cache.ctx, True)
    st2a = cache.sync()
    for t in range(args.warmup + n_value, args.warmup + n_value + n_prof):
        do_step(sel_dev[t], steps[t][1], rows_dev[t])
    st2 = cache.sync()
    prof = ula.ula_profile_read(cache.ctx, reset=True)
    ula.ula_profile_enable(cache.ctx, False)

    # ---- per-layer ready times (one step at a time): from the group call to its
    # layer_ready events (CUDA events on the caller's stream side), and, with the
    # layer signal, to each layer's device flag (globaltimer in the kernels)
    ev_ms = [[] for _ in range(L)]
    flag_ms = [[] for _ in range(L)]
    t0_ev = torch.cuda.Event(enable_timing=True)
    lr_ev = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
    for t in range(n_dev - n_lat, n_dev):
        sel_t, ev, rows_t = sel_dev[t], steps[t][1], rows_dev[t]
        for g in range(G):
            torch.cuda.synchronize()
            t0_ev.record(stream)
            cache.step_group(g, sel_t[g], outs[g], entry_row[g], req_off[g], layer_ready=lr_ev)
            cache.sync()
            torch.cuda.synchronize()
            for j in range(L):
                ev_ms[j].append(t0_ev.elapsed_time(lr_ev[j]))
            if args.layer_signal:
                ns = ula.ula_debug_layer_times(cache.ctx, g, L)
                for j in range(L):
                    flag_ms[j].append((int(ns[j]) - int(ns[L])) / 1e6)
        apply_step_events(cache, ev, rows_t)
    cache.sync()
    layer_ready = {"layer_ready_event_ms": [round(float(np.median(x)), 4) for x in ev_ms],
                   "how": "median over groups and steps; one group call at a time, from an "
                          "event recorded before the call to its layer_ready events"}
    if args.layer_signal:
        layer_ready["layer_flag_ms"] = [round(float(np.median(x)), 4) for x in flag_ms]
        layer_ready["flag_how"] = ("device globaltimer from the step's first kernel to the "
                                   "store of each layer's flag")

    # ---- e2e: host buffers through the C ABI
    e2e = None
    if n_e2e:
        sel_host = torch.from_numpy(np.stack([s[0] for s in steps[n_dev:]]).view(np.int32))
        sel_host = sel_host.pin_memory()
        rows_host = [rows_to(s[2], lambda r: torch.from_numpy(r.reshape(-1)).pin_memory())
                     for s in steps[n_dev:]]
        sel_buf = [torch.empty((G, R, Q, K), dtype=torch.int32, device=dev) for _ in range(2)]
        res_host = torch.empty((n_e2e, G, R + 1), dtype=torch.int32, pin_memory=True)
        h2d_bytes = d2h_bytes = 0
        # Each step's selections go up on a stream of their own into one of two device
        # buffers; each group's calls wait for their upload, and each group reads its CSR
        # offsets back on its own stream right after its call, so that steps overlap as in
        # the timed regions.  A buffer is refilled once every group's call of two steps
        # before has ended.
        up = stream if args.one_stream else torch.cuda.Stream(dev)
        up_evt = [torch.cuda.Event() for _ in range(2)]
        used = [[torch.cuda.Event() for _ in range(G)] for _ in range(2)]
        # `reps` regions of NS steps, like the timed regions; the median region is reported
        regions = []
        for rep in range(reps):
            sa = cache.sync()
            torch.cuda.synchronize()
            e0.record(stream)
            up.wait_stream(stream)
            for g in range(G):
                gstreams[g].wait_stream(stream)
            for i in range(rep * NS, (rep + 1) * NS):
                b = i % 2
                buf = sel_buf[b]
                if i >= 2 and not args.one_stream:
                    for g in range(G):
                        up.wait_event(used[b][g])
                with torch.cuda.stream(up):
                    buf.copy_(sel_host[i], non_blocking=True)
                up_evt[b].record(up)
                h2d_bytes += buf.numel() * 4
                for g in range(G):
                    gs = gstreams[g]
                    gs.wait_event(up_evt[b])
                    cache.step_group(g, buf[g], outs[g], entry_row[g], req_off[g], stream=gs)
                    with torch.cuda.stream(gs):
                        res_host[i, g].copy_(req_off[g], non_blocking=True)
                    used[b][g].record(gs)
                    d2h_bytes += (R + 1) * 4
                ev = steps[n_dev + i][1]
                apply_step_events(cache, ev, rows_host[i])  # rows read from pinned host memory
                h2d_bytes += sum(r.numel() for r in rows_host[i] if r is not None)
            join_groups()
            stream.wait_stream(up)
            e1.record(stream)
            sb = cache.sync()
            torch.cuda.synchronize()
            regions.append((e0.elapsed_time(e1), sb["rows_gathered"] - sa["rows_gathered"]))
        assert int(res_host[-1, 0, -1]) > 0
        e2e_ms, rows_e2e = sorted(regions)[len(regions) // 2]
        e2e = {"rows": rows_e2e, "e2e_ms": e2e_ms, "h2d": h2d_bytes / n_e2e,
               "d2h": d2h_bytes / n_e2e,
               "regions_rows_per_s": [round(r / (ms / 1e3)) for ms, r in regions]}
    clk = clocks.stop()

    # ---- roofline of the gather (the dominant HBM bytes): one launch per group-step gathers
    # every layer of the step's hit rows (algorithmic bytes: each layer's row read from the
    # pool and written to out; missed rows' outputs are written by the move from the bytes
    # it moves).  Durations are the launches' device spans in the median timed region.
    hbm_peak, hbm_src = measured_peaks()
    sp = med["spans"]
    ga = sp.get("gather", {"launches": 0, "sum_us": 0.0, "union_us": 0.0})
    hit_rows = med["stats"]["hits"] * L
    g_bytes = hit_rows * 2 * W
    avg_launch_us = ga["sum_us"] / max(1, ga["launches"])
    achieved = g_bytes / (ga["sum_us"] * 1e3) if ga["sum_us"] else 0.0  # bytes/ns = GB/s
    iso = isolated_gather(cache, ula, torch, dev, stream, W, L)
    roof = {"bound": "hbm", "kernel": "k_gather_bulk", "achieved": round(achieved, 1),
            "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
            "traffic": traffic_per_launch(med["stats"]["hits"], ga["launches"], args.workload),
            "traffic_read_per_hit_row": (round(GATHER_TRAFFIC["read_bytes_per_hit"], 1)
                                         if traffic_per_launch(1, 1, args.workload) else None),
            "algorithmic_read_per_hit_row": L * W,
            "peak_source": f"{hbm_src} (hbm_gbs, STREAM-style copy)",
            "avg_launch_us": round(avg_launch_us, 2),
            "bytes_per_launch": round(g_bytes / max(1, ga["launches"])),
            "rows_per_launch": round(hit_rows / max(1, ga["launches"]), 1), "bytes_per_row": 2 * W,
            "union_us_per_step": round(ga["union_us"] / NS, 2),
            "timing": ("in the timed region (median repeat): device globaltimer span of each "
                       "gather launch, first warp start to last warp end; achieved = hit-gather "
                       "bytes / summed spans (the launches do not overlap: union "
                       f"{ga['union_us']:.1f} us, sum {ga['sum_us']:.1f} us)"),
            "isolated": iso}
    # ---- host link: the move kernel moves fills (H2D) and write-backs (D2H) at once;
    # its device spans in the same timed region
    mv = sp.get("move", {"launches": 0, "sum_us": 0.0, "union_us": 0.0})
    # the link is shared with the machine's other work: its capacity is the best the copy
    # engines showed in this run (at set-up, and after every timed region)
    link = dict(link, bidir_gbs=max([link["bidir_gbs"]] + [r["ce_bidir_gbs"] for r in repeats]),
                h2d_beside_d2h_gbs=max([link["h2d_beside_d2h_gbs"]] +
                                       [r["ce_h2d_beside_d2h_gbs"] for r in repeats]))
    mv_s = mv["sum_us"] / 1e6
    h2d_b, d2h_b = med["stats"]["bytes_h2d"], med["stats"]["bytes_d2h"]
    host = {"kernel": "k_move_layers + k_commit" if args.layer_signal else "k_move",
            "fill_gbs": round(h2d_b / mv_s / 1e9, 1) if mv_s else 0,
            "writeback_gbs": round(d2h_b / mv_s / 1e9, 1) if mv_s else 0,
            "total_gbs": round((h2d_b + d2h_b) / mv_s / 1e9, 1) if mv_s else 0,
            "peak_h2d_gbs": round(link["h2d_gbs"], 1), "peak_d2h_gbs": round(link["d2h_gbs"], 1),
            "peak_bidir_gbs": round(link["bidir_gbs"], 1),
            "peak_h2d_beside_d2h_gbs": round(link["h2d_beside_d2h_gbs"], 1),
            "peak_source": ("measured in this run: pinned cudaMemcpyAsync, 1 GiB each way at "
                            "set-up, 256 MiB each way after every timed region (both directions: "
                            "the best of these)"),
            "timing": "device spans of the move launches in the median timed region",
            "move_us_per_step": round(mv["sum_us"] / NS, 2)}
    if mv_s:
        # fills against the H2D copy alone, and against H2D while a D2H copy runs beside
        # it (the move's write-backs share the link with its fills); fills and write-backs
        # together against both directions at once
        host["frac_fill"] = round(h2d_b / mv_s / 1e9 / link["h2d_gbs"], 4)
        host["frac_fill_beside_d2h"] = round(h2d_b / mv_s / 1e9 / link["h2d_beside_d2h_gbs"], 4)
        host["frac_total"] = round((h2d_b + d2h_b) / mv_s / 1e9 / link["bidir_gbs"], 4)
    rep_lines = []
    for r in repeats:
        m = r["spans"].get("move", {"sum_us": 0.0})
        gsp = r["spans"].get("gather", {"sum_us": 0.0})
        mb = r["stats"]["bytes_h2d"] + r["stats"]["bytes_d2h"]
        gb = r["stats"]["hits"] * L * 2 * W
        mg = mb / (m["sum_us"] * 1e3) if m["sum_us"] else None
        rep_lines.append({"value": r["stats"]["rows_gathered"] / (r["ms"] / 1e3),
                          "ms_per_step": round(r["ms"] / NS, 4),
                          "move_gbs": round(mg, 1) if mg else None,
                          "ce_bidir_gbs_after": round(r["ce_bidir_gbs"], 1),
                          "move_frac_of_ce_after": round(mg / r["ce_bidir_gbs"], 4) if mg else None,
                          "gather_gbs": round(gb / (gsp["sum_us"] * 1e3), 1) if gsp["sum_us"] else None})
    phases = {k: round(v["ms"] / max(1, n_prof), 4) for k, v in prof.items() if v["timed"]}

    agg = aggregate({"rows": rows_value, "value_ms": value_ms}, world, dev)
    res = {
        "rows": agg["rows"], "value_ms": agg["value_ms"], "launches": launches,
        "roofline": roof, "host_link": host, "clocks": clk, "phases": phases, "e2e": e2e,
        "layer_ready": layer_ready, "repeats": rep_lines,
        "spans_us_per_step": {k: round(v["sum_us"] / NS, 2) for k, v in sp.items()},
        "metadata_beside_copies": (round(sp["select"]["beside_copies_us"] /
                                         max(1e-9, sp["select"]["union_us"]), 4)
                                   if "select" in sp else None),
        "setup_s": setup_s, "stats": med["stats"],
        "host_huge": [None if f is None else round(f, 3) for f in cache.host_huge_fraction],
    }
    if e2e is not None:
        a = aggregate({"rows": e2e["rows"], "e2e_ms": e2e["e2e_ms"]}, world, dev)
        res["e2e"] = {"value": a["rows"] / (a["e2e_ms"] / 1e3), "unit": "rows/s",
                      "h2d_bytes_per_step": int(e2e["h2d"]), "d2h_bytes_per_step": int(e2e["d2h"]),
                      "ms_per_step": round(a["e2e_ms"] / NS, 4),
                      "regions": e2e["regions_rows_per_s"],
                      "timing": "median of the regions (as for value), NS steps each"}
    cache.close()
    return res


def isolated_gather(cache, ula, torch, dev, stream, W, L, reps=20):
    """The gather kernel alone, in the step's launch (every layer of group 0's last hit
    rows), L2 flushed before each launch, CUDA events on the launching stream; with the
    step's grid and with every block that fits on the SMs."""
    st = cache.export(0)
    hits = st["hits"]
    out = cache.out_buffer(0, max(1, st["U"]))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    peak, _ = measured_peaks()
    kinds = [(0, L)]
    res = {}
    for name, bps in (("step_grid", 0), ("full_grid", 64)):
        ms = {k: [] for k in kinds}
        for i in range(reps + 2):
            for k in kinds:
                flush.zero_()
                e0.record(stream)
                ula.ula_debug_regather(cache.ctx, 0, k[0], out.data_ptr(), out.shape[1],
                                       stream.cuda_stream, blocks_per_sm=bps, n_layers=k[1])
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    ms[k].append(e0.elapsed_time(e1))
        avg = {k: sum(v) / len(v) for k, v in ms.items()}
        ach = hits * L * 2 * W / (sum(avg.values()) / 1e3) / 1e9
        res[name] = {"achieved": round(ach, 1), "frac": round(ach / peak, 4),
                     "avg_launch_us": round(sum(avg.values()) / len(avg) * 1e3, 2),
                     "launch_us": {f"layers {k[0]}..{k[0] + k[1] - 1}": round(v * 1e3, 2)
                                   for k, v in avg.items()}}
    res.update({"hit_rows": hits, "launches": reps * len(kinds),
                "l2": "flushed (512 MB write) before each launch"})
    return res


def union_ns(iv) -> int:
    """Length of the union of [a, b) intervals."""
    tot, c0, c1 = 0, None, None
    for a, b in sorted(iv):
        if c1 is None or a > c1:
            if c1 is not None:
                tot += c1 - c0
            c0, c1 = a, b
        else:
            c1 = max(c1, b)
    if c1 is not None:
        tot += c1 - c0
    return tot


def merged(iv):
    """The union of [a, b) intervals as sorted disjoint intervals."""
    out = []
    for a, b in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def overlap_ns(x, y) -> int:
    """Length of the intersection of two unions of intervals."""
    xs, ys = merged(x), merged(y)
    i = j = tot = 0
    while i < len(xs) and j < len(ys):
        lo, hi = max(xs[i][0], ys[j][0]), min(xs[i][1], ys[j][1])
        if hi > lo:
            tot += hi - lo
        if xs[i][1] < ys[j][1]:
            i += 1
        else:
            j += 1
    return tot


def span_summary(spans, d, L, W, group_steps):
    """Per kernel kind of one timed region: launches, summed and united device spans (us);
    for the metadata ("select": dedup through victim emission), how much of it ran while
    the copy kernels (gather, staging, move) were running."""
    by = {}
    for ph, _g, t0, t1 in spans:
        if t1 >= t0 > 0:
            by.setdefault(ph, []).append((t0, t1))
    out = {ph: {"launches": len(iv), "sum_us": sum(b - a for a, b in iv) / 1e3,
                "union_us": union_ns(iv) / 1e3} for ph, iv in by.items()}
    if "select" in by:
        copies = [x for ph in ("gather", "stage", "move") for x in by.get(ph, [])]
        out["select"]["beside_copies_us"] = overlap_ns(by["select"], copies) / 1e3
    return out


# DRAM traffic of the gather kernel measured by ncu (dram__bytes_read.sum and
# dram__bytes_write.sum of one launch), per hit row, with the case it was taken on and
# the hash of the gather kernel's source (its launch-shape defaults and its body).
# Reported only while that source is unchanged and for the workload it was taken on.
GATHER_TRAFFIC = {"source_sha256": "0001e758e1cafa8159303f83b95ab22d89bcb7de0a46017016194da97a457ee6",
                  "workload": "longdoc",  # the recipe; the case had 12 of its 32 requests
                  "case": "long-document recipe with 12 requests: group 0's hit rows after 3 "
                          "steps, re-gathered in the step's one all-layer launch, L2 flushed",
                  "hit_rows": 24255,
                  "read_bytes_per_hit": 64330240 / 24255,   # 2,652 B per 2,624-B slot read
                  "write_bytes_per_hit": 10951936 / 24255}  # written rows mostly stay in L2


def gather_source_sha256() -> str | None:
    """Hash of the hit gather's source (its shared-memory constants and helpers, the kernel,
    and the step grid's constant), or None where the source does not have that shape."""
    src = os.path.join(ROOT, "serving_step_sparse_gb300", "csrc")
    lines = open(os.path.join(src, "ula_kernels.cu")).read().splitlines()
    try:
        start = next(i for i, ln in enumerate(lines) if ln.startswith("constexpr int kBulkThreads"))
        body = next(i for i, ln in enumerate(lines) if "k_gather_bulk(GatherParams p) {" in ln)
        end = next(i for i in range(body, len(lines)) if lines[i] == "}")
    except StopIteration:
        return None
    keep = lines[start:end + 1]
    keep += [ln for ln in open(os.path.join(src, "ula_api.cu")).read().splitlines()
             if ln.startswith("constexpr uint32_t kGatherRowsPerBlock")]
    return hashlib.sha256("\n".join(keep).encode()).hexdigest()


def traffic_per_launch(hits, launches, workload):
    """DRAM bytes (read + write) per gather launch in the step, from the ncu figures per
    hit row scaled by the hits (reads grow in proportion to the rows gathered); None when
    they were taken on another gather source or another workload's recipe."""
    t = GATHER_TRAFFIC
    if (not launches or t["source_sha256"] is None or t["source_sha256"] != gather_source_sha256()
            or t["workload"] != workload):
        return None
    return round(hits * (t["read_bytes_per_hit"] + t["write_bytes_per_hit"]) / launches)


# ------------------------------------------------------------- CPU oracle arm

def run_oracle(w, warmup, steps=None, seconds=None):
    """The oracle as it stands, single-threaded and pinned to one host core, on the same
    workload `w` (its exact-LRU mode for an exact-LRU workload), for `steps` steps or until `seconds`
    of oracle time.  It runs in content-id mode (8-byte rows naming their address, group
    and layer: exact, since a row's bytes are a function of those): the byte mode needs
    about 40 GB and a quarter of an hour to set up the long-document pools, and moving
    8 instead of 656 bytes per row only makes the oracle faster.  The clock covers the
    oracle's group steps and its alloc/free of the step's events; the selections and the
    rows of joining requests and appended tokens are generated before it starts."""
    from oracle import ExactLru
    from oracle.replay import OracleRun, alloc_rows, apply_events

    run = OracleRun(w, "id")
    # the exact-LRU hit rate on the same trace: the companion (hit counts only), or, where
    # the overflow bypass is on (the companion has none), the oracle's exact-LRU mode
    lru = ExactLru(w.n_groups, w.gpu_slots, w.max_logical) if not w.bypass else None
    exact_run = OracleRun(w.replace(exact_lru=True), "id") if w.bypass else None
    exact_acc = [0, 0]  # unique, hits (timed steps)
    if lru is not None:
        for b, n in [(int(b), int(c)) for b, c in zip(*run.trace.initial()[1::-1])]:
            lru.alloc(n)
    t_oracle = 0.0
    rows = hits = uniq = 0
    n_done = 0
    limit = steps if steps is not None else 10 ** 9
    allowed = os.sched_getaffinity(0)
    core = max(allowed)
    os.sched_setaffinity(0, {core})  # this thread only, for the timed loop
    try:
        while n_done < warmup + limit:
            if n_done == warmup and lru is not None:
                lru.acc[:] = 0  # hit rates over the timed steps only
            sel, ev = run.trace.step()
            rows_of = {ev[f"{k}_base"]: alloc_rows(w, ev[f"{k}_base"], ev[f"{k}_n"], "id")
                       for k in ("join", "append") if ev[f"{k}_n"]}
            t0 = time.perf_counter()
            res = [run.o.step_group(g, sel[g]) for g in range(w.n_groups)]
            apply_events(lambda base, n: run.o.alloc(n, rows_of[base]), run.o.free, ev)
            dt = time.perf_counter() - t0
            if lru is not None:
                for g in range(w.n_groups):
                    lru.step_group(g, sel[g])
                if ev["free_n"]:
                    lru.free(ev["free_base"], ev["free_n"])
                for k in ("join", "append"):
                    if ev[f"{k}_n"]:
                        lru.alloc(ev[f"{k}_n"])
            else:
                xr = [exact_run.o.step_group(g, sel[g]) for g in range(w.n_groups)]
                apply_events(lambda base, n: exact_run.o.alloc(n, rows_of[base]),
                             exact_run.o.free, ev)
                if n_done >= warmup:
                    exact_acc[0] += sum(r["counters"]["uniq"] for r in xr)
                    exact_acc[1] += sum(r["counters"]["hits"] for r in xr)
            if n_done >= warmup:
                t_oracle += dt
                for r in res:
                    rows += r["counters"]["rows_gathered"]
                    hits += r["counters"]["hits"]
                    uniq += r["counters"]["uniq"]
            n_done += 1
            if seconds is not None and t_oracle >= seconds and n_done >= warmup + 4:
                break
    finally:
        os.sched_setaffinity(0, allowed)
    timed_steps = n_done - warmup
    return {"value": rows / t_oracle if t_oracle else 0.0, "unit": "rows/s", "cores": 1,
            "pinned_core": core, "host_cores": os.cpu_count(), "kind": "oracle",
            "steps": timed_steps, "seconds": round(t_oracle, 3),
            "sample": (f"{w.description}: the whole workload ({w.n_live} requests, "
                       f"S={w.gpu_slots}, H={w.host_slots}), {timed_steps} decode steps after "
                       f"{warmup} warm-up, rows as 8-byte content ids, single-threaded, pinned "
                       f"to host core {core} of {os.cpu_count()}"),
            "rows": "content ids (8 B per row)",
            "policy": "exact LRU" if w.exact_lru else "PB-LRU",
            "hit_rate": hits / max(1, uniq),
            "exact_lru_hit_rate": (lru.hit_rate if lru is not None
                                   else exact_acc[1] / max(1, exact_acc[0]))}


# -------------------------------------------------------------------- main

def workload_for(args):
    from synth.configs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.policy == "exact":
        w = w.replace(exact_lru=True, name=w.name + "_exact",
                      description=w.description + " (exact LRU)")
    if args.pool_frac is not None:
        w = w.replace(gpu_frac=args.pool_frac, gpu_slots_explicit=None, host_slots_explicit=None,
                      name=w.name + f"_pool{args.pool_frac:g}",
                      description=w.description + f" (GPU pool {args.pool_frac:g} of history)")
    if args.requests is not None and args.requests != w.n_live:
        w = w.replace(n_live=args.requests, name=f"{w.name}_r{args.requests}",
                      description=w.description + f" (recipe with {args.requests} requests)")
    return w


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    w = workload_for(args)
    config = dict(w.summary())
    config["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    if args.layer_signal:
        config["layer_signal"] = True
    config["l2"] = ("inputs larger than L2: GPU pool "
                    f"{w.gpu_slots * w.n_groups * w.layers_per_group * w.row_bytes / 1e9:.1f} GB, "
                    "rows gathered at random slots")

    if args.hit_rates:  # the policy comparison over the whole trace, on the host
        cb = run_oracle(w, 0, steps=w.steps)
        print(json.dumps({"workload": w.name, "steps": cb["steps"], "pblru_hit_rate": cb["hit_rate"],
                          "exact_lru_hit_rate": cb["exact_lru_hit_rate"],
                          "difference_pp": round(100 * (cb["exact_lru_hit_rate"] - cb["hit_rate"]), 4),
                          "oracle_rows_per_s": cb["value"], "config": config}), flush=True)
        return 0
    if args.impl == "reference":
        if rank != 0:
            return 0
        cb = run_oracle(w, args.warmup, steps=args.steps)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "rows/s",
                "n_gpus": args.gpus, "steps": cb["steps"], "warmup": args.warmup,
                "ms_per_step": round(cb["seconds"] / max(1, cb["steps"]) * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                "data": "synthetic", "config": config, "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    if args.tp > 1:
        if rank == 0:
            print(json.dumps(run_tp(args, local)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    r = run_gpu(args, rank, world, local)
    if rank == 0:
        value = r["rows"] / (r["value_ms"] / 1e3)
        line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(r["value_ms"] / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                "data": "synthetic (seeded trace; rows are seeded random bytes)",
                "config": config, "roofline": r["roofline"], "host_link": r["host_link"],
                "gpu_launches": r["launches"], "clocks": r["clocks"],
                "phases_ms_per_step": r["phases"],
                "layer_ready": r["layer_ready"],
                "scheduling_ms_per_step": round(sum(r["phases"].get(k, 0.0)
                                                    for k in ("rotate", "mark", "select")), 4),
                "metadata_ms_per_step": round(sum(r["phases"].get(k, 0.0)
                                                  for k in ("dedup", "rotate", "mark", "select")), 4),
                "hit_rate": r["stats"]["hits"] / max(1, r["stats"]["uniq"]),
                "repeats": r["repeats"], "value_median": value,
                "value_spread": [min(x["value"] for x in r["repeats"]),
                                 max(x["value"] for x in r["repeats"])],
                "spans_us_per_step": r["spans_us_per_step"],
                "metadata_beside_copies": r["metadata_beside_copies"]}
        line["config"]["host_pool_huge_page_fraction"] = r["host_huge"]
        if args.gather_beside:
            line["config"]["gather"] = "beside the move"
        line["config"]["group_calls"] = ("one caller stream" if args.one_stream else
                                         "one caller stream per group (later groups issued ahead)")
        if r["e2e"] is not None:
            line["e2e"] = r["e2e"]
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = run_oracle(w, 2, seconds=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
