"""Benchmark: MoE top-k dispatch + combine on one GB300 (or N replicas).

One step is the whole hot path on one batch of synthetic input: the routing
metadata (compute_send_counts + build_send_layout of the axolotl
``integrations.expert_parallel.torch_dispatch`` page), dispatch (row scatter)
and combine (per-token sum of the expert outputs).  The timed step uses the
no-host-sync form (worst-case row buffers, the "num_worst_tokens" mode of the
NeMo ``uccl_ep.buffer`` page); the pages' host-synchronising call order
(counts -> device->host copy -> layout(num_send)) is timed too and reported
under ``host_sync_path``, and a CUDA-graph replay of the step under
``graph_replay``.

on the large skewed workload (T=16384, H=7168 bf16, E=256, K=8, P=8 logical
ranks, Zipf(1.2) routing).  Inputs are resident in HBM when a step starts; L2
is flushed between steps (512 MiB write, then a 256 MiB read that leaves L2
clean), outside the timed events.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(plain C, one core) on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (evicts every line
    the step could reuse), then read another one, so that the lines L2 holds
    are clean and the next step pays for no write-back of the flush's data."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)   # summed as is: one read
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.wbuf.zero_()
        self.torch.sum(self.rbuf, dim=0, out=self.acc)


# ------------------------------------------------------------ host helpers --
def workload_name(w) -> str:
    """The workload as both arms name it in config.workload."""
    return (f"{w.name}: T={w.T} H={w.H} E={w.E} K={w.K} P={w.P} E_local={w.E_local} "
            f"routing={w.routing}({w.zipf_s}) weights={w.weights}")


def algorithmic_bytes(T: int, H: int, N: int, K: int, P: int) -> dict:
    """Bytes the method must move (each source row read once, each
    destination row written once), per kernel of one step."""
    row = H * 2
    return {
        "counts": T * K * 8 + T * K * 4 + T * P,                       # idx in; dest, is_in_rank out
        "layout": T * K * 8 + T * K * 4 + T * K * 4 + 2 * T * P + T * P * 4 + N * (8 + K * 12),
        "dispatch": T * row + N * row + T * P * 4,
        "combine": N * row + T * row + T * P * 4,
    }


def aggregate(local_seconds: float, local_units: float, world: int, dist=None) -> tuple:
    """Whole-job throughput of N replicas: units summed over ranks, time is the
    slowest rank's.  Returns (units_per_second, max_seconds)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([local_seconds], dtype=torch.float64)
        u = torch.tensor([local_units], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t, u = t.cuda(), u.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        local_seconds, local_units = float(t.item()), float(u.item())
    return local_units / local_seconds, local_seconds


def measured_peak() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


# Source files of the kernels whose DRAM traffic profiles/traffic.json records.
KERNEL_SOURCES = {
    "dispatch": ["ep_move.cu", "ep_rows.cuh", "ep_device.cuh", "ep_internal.h"],
    "combine": ["ep_combine.cu", "ep_rows.cuh", "ep_device.cuh", "ep_internal.h"],
    "route": ["ep_route.cu", "ep_barrier.cuh", "ep_slots.cuh", "ep_device.cuh", "ep_internal.h"],
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_send_counts_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + ["../../include/ep.h"]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(os.path.basename(name).encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per full-size launch from the committed ncu capture, if it was
    taken on the kernel's current sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            k = json.load(f)["kernels"][kernel]
    except Exception:
        return None
    if k.get("source_hash") != kernel_source_hash(kernel):
        return None
    return k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm --
class SendPath:
    """All device buffers of the send-layout path, allocated once.

    Two ways through the same kernels:
      nosync -- ep_route_nosync (counts + layout, rows sized for the worst
                case T*min(K,P), no host round trip) -> ep_dispatch ->
                ep_combine; 4 launches, nothing waits on the host;
      sync   -- ep_compute_send_counts -> device-to-host copy of the counts and
                a host wait -> ep_build_send_layout(num_send) -> ep_dispatch ->
                ep_combine; 6 launches.
    """

    def __init__(self, ep, torch, w, x, idx, wts, dev):
        self.ep, self.torch, self.w = ep, torch, w
        T, K, P, El = w.T, w.K, w.P, w.E_local
        self.x, self.idx, self.wts = x, idx, wts
        i32, u8 = torch.int32, torch.uint8
        self.dest = torch.empty((T, K), dtype=i32, device=dev)
        self.is_in_rank = torch.empty((T, P), dtype=u8, device=dev)
        self.send_counts = torch.empty((1, P), dtype=i32, device=dev)
        self.rank_offsets = torch.empty((1, P + 1), dtype=i32, device=dev)
        self.counts_h = torch.empty((1, P), dtype=i32, pin_memory=True)
        self.ws = ep.workspace(T, K, P, El, 1, dev)
        self.cws = ep.combine_ws(dev)
        self.err = ep.error_word(dev)
        self.token_pos = torch.empty((T, P), dtype=i32, device=dev)
        self.N = None

    def alloc_rows(self, N):
        torch, w, dev = self.torch, self.w, self.x.device
        self.N = N
        self.W = w.T * min(w.K, w.P)          # worst-case rows of the no-sync path
        W = self.W
        self.send_token_idx = torch.empty(W, dtype=torch.int32, device=dev)
        self.send_rank = torch.empty(W, dtype=torch.int32, device=dev)
        self.send_idx = torch.empty((W, w.K), dtype=torch.int64, device=dev)
        self.send_w = torch.empty((W, w.K), dtype=torch.float32, device=dev)
        self.recv_x = torch.empty((W, w.H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)

    def step_nosync(self, y, stream, ev=None, split=False, io=None):
        """The no-sync step.  Default: ep_dispatch_nosync (route, then the
        dispatch launched as its programmatic dependent) and ep_combine; ev: 3
        events (start, after route + dispatch, after combine) or None.
        split: ep_route_nosync and ep_dispatch as separate ordinary launches
        (per-kernel times); ev: 4 events (start, route, dispatch, combine).
        io: (x, topk_idx, topk_weights, out) to use instead of this path's own."""
        ep, w = self.ep, self.w
        T, K, P, El, H, W = w.T, w.K, w.P, w.E_local, w.H, self.W
        x, idx, wts, out = io if io is not None else (self.x, self.idx, self.wts, self.out)
        rec = (lambda i: ev[i].record(stream)) if ev is not None else (lambda i: None)
        rec(0)
        if split:
            ep.ep_route_nosync(idx, wts, T, K, P, El, W, self.dest, self.is_in_rank, self.send_counts,
                               self.rank_offsets, None, self.send_token_idx, self.send_rank, self.send_idx,
                               self.send_w, self.token_pos, self.ws, self.err, stream)
            rec(1)
            ep.ep_dispatch(x, T, H, self.token_pos, P, W, self.recv_x, None, 0, self.err, stream)
            rec(2)
        else:
            ep.ep_dispatch_nosync(x, idx, wts, T, K, H, P, El, W, 0, self.dest, self.is_in_rank,
                                  self.send_counts, self.rank_offsets, None, self.send_token_idx, self.send_rank,
                                  self.send_idx, self.send_w, self.token_pos, self.recv_x, None, self.ws, self.err,
                                  stream)
            rec(1)
        ep.ep_combine(y, T, H, self.token_pos, P, W, out, 0, self.cws, self.err, stream)
        rec(3 if split else 2)

    def step_sync(self, y, stream, ev=None):
        """ev: 6 events (start, counts, host sync, layout, dispatch, combine) or None."""
        ep, w = self.ep, self.w
        T, K, P, El, H = w.T, w.K, w.P, w.E_local, w.H
        rec = (lambda i: ev[i].record(stream)) if ev is not None else (lambda i: None)
        rec(0)
        ep.ep_compute_send_counts(self.idx, T, K, P, El, None, 1, self.dest, self.is_in_rank, self.send_counts,
                                  self.rank_offsets, None, self.ws, self.err, stream)
        rec(1)
        self.counts_h.copy_(self.send_counts, non_blocking=True)
        stream.synchronize()
        num_send = int(self.counts_h.sum())
        if num_send != self.N:
            raise RuntimeError(f"routed rows changed: {num_send} != {self.N}")
        rec(2)
        ep.ep_build_send_layout(self.idx, self.wts, self.dest, self.is_in_rank, T, K, P, El, num_send,
                                self.send_token_idx, self.send_rank, self.send_idx, self.send_w,
                                self.token_pos, self.ws, self.err, stream)
        rec(3)
        ep.ep_dispatch(self.x, T, H, self.token_pos, P, num_send, self.recv_x, None, 0, self.err, stream)
        rec(4)
        ep.ep_combine(y, T, H, self.token_pos, P, num_send, self.out, 0, self.cws, self.err, stream)
        rec(5)


LAUNCHES_PER_STEP = 3   # route (one cooperative kernel), dispatch, combine


def _timed_steps(torch, steps, flush, step, n_events):
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(steps)]
    for k in range(steps):
        flush()                # outside the events; the step is enqueued while it runs
        step(evs[k])
    torch.cuda.synchronize()
    return evs


def _kernel_table(ab, parts):
    kern = {}
    for name, times in parts.items():
        us = statistics.mean(times) * 1e3
        kern[name] = {"us": round(us, 2)}
        if name in ab:
            kern[name]["algorithmic_bytes"] = ab[name]
            kern[name]["gbs"] = round(ab[name] / (us * 1e-6) / 1e9, 1)
    return kern


def _graph_replay(torch, sp, y, stream, flush, dev, steps, T, step_bytes):
    """Capture the no-sync step once and time its replays."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        sp.step_nosync(y, side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=side):
        sp.step_nosync(y, side)
    torch.cuda.synchronize()
    gt = []
    for _ in range(steps):
        flush()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        g.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        gt.append(a0.elapsed_time(a1))
    return {"value": round(T * len(gt) / (sum(gt) / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(statistics.mean(gt), 4),
            "hbm_gbs": round(step_bytes / (statistics.mean(gt) * 1e-3) / 1e9, 1)}


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import combine_send_counts_gb300 as ep
    from combine_send_counts_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    ep.load()

    w = wl.WORKLOADS[args.workload]
    if args.tokens:
        w = w.scaled(T=args.tokens)
    x_h, idx_h, w_h = wl.make(w)
    x, idx, wts = x_h.to(dev), idx_h.to(dev), w_h.to(dev)
    sp = SendPath(ep, torch, w, x, idx, wts, dev)
    stream = torch.cuda.current_stream(dev)

    # size the rows from one count pass, then draw the expert outputs
    ep.ep_compute_send_counts(idx, w.T, w.K, w.P, w.E_local, None, 1, sp.dest, sp.is_in_rank, sp.send_counts,
                              sp.rank_offsets, None, sp.ws, sp.err, stream)
    N = int(sp.send_counts.sum().item())
    sp.alloc_rows(N)
    y_h = wl.expert_outputs(w, N)
    y = torch.empty((sp.W, w.H), dtype=torch.bfloat16, device=dev)   # expert outputs in worst-case rows
    y[:N].copy_(y_h)
    flush = L2Flush(torch, dev)

    for _ in range(max(args.warmup, 0)):
        flush()
        sp.step_nosync(y, stream)
        flush()
        sp.step_sync(y, stream)
    torch.cuda.synchronize()
    if int(sp.err.item()) != 0:
        raise ep.EPError(int(sp.err.item()), "warmup")

    # ---- timed region: the no-sync path
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        evs = _timed_steps(torch, args.steps, flush, lambda e: sp.step_nosync(y, stream, e), 3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if int(sp.err.item()) != 0:
        raise ep.EPError(int(sp.err.item()), "timed steps")
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    combine_ms = [e[1].elapsed_time(e[2]) for e in evs]
    # per-kernel times: the same step with route and dispatch as separate
    # ordinary launches (the timed step overlaps them), outside the timed region
    evs_b = _timed_steps(torch, args.steps, flush, lambda e: sp.step_nosync(y, stream, e, split=True), 4)
    parts = {"route": [e[0].elapsed_time(e[1]) for e in evs_b],
             "dispatch": [e[1].elapsed_time(e[2]) for e in evs_b],
             "combine": combine_ms}
    total_s = sum(step_ms) / 1e3
    tok_s, max_s = aggregate(total_s, float(w.T * args.steps), world, dist if world > 1 else None)

    peak, peak_src = measured_peak()
    ab = algorithmic_bytes(w.T, w.H, N, w.K, w.P)
    ab["route"] = ab.pop("counts") + ab.pop("layout")
    kern = _kernel_table(ab, parts)
    # the roofline kernel: combine, the largest kernel of the step, timed inside the timed steps
    dom = "combine"
    step_bytes = sum(ab.values())
    achieved_step = step_bytes / (statistics.mean(step_ms) * 1e-3) / 1e9

    # ---- the same step through the host-synchronising calls (pages' call order)
    evs_s = _timed_steps(torch, args.steps, flush, lambda e: sp.step_sync(y, stream, e), 6)
    ms_s = [e[0].elapsed_time(e[5]) for e in evs_s]
    ab_s = algorithmic_bytes(w.T, w.H, N, w.K, w.P)
    sync_path = {
        "value": round(w.T * len(ms_s) / (sum(ms_s) / 1e3), 1), "unit": "tokens/s",
        "ms_per_step": round(statistics.mean(ms_s), 4),
        "path": "ep_compute_send_counts -> D2H counts + host wait -> ep_build_send_layout(num_send) -> "
                "ep_dispatch -> ep_combine",
        "kernels": _kernel_table(ab_s, {
            "counts": [e[0].elapsed_time(e[1]) for e in evs_s],
            "counts_d2h_host_wait": [e[1].elapsed_time(e[2]) for e in evs_s],
            "layout": [e[2].elapsed_time(e[3]) for e in evs_s],
            "dispatch": [e[3].elapsed_time(e[4]) for e in evs_s],
            "combine": [e[4].elapsed_time(e[5]) for e in evs_s]}),
    }

    # ---- the no-sync step replayed from a CUDA graph
    graph_path = None
    if not args.no_graph:
        try:
            graph_path = _graph_replay(torch, sp, y, stream, flush, dev, args.steps, w.T, step_bytes)
        except Exception as exc:   # capture unsupported here: report why, keep the eager numbers
            torch.cuda.synchronize()
            graph_path = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
        if int(sp.err.item()) != 0:
            raise ep.EPError(int(sp.err.item()), "graph replay")

    result = {
        "metric": METRIC,
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(w),
                   "N_rows": N, "worst_case_rows": sp.W,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps, outside the timed events: a 512 MiB write, then a 256 MiB "
                         "read so that L2 holds no dirty lines; working set 1.8 GB > L2",
                   "path": "ep_dispatch_nosync (ep_route_nosync: counts + layout, worst-case rows, no host "
                           "round trip; then the dispatch, launched as the route's programmatic dependent) -> "
                           "ep_combine",
                   "seed": w.seed},
        "hbm_gbs": round(achieved_step, 1),
        "hbm_frac_of_peak": round(achieved_step / peak, 4),
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["gbs"], "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(kern[dom]["gbs"] / peak, 4),
                     "traffic": committed_traffic(dom),
                     "algorithmic_bytes_per_launch": ab[dom]},
        "kernels": kern,
        "kernels_note": "combine from the timed steps; route and dispatch from the same number of steps run "
                        "with the two as separate ordinary launches (the timed step overlaps them)",
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks.summary(),
        "host_sync_path": sync_path,
        "graph_replay": graph_path,
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, ep, torch, w, sp, x_h, idx_h, w_h, y_h, y, stream, world, dist)
    if not args.no_other_paths and not args.tokens:
        del sp, y
        torch.cuda.empty_cache()
        result["other_paths"] = run_other_paths(ep, torch, wl, dev, flush, peak, iters=10)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, x_h, idx_h, w_h, y_h, args.cpu_steps, full=True)
        result["cpu_baseline_threads"] = cpu_baseline_threads(w, x_h, idx_h, w_h, y_h, args.cpu_steps)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def _event_time_us(torch, flush, fn, iters, warmup=2):
    ts = []
    for i in range(warmup + iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        if i >= warmup:
            ts.append(a.elapsed_time(b) * 1e3)
    return statistics.mean(ts)


def _graph_time_us(torch, flush, fn, iters, dev, warmup=2):
    """Capture fn once (after one eager call) and time its replays."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize()
    return _event_time_us(torch, flush, g.replay, iters, warmup)


def run_other_paths(ep, torch, wl, dev, flush, peak, iters):
    """The other rows of the path, each on its own workload: expert-batched
    prepare and combine (batched workload), fp8 dispatch of one chunk and the
    native chunked fp8 forward (chunked fp8 workload).  Routing follows each
    workload's recipe; row values are drawn on the device (they do not change
    the work)."""
    out = {}
    g = torch.Generator(device=dev).manual_seed(0)
    err = ep.error_word(dev)
    cws = ep.combine_ws(dev)

    w = wl.WORKLOADS["batched"]
    idx, wts = (t.to(dev) for t in wl.routing(w))
    x = torch.randn((w.T, w.H), device=dev, generator=g).to(torch.bfloat16)
    r = ep.batched_prepare(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, err=err)
    hits = int(r["tokens_per_expert"].sum().item())
    # tokens with at least one local slot: the only rows a prepare must read
    t_hit = int((r["slot"] >= 0).any(dim=1).sum().item())
    ws = ep.workspace(w.T, w.K, w.P, w.E_local, 1, dev)
    ab = (t_hit + hits) * w.H * 2
    us = _event_time_us(torch, flush, lambda: ep.ep_batched_prepare(
        x, idx, w.T, w.K, w.H, w.E, w.E_local, w.rank, w.max_num_tokens, r["b_x"], r["tokens_per_expert"],
        r["slot"], 0, ws, err), iters)
    out["batched_prepare"] = {"workload": "batched", "us": round(us, 2), "algorithmic_bytes": ab,
                              "gbs": round(ab / us / 1e3, 1), "frac": round(ab / us / 1e3 / peak, 4),
                              "local_hits": hits, "tokens_with_a_local_slot": t_hit}
    y = torch.randn((w.E_local, w.max_num_tokens, w.H), device=dev, generator=g).to(torch.bfloat16)
    o = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    us = _event_time_us(torch, flush, lambda: ep.ep_batched_combine(
        y, idx, wts, r["slot"], w.T, w.K, w.H, w.E_local, w.rank, w.max_num_tokens, o, cws, err), iters)
    abc = (w.T + hits) * w.H * 2   # every token's output row is written
    out["batched_combine"] = {"workload": "batched", "us": round(us, 2), "algorithmic_bytes": abc,
                              "gbs": round(abc / us / 1e3, 1), "frac": round(abc / us / 1e3 / peak, 4)}
    # fp8 expert-batched prepare: codes + column-major scales (fp32, or
    # power-of-two UE8M0 packed four per int)
    ab8 = t_hit * w.H * 2 + hits * (w.H + w.H // 32)
    for name, fmt, rs in (("batched_prepare_fp8_col_f32", ep.EP_SCALE_COL_F32, 0),
                          ("batched_prepare_fp8_ue8m0", ep.EP_SCALE_COL_UE8M0, 1)):
        r8 = ep.batched_prepare_fp8(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, fmt, bool(rs), err=err)
        us = _event_time_us(torch, flush, lambda: ep.ep_batched_prepare_fp8(
            x, idx, w.T, w.K, w.H, w.E, w.E_local, w.rank, w.max_num_tokens, r8["b_q"], r8["b_scale"], fmt, rs,
            r8["tokens_per_expert"], r8["slot"], 0, ws, err), iters)
        out[name] = {"workload": "batched", "us": round(us, 2), "algorithmic_bytes": ab8,
                     "gbs": round(ab8 / us / 1e3, 1), "frac": round(ab8 / us / 1e3 / peak, 4)}
        del r8
    # capacity factor 1.0 and receive alignment 128 (bf16 rows): kept rows are
    # copied, the alignment rows zero-filled
    C = ep.expert_capacity(w.T, w.K, w.E, 1.0)
    rx = ep.batched_prepare_ex(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, capacity=C, alignment=128, err=err)
    kept = int((rx["tokens_per_expert"]).sum().item())   # kept rows plus alignment rows
    t_kept = int((rx["slot"] >= 0).any(dim=1).sum().item())
    abx = t_kept * w.H * 2 + kept * w.H * 2
    us = _event_time_us(torch, flush, lambda: ep.ep_batched_prepare_ex(
        x, idx, w.T, w.K, w.H, w.E, w.E_local, w.rank, w.max_num_tokens, C, 128, rx["b_rows"], None, -1, 0,
        rx["tokens_per_expert"], rx["slot"], rx["dropped"], 0, ws, err), iters)
    out["batched_prepare_capacity_align"] = {
        "workload": "batched, capacity factor 1.0 (%d per expert), alignment 128" % C, "us": round(us, 2),
        "algorithmic_bytes": abx, "gbs": round(abx / us / 1e3, 1), "frac": round(abx / us / 1e3 / peak, 4),
        "dropped": int(rx["dropped"].sum().item())}
    del rx
    # the same with fp8 rows and column-major fp32 scales (kept rows quantised,
    # alignment rows and their scales zero-filled)
    rx = ep.batched_prepare_ex(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, capacity=C, alignment=128,
                               scale_fmt=ep.EP_SCALE_COL_F32, err=err)
    abx8 = t_kept * w.H * 2 + kept * (w.H + w.H // 32)
    us = _event_time_us(torch, flush, lambda: ep.ep_batched_prepare_ex(
        x, idx, w.T, w.K, w.H, w.E, w.E_local, w.rank, w.max_num_tokens, C, 128, rx["b_rows"], rx["b_scale"],
        ep.EP_SCALE_COL_F32, 0, rx["tokens_per_expert"], rx["slot"], rx["dropped"], 0, ws, err), iters)
    out["batched_prepare_fp8_capacity_align"] = {
        "workload": "batched, fp8 with column-major fp32 scales, capacity factor 1.0, alignment 128",
        "us": round(us, 2), "algorithmic_bytes": abx8, "gbs": round(abx8 / us / 1e3, 1),
        "frac": round(abx8 / us / 1e3 / peak, 4)}
    del rx
    del x, y, o, r

    # metadata views of the large workload's routing: multihot map + dense
    # probabilities, and the send layout with rank segments aligned to 128
    w = wl.WORKLOADS["large"]
    idx, wts = (t.to(dev) for t in wl.routing(w))
    rm = torch.empty((w.T, w.E), dtype=torch.bool, device=dev)
    pr = torch.empty((w.T, w.E), dtype=torch.float32, device=dev)
    abm = w.T * w.K * 12 + w.T * w.E * 5
    us = _event_time_us(torch, flush, lambda: ep.ep_indices_to_multihot(idx, wts, w.T, w.K, w.E, rm, pr, err), iters)
    out["indices_to_multihot"] = {"workload": "large (T=16384, K=8, E=256)", "us": round(us, 2),
                                  "algorithmic_bytes": abm, "gbs": round(abm / us / 1e3, 1),
                                  "frac": round(abm / us / 1e3 / peak, 4)}
    for A in (1, 128):
        ra = ep.route_nosync(idx, wts, w.P, w.E_local, alignment=A, err=err)
        wsr = ep.workspace(w.T, w.K, w.P, w.E_local, 1, dev)
        us = _event_time_us(torch, flush, lambda: ep.ep_route_nosync_aligned(
            idx, wts, w.T, w.K, w.P, w.E_local, ra["num_worst_rows"], A, ra["dest"], ra["is_in_rank"],
            ra["send_counts"], ra["rank_offsets"], None, ra["send_token_idx"], ra["send_rank"], ra["send_idx"],
            ra["send_w"], ra["token_pos"], wsr, err), iters)
        out["route_nosync" + ("_aligned128" if A > 1 else "")] = {"workload": "large", "us": round(us, 2)}
    del rm, pr, ra

    w = wl.WORKLOADS["chunk_fp8"]
    idx, wts = (t.to(dev) for t in wl.routing(w))
    x = torch.randn((w.T, w.H), device=dev, generator=g).to(torch.bfloat16)
    Tc = w.T // w.chunks
    rr = ep.route_nosync(idx[:Tc], wts[:Tc], w.P, w.E_local, err=err)
    N = int(rr["rank_offsets"][w.P].item())
    q = torch.empty((N, w.H), dtype=torch.uint8, device=dev)
    sc = torch.empty((N, w.H // 128), dtype=torch.float32, device=dev)
    ab = Tc * w.H * 2 + N * (w.H + w.H // 32)
    us = _event_time_us(torch, flush, lambda: ep.ep_dispatch(x[:Tc], Tc, w.H, rr["token_pos"], w.P, N, q, sc, 1,
                                                             err), iters)
    out["fp8_dispatch"] = {"workload": f"chunk_fp8, one chunk of {Tc} tokens", "us": round(us, 2),
                           "algorithmic_bytes": ab, "gbs": round(ab / us / 1e3, 1),
                           "frac": round(ab / us / 1e3 / peak, 4), "rows": N}
    # the synthetic fp8 expert on that chunk's rows: codes + scales + the rows'
    # expert ids and weights read, bf16 rows written
    out_l = torch.empty((N, w.H), dtype=torch.bfloat16, device=dev)
    sidx, sw = rr["send_idx"][:N], rr["send_w"][:N]
    abl = N * (w.H + w.H // 32 + w.K * 12 + 2 * w.H)
    us = _event_time_us(torch, flush, lambda: ep.ep_local_expert_fp8(q, sc, sidx, sw, N, w.K, w.H, out_l, err),
                        iters)
    out["local_expert_fp8"] = {"workload": f"chunk_fp8, one chunk of {Tc} tokens (the dispatched rows)",
                               "us": round(us, 2), "algorithmic_bytes": abl, "gbs": round(abl / us / 1e3, 1),
                               "frac": round(abl / us / 1e3 / peak, 4), "rows": N}
    del out_l
    us = _event_time_us(torch, flush, lambda: ep.dispatch_chunked_forward(
        x, idx, wts, num_local_experts=w.E_local, num_ranks=w.P, chunks=w.chunks, fp8=True, err=err),
        max(2, iters // 4), warmup=1)
    out["chunked_fp8_forward"] = {"workload": "chunk_fp8 (T=32768, 4 chunks, synthetic fp8 expert included)",
                                  "path": "one count pass, one D2H + host wait, then per chunk layout -> fp8 "
                                          "dispatch -> expert -> combine",
                                  "us": round(us, 1), "tokens_per_s": round(w.T / us * 1e6, 1)}
    # the same forward without a host round trip: one row set in order, two
    # row sets pipelined over two streams, and the pipelined form replayed
    # from a CUDA graph
    o = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    for n_sets in (1, 2):
        f = ep.ChunkedForward(w.T, w.K, w.H, num_ranks=w.P, num_local_experts=w.E_local, chunks=w.chunks, fp8=True,
                              n_sets=n_sets, device=dev)
        us = _event_time_us(torch, flush, lambda: f(x, idx, wts, out=o, err=err), max(2, iters // 4))
        key = "chunked_fp8_forward_nosync" + ("_pipelined" if n_sets == 2 else "")
        out[key] = {"workload": "chunk_fp8 (T=32768, 4 chunks, synthetic fp8 expert included)",
                    "path": f"ep_dispatch_chunked_forward_nosync, {n_sets} row set(s)",
                    "us": round(us, 1), "tokens_per_s": round(w.T / us * 1e6, 1)}
    us = _graph_time_us(torch, flush, lambda: f(x, idx, wts, out=o, err=err), max(2, iters // 4), dev)
    out["chunked_fp8_forward_nosync_graph"] = {
        "workload": "chunk_fp8 (T=32768, 4 chunks, synthetic fp8 expert included)",
        "path": "ep_dispatch_chunked_forward_nosync, 2 row sets, replayed from a CUDA graph",
        "us": round(us, 1), "tokens_per_s": round(w.T / us * 1e6, 1)}
    del f
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise ep.EPError(int(err.item()), "other paths")
    return out


def run_e2e(args, ep, torch, w, sp, x_h, idx_h, w_h, y_h, y_dev, stream, world, dist):
    """The same no-sync step through the C ABI from pinned HOST buffers: every
    step copies its inputs and expert outputs host -> device, runs the path and
    copies the combined result device -> host, all inside the timed region.
    Steps are pipelined over two device buffer sets and three streams (copies
    in, compute, copies out), so step k+1's uploads overlap step k's compute
    and download; the timed region runs from the first upload to the last
    download, and the value is the tokens of all steps over that time."""
    dev = y_dev.device
    xp, ip, wp, yp = (t.pin_memory() for t in (x_h, idx_h, w_h, y_h))
    outp = torch.empty((w.T, w.H), dtype=torch.bfloat16, pin_memory=True)
    N = y_h.shape[0]
    h2d = sum(t.numel() * t.element_size() for t in (xp, ip, wp, yp))
    d2h = outp.numel() * outp.element_size()
    sets = [(sp.x, sp.idx, sp.wts, y_dev, sp.out)]
    sets.append((torch.empty_like(sp.x), torch.empty_like(sp.idx), torch.empty_like(sp.wts),
                 torch.empty_like(y_dev), torch.empty_like(sp.out)))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_c = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]

    def run(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        a.record(s_in)
        for k in range(steps):
            j = k % 2
            x_d, i_d, w_d, y_d, o_d = sets[j]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_c[j])      # step k-2's compute is done with set j
                x_d.copy_(xp, non_blocking=True)
                i_d.copy_(ip, non_blocking=True)
                w_d.copy_(wp, non_blocking=True)
                y_d[:N].copy_(yp, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if k >= 2:
                stream.wait_event(ev_out[j])      # step k-2's download has read out_j
            sp.step_nosync(y_d, stream, io=(x_d, i_d, w_d, o_d))
            ev_c[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[j])
                outp.copy_(o_d, non_blocking=True)
                ev_out[j].record(s_out)
        s_out.wait_stream(stream)
        b.record(s_out)
        b.synchronize()
        return a.elapsed_time(b) / 1e3

    ref = sp.out.cpu()   # every step has the same inputs: each download must equal the device result
    run(args.e2e_warmup)
    total = run(args.e2e_steps)
    if not torch.equal(outp.view(torch.int16), ref.view(torch.int16)):
        raise RuntimeError("end-to-end result differs from the device-timed steps' result")
    tok_s, _ = aggregate(total, float(w.T * args.e2e_steps), world, dist if world > 1 else None)
    return {"value": round(tok_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "pipelined": "uploads of step k+1 overlap step k's compute and download"}


# ------------------------------------------------------------------ CPU arm --
def oracle_step(oracle, w, x, idx, wts, y):
    o = oracle.send_path(x, idx, wts, None, w.P, w.E_local)
    return oracle.combine(y[:o["layout"]["n"]], o["layout"]["token_pos"])


def cpu_baseline(w, x, idx, wts, y, steps, full=True, T_sample=None):
    import oracle
    if T_sample is not None and T_sample < w.T:
        x, idx, wts = x[:T_sample], idx[:T_sample], wts[:T_sample]
    T = x.shape[0]
    oracle_step(oracle, w, x[:64], idx[:64], wts[:64], y)   # load / build
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(oracle, w, x, idx, wts, y)
    dt = time.perf_counter() - t0
    return {"value": round(T * steps / dt, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} step(s) of the send path (counts, layout, dispatch, combine) on the first "
                      f"{T} of {w.T} tokens of the {w.name} workload, single-threaded C oracle"}


def oracle_step_threads(oracle, w, x, idx, wts, y, pool, parts):
    """The same send path with the oracle's own functions, its independent
    parts split over threads (ctypes releases the GIL): counts and layout
    once, then the row gather on contiguous row ranges and the combine on
    contiguous token ranges (each row and each token depends on nothing
    else), so the result is the single-threaded one, bit for bit."""
    import numpy as np
    c = oracle.compute_send_counts(idx, w.P, w.E_local)
    lay = oracle.build_send_layout(idx, wts, c["dest"], c["is_in_rank"], w.E_local)
    sti, tp = lay["send_token_idx"], lay["token_pos"]
    N, T = sti.size, tp.shape[0]
    rb = [N * i // parts for i in range(parts + 1)]
    tb = [T * i // parts for i in range(parts + 1)]
    recv = list(pool.map(lambda i: oracle.dispatch(x, sti[rb[i]:rb[i + 1]]), range(parts)))
    out = list(pool.map(lambda i: oracle.combine(y[:N], tp[tb[i]:tb[i + 1]]), range(parts)))
    return recv, np.concatenate(out)


def cpu_baseline_threads(w, x, idx, wts, y, steps):
    """The oracle's send path over the host's cores (see oracle_step_threads);
    checked bit for bit against the single-threaded oracle first."""
    import concurrent.futures as cf
    import numpy as np
    import oracle
    cores = max(1, min(os.cpu_count() or 1, 64))
    with cf.ThreadPoolExecutor(cores) as pool:
        _, out = oracle_step_threads(oracle, w, x, idx, wts, y, pool, cores)
        if not np.array_equal(out, oracle_step(oracle, w, x, idx, wts, y)):
            return {"unavailable": "the threaded oracle differs from the single-threaded one"}
        t0 = time.perf_counter()
        for _ in range(steps):
            oracle_step_threads(oracle, w, x, idx, wts, y, pool, cores)
        dt = time.perf_counter() - t0
    return {"value": round(w.T * steps / dt, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{steps} step(s) of the send path on all {w.T} tokens of the {w.name} workload: the "
                      f"single-threaded C oracle's counts and layout, then its row gather and combine on "
                      f"{cores} row and token ranges in {cores} threads (same bits as one thread)"}


def run_reference(args):
    """The oracle as the reference arm: each step is the send path on the same
    workload as the GPU arm (all of its tokens, about half a second per step on
    one host core), or on its first --reference-tokens tokens if that is set."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from combine_send_counts_gb300 import workloads as wl
    import oracle
    w = wl.WORKLOADS[args.workload]
    x, idx, wts = wl.make(w)
    Ts = w.T if args.reference_tokens <= 0 else min(args.reference_tokens, w.T)
    x, idx, wts = x[:Ts], idx[:Ts], wts[:Ts]
    c = oracle.compute_send_counts(idx, w.P, w.E_local, with_tokens_per_expert=False)
    y = wl.expert_outputs(w, int(c["send_counts"].sum()))
    for _ in range(max(args.warmup, 0)):
        oracle_step(oracle, w, x, idx, wts, y)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(oracle, w, x, idx, wts, y)
        times.append(time.perf_counter() - t0)
    tok_s = Ts * len(times) / sum(times)
    which = f"all {w.T} tokens" if Ts == w.T else f"first {Ts} of {w.T} tokens"
    sample = (f"{which} of the {w.name} workload per step; send path (counts, layout, dispatch, combine) in the "
              f"single-threaded C oracle")
    config = {"workload": workload_name(w)}
    if Ts < w.T:
        config["T_sample"] = Ts
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": round(tok_s, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(tok_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload's recipe with this many tokens instead (reduced cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-other-paths", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--e2e-warmup", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=20, help="oracle steps of the CPU baseline (about 0.5 s each on one core)")
    ap.add_argument("--reference-tokens", type=int, default=0,
                    help="reference arm: time the oracle on the first N tokens only (0 = the whole workload)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
