#!/usr/bin/env python3
"""Benchmark: exhaustive SIFT matching of one 8,192 x 8,192 descriptor pair per step.

One step = one pass of the whole path (staging, fused tensor-core GEMM + row/column
top-2 merged into per-row and per-column keys, ratio / distance / mutual test with
compaction) over the seeded 8,192 x 8,192 pair (25% planted matches at sigma 0.08).
Inputs are resident in HBM when the timed region starts; L2 is flushed (256 MiB
write) before every timed step, outside the step's events; steps are enqueued back
to back (the host does not wait for one step before enqueuing the next).  The step
is captured once in a CUDA graph and replayed; every replay launches the library's
own kernels.

Also reported on the same JSON line:
  roofline      the fused kernel's int8-equivalent TFLOP/s (2 * n_a * n_b * 128 per
                launch) against the measured bf16 tensor peak, from CUDA events
                recorded around that launch in a second pass of the same steps;
  e2e           the same metric through the public API with host buffers: the
                descriptors stay in pinned host memory and the staging kernel reads
                them over the host link, the match kernel writes the count and the
                match list into pinned host memory, all inside the timed region;
  cpu_baseline  the CPU oracle on this host's cores (full pairs, bounded in time);
  clocks        nvidia-smi samples taken while the timed loop ran.

--workload selects the batch workloads instead (ring, ragged, 100-image survey), one
match_batch over the whole workload per step, with the same keys.

--impl reference times the CPU oracle itself on the same workload and metric (the
pages publish no runnable reference for this path; the oracle is the baseline arm).

Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no data-path collective); time is the max over ranks.  --shard (batch
workloads) splits the workload's pairs over the ranks by cost instead (strong
scaling); rank 0 then gathers every pair's match list after the timed steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "image pairs/sec at 8192×8192 SIFT (int8 TOPS vs tensor peak), bit-exact"
UNIT = "pairs/s"
N_A = N_B = 8192
OPS_PER_PAIR = 2 * N_A * N_B * 128
WORKLOAD = "single pair 8192x8192 SIFT-shaped u8 descriptors, 25% planted at sigma 0.08, seed 0"
WORKLOAD_2000 = "single pair 2000x2000 SIFT-shaped u8 descriptors, 30% planted at sigma 0.05, seed 0"
# DRAM bytes (read + write) of one fused_top2_kernel launch on the 8192 x 8192 pair, as
# measured by the latest ncu capture of the kernel as it stands (dram__bytes_read.sum +
# dram__bytes_write.sum); None whenever the kernel has changed since that capture
FUSED_TRAFFIC_8192 = 4482560
# the arithmetic of the path: u8 inputs, exact integer scores formed on the tensor
# cores from bf16 operands with f32 accumulation (every partial sum < 2^24)
DTYPE = "u8 exact (bf16 operands, f32 accumulate)"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("hbm_gbs", 6800.0)), "measured"
    return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples every 100 ms while running.  Samples are time-stamped; those
    inside the marked timed window are reported as such.  A timed window shorter than
    the sampling period is followed by an untimed continuation of the same steps (see
    hold_load) so that the clocks under that load are still seen."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    MIN_WINDOW_S = 0.5

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.window = None
        self.path = os.path.join("/tmp", f"serac_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # wait for the first sample so that sampling runs before the timed window opens
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def hold_load(self, fn, t_begin: float):
        """Run fn (one untimed step, enqueued) until MIN_WINDOW_S has passed since t_begin."""
        import torch
        while time.time() - t_begin < self.MIN_WINDOW_S:
            for _ in range(8):
                fn()
            torch.cuda.synchronize()

    @staticmethod
    def _stamp(x: str):
        import datetime
        try:
            return datetime.datetime.strptime(x.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append((self._stamp(parts[0]), float(parts[2]), float(parts[3]),
                                 {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
                except ValueError:
                    continue
        os.unlink(self.path)
        w0, w1 = self.window if self.window else (None, None)
        inside = [r for r in rows if w0 is not None and r[0] is not None and w0 <= r[0] <= w1]
        # the timed window and its untimed continuation under the same load
        loaded = [r for r in rows if w0 is not None and r[0] is not None and r[0] >= w0] or rows
        use = inside or loaded
        reasons = set().union(*[r[3] for r in use]) if use else set()
        out = {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
               "sm_max_mhz": max(r[2] for r in use) if use else None,
               "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_window": len(inside)}
        if w0 is not None:
            out["timed_window_ms"] = round((w1 - w0) * 1e3, 1)
        if not inside:
            out["note"] = "timed window shorter than the 100 ms sampling period: samples from its untimed continuation"
        return out


def _on_stream(stream, flush, fn):
    """One untimed step (L2 flush, then fn) on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        flush.fill_(0)
        fn()


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (x itself on a single process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_baseline(a, b, budget_s: float = 12.0):
    """The oracle as it stands on this host: full pairs, repeated for about budget_s."""
    import oracle
    oracle.build_library()
    t0 = time.perf_counter()
    ref = oracle.match(a, b)
    n = 1
    while time.perf_counter() - t0 < budget_s:
        oracle.match(a, b)
        n += 1
    dt = time.perf_counter() - t0
    return ref, {"value": n / dt, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                 "sample": f"{n} full {a.shape[0]}x{b.shape[0]} pairs (rows and columns, all threads), {dt:.1f} s"}


def run_reference(args):
    """The oracle arm: each step matches a bounded sample of the pair's rows (their
    top-2, their best column's full top-2, the decision); the rate is scaled by the
    sampled fraction of the pair's work."""
    import numpy as np

    import oracle
    import sift_synth
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    oracle.build_library()
    p = sift_synth.single_pair_8192(0)
    params = oracle.Params()
    t0 = time.perf_counter()
    oracle.accept_rows(p.a, p.b, np.arange(256, dtype=np.int32), params)
    per_row = (time.perf_counter() - t0) / 256
    budget = 150.0 / max(args.steps + args.warmup, 1)
    m = int(max(64, min(N_A, budget / max(per_row, 1e-9))))
    rng = np.random.default_rng(0)
    times = []
    for s in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(N_A, m, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.accept_rows(p.a, p.b, rows, params)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    frac = m / N_A
    total = sum(times)
    value = args.steps * frac / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "n_a": N_A, "n_b": N_B,
                                             "sample_rows_per_step": m},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{m} of {N_A} rows per step (row top-2, best column's top-2, "
                                       f"decision); rate scaled by {frac:.4f} of a pair"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import sift_synth
    import top_ratio_test_gb300 as serac

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    st = serac.device_check()
    if st != serac.OK:
        raise SystemExit(f"device check failed: {serac.status_str(st)}")

    if args.n:
        pair = sift_synth.make_pair(0, 1, args.n, args.n, args.n, 0.25, 0.08)
    elif args.workload == "pair8192":
        pair = sift_synth.single_pair_8192(0)
    else:
        pair = sift_synth.single_pair_2000(0)
    n_a, n_b = pair.a.shape[0], pair.b.shape[0]
    ops_per_pair = 2 * n_a * n_b * 128
    a_host = torch.from_numpy(pair.a).pin_memory()
    b_host = torch.from_numpy(pair.b).pin_memory()
    a = a_host.to(dev)
    b = b_host.to(dev)
    params = serac.default_params()
    stream = torch.cuda.Stream(device=dev)
    ws = serac.workspace(serac.pair_workspace_size(n_a, n_b), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev_fb = torch.cuda.Event(enable_timing=True)
    ev_fe = torch.cuda.Event(enable_timing=True)
    ev_fb.record(stream)  # torch creates the CUDA events on first record
    ev_fe.record(stream)

    # one step, captured once
    with torch.cuda.stream(stream):
        out = serac.match_pair(a, b, params, workspace_t=ws, stream=stream)  # warm the library
        stream.synchronize()
        launches = serac.last_launch_count()
        # the timed step: no event nodes between the kernels (they would break the
        # programmatic dependent launches that overlap one kernel's start with the last)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            out = serac.match_pair(a, b, params, workspace_t=ws, stream=stream)
        # the same step with events around the fused kernel, for its duration
        serac.set_profile_events(ev_fb, ev_fe)
        g_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prof, stream=stream):
            serac.match_pair(a, b, params, workspace_t=ws, stream=stream)
        serac.set_profile_events(None, None)
    stream.synchronize()

    def timed(fn, steps, warmup, fused_events=False):
        """Per-step device time between events recorded right before and after the
        step, with an L2 flush before every step (outside the events).  Steps are
        enqueued without waiting for the previous one (the host runs ahead), except
        when the fused-kernel events, reused by every step, must be read each time."""
        t_step, t_fused, evs = [], [], []
        for s in range(warmup + steps):
            with torch.cuda.stream(stream):
                flush.fill_(s & 0xFF)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            if s >= warmup:
                evs.append((e0, e1))
            if fused_events:
                stream.synchronize()
                if s >= warmup:
                    t_fused.append(ev_fb.elapsed_time(ev_fe))
        stream.synchronize()
        t_step = [e0.elapsed_time(e1) for e0, e1 in evs]
        return t_step, t_fused

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_w0 = time.time()
    t_step, _ = timed(g.replay, args.steps, args.warmup)
    torch.cuda.synchronize()
    clocks.mark(t_w0, time.time())
    clocks.hold_load(lambda: _on_stream(stream, flush, g.replay), t_w0)
    clk = clocks.stop()
    t_step_prof, t_fused = timed(g_prof.replay, args.steps, args.warmup, fused_events=True)

    # parity of the timed output (the last replay) against the oracle, on rank 0
    n = int(out.count.item())
    got = out.matches[:n].cpu().numpy()
    total_ms = max_over_ranks(sum(t_step), dev)

    # e2e through the public API with host buffers: the descriptors stay in pinned host
    # memory and the staging kernel reads them over the host link; the match kernel
    # writes the count and the match list straight into pinned host memory
    e2e_steps = max(3, min(args.steps, 200))
    e2e_out = serac.match_pair(a_host, b_host, params, workspace_t=ws, stream=stream, host_out=True)
    stream.synchronize()

    def e2e_step():
        serac.match_pair(a_host, b_host, params, workspace_t=ws, stream=stream, out=e2e_out)

    e2e_t, _ = timed(e2e_step, e2e_steps, 3)
    e2e_ms = max_over_ranks(sum(e2e_t), dev)

    peak_tflops, _, peak_kind = _peaks()
    fused_ms = statistics.mean(t_fused)
    achieved = ops_per_pair / (fused_ms * 1e-3) / 1e12
    value = world * args.steps / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": (f"single pair {n_a}x{n_b} SIFT-shaped u8 descriptors, 25% planted at sigma 0.08, "
                                f"seed 0" if args.n else WORKLOAD if args.workload == "pair8192" else WORKLOAD_2000),
                   "n_a": n_a, "n_b": n_b,
                   "l2": "flushed before every step (256 MiB write)",
                   "graph": "one CUDA graph per step, replayed; kernels chained by programmatic dependent launch",
                   "parallelism": f"replicas x{world}"},
        "int8_equiv_tops": value * ops_per_pair / 1e12,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops,
                     "traffic": FUSED_TRAFFIC_8192 if args.workload == "pair8192" and not args.n else None,
                     "kernel": "fused_top2_kernel", "peak_kind": f"bf16 dense burst, {peak_kind}",
                     "fused_ms": fused_ms, "timing": "fused-kernel events in a second timed pass of the "
                     "same steps (event nodes in the step graph would serialise its launches)",
                     "ms_per_step_with_events": statistics.mean(t_step_prof)},
        "e2e": {"value": world * e2e_steps / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": (n_a + n_b) * 128, "d2h_bytes_per_step": 4 + 8 * int(e2e_out.count.item()),
                "path": "match_pair on pinned host descriptors, outputs in pinned host memory "
                        "(kernels read and write the host directly)"},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref, cb = cpu_baseline(pair.a, pair.b)
        line["cpu_baseline"] = cb
        line["bit_exact"] = bool(np.array_equal(got, ref.matches))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _batch_workload(name):
    """(description, list of (a, b) numpy pairs sharing image arrays where the workload does)."""
    import sift_synth
    if name == "ring12":
        r = sift_synth.ring_12x8192(0)
        return ("12 images x 8192 descriptors on a ring (20% shared with 3 neighbours, sigma 0.06), all 66 pairs",
                r.images, [(int(i), int(j)) for i, j in r.pairs])
    if name == "survey100":
        r = sift_synth.survey_100x8192(0)
        return ("100 images x 8192 descriptors (10% shared with the 6 nearest indices, sigma 0.05), all 4950 pairs",
                r.images, [(int(i), int(j)) for i, j in r.pairs])
    sizes = sift_synth.ragged_sizes(0)
    imgs, pairs = [], []
    for k in range(sizes.shape[0]):
        pr = sift_synth.ragged_pair(0, k, sizes)
        imgs += [pr.a, pr.b]
        pairs.append((2 * k, 2 * k + 1))
    return ("256 ragged pairs, 1000..16384 descriptors per image, 15% planted at sigma 0.05", imgs, pairs)


def run_batch(args):
    """One step = match_batch over the whole workload (images staged once per step)."""
    import numpy as np
    import torch

    import top_ratio_test_gb300 as serac

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    desc, imgs_np, all_idx = _batch_workload(args.workload)
    # replicas: every rank matches the whole workload (weak scaling); --shard: the pairs
    # are split over the ranks by cost and every rank matches its own share (strong)
    shard = args.shard and world > 1
    mine = list(range(len(all_idx)))
    if shard:
        sizes = [(imgs_np[i].shape[0], imgs_np[j].shape[0]) for i, j in all_idx]
        mine = serac.shard_pairs(sizes, world)[rank]
    pairs_idx = [all_idx[k] for k in mine]
    imgs = [torch.from_numpy(x).to(dev) for x in imgs_np]
    pairs = [(imgs[i], imgs[j]) for i, j in pairs_idx]
    ops_all = sum(2 * imgs_np[i].shape[0] * imgs_np[j].shape[0] * 128 for i, j in all_idx)
    ops = sum(2 * imgs_np[i].shape[0] * imgs_np[j].shape[0] * 128 for i, j in pairs_idx)
    params = serac.default_params()
    stream = torch.cuda.Stream(device=dev)
    ws = serac.workspace(serac.batch_workspace_size(pairs), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        outs = serac.match_batch(pairs, params, workspace_t=ws, stream=stream)
        stream.synchronize()
        launches = serac.last_launch_count()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            outs = serac.match_batch(pairs, params, workspace_t=ws, stream=stream)
    stream.synchronize()
    evs = []
    clocks = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(dev).uuid))
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_w0 = time.time()
    for st in range(args.warmup + args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(st & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        if st >= args.warmup:
            evs.append((e0, e1))
    stream.synchronize()
    clocks.mark(t_w0, time.time())
    clocks.hold_load(lambda: _on_stream(stream, flush, g.replay), t_w0)
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs), dev)
    n_pairs = len(pairs)
    # pairs and ops of the whole job: every rank's replica, or the one sharded workload
    job_pairs = len(all_idx) if shard else world * n_pairs
    job_ops = ops_all if shard else world * ops
    value = job_pairs * args.steps / (total_ms * 1e-3)
    tops = job_ops * args.steps / (total_ms * 1e-3) / 1e12
    peak_tflops, _, peak_kind = _peaks()
    line = {"metric": "image pairs/sec (batch), int8-equivalent TOPS", "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "strong" if shard else "weak", "vs_baseline": None,
            "dtype": DTYPE,
            "data": "synthetic", "config": {"workload": desc, "pairs": len(all_idx),
                                             "l2": "flushed before every step (256 MiB write)",
                                             "graph": "one CUDA graph per step (match_batch), replayed",
                                             "parallelism": (f"pairs sharded by cost over {world} GPUs" if shard
                                                             else f"replicas x{world}")},
            "int8_equiv_tops": tops,
            "roofline": {"bound": "tensor", "achieved": tops, "peak": peak_tflops, "unit": "TFLOP/s",
                         "frac": tops / world / peak_tflops, "traffic": None,
                         "kernel": "whole step (all launches of match_batch)",
                         "peak_kind": f"bf16 dense burst, {peak_kind}"},
            "e2e": None, "gpu_launches": launches * args.steps, "clocks": clk}
    # e2e through the public API from host buffers: the images stay in pinned host
    # memory (the staging kernel reads each image once per step over the host link)
    # and the kernels write counts and match lists straight into pinned host memory
    imgs_host = [torch.from_numpy(x).pin_memory() for x in imgs_np]
    pairs_host = [(imgs_host[i], imgs_host[j]) for i, j in pairs_idx]
    ws_h = serac.workspace(serac.batch_workspace_size(pairs_host), dev)
    with torch.cuda.stream(stream):
        e2e_outs = serac.match_batch(pairs_host, params, workspace_t=ws_h, stream=stream, host_out=True)
    stream.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    e2e_evs = []
    for st in range(3 + e2e_steps):
        with torch.cuda.stream(stream):
            flush.fill_(st & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            serac.match_batch(pairs_host, params, workspace_t=ws_h, stream=stream, outs=e2e_outs)
            e1.record(stream)
        if st >= 3:
            e2e_evs.append((e0, e1))
    stream.synchronize()
    e2e_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in e2e_evs), dev)
    same = all(torch.equal(o.result(), h.result()) for o, h in zip(outs, e2e_outs))
    if shard:
        # collect every pair's match list on rank 0 (host side, after the timed work)
        got = serac.gather_matches(mine, outs, len(all_idx))
        if rank == 0:
            line["gathered_pairs"] = sum(1 for m in got if m is not None)
    line["e2e"] = {"value": job_pairs * e2e_steps / (e2e_ms * 1e-3), "unit": UNIT,
                   "h2d_bytes_per_step": sum(x.shape[0] * 128 for x in imgs_np),
                   "d2h_bytes_per_step": sum(4 + 8 * int(h.count.item()) for h in e2e_outs),
                   "steps": e2e_steps, "equals_device_resident_result": bool(same),
                   "path": "match_batch on pinned host images, outputs in pinned host memory "
                           "(kernels read and write the host directly)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build_library()
        rng = np.random.default_rng(0)
        check = rng.choice(n_pairs, min(6, n_pairs), replace=False)
        exact = True
        t0, done_ops, n_done = time.perf_counter(), 0, 0
        for k in check:
            i, j = pairs_idx[k]
            ref = oracle.match(imgs_np[i], imgs_np[j])
            exact &= bool(np.array_equal(outs[k].result().numpy(), ref.matches))
            done_ops += 2 * imgs_np[i].shape[0] * imgs_np[j].shape[0] * 128
            n_done += 1
        dt = time.perf_counter() - t0
        line["bit_exact"] = exact
        line["bit_exact_sample"] = f"{n_done} seeded pairs against the oracle"
        # pairs/s of the oracle, scaled from the sampled pairs' work to the mean pair
        line["cpu_baseline"] = {"value": n_done / dt * (done_ops / n_done) / (ops / n_pairs), "unit": UNIT,
                                "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": f"{n_done} pairs in {dt:.1f} s, scaled to the workload's mean pair"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_topk(args):
    """--topk K: one step = serac_topk_pair (row top-k of the pair, the guided-matching
    candidate lists), same timing rules as the match step."""
    import numpy as np
    import torch

    import sift_synth
    import top_ratio_test_gb300 as serac

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    k = args.topk
    pair = sift_synth.single_pair_8192(0) if args.workload == "pair8192" else sift_synth.single_pair_2000(0)
    n_a, n_b = pair.a.shape[0], pair.b.shape[0]
    ops_per_pair = 2 * n_a * n_b * 128
    a_host = torch.from_numpy(pair.a).pin_memory()
    b_host = torch.from_numpy(pair.b).pin_memory()
    a, b = a_host.to(dev), b_host.to(dev)
    stream = torch.cuda.Stream(device=dev)
    ws = serac.workspace(serac.topk_workspace_size(n_a, n_b, k), dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev_fb, ev_fe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_fb.record(stream)
    ev_fe.record(stream)
    with torch.cuda.stream(stream):
        out = serac.topk_pair(a, b, k, workspace_t=ws, stream=stream)
        stream.synchronize()
        launches = serac.last_launch_count()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            serac.topk_pair(a, b, k, workspace_t=ws, stream=stream, out=out)
        serac.set_profile_events(ev_fb, ev_fe)
        g_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prof, stream=stream):
            serac.topk_pair(a, b, k, workspace_t=ws, stream=stream, out=out)
        serac.set_profile_events(None, None)
    stream.synchronize()

    def timed(fn, steps, warmup, fused_events=False):
        t_fused, evs = [], []
        for s_ in range(warmup + steps):
            with torch.cuda.stream(stream):
                flush.fill_(s_ & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            if s_ >= warmup:
                evs.append((e0, e1))
            if fused_events:
                stream.synchronize()
                if s_ >= warmup:
                    t_fused.append(ev_fb.elapsed_time(ev_fe))
        stream.synchronize()
        return [x.elapsed_time(y) for x, y in evs], t_fused

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_w0 = time.time()
    t_step, _ = timed(g.replay, args.steps, args.warmup)
    torch.cuda.synchronize()
    clocks.mark(t_w0, time.time())
    clocks.hold_load(lambda: _on_stream(stream, flush, g.replay), t_w0)
    clk = clocks.stop()
    _, t_fused = timed(g_prof.replay, args.steps, args.warmup, fused_events=True)
    total_ms = max_over_ranks(sum(t_step), dev)
    assert int(out.status.item()) == serac.OK
    got_s, got_i = out.scores.cpu().numpy(), out.index.cpu().numpy()

    e2e_steps = max(3, min(args.steps, 200))
    e2e_out = serac.topk_pair(a_host, b_host, k, workspace_t=ws, stream=stream, host_out=True)
    stream.synchronize()
    e2e_t, _ = timed(lambda: serac.topk_pair(a_host, b_host, k, workspace_t=ws, stream=stream, out=e2e_out),
                     e2e_steps, 3)
    e2e_ms = max_over_ranks(sum(e2e_t), dev)

    peak_tflops, _, peak_kind = _peaks()
    fused_ms = statistics.mean(t_fused)
    achieved = ops_per_pair / (fused_ms * 1e-3) / 1e12
    value = world * args.steps / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": (WORKLOAD if args.workload == "pair8192" else WORKLOAD_2000)
                   + f"; row top-{k} of A against B (guided-matching candidates) instead of the match list",
                   "n_a": n_a, "n_b": n_b, "k": k,
                   "l2": "flushed before every step (256 MiB write)",
                   "graph": "one CUDA graph per step, replayed", "parallelism": f"replicas x{world}"},
        "int8_equiv_tops": value * ops_per_pair / 1e12,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops, "traffic": None,
                     "kernel": f"fused_top2_kernel (row top-{4 if k <= 4 else 8} mode)",
                     "peak_kind": f"bf16 dense burst, {peak_kind}", "fused_ms": fused_ms},
        "e2e": {"value": world * e2e_steps / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": (n_a + n_b) * 128, "d2h_bytes_per_step": 4 + 8 * n_a * k,
                "path": "serac_topk_pair on pinned host descriptors, outputs in pinned host memory"},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build_library()
        rows = np.random.default_rng(0).choice(n_a, 512, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        rs, ri = oracle.row_topk(pair.a, pair.b, k, rows=rows)
        n = 1
        while time.perf_counter() - t0 < 10.0:
            oracle.row_topk(pair.a, pair.b, k, rows=rows)
            n += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": n * rows.shape[0] / n_a / dt, "unit": UNIT, "cores": oracle.max_threads(),
                                "kind": "oracle", "sample": f"{n} x 512 sampled rows' top-{k}, scaled to the pair, "
                                f"{dt:.1f} s"}
        line["bit_exact"] = bool(np.array_equal(got_s[rows], rs) and np.array_equal(got_i[rows], ri))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["pair8192", "pair2000", "ring12", "ragged256", "survey100"],
                    default="pair8192", help="pair8192 is the headline; the others are batch lines "
                    "for the tables (match_batch over the whole workload per step)")
    ap.add_argument("--shard", action="store_true",
                    help="batch workloads on several GPUs: split the pairs over the ranks by cost "
                    "(strong scaling) instead of running a replica per rank")
    ap.add_argument("--n", type=int, default=0,
                    help="a single n x n pair (same recipe as the 8192 x 8192 one) instead of the workload")
    ap.add_argument("--topk", type=int, default=0,
                    help="pair workloads: time the row top-k path (k = 1..8) instead of the match step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.topk and args.workload in ("pair8192", "pair2000"):
        return run_topk(args)
    if args.n or args.workload in ("pair8192", "pair2000"):
        return run_ours(args)
    return run_batch(args)


if __name__ == "__main__":
    sys.exit(main())
