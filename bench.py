#!/usr/bin/env python3
"""Benchmark: batched exact top-k / top-p truncation and sampling.

One step = one smp_sample call (temperature, mask, top-k, top-p, draw, kept
mask + count) over one batch of the named workload.  Default workload:
B=256 rows x V=128256 bf16 logits with mixed per-row parameters.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints one JSON line.  `value` = rows/s over all ranks, device-timed with CUDA
events, inputs resident in HBM and rotated over enough copies to exceed L2.
`e2e` = the same metric through the C ABI with the logits and parameters
copied from pinned host memory and the results read back every step.
`--impl reference` times the CPU oracle (plain full-sort reference) on the
host cores on a bounded sample of the same workload.
Multi-GPU (torchrun): rows are independent, every rank runs its own batch,
no collective on the data path (weak scaling).
"""
import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rows/sec and achieved HBM GB/s (fraction of roofline), B=256 V=128256 bf16"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["top_selection_stats_gb300/csrc/" + f for f in (
    "smp_philox.cuh", "smp_device.cuh", "smp_core.cuh", "smp_list.cuh", "smp_stream_passes.cuh",
    "smp_general.cuh", "smp_kernel.cuh", "smp_api.cu")]


# the verification kernel, its launch plan and its enqueue all live in one file
VERIFY_SOURCES = ["top_selection_stats_gb300/csrc/" + f for f in ("smp_verify.cu",
                                                                  "smp_philox.cuh")]


def kernel_source_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


TOPLP_SOURCES = ["top_selection_stats_gb300/csrc/smp_toplp.cu"]
SPLIT_SOURCES = ["top_selection_stats_gb300/csrc/" + f for f in (
    "smp_device.cuh", "smp_philox.cuh", "smp_split.cuh", "smp_x_bf16.cu", "smp_x_f16.cu", "smp_api.cu")]
GUMBEL_SOURCES = ["top_selection_stats_gb300/csrc/" + f for f in ("smp_gumbel.cu", "smp_philox.cuh")]
PENALTY_SOURCES = ["top_selection_stats_gb300/csrc/smp_penalty.cu"]


def profiled_entry(key, sources=KERNEL_SOURCES):
    """The committed ncu summary's entry for `key` (a workload, or
    "kernel:workload"), if it was taken on the current kernel source; else
    None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(key)
    if not e or e.get("kernel_source_sha") != kernel_source_hash(sources):
        return None
    return e


def profiled_traffic(workload, sources=KERNEL_SOURCES):
    """DRAM bytes (read + write) per launch from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    e = profiled_entry(workload, sources)
    return None if e is None else e.get("dram_bytes_per_launch")


def passes_over_hbm(entry, logits_bytes):
    """DRAM bytes read per launch over the logits' bytes (None without a
    current capture)."""
    if entry is None or not entry.get("dram_bytes_read_per_launch"):
        return None
    return entry["dram_bytes_read_per_launch"] / float(logits_bytes)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    rank, world, local = 0, 1, 0
    if n_gpus > 1 or "RANK" in os.environ:
        import torch.distributed as dist
        rank = int(os.environ.get("RANK", 0))
        world = int(os.environ.get("WORLD_SIZE", 1))
        local = int(os.environ.get("LOCAL_RANK", 0))
        if world > 1:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(local)
            dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def row_bytes(V, has_mask, write_mask, esize):
    W = (V + 31) // 32
    b = V * esize + 28 + 12  # logits, params (t, k, p, seed, offset), token + status + count
    if has_mask:
        b += 4 * W
    if write_mask:
        b += 4 * W
    return b


def cpu_oracle_rate(case, rows, threads=None):
    import oracle
    from top_selection_stats_gb300 import workloads
    x = workloads.bits_numpy(case["logits"])
    bm = None if case["bitmask"] is None else case["bitmask"].cpu().numpy().view(np.uint32)
    sel = np.arange(rows)
    p = {k: case[k].cpu().numpy()[sel] for k in ("temperature", "top_k", "top_p", "seed",
                                                 "offset")}
    cores = threads or oracle.host_cores()
    xs = np.ascontiguousarray(x[sel])
    bms = None if bm is None else np.ascontiguousarray(bm[sel])
    t0 = time.perf_counter()
    oracle.run_batch(xs, case["dtype"], case["V"], bitmask=bms, n_threads=cores, **p)
    dt = time.perf_counter() - t0
    return rows / dt, cores, dt


def cpu_oracle_sample(case, rows, min_seconds=10.0, max_passes=1000, threads=None):
    """The oracle over the first `rows` rows, repeated until about min_seconds
    of host time have been spent; returns (rows/s, cores, passes, seconds)."""
    passes, total, cores = 0, 0.0, 1
    while passes < max_passes and (passes == 0 or total < min_seconds):
        _, cores, dt = cpu_oracle_rate(case, rows, threads)
        total += dt
        passes += 1
    return rows * passes / total, cores, passes, total


def run_reference(args, rank, world):
    """CPU oracle arm: rank 0 alone, each step a bounded sample of the workload."""
    if rank != 0:
        return
    from top_selection_stats_gb300 import workloads
    case = workloads.make(args.workload, device="cpu")
    rows = min(case["B"], args.ref_rows)
    for _ in range(args.warmup):
        cpu_oracle_rate(case, rows)
    t0 = time.perf_counter()
    cores = 1
    for _ in range(args.steps):
        _, cores, _ = cpu_oracle_rate(case, rows)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": case["B"], "V": case["V"],
                   "logits": case["dtype"]},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} rows of {args.workload} per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


VERIFY_METRIC = ("sequences/sec and achieved HBM GB/s (fraction of roofline), speculative "
                 "verification, B=256 G=4 V=128256 f32")


def verify_bytes(B, G, V, n_acc):
    """Algorithmic bytes of one verification launch given its outcomes: per
    sequence the drawn row (p_j and q_j after a rejection, p_G after G
    acceptances) once, plus draft token, p and q at it per draft position,
    seed, offset and the outputs."""
    rows = np.where(np.asarray(n_acc) < G, 2, 1)
    per = rows * V * 4 + G * 12 + 16 + 4 * (G + 1) + 8
    return int(per.sum())


def verify_oracle_rate(c, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.spec_verify(c["p"][:rows].numpy(), c["q"][:rows].numpy(), c["d"][:rows].numpy(),
                       c["seed"][:rows].numpy().view(np.uint64),
                       c["offset"][:rows].numpy().view(np.uint64), n_threads=oracle.host_cores())
    return time.perf_counter() - t0, oracle.host_cores()


def run_verify_reference(args, rank, world):
    if rank != 0:
        return
    from top_selection_stats_gb300 import workloads
    c = workloads.make_verify(args.workload)
    rows = c["B"]
    for _ in range(args.warmup):
        verify_oracle_rate(c, rows)
    total, cores = 0.0, 1
    for _ in range(args.steps):
        dt, cores = verify_oracle_rate(c, rows)
        total += dt
    value = rows * args.steps / total
    line = {
        "impl": "reference", "metric": VERIFY_METRIC, "value": value, "unit": "sequences/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "B": c["B"], "G": c["G"], "V": c["V"]},
        "cpu_baseline": {"value": value, "unit": "sequences/s", "cores": cores, "kind": "oracle",
                         "sample": f"all {rows} sequences of {args.workload} per step"},
        "e2e": {"value": value, "unit": "sequences/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_verify(args, rank, world, local):
    """Speculative-decoding verification (smp_spec_verify) on a named
    workload: one step = one call over B sequences of G draft tokens."""
    from top_selection_stats_gb300 import Sampler, workloads
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    c = workloads.make_verify(args.workload)
    B, G, V = c["B"], c["G"], c["V"]
    stream = torch.cuda.current_stream(dev)
    nbuf = 2  # each step draws up to 2 rows of 0.5 MB per sequence: > L2 between reuses
    ps = [c["p"].to(dev) for _ in range(nbuf)]
    qs = [c["q"].to(dev) for _ in range(nbuf)]
    d = c["d"].to(dev)
    seed = c["seed"].to(dev)
    total = args.warmup + args.steps
    offsets = [(c["offset"] + s * B * (G + 1)).to(dev) for s in range(total)]
    smp = Sampler(local, max_batch=max(B, 64), max_vocab=max(V, 1024))
    out_t = torch.empty((B, G + 1), dtype=torch.int32, device=dev)
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)

    def step(s):
        smp.spec_verify(ps[s % nbuf], qs[s % nbuf], d, seed, offsets[s], out_tokens=out_t,
                        n_accepted=n_acc, status=st)

    # algorithmic bytes: the drawn rows depend on the outcomes of each step
    bytes_per = []
    for s in range(total):
        step(s)
        bytes_per.append(verify_bytes(B, G, V, n_acc.cpu().numpy()))
    torch.cuda.synchronize(dev)
    alg_bytes = float(np.mean(bytes_per[args.warmup:]))
    clk = ClockSampler(local) if rank == 0 else None
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                step(args.warmup + i)
    stream.wait_stream(cap)
    graph.replay()  # untimed: the first replay also uploads the graph
    torch.cuda.synchronize(dev)
    if clk:
        clk.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    graph.replay()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = clk.stop() if clk else None
    elapsed_ms = max_over_ranks(g0.elapsed_time(g1), world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = B * world / (ms_per_step / 1000.0)

    # end to end: probabilities, drafts and offsets from pinned host memory,
    # outputs read back, every step
    hp, hq, hd = (x.pin_memory() for x in (c["p"], c["q"], c["d"]))
    hseed = c["seed"].pin_memory()
    hoff = [o.pin_memory() for o in (c["offset"] + s * B * (G + 1) for s in range(4))]
    ho = [torch.empty(x.shape, dtype=torch.int32).pin_memory() for x in (out_t, n_acc, st)]
    dp, dq = torch.empty_like(ps[0]), torch.empty_like(qs[0])
    dd, dseed = torch.empty_like(d), torch.empty_like(seed)
    doff = torch.empty_like(offsets[0])

    def e2e_step(s):
        dp.copy_(hp, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dd.copy_(hd, non_blocking=True)
        dseed.copy_(hseed, non_blocking=True)
        doff.copy_(hoff[s % 4], non_blocking=True)
        smp.spec_verify(dp, dq, dd, dseed, doff, out_tokens=out_t, n_accepted=n_acc, status=st)
        for h, x in zip(ho, (out_t, n_acc, st)):
            h.copy_(x, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_steps = 5
    for s in range(2):
        e2e_step(s)
    barrier(world)
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        e2e_step(s)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = sum(x.numel() * x.element_size() for x in (hp, hq, hd, hseed)) + B * 8
    d2h = sum(x.numel() * 4 for x in ho)
    e2e = {"value": B * world * e2e_steps / e2e_s, "unit": "sequences/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (ms_per_step / 1000.0) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(args.workload, VERIFY_SOURCES),
            "peak_kind": peak_kind, "algorithmic_bytes_per_launch": alg_bytes,
            "kernel_ms": ms_per_step}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        secs, passes, cores = 0.0, 0, 1
        while passes == 0 or (secs < 5.0 and passes < 1000):
            dt, cores = verify_oracle_rate(c, B)
            secs += dt
            passes += 1
        cpu = {"value": B * passes / secs, "unit": "sequences/s", "cores": cores,
               "kind": "oracle", "sample": f"all {B} sequences of {args.workload}, {passes} "
                                           f"passes ({secs:.1f} s)"}
    if rank == 0:
        n = n_acc.cpu().numpy()
        line = {
            "metric": VERIFY_METRIC, "value": value, "unit": "sequences/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "G": G, "V": V,
                       "l2": f"inputs rotated over {nbuf} copies of "
                             f"{(c['p'].numel() + c['q'].numel()) * 4 / 1e6:.0f} MB",
                       "rejected_sequences_last_step": int((n < G).sum()),
                       "timing": "cuda graph of the K launches, replayed once untimed first"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps,
        }
        print(json.dumps(line), flush=True)
    smp.close()


def run_decode_loop(args, rank, world, local):
    """The repeated decode loop: args.steps steps (default 200) of the decode
    workload, fresh logits generated for every step outside the timed region,
    the Philox offsets advanced by the B blocks each step consumes, kept masks
    returned.  Each step's launch is timed alone with CUDA events after an L2
    flush; the line reports the per-step distribution and the loop total."""
    from top_selection_stats_gb300 import Sampler, workloads
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    first = workloads.make(args.workload, step=0, device="cuda")
    B, V = first["B"], first["V"]
    esize = 4 if first["dtype"] == "f32" else 2
    W = (V + 31) // 32
    smp = Sampler(local, max_batch=max(B, 64), max_vocab=max(V, 1024))
    smp.set_kernel(args.kernel)
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    kmask = torch.empty((B, W), dtype=torch.int32, device=dev)
    kcount = torch.empty(B, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    del first

    def launch(c):
        smp.sample(c["logits"], c["temperature"], c["top_k"], c["top_p"], c["seed"],
                   c["offset"], bitmask=c["bitmask"], kept_mask=kmask, kept_count=kcount,
                   tokens=tokens, status=status)

    # warm-up on steps of their own (before step 0 of the loop)
    for w in range(args.warmup):
        launch(workloads.rank_shard(workloads.make(args.workload, step=args.steps + w,
                                                   device="cuda"), rank, world))
    torch.cuda.synchronize(dev)
    clk = ClockSampler(local) if rank == 0 else None
    if clk:
        clk.start()
        time.sleep(0.3)
    barrier(world)
    per_step = []
    bad = 0
    for st in range(args.steps):
        c = workloads.rank_shard(workloads.make(args.workload, step=st, device="cuda"), rank, world)
        flush.zero_()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch(c)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per_step.append(e0.elapsed_time(e1))
        bad += int((status != 0).sum())
    barrier(world)
    clocks = clk.stop() if clk else None
    total_ms = max_over_ranks(float(np.sum(per_step)), world, dev)
    ms = np.asarray(per_step)
    ms_per_step = total_ms / args.steps
    value = B * world / (ms_per_step / 1000.0)

    # end to end through the public API: each step's logits from pinned host
    # memory, the tokens, statuses, counts and kept masks back to the host
    e2e_steps = min(args.steps, 20)
    host_logits = torch.empty((B, V), dtype=torch.float16 if esize == 2 else torch.float32)
    host_logits = host_logits.pin_memory()
    out = [torch.empty(B, dtype=torch.int32).pin_memory() for _ in range(3)]
    out_mask = torch.empty((B, W), dtype=torch.int32).pin_memory()
    dl = torch.empty((B, V), dtype=host_logits.dtype, device=dev)
    e2e_s = 0.0
    for st in range(e2e_steps):
        c = workloads.rank_shard(workloads.make(args.workload, step=st, device="cuda"), rank,
                                 world)
        host_logits.copy_(c["logits"])
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        dl.copy_(host_logits, non_blocking=True)
        c2 = dict(c, logits=dl)
        launch(c2)
        for o, d in zip(out, (tokens, status, kcount)):
            o.copy_(d, non_blocking=True)
        out_mask.copy_(kmask, non_blocking=True)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e = {"value": B * world * e2e_steps / e2e_s, "unit": "rows/s",
           "h2d_bytes_per_step": B * V * esize, "d2h_bytes_per_step": B * 12 + B * W * 4,
           "steps": e2e_steps, "params": "on the device (per-row parameters do not change)"}
    peak, peak_kind = measured_peaks()
    alg_bytes = B * row_bytes(V, False, True, esize)
    achieved = alg_bytes / (ms_per_step / 1000.0) / 1e9
    prof = (profiled_entry(args.workload) if args.kernel == "board"
            else profiled_entry("split:" + args.workload, SPLIT_SOURCES))
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": None if prof is None else prof.get("dram_bytes_per_launch"),
            "passes_over_hbm": passes_over_hbm(prof, B * V * esize), "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": ms_per_step}
    if rank == 0:
        line = {
            "metric": f"rows/sec over a {args.steps}-step decode loop, B={B} V={V} "
                      f"{workloads.WORKLOADS[args.workload]['dtype']}",
            "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": workloads.WORKLOADS[args.workload]["dtype"],
            "arith": "f32 weights, 64-bit fixed-point masses", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "V": V, "kernel": args.kernel,
                       "kept_mask": True, "fresh_logits_per_step": True,
                       "offset_advance": f"{B} Philox blocks per step (one per row)",
                       "l2": "flushed (2x L2 written) before every step",
                       "timing": "each step's launch alone, CUDA events on the launch stream",
                       "per_step_ms": {"mean": float(ms.mean()), "p50": float(np.median(ms)),
                                       "p90": float(np.percentile(ms, 90)),
                                       "max": float(ms.max()), "min": float(ms.min())},
                       "total_ms": total_ms, "error_rows": bad},
            "roofline": roof, "cpu_baseline": None, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps,
        }
        print(json.dumps(line), flush=True)
    smp.close()


def run_ours(args, rank, world, local):
    from top_selection_stats_gb300 import Sampler, binding, workloads
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = workloads.rank_shard(workloads.make(args.workload, device="cpu"), rank, world)
    B, V = case["B"], case["V"]
    esize = 4 if case["dtype"] == "f32" else 2
    bytes_logits = B * V * esize
    nbuf = max(2, -(-3 * L2_BYTES // bytes_logits))
    stream = torch.cuda.current_stream(dev)
    logits = [case["logits"].to(dev) for _ in range(nbuf)]
    bitmask = None if case["bitmask"] is None else case["bitmask"].to(dev)
    t = case["temperature"].to(dev)
    k = case["top_k"].to(dev)
    p = case["top_p"].to(dev)
    seed = case["seed"].to(dev)
    total = args.warmup + args.steps
    offsets = [(case["offset"] + s * B).to(dev) for s in range(total)]
    smp = Sampler(local, max_batch=max(B, 64), max_vocab=max(V, 1024))
    smp.set_kernel(args.kernel)
    plan = smp.plan(case["logits"].dtype, V, B=B)
    W = (V + 31) // 32
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    kmask = torch.empty((B, W), dtype=torch.int32, device=dev)
    kcount = torch.empty(B, dtype=torch.int32, device=dev)

    logprobs = torch.empty(B, dtype=torch.float32, device=dev) if args.logprob else None
    pen_hist = pen_theta = pen_status = None
    pen_bytes = 0
    if args.repetition_penalty:
        # a history of H token ids per row (repeats included) and a per-row penalty
        rng = np.random.Generator(np.random.PCG64(11))
        Hn = args.repetition_penalty
        hist = rng.integers(0, V, size=(B, Hn)).astype(np.int32)
        hist[:, Hn // 2:] = hist[:, :Hn - Hn // 2][:, :Hn // 2]
        pen_hist = torch.as_tensor(hist).to(dev)
        pen_theta = torch.as_tensor(rng.choice(np.array([1.1, 1.2, 1.3], np.float32),
                                               size=B)).to(dev)
        pen_status = torch.empty(B, dtype=torch.int32, device=dev)
        distinct = sum(len(np.unique(hist[r])) for r in range(B))
        pen_bytes = B * (Hn * 4 + 4 + 4) + distinct * 2 * esize
        # every rotated buffer is penalised once, as a decode step's fresh
        # logits would be; the timed launches then run the same kernel with
        # theta = 1 (the same loads, arithmetic and stores) so that repeated
        # steps on a buffer do not compound the penalty
        for buf in logits:
            smp.repetition_penalty(buf, pen_hist, pen_theta, status=pen_status)
        pen_theta = torch.ones(B, dtype=torch.float32, device=dev)
        torch.cuda.synchronize(dev)

    def step(s, lg=None):
        if pen_hist is not None:
            smp.repetition_penalty(logits[s % nbuf] if lg is None else lg, pen_hist, pen_theta,
                                   status=pen_status)
        smp.sample(logits[s % nbuf] if lg is None else lg, t, k, p, seed, offsets[s],
                   bitmask=bitmask, kept_mask=kmask, kept_count=kcount, tokens=tokens,
                   status=status, logprobs=logprobs)

    # path statistics (untimed)
    smp.set_row_info(True, max_batch=B)
    step(0)
    torch.cuda.synchronize(dev)
    info = smp.row_info(B).cpu().numpy()
    smp.set_row_info(False)
    paths = {name: int((info[:, 0] == code).sum())
             for code, name in {0: "error", 1: "greedy", 2: "all", 3: "sigma", 4: "full"}.items()}

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(local) if rank == 0 else None
    # The K timed launches are captured in one CUDA graph (each with its own
    # input copy and Philox offsets) so that host-side launch overhead does not
    # sit between them; the replay is timed with events on the launch stream.
    graph = None
    timing = "cuda graph of the K launches"
    try:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for i in range(args.steps):
                    step(args.warmup + i)
        stream.wait_stream(cap)
        graph.replay()  # untimed: the first replay also uploads the graph
        torch.cuda.synchronize(dev)
        timing += ", replayed once untimed first"
    except Exception as exc:  # capture unavailable: eager launches
        graph = None
        timing = f"eager launches ({type(exc).__name__})"
    if clk:
        clk.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(args.warmup + i)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = clk.stop() if clk else None
    elapsed_ms = g0.elapsed_time(g1)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    kern_ms = elapsed_ms / args.steps
    ms_per_step = elapsed_ms / args.steps
    value = B * world / (ms_per_step / 1000.0)

    # end to end through the C ABI with host buffers
    host_logits = case["logits"].pin_memory()
    host_par = [x.pin_memory() for x in (case["temperature"], case["top_k"], case["top_p"],
                                         case["seed"])]
    host_off = [o.cpu().pin_memory() for o in offsets]
    host_mask = None if case["bitmask"] is None else case["bitmask"].pin_memory()
    out_tok = torch.empty(B, dtype=torch.int32).pin_memory()
    out_st = torch.empty(B, dtype=torch.int32).pin_memory()
    out_mask = torch.empty((B, W), dtype=torch.int32).pin_memory()
    out_cnt = torch.empty(B, dtype=torch.int32).pin_memory()
    dl = torch.empty_like(logits[0])
    dpar = [torch.empty_like(x, device=dev) for x in host_par]
    doff = torch.empty(B, dtype=torch.int64, device=dev)
    dmask = None if host_mask is None else torch.empty_like(host_mask, device=dev)

    def e2e_step(s):
        dl.copy_(host_logits, non_blocking=True)
        for d_, h_ in zip(dpar, host_par):
            d_.copy_(h_, non_blocking=True)
        doff.copy_(host_off[s], non_blocking=True)
        if dmask is not None:
            dmask.copy_(host_mask, non_blocking=True)
        smp.sample(dl, dpar[0], dpar[1], dpar[2], dpar[3], doff, bitmask=dmask,
                   kept_mask=kmask, kept_count=kcount, tokens=tokens, status=status)
        out_tok.copy_(tokens, non_blocking=True)
        out_st.copy_(status, non_blocking=True)
        out_mask.copy_(kmask, non_blocking=True)
        out_cnt.copy_(kcount, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_steps = min(args.steps, max(3, args.steps // 2))
    for s in range(min(3, args.warmup)):
        e2e_step(s)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        e2e_step(s % total)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = bytes_logits + B * 28 + (0 if host_mask is None else host_mask.numel() * 4)
    d2h = B * 4 * 3 + B * W * 4
    e2e = {"value": B * world * e2e_steps / e2e_s, "unit": "rows/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    peak, peak_kind = measured_peaks()
    alg_bytes = B * (row_bytes(V, bitmask is not None, True, esize) + (4 if args.logprob else 0))
    alg_bytes += pen_bytes
    pen_info = None
    if pen_hist is not None:
        # the penalty kernel alone, same rotation, timed the same way
        pg = torch.cuda.CUDAGraph()
        cap2 = torch.cuda.Stream(dev)
        cap2.wait_stream(stream)
        with torch.cuda.stream(cap2):
            with torch.cuda.graph(pg, stream=cap2):
                for i in range(args.steps):
                    smp.repetition_penalty(logits[i % nbuf], pen_hist, pen_theta,
                                           status=pen_status)
        stream.wait_stream(cap2)
        pg.replay()
        torch.cuda.synchronize(dev)
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        pg.replay()
        q1.record(stream)
        torch.cuda.synchronize(dev)
        pen_ms = q0.elapsed_time(q1) / args.steps
        pen_info = {"history_per_row": args.repetition_penalty, "kernel_us": 1000 * pen_ms,
                    "timed_theta": "1 (buffers penalised once with 1.1-1.3 before timing)",
                    "algorithmic_bytes": pen_bytes,
                    "gbs": pen_bytes / (pen_ms / 1000.0) / 1e9,
                    "traffic": profiled_traffic("penalty:" + args.workload, PENALTY_SOURCES)}
    achieved = alg_bytes / (kern_ms / 1000.0) / 1e9
    prof = (profiled_entry(args.workload) if args.kernel == "board"
            else profiled_entry("split:" + args.workload, SPLIT_SOURCES))
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": None if prof is None else prof.get("dram_bytes_per_launch"),
            "passes_over_hbm": passes_over_hbm(prof, bytes_logits), "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": kern_ms}

    toplp_info = None
    if args.top_logprobs:
        # the n best kept tokens and their logprobs from the last step's outputs
        tl_ids = torch.empty((B, args.top_logprobs), dtype=torch.int32, device=dev)
        tl_lp = torch.empty((B, args.top_logprobs), dtype=torch.float32, device=dev)
        last = args.warmup + args.steps - 1

        def toplp(i):
            smp.lib.smp_top_logprobs(smp.h, binding._ptr(logits[last % nbuf]),
                                     binding._DTYPES[logits[0].dtype], B, V, V,
                                     binding._ptr(kmask), binding._ptr(t), binding._ptr(tokens),
                                     binding._ptr(logprobs), args.top_logprobs,
                                     binding._ptr(tl_ids), binding._ptr(tl_lp), smp._stream())

        tg = torch.cuda.CUDAGraph()
        cap4 = torch.cuda.Stream(dev)
        cap4.wait_stream(stream)
        with torch.cuda.stream(cap4):
            with torch.cuda.graph(tg, stream=cap4):
                for i in range(args.steps):
                    toplp(i)
        stream.wait_stream(cap4)
        tg.replay()
        torch.cuda.synchronize(dev)
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        tg.replay()
        q1.record(stream)
        torch.cuda.synchronize(dev)
        toplp_info = {"n": args.top_logprobs,
                      "kernel_us": 1000 * q0.elapsed_time(q1) / args.steps,
                      "note": "one buffer (its kept masks in L2 between launches)",
                      "traffic": profiled_traffic("toplp:" + args.workload, TOPLP_SOURCES)}

    gumbel_info = None
    if args.gumbel:
        # the sort-free second sampler: the kept set from smp_topk_topp_mask,
        # then a Gumbel-max draw over it (two launches per step), against the
        # fused smp_sample timed above
        mk = smp.topk_topp_mask(logits[0], t, k, p, bitmask=bitmask)["kept_mask"]
        gtok = torch.empty(B, dtype=torch.int32, device=dev)
        gst = torch.empty(B, dtype=torch.int32, device=dev)
        gbuf = torch.empty((B, W), dtype=torch.int32, device=dev)
        gcnt = torch.empty(B, dtype=torch.int32, device=dev)
        gstat = torch.empty(B, dtype=torch.int32, device=dev)

        def gumbel_only(i):
            smp.gumbel_sample(logits[i % nbuf], t, seed, offsets[i], kept_mask=mk, tokens=gtok,
                              status=gst)

        def mask_then_gumbel(i):
            smp.lib.smp_topk_topp_mask(
                smp.h, binding._ptr(logits[i % nbuf]), binding._DTYPES[logits[0].dtype], B, V, V,
                binding._ptr(bitmask), ctypes.byref(binding.RowParams(
                    t.data_ptr(), k.data_ptr(), p.data_ptr(), None, None)),
                binding._ptr(gbuf), binding._ptr(gcnt), binding._ptr(gstat), None,
                smp._stream())
            smp.gumbel_sample(logits[i % nbuf], t, seed, offsets[i], kept_mask=gbuf, tokens=gtok,
                              status=gst)

        gumbel_info = {}
        for name, fn in (("gumbel_kernel_us", gumbel_only), ("mask_plus_gumbel_us",
                                                              mask_then_gumbel)):
            gg = torch.cuda.CUDAGraph()
            cap3 = torch.cuda.Stream(dev)
            cap3.wait_stream(stream)
            with torch.cuda.stream(cap3):
                with torch.cuda.graph(gg, stream=cap3):
                    for i in range(args.steps):
                        fn(args.warmup + i)
            stream.wait_stream(cap3)
            gg.replay()
            torch.cuda.synchronize(dev)
            q0 = torch.cuda.Event(enable_timing=True)
            q1 = torch.cuda.Event(enable_timing=True)
            q0.record(stream)
            gg.replay()
            q1.record(stream)
            torch.cuda.synchronize(dev)
            gumbel_info[name] = 1000 * q0.elapsed_time(q1) / args.steps
        gumbel_info["fused_smp_sample_us"] = 1000 * kern_ms
        gumbel_info["traffic"] = profiled_traffic("gumbel:" + args.workload, GUMBEL_SOURCES)

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline:
        rows = min(B, args.cpu_rows)
        rate, cores, passes, secs = cpu_oracle_sample(case, rows)
        rows1 = min(rows, 16)
        rate1, _, passes1, secs1 = cpu_oracle_sample(case, rows1, min_seconds=5.0, threads=1)
        cpu = {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"first {rows} rows of {args.workload}, {passes} passes "
                         f"({secs:.1f} s wall)",
               "single_thread": {"value": rate1, "unit": "rows/s", "cores": 1,
                                 "sample": f"first {rows1} rows, {passes1} passes "
                                           f"({secs1:.1f} s wall)"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": case["dtype"], "data": "synthetic",
            "arith": "f32 weights, 64-bit fixed-point masses",
            "config": {"workload": args.workload, "B": B, "V": V, "logits": case["dtype"],
                       "kernel": args.kernel,
                       "kept_mask": True,
                       "l2": f"inputs rotated over {nbuf} copies ({nbuf * bytes_logits / 1e6:.0f} MB > L2)",
                       "cluster": plan["cluster"], "slice": plan["slice"],
                       "smem_per_cta": plan["smem"], "paths": paths, "timing": timing,
                       "logprob": bool(args.logprob), "repetition_penalty": pen_info,
                       "gumbel": gumbel_info, "top_logprobs": toplp_info},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps * (2 if pen_hist is not None else 1),
        }
        print(json.dumps(line), flush=True)
    smp.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed256x128256_bf16")
    ap.add_argument("--cpu-rows", type=int, default=256)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repetition-penalty", type=int, default=0, metavar="H",
                    help="apply the repetition penalty (H history ids per row) before each "
                         "sample call, in place on the step's logits")
    ap.add_argument("--top-logprobs", type=int, default=0, metavar="N",
                    help="also time smp_top_logprobs (N best kept tokens; implies --logprob)")
    ap.add_argument("--gumbel", action="store_true",
                    help="also time the Gumbel-max sampler (kept mask + smp_gumbel_sample)")
    ap.add_argument("--kernel", default="board", choices=["board", "split"],
                    help="sampler kernel (smp_set_kernel): job board, or split rows over clusters")
    ap.add_argument("--logprob", action="store_true",
                    help="also return each drawn token's log-probability (smp_sample_logprob)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.top_logprobs:
        args.logprob = True
    rank, world, local = dist_setup(args.gpus)
    verify = args.workload.startswith("verify")
    if args.impl == "reference":
        (run_verify_reference if verify else run_reference)(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --impl ours needs a CUDA GPU")
        if args.workload.startswith("decode"):
            run_decode_loop(args, rank, world, local)
        else:
            (run_verify if verify else run_ours)(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
