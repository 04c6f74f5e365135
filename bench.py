"""Benchmark of the ZeRO-1 optimizer step: params/s and achieved HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = the whole hot path over one batch: reduce-scatter of W emulated
ranks' bf16 gradients + global norm + clip + AdamW on the fp32 shards + bf16
all-gather into W replicas, through the C ABI (zero1_step).  Inputs are
seeded synthetic tensors already resident in HBM (two gradient sets used
alternately); the working set is far larger than L2, so no flush is needed.

Multi-GPU (torchrun, one process per GPU): every GPU runs its own emulated
W-rank problem ("replicas only"); no data crosses GPUs, the process group
serves only the barrier and the max-over-ranks time.  value = params of all
GPUs / max time.

--impl reference times the CPU oracle (single-threaded C) on the host cores,
each step a bounded sample of the same workload; rank 0 only.
"""
from __future__ import annotations

import argparse
import datetime as dt
import hashlib
import re
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as WL  # noqa: E402

METRIC = "ZeRO-1 step params/s and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "zero_sharded_adamw_gb300", "csrc")
# The sources the step's kernels are compiled from; a committed ncu summary
# counts for the current build only if it carries their digest.
KERNEL_SRCS = [os.path.join(CSRC, f) for f in ("zero1_kernels.cu", "zero1_ptx.cuh", "zero1_internal.h")]


def kernel_source_digest(paths=KERNEL_SRCS) -> str:
    """sha256 over the sources with comments and whitespace runs removed, so
    that an edit to a comment does not orphan counters taken on the same code."""
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


# ------------------------------------------------------------- helpers

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(world_size: int, backend: str):
    if world_size > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world_size: int):
    if world_size > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world_size: int, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (identity on one rank)."""
    if world_size == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def host_available_bytes() -> int | None:
    """Host memory available to new allocations (Linux), or None if unknown."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def host_memory_short(pinned_per_rank: int, local_ranks: int, world_size: int, device="cpu",
                      available: int | None = None) -> bool:
    """True on every rank if any rank's node cannot pin `local_ranks` x
    pinned_per_rank bytes within 80% of its available memory (collective,
    so that all ranks take the same branch)."""
    avail = host_available_bytes() if available is None else available
    short = avail is not None and pinned_per_rank * local_ranks > 0.8 * avail
    return reduce_max(1.0 if short else 0.0, world_size, device) > 0


def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _summary_fields(path: str) -> dict:
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    return fields


def kernel_traffic(workload: str, n: int) -> tuple[float | None, str | None]:
    """DRAM bytes per launch of the update kernel at n parameters, from the
    committed ncu summary of the workload's recipe taken on the current
    kernel sources: a one-kernel capture on a small case (a few GB on the
    device), whose DRAM bytes per parameter are scaled by n (the kernel
    streams every parameter once, so its traffic grows in proportion to n).
    (None, None) when no summary matches the current sources."""
    sha = kernel_source_digest()
    fname = f"dram_{workload.split('@')[0]}.txt"
    path = os.path.join(ROOT, "profiles", fname)
    if not os.path.exists(path):
        return None, None
    fields = _summary_fields(path)
    if fields.get("kernel_source_digest") != sha:
        return None, None
    try:
        return float(fields["zero1_adamw_ag_kernel.dram_bytes_per_param"]) * n, "profiles/" + fname
    except (KeyError, ValueError):
        return None, None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms, kept with timestamps."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        smi = shutil.which("nvidia-smi")
        if smi is None:
            return
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            gpu = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            gpu = str(device_index)
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        self.proc = subprocess.Popen([smi, "-i", gpu, f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=self.out, stderr=subprocess.DEVNULL)

    def stop(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        used = inside or rows
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in used for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples": len(used), "in_timed_region": bool(inside)}


# -------------------------------------------------------- oracle timing

def oracle_rate(w: WL.Workload, n_sample: int, steps: int, seconds: float | None = None) -> tuple[float, int, int]:
    """Time the CPU oracle on the first n_sample parameters of workload w.
    Runs `steps` steps (or until `seconds` have passed, if given).  Returns
    (params/s, steps run, n_sample)."""
    import numpy as np
    from oracle import zero1_oracle as o
    ws = w.with_n(n_sample)
    hp = o.HP(**w.hparams())
    sets = []
    for t in (1, 2):
        g = WL.grads(ws, t, "cpu")
        sets.append([x.view(torch.int16).numpy().view(np.uint16) for x in g])
    st = o.State(WL.master(ws, "cpu").numpy())
    done, t_start = 0, time.perf_counter()
    while True:
        o.step(st, sets[done % 2], hp)
        done += 1
        el = time.perf_counter() - t_start
        if (seconds is None and done >= steps) or (seconds is not None and el >= seconds and done >= 1):
            break
    return n_sample * done / el, done, n_sample


def reference_arm(args, w: WL.Workload, cfg: dict):
    rank, world_size, _ = dist_env()
    if rank != 0:
        return
    # Size each step's sample so that warmup + timed steps end in ~60 s.
    rate, _, _ = oracle_rate(w, 1 << 18, 1)
    per_step = 60.0 / max(1, args.steps + args.warmup)
    n_sample = int(min(w.n, max(4096, rate * per_step)))
    oracle_rate(w, n_sample, max(1, args.warmup))
    value, done, n_sample = oracle_rate(w, n_sample, args.steps)
    sample = (f"first {n_sample:,} parameters of the {w.name} recipe, W={w.world}, "
              f"{done} steps, single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * n_sample / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our arm

def ours_arm(args, w: WL.Workload, cfg: dict):
    import zero_sharded_adamw_gb300 as z

    rank, world_size, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    init_dist(world_size, "nccl")
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)

    hp = z.Hparams(**w.hparams())
    opts = z.Options(args.decay_first, args.clip_eps, args.moments_bf16, small_step=args.small_step,
                     capturable=args.graph, host_chunk=args.host_chunk, load_phase_gbs=args.load_phase_gbs)
    grad_sets = [WL.grads(w, t, dev) for t in range(1, args.grad_sets + 1)]
    reps = [torch.empty(w.n, dtype=torch.bfloat16, device=dev) for _ in range(w.world)]
    opt = z.Zero1(w.n, w.world, hp, opts)
    opt.set_state(WL.master(w, dev), stream=stream)
    torch.cuda.synchronize(dev)

    # pointer tables built once: the timed loop marshals no per-step arguments
    tables = [z.PtrTable(g) for g in grad_sets]
    rep_table = z.PtrTable(reps)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == 0:
            w0.record(stream)
        opt.step(grad_sets[i % len(grad_sets)], reps, stream)
        if i == 0:
            w1.record(stream)
    torch.cuda.synchronize(dev)
    first_ms = w0.elapsed_time(w1) if args.warmup else None

    clocks = ClockSampler(local_rank)
    time.sleep(0.3 if clocks.proc else 0.0)
    z.zero1_profile_start(opt.handle, args.steps)
    barrier(world_size)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    h0 = time.perf_counter()
    for i in range(args.steps):
        opt.step(tables[i % len(tables)], rep_table, stream)
    host_enqueue_s = time.perf_counter() - h0
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world_size)
    t1 = time.time()
    local_ms = ev0.elapsed_time(ev1)
    per_rs, per_upd = z.zero1_profile_read(opt.handle, args.steps)
    per_step = sorted(x + y for x, y in zip(per_rs, per_upd))
    rs_ms, upd_ms, prof_steps = z.zero1_profile_stop(opt.handle)
    clk = clocks.stop(t0, t1)
    ms = reduce_max(local_ms, world_size, dev)
    norm, clip = opt.grad_norm(stream)

    ms_per_step = ms / args.steps
    value = world_size * w.n * args.steps / (ms / 1e3)
    state_rw = 16 if args.moments_bf16 else 24          # master, m, v read + write
    alg_step = (4 * w.world + state_rw) * w.n
    peak, peak_kind = measured_peak()
    upd_avg = upd_ms / max(1, prof_steps)
    rs_avg = rs_ms / max(1, prof_steps)
    upd_bytes = (state_rw + 2 * w.world) * w.n    # state read+write, replica writes
    rs_bytes = (2 * w.world) * w.n                # gradient reads
    # the committed captures are of the default variant (fp32 moments)
    traffic, traffic_src = (None, None) if args.moments_bf16 else kernel_traffic(w.name, w.n)
    achieved = upd_bytes / (upd_avg / 1e3) / 1e9
    launches = opt.launches_per_step()
    if launches == 1:
        # one-launch small-n path: the step's one kernel moves every byte
        achieved = alg_step / (rs_avg / 1e3) / 1e9
        kernels = {"zero1_small_step_kernel": {"avg_launch_ms": rs_avg, "algorithmic_bytes": alg_step,
                                               "gbs": achieved},
                   "launches_timed": prof_steps}
        roof_kernel, roof_bytes, roof_ms = "zero1_small_step_kernel", alg_step, rs_avg
        traffic, traffic_src = None, None
    else:
        kernels = {"zero1_rs_norm_kernel": {"avg_launch_ms": rs_avg, "algorithmic_bytes": rs_bytes,
                                            "gbs": rs_bytes / (rs_avg / 1e3) / 1e9},
                   "zero1_adamw_ag_kernel": {"avg_launch_ms": upd_avg, "algorithmic_bytes": upd_bytes,
                                             "gbs": achieved},
                   "launches_timed": prof_steps}
        roof_kernel, roof_bytes, roof_ms = "zero1_adamw_ag_kernel", upd_bytes, upd_avg

    # Graph replay (capturable handle): G consecutive steps captured in one
    # CUDA graph (each replay advances the device step counter G times),
    # replayed until K steps ran, so the host enqueues one graph launch per
    # G steps instead of each step's kernel launches and profile events.
    graph = None
    if args.graph:
        gsteps = max(1, min(args.graph_steps, args.steps))
        reps_n = -(-args.steps // gsteps)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            for i in range(gsteps):
                opt.step(tables[i % len(tables)], rep_table, cs)
        for _ in range(3):
            g.replay()
        barrier(world_size)
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps_n):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        gms = reduce_max(g0.elapsed_time(g1), world_size, dev)
        done = reps_n * gsteps
        graph = {"ms_per_step": gms / done, "value": world_size * w.n * done / (gms / 1e3),
                 "unit": "params/s", "steps": done, "steps_per_graph": gsteps,
                 "note": "consecutive zero1_step calls (capturable handle) captured in one CUDA graph "
                         "and replayed; the two gradient sets alternate"}
        del g

    # End to end through the host-buffer entry points: every step uploads
    # every rank's gradient from pinned memory, runs the step and downloads
    # every rank's replica.  The pipelined entry point overlaps step t's
    # download with step t+1's upload; the blocking one is reported beside it.
    # The device-resident gradient and replica buffers are released first:
    # the host path needs only the optimizer state, its scratch and two
    # bounded rings on the device.
    e2e = None
    # Every local rank pins W gradient and W replica buffers of n bf16 at
    # once; leave the leg out (with the reason) where the node cannot hold
    # them all, rather than exhaust its memory.
    pinned = 4 * w.world * w.n
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", 1))
    short = host_memory_short(pinned, local_ranks, world_size, dev)
    if not args.no_e2e and short:
        e2e = {"value": None, "skipped": f"host memory: {local_ranks} rank(s) x {pinned / 1e9:.0f} GB pinned "
                                         f"> 80% of the node's available memory"}
    elif not args.no_e2e:
        hg = []
        for g in grad_sets[0]:
            hg.append(torch.empty(w.n, dtype=torch.bfloat16, pin_memory=True))
            hg[-1].copy_(g)
        hr = [torch.empty(w.n, dtype=torch.bfloat16, pin_memory=True) for _ in range(w.world)]
        del tables, rep_table, grad_sets, reps
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        k_e2e = args.e2e_steps or max(3, min(args.steps, 20))
        rates = {}
        for name in ("zero1_step_host", "zero1_step_host_async"):
            run = opt.step_host if name == "zero1_step_host" else opt.step_host_async
            for _ in range(2):                     # sets up the rings, streams and events
                run(hg, hr, stream)
            opt.host_sync()
            barrier(world_size)
            torch.cuda.synchronize(dev)
            s0 = time.perf_counter()
            for _ in range(k_e2e):
                run(hg, hr, stream)
            opt.host_sync()
            torch.cuda.synchronize(dev)
            e2e_s = reduce_max(time.perf_counter() - s0, world_size, dev)
            rates[name] = world_size * w.n * k_e2e / e2e_s
        e2e = {"value": rates["zero1_step_host_async"], "unit": "params/s",
               "h2d_bytes_per_step": 2 * w.world * w.n, "d2h_bytes_per_step": 2 * w.world * w.n,
               "steps": k_e2e, "entry_point": "zero1_step_host_async + zero1_host_sync",
               "blocking_value": rates["zero1_step_host"]}
        del hg, hr

    cpu = None
    if rank == 0 and world_size == 1 and not args.no_cpu_baseline:
        rate, done, n_s = oracle_rate(w, 1 << 20, 1, seconds=10.0)
        cpu = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n_s:,} parameters of the {w.name} recipe, W={w.world}, {done} steps "
                         f"(~10 s), single-threaded C oracle"}

    line = {
        "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world_size,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": cfg,
        "hbm": {"algorithmic_bytes_per_step": alg_step,
                "algorithmic_gbs": world_size * alg_step / (ms_per_step / 1e3) / 1e9,
                "frac_of_peak": (alg_step / (ms_per_step / 1e3) / 1e9) / peak,
                "peak_gbs": peak, "peak_kind": peak_kind},
        "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_ms": roof_ms,
                     "peak_kind": peak_kind},
        "kernels": kernels,
        # per-step K1 + K2 device time from the same events (gaps between
        # steps excluded), and the first warm-up step on its own
        "step_kernel_ms": {"median": per_step[len(per_step) // 2] if per_step else None,
                           "min": per_step[0] if per_step else None,
                           "first_warmup_step": first_ms,
                           # host time to enqueue one step (binding + C ABI + launches + profile
                           # events); when it reaches ms_per_step the GPU waits on the host
                           "host_enqueue_per_step": 1e3 * host_enqueue_s / args.steps},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "graph_replay": graph,
        "gpu_launches": launches * args.steps,
        "last_step": {"grad_norm": norm, "clip_coef": clip},
    }
    opt.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world_size > 1:
        torch.distributed.destroy_process_group()


def allreduce_arm(args):
    """The DDP all-reduce path: one zero1_allreduce per step over W emulated
    ranks' buffers (inputs and outputs distinct).  Reports HBM GB/s of the
    algorithmic traffic (read W buffers, write W buffers) and, for context
    with the lecture's figures, the bus bandwidth in the usual convention
    size * 2(W-1)/W / t."""
    import zero_sharded_adamw_gb300 as z

    rank, world_size, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    init_dist(world_size, "nccl")
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    w = WL.ALLREDUCE_WORKLOADS[args.ar_workload]
    code = z.DTYPE_BF16 if w.dtype == torch.bfloat16 else z.DTYPE_F32
    op = z.OP_AVG if w.average else z.OP_SUM
    ins = WL.allreduce_inputs(w, dev)
    outs = [torch.empty_like(ins[0]) for _ in range(w.world)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        z.zero1_allreduce(w.n, w.world, code, op, ins, outs, err, stream)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local_rank)
    time.sleep(0.3 if clocks.proc else 0.0)
    barrier(world_size)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        z.zero1_allreduce(w.n, w.world, code, op, ins, outs, err, stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world_size)
    t1 = time.time()
    ms = reduce_max(ev0.elapsed_time(ev1), world_size, dev) / args.steps
    clk = clocks.stop(t0, t1)
    assert int(err.item()) == 0, "a kernel pipeline wait gave up"
    size = w.n * ins[0].element_size()
    hbm_bytes = 2 * w.world * size
    peak, peak_kind = measured_peak()
    achieved = hbm_bytes / (ms / 1e3) / 1e9
    line = {
        "metric": "emulated DDP all-reduce HBM GB/s at 1 GPU", "value": world_size * achieved, "unit": "GB/s",
        "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_elements": w.n, "emulated_ranks": w.world,
                   "element": str(w.dtype).replace("torch.", ""), "op": "avg" if w.average else "sum",
                   "l2": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "kernel": "zero1_allreduce_kernel", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": hbm_bytes, "avg_launch_ms": ms, "peak_kind": peak_kind},
        "busbw_gbs": size * 2 * (w.world - 1) / w.world / (ms / 1e3) / 1e9,
        "algbw_gbs": size / (ms / 1e3) / 1e9,
        "clocks": clk, "gpu_launches": args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world_size > 1:
        torch.distributed.destroy_process_group()


def zero2_arm(args, w: WL.Workload):
    """The bucketed (ZeRO-2-style) step overlapped with an emulated backward.

    The backward is emulated as, per bucket of P parameters (last layer
    first), the two GEMMs a layer's backward runs on T tokens (2*T*P flops
    each, bf16 on cuBLAS) on a compute stream; each bucket is handed to
    zero1_bucket_reduce on a second stream as soon as its GEMMs finish, and
    zero1_bucket_finish runs after the backward.  With --bucket-update
    (clipping off in every schedule) each bucket is reduced and updated at
    once by zero1_bucket_update.  Reported: the backward alone, backward +
    zero1_step back to back (the ZeRO-1 schedule), and the overlapped
    schedule; the optimizer time left exposed after the backward is the
    figure of merit."""
    import zero_sharded_adamw_gb300 as z

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    hpd = w.hparams()
    if args.bucket_update:
        hpd["max_norm"] = 0.0                   # an update per bucket needs no global norm
    hp = z.Hparams(**hpd)
    grads = WL.grads(w, 1, dev)
    reps = [torch.empty(w.n, dtype=torch.bfloat16, device=dev) for _ in range(w.world)]
    per_bucket = max(8, (int(args.bucket_mb * 1e6) // 2) // 8 * 8)
    cuts = [(lo, min(per_bucket, w.n - lo)) for lo in range(0, w.n, per_bucket)][::-1]
    d_model = 768
    x = torch.randn(args.tokens, d_model, device=dev, dtype=torch.bfloat16)
    mats = {cnt: torch.randn(d_model, max(128, cnt // d_model // 128 * 128), device=dev, dtype=torch.bfloat16)
            for _, cnt in cuts}
    # --partition K: the device's SMs split into two green contexts, K (or
    # the driver's rounding of it) for the bucket reduces and the rest for
    # the backward, whose persistent GEMMs would otherwise hold every SM.
    part = z.SmPartition(args.partition) if args.partition > 0 else None
    bucket_ctas = part.sms_a if part else args.bucket_ctas
    opt = z.Zero1(w.n, w.world, hp, z.Options(bucket_ctas=bucket_ctas))
    opt.set_state(WL.master(w, dev))
    # Ordinary (non-default) streams: the legacy default stream would
    # serialise against the others.  The optimizer's closing kernel runs on
    # `main` with every SM; the backward runs on `bwd`.
    main = torch.cuda.Stream(dev)
    if part:
        comm = torch.cuda.ExternalStream(part.stream_a, device=dev)
        bwd = torch.cuda.ExternalStream(part.stream_b, device=dev)
    else:
        comm = torch.cuda.Stream(dev, priority=-1)  # bucket reduces get SMs as soon as they free up
        bwd = main

    sleep_cycles = int(args.sleep_us * 1e-6 * 2.07e9)

    def backward_bucket(cnt):
        if args.backward == "sleep":            # a latency-bound backward that holds one SM
            torch.cuda._sleep(sleep_cycles)
            return None
        y = x @ mats[cnt]                       # dgrad-sized GEMM
        return y.t() @ x                        # wgrad-sized GEMM

    def run(mode):
        evs = []
        bwd.wait_stream(main)                   # this iteration's backward follows the last update
        with torch.cuda.stream(bwd):
            for off, cnt in cuts:
                backward_bucket(cnt)
                if mode == "overlap":
                    ev = torch.cuda.Event()
                    ev.record(bwd)
                    evs.append((off, cnt, ev))
        main.wait_stream(bwd)
        if mode == "seq":
            opt.step(grads, reps, main)
        elif mode == "overlap":
            z.zero1_bucket_begin(opt.handle)
            for off, cnt, ev in evs:
                comm.wait_event(ev)
                if args.bucket_update:
                    z.zero1_bucket_update(opt.handle, off, cnt, [g[off:off + cnt] for g in grads],
                                          [r[off:off + cnt] for r in reps], comm)
                else:
                    z.zero1_bucket_reduce(opt.handle, off, cnt, [g[off:off + cnt] for g in grads], comm)
            main.wait_stream(comm)
            z.zero1_bucket_finish(opt.handle, None if args.bucket_update else reps, main)

    out = {}
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(main):
        for mode in ("bwd", "seq", "overlap"):
            for _ in range(args.warmup):
                run(mode)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            for _ in range(args.steps):
                run(mode)
            e1.record(main)
            torch.cuda.synchronize(dev)
            out[mode] = e0.elapsed_time(e1) / args.steps
    opt.close()
    sms = {"bucket_group": part.sms_a, "backward_group": part.sms_b} if part else None
    if part:
        torch.cuda.synchronize(dev)
        part.close()
    line = {
        "metric": "ZeRO-2 bucketed step: optimizer ms exposed after an emulated backward", "value":
            out["overlap"] - out["bwd"], "unit": "ms", "higher_is_better": False, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_params": w.n, "emulated_ranks": w.world, "buckets": len(cuts),
                   "bucket_params": per_bucket, "tokens": args.tokens, "bucket_ctas": bucket_ctas,
                   "sm_partition": sms, "backward": args.backward,
                   "bucket_update": args.bucket_update, "max_norm": hpd["max_norm"],
                   "sleep_us_per_bucket": args.sleep_us if args.backward == "sleep" else None},
        "ms": {"backward_alone": out["bwd"], "backward_then_step": out["seq"], "overlapped": out["overlap"]},
        "exposed_ms": {"zero1_schedule": out["seq"] - out["bwd"], "zero2_overlapped": out["overlap"] - out["bwd"]},
    }
    print(json.dumps(line), flush=True)


def ddp_arm(args, w: WL.Workload):
    """The DDP baseline the ZeRO-1 step is measured against: the bf16
    gradients all-reduced (mean, in place, zero1_allreduce), then every rank
    runs the full AdamW on its own replicated optimizer state (W handles of
    world 1, zero1_step).  Emulated on one GPU the W ranks' work is summed,
    so the figure compares total GPU work and optimizer-state memory:
    DDP holds W copies of master/m/v, ZeRO-1 one sharded copy."""
    import zero_sharded_adamw_gb300 as z

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    hp = z.Hparams(**w.hparams())
    grads = WL.grads(w, 1, dev)
    reps = [torch.empty(w.n, dtype=torch.bfloat16, device=dev) for _ in range(w.world)]
    m0 = WL.master(w, dev)
    ranks = [z.Zero1(w.n, 1, hp, z.Options(small_step=-1)) for _ in range(w.world)]
    for h in ranks:
        h.set_state(m0, stream=stream)
    zero1 = z.Zero1(w.n, w.world, hp)
    zero1.set_state(m0, stream=stream)
    rep_tables = [z.PtrTable([r]) for r in reps]
    grad_tables = [z.PtrTable([g]) for g in grads]
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def ddp_step():
        z.zero1_allreduce(w.n, w.world, z.DTYPE_BF16, z.OP_AVG, grads, grads, err, stream)
        for q, h in enumerate(ranks):
            h.step(grad_tables[q], rep_tables[q], stream)

    def zero1_step():
        zero1.step(grads, reps, stream)

    out = {}
    for name, fn in (("ddp", ddp_step), ("zero1", zero1_step)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = e0.elapsed_time(e1) / args.steps
    assert int(err.item()) == 0, "a kernel pipeline wait gave up"
    state_ddp = sum(h.layout()[2] for h in ranks)
    state_zero1 = zero1.layout()[2]
    for h in ranks + [zero1]:
        h.close()
    line = {
        "metric": "DDP baseline vs ZeRO-1: step ms (all W emulated ranks' work) and optimizer-state bytes",
        "value": out["ddp"], "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_params": w.n, "emulated_ranks": w.world,
                   "ddp": "bf16 all-reduce (mean, in place) + W replicated AdamW updates",
                   "note": "the gradients are overwritten by their mean each step (timing only)"},
        "ms": {"ddp_step": out["ddp"], "zero1_step": out["zero1"]},
        "optimizer_state_bytes": {"ddp_all_ranks": state_ddp, "zero1_all_ranks": state_zero1},
        "gpu_launches": args.steps * (1 + 2 * w.world),
    }
    print(json.dumps(line), flush=True)


def fsdp_arm(args):
    """ZeRO-3 / FSDP forward over the GPT-2-small layers (embeddings + 12
    blocks), W = 8 emulated ranks: each layer's bf16 parameters are sharded
    and all-gathered (zero1_allgather) onto every rank before the layer
    runs.  Schedules: compute alone; gather then compute, layer by layer;
    and prefetch -- layer l+1's gather on a side stream while layer l
    computes, into the other of two staging sets.  The layer compute is
    emulated by a one-SM latency-bound kernel (args.layer_us per layer) or
    by bf16 GEMMs on args.tokens tokens."""
    import zero_sharded_adamw_gb300 as z

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    world = 8
    shapes = WL.gpt2_small_shapes()
    sizes = [shapes[0][0] * shapes[0][1] + shapes[1][0] * shapes[1][1]]
    for b in range(12):
        blk = shapes[2 + 8 * b: 10 + 8 * b]
        sizes.append(sum(int(torch.tensor(s).prod()) for s in blk))
    layers = []
    g = torch.Generator(device=dev).manual_seed(77)
    for p in sizes:
        s = -(-(-(-p // world)) // 8) * 8
        shards = [torch.randn(max(0, min(s, p - r * s)), generator=g, device=dev).to(torch.bfloat16)
                  for r in range(world)]
        layers.append((p, s, shards))
    pmax = max(sizes)
    staging = [[torch.empty(pmax, dtype=torch.bfloat16, device=dev) for _ in range(world)] for _ in range(2)]
    x = torch.randn(args.tokens, 768, device=dev, dtype=torch.bfloat16)
    mats = [torch.randn(768, max(128, p // 768 // 128 * 128), device=dev, dtype=torch.bfloat16) for p in sizes]
    sleep_cycles = int(args.layer_us * 1e-6 * 2.07e9)
    main, side = torch.cuda.Stream(dev), torch.cuda.Stream(dev, priority=-1)

    def compute(l):
        if args.backward == "sleep":
            torch.cuda._sleep(sleep_cycles)
        else:
            y = x @ mats[l]
            y.t() @ x

    def gather(l, buf, stream):
        p, s, shards = layers[l]
        z.zero1_allgather(p, world, s, z.DTYPE_BF16, [t if t.numel() else None for t in shards],
                          staging[buf], None, stream)

    def run(mode):
        if mode == "compute":
            for l in range(len(layers)):
                compute(l)
        elif mode == "gather":
            for l in range(len(layers)):
                gather(l, l % 2, main)
        elif mode == "seq":
            for l in range(len(layers)):
                gather(l, l % 2, main)
                compute(l)
        else:
            done = [torch.cuda.Event() for _ in layers]
            used = [torch.cuda.Event() for _ in layers]
            side.wait_stream(main)
            gather(0, 0, side)
            done[0].record(side)
            for l in range(len(layers)):
                if l + 1 < len(layers):
                    if l >= 1:
                        side.wait_event(used[l - 1])          # staging set (l+1)%2 is free
                    gather(l + 1, (l + 1) % 2, side)
                    done[l + 1].record(side)
                main.wait_event(done[l])
                compute(l)
                used[l].record(main)

    out = {}
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(main):
        for mode in ("compute", "gather", "seq", "prefetch"):
            for _ in range(args.warmup):
                run(mode)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            for _ in range(args.steps):
                run(mode)
            e1.record(main)
            torch.cuda.synchronize(dev)
            out[mode] = e0.elapsed_time(e1) / args.steps
    total = sum(sizes)
    ag_bytes = (1 + world) * 2 * total          # read every shard once, write W full copies
    peak, peak_kind = measured_peak()
    gbs = ag_bytes / (out["gather"] / 1e3) / 1e9
    line = {
        "metric": "FSDP forward: per-layer all-gather ms exposed, gather then compute vs prefetch",
        "value": out["prefetch"] - out["compute"], "unit": "ms", "higher_is_better": False, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "gpt2_small layers (embeddings + 12 blocks)", "n_params": total,
                   "emulated_ranks": world, "layers": len(sizes), "compute": args.backward,
                   "layer_us": args.layer_us if args.backward == "sleep" else None, "tokens": args.tokens},
        "ms": out,
        "exposed_ms": {"gather_then_compute": out["seq"] - out["compute"],
                       "prefetch": out["prefetch"] - out["compute"]},
        "allgather": {"gbs": gbs, "peak": peak, "frac": gbs / peak, "peak_kind": peak_kind,
                      "bytes_per_forward": ag_bytes, "gpu_launches_per_forward": len(sizes)},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    # The metric names no configuration, so the default is the largest
    # workload one GPU holds: 7B parameters of fp32 AdamW state, W = 2.
    ap.add_argument("--workload", default="state_7b", choices=sorted(WL.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="step", choices=["step", "allreduce", "zero2", "fsdp", "ddp"],
                    help="step: the ZeRO-1 optimizer step (default); allreduce: the DDP all-reduce; "
                         "zero2: the bucketed step overlapped with an emulated backward; "
                         "fsdp: per-layer parameter all-gather with prefetch")
    ap.add_argument("--bucket-mb", type=float, default=25.0, help="zero2: bucket size per rank (MB of bf16)")
    ap.add_argument("--tokens", type=int, default=8192, help="zero2: tokens of the emulated backward")
    ap.add_argument("--bucket-ctas", type=int, default=32, help="zero2: CTAs per bucket reduce (0 = one per SM)")
    ap.add_argument("--partition", type=int, default=0,
                    help="zero2: SMs for the bucket reduces; the backward runs on the rest (green contexts)")
    ap.add_argument("--bucket-update", action="store_true",
                    help="zero2: clipping off; reduce and update each bucket at once (zero1_bucket_update)")
    ap.add_argument("--backward", default="gemm", choices=["gemm", "sleep"],
                    help="zero2: emulated backward: bf16 GEMMs, or a one-SM latency-bound kernel per bucket")
    ap.add_argument("--sleep-us", type=float, default=240.0, help="zero2: sleep backward, microseconds per bucket")
    ap.add_argument("--layer-us", type=float, default=150.0, help="fsdp: sleep compute, microseconds per layer")
    ap.add_argument("--ar-workload", default="lecture_fp32_w4", choices=sorted(WL.ALLREDUCE_WORKLOADS))
    ap.add_argument("--n", type=int, default=None,
                    help="override the workload's parameter count (same recipe; small profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="e2e: timed steps per host entry point (0: min(steps, 20))")
    ap.add_argument("--host-chunk", type=int, default=0,
                    help="e2e: parameters per chunk of the host-buffer step (0 = the library's default)")
    ap.add_argument("--grad-sets", type=int, default=2, choices=[1, 2],
                    help="gradient sets used in turn (2: consecutive steps never reuse inputs; 1 halves the "
                         "device footprint, for profiler captures of one launch)")
    ap.add_argument("--moments-bf16", action="store_true", help="variant: m and v stored in bf16")
    ap.add_argument("--decay-first", action="store_true", help="variant: torch.optim.AdamW's decay order")
    ap.add_argument("--clip-eps", type=float, default=0.0, help="variant: clip eps (torch uses 1e-6)")
    ap.add_argument("--load-phase-gbs", type=float, default=0.0,
                    help="update-kernel load phasing: 0 = built-in rule, > 0 = device-wide rate in GB/s, < 0 = off")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capturable handle; also time steps captured in a CUDA graph and replayed")
    ap.add_argument("--graph-steps", type=int, default=20, help="--graph: steps captured per graph")
    ap.add_argument("--small-step", type=int, default=0, choices=[-1, 0, 1],
                    help="one-launch small-n path: 0 automatic, 1 whenever n fits, -1 never")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WL.WORKLOADS[args.workload]
    if args.n is not None:
        w = w.with_n(args.n)
    cfg = {"workload": w.name, "n_params": w.n, "emulated_ranks": w.world,
           "bytes_per_param": 4 * w.world + (16 if args.moments_bf16 else 24), "hparams": w.hparams(),
           "variant": {"moments_bf16": args.moments_bf16, "decay_first": args.decay_first,
                       "clip_eps": args.clip_eps, "small_step": args.small_step, "capturable": args.graph,
                       "load_phase_gbs": args.load_phase_gbs},
           "parallelism": f"zero1 over {w.world} emulated ranks per GPU; GPUs run independent replicas",
           "gradient_sets": args.grad_sets,
           "l2": "inputs larger than L2 (no flush)" if w.bytes_per_step() > 4 * (126 << 20)
                 else "working set fits in L2 (launch-latency bound)"}
    if args.path == "allreduce" and args.impl == "ours":
        allreduce_arm(args)
    elif args.path == "zero2" and args.impl == "ours":
        zero2_arm(args, w)
    elif args.path == "fsdp" and args.impl == "ours":
        fsdp_arm(args)
    elif args.path == "ddp" and args.impl == "ours":
        ddp_arm(args, w)
    elif args.impl == "reference":
        reference_arm(args, w, cfg)
    else:
        ours_arm(args, w, cfg)


if __name__ == "__main__":
    main()
