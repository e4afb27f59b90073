#!/usr/bin/env python
"""Throughput benchmark of the Q8_0 decode matvec on GB300.

One step is one call of the whole path, C = matvec(A, W, S), on the LM head
with a ragged K (K = 4100, N = 128256, the largest decode shape) unless
``--workload`` says otherwise; with ``--rows M`` a step is one batched call of M activation rows
against the same weights, with ``--epilogue ACT`` the call also applies the
fused epilogue C = act(product + bias) + residual as it writes C, and with
``--transposed`` the weights are stored one output row per row (Wt [N, K],
St [N, KB]); ``--a-int8`` (with ``--transposed``) quantizes the activations
to int8 per 32-element block inside the kernel and multiplies with dp4a.  The timed region replays CUDA graphs of back-to-back calls that
rotate over enough distinct copies of the inputs to exceed twice the L2, so
every call streams its weights from HBM.

Printed (rank 0, one JSON line): effective HBM GB/s over the algorithmic
bytes K*N + 4*KB*N + 4*K + 4*N per call, microseconds per call, the roofline
of the kernel against the measured HBM copy bandwidth, the fp64 CPU oracle
timed on the host cores (one core, and every core of the affinity mask), an
end-to-end figure with host buffers, the SM clocks seen during the timed
region, the number of kernel launches and, under ``per_config``, the same
timing (microseconds per call, GB/s, fraction of the peak, plan, and the
oracle on one core) for every decode shape.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload attn]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

With N > 1 (under torchrun) every rank runs an independent replica on its own
GPU: the matvec has no exchange step, so there is no collective on the data
path; the process group only provides the barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "Q8_0 matvec effective HBM GB/s and % of GB300 peak; µs per call"
UNIT = "GB/s"
CSRC = os.path.join(ROOT, "q8_matrix_vector_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
GRAPH_CALLS = 1000  # calls captured per CUDA graph (rounded to the rotation length)
CPU_BASELINE_SECONDS = 8.0        # single-thread oracle on the headline workload
CPU_ALL_CORES_SECONDS = 4.0       # the oracle on every core of the affinity mask
PER_CONFIG_ORACLE_SECONDS = 0.6   # single-thread oracle sample per config
PER_CONFIG_TARGET_S = 0.03        # device time of one timed repetition per config


# ----------------------------------------------------------------------------
# process group (replicas only: barrier and max/sum over ranks)
# ----------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local_rank, world


def init_group(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(group):
    if group is not None:
        group.barrier()


def reduce_over_ranks(group, value: float, op: str, device=None) -> float:
    """max or sum of a float over all ranks (the identity with one rank)."""
    if group is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    group.all_reduce(t, op=group.ReduceOp.MAX if op == "max" else group.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------
# peaks, clocks, profile data
# ----------------------------------------------------------------------------
def read_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name: str) -> str:
    with open(os.path.join(CSRC, name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


KERNEL_NAMES = {1: "regs", 2: "stream", 4: "rows", 5: "rows_i8", 6: "mma", 7: "tc"}


def traffic_key(workload: str, rows: int, transposed: bool = False, a_int8: bool = False, kernel: int = 1) -> str:
    """Key of a recorded ncu capture: workload, activation rows (or the
    transposed layout) and, for batched calls, the kernel that ran."""
    if transposed:
        return f"{workload}_t" + ("8" if a_int8 else "")
    if rows == 1:
        return f"{workload}_stream" if kernel == 2 else workload
    return f"{workload}_m{rows}_{KERNEL_NAMES.get(kernel, str(kernel))}"


def launches_per_call(info) -> int:
    """Kernels one call launches: the tcgen05 path splits the activations into
    bf16 parts first."""
    return 2 if info.get("kernel") == 7 else 1


def recorded_traffic(key: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("workloads", {}).get(key)
    if not entry:
        return None
    try:
        if kernel_source_hash(entry["kernel_source"]) != entry["kernel_source_sha256"]:
            return None
    except (OSError, KeyError):
        return None
    return entry.get("dram_bytes_per_launch")


CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let it start before the timed region
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(text: str):
    sm, sm_max, power = [], [], []
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) != len(CLOCK_FIELDS):
            continue
        try:
            sm.append(float(parts[1]))
            sm_max.append(float(parts[2]))
            power.append(float(parts[3]))
        except ValueError:
            continue
        for name, val in zip(names, parts[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(sm_max), "samples": len(sm),
            "power_w_max": max(power), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, rank, local_rank, world):
    import numpy as np
    import torch

    import q8_matrix_vector_gb300 as q8mv

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the q8mv arm")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    group = init_group(world, "nccl")
    wl = workloads.WORKLOADS[args.workload]
    if args.limit_k:
        # the workload's recipe (distributions, seed, N) at a smaller K: a smaller case for profiling
        wl = dataclasses.replace(wl, K=args.limit_k, name=f"{wl.name}_k{args.limit_k}",
                                 description=f"{wl.description}, drawn at K={args.limit_k} instead")
    K, N, KB = wl.K, wl.N, wl.KB
    M = args.rows
    bytes_per_call = workloads.batched_bytes(K, N, M)
    fused = args.epilogue != "none"
    if fused:
        bytes_per_call += 4 * N + 4 * M * N  # bias and residual read once per call

    A, W, S = workloads.make_inputs(wl)
    if M > 1:
        A = workloads.make_rows(wl, M)
    if args.transposed:
        W, S = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    bias_h, res_h = epilogue_inputs(N, M) if fused else (None, None)
    kernel = {"auto": q8mv.KERNEL_AUTO, "regs": q8mv.KERNEL_REGS, "stream": q8mv.KERNEL_STREAM,
              "mma": q8mv.KERNEL_MMA,
              "tc": q8mv.KERNEL_TC}[args.kernel]
    overlap = not args.no_overlap
    plan_opts = dict(kernel=kernel, split_k=args.split, stages=args.stages, threads_n=args.threads_n,
                     cta_threads=args.cta_threads, vec_bytes=args.vec_bytes)
    if args.transposed:
        plan_opts = dict(kernel=q8mv.KERNEL_ROWS_I8 if args.a_int8 else 0)
    plan = q8mv.Plan(K, N, device=local_rank, rows=M, transposed=args.transposed, overlap=int(overlap), **plan_opts)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0)) or 126 * 1024 * 1024
    # distinct copies so that a copy is reused only after > 2 x L2 of other traffic
    copies = max(2, math.ceil(2 * l2 / bytes_per_call) + 1)
    Ah, Wh, Sh = torch.from_numpy(A), torch.from_numpy(W), torch.from_numpy(S)
    bufs = []
    for _ in range(copies):
        bufs.append((Ah.to(dev), Wh.to(dev), Sh.to(dev), torch.empty((M, N), dtype=torch.float32, device=dev)))
    ptrs = [(a.data_ptr(), w.data_ptr(), s.data_ptr(), c.data_ptr()) for a, w, s, c in bufs]
    epis = None
    if fused:
        epi_bufs = [(torch.from_numpy(bias_h).to(dev), torch.from_numpy(res_h).to(dev)) for _ in range(copies)]
        epis = [q8mv.Epilogue(1.0, 0.0, b.data_ptr(), r.data_ptr(), EPILOGUE_ACTS[args.epilogue])
                for b, r in epi_bufs]
    launch = make_launcher(plan, ptrs, epis)
    stream = torch.cuda.Stream(dev)

    # warm-up steps (eager launches through the C library)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(i, stream.cuda_stream)
    stream.synchronize()

    # graphs of back-to-back calls; the rotation restarts at copy 0 in each graph
    chunk = max(copies, (min(GRAPH_CALLS, max(args.steps, 1)) // copies) * copies)
    full, rest = divmod(args.steps, chunk)

    def capture(ncalls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s = torch.cuda.current_stream().cuda_stream
            for i in range(ncalls):
                launch(i, s)
        return g

    g_full = capture(chunk) if full else None
    g_rest = capture(rest) if rest else None
    with torch.cuda.stream(stream):  # one untimed replay uploads the graphs
        if g_full:
            g_full.replay()
        if g_rest:
            g_rest.replay()
    stream.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(group)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rest:
            g_rest.replay()
        end.record(stream)
    end.synchronize()
    wall = time.perf_counter() - wall0
    torch.cuda.synchronize(dev)
    barrier(group)
    clocks = sampler.stop()
    ms = start.elapsed_time(end)
    ms_max = reduce_over_ranks(group, ms, "max", dev)
    total_bytes = reduce_over_ranks(group, float(bytes_per_call) * args.steps, "sum", dev)
    value = total_bytes / (ms_max * 1e-3) / 1e9 if ms_max > 0 else 0.0

    # roofline of the call (for the tcgen05 path: its parts kernel and product kernel)
    per_launch_s = ms * 1e-3 / max(args.steps, 1)
    achieved = bytes_per_call / per_launch_s / 1e9 if per_launch_s > 0 else 0.0
    peak, peak_kind = read_hbm_peak()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} copy bandwidth",
                "traffic": recorded_traffic(traffic_key(args.workload, M, args.transposed, args.a_int8,
                                                        plan.info["kernel"])),
                "algorithmic_bytes_per_launch": bytes_per_call}

    # end to end through the public binding: pinned host inputs in, result out
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    Ap, Wp, Sp = Ah.pin_memory(), Wh.pin_memory(), Sh.pin_memory()
    Cp = torch.empty((M, N), dtype=torch.float32).pin_memory()
    Ad, Wd, Sd, Cd = bufs[0]
    epi_kw, epi_copies = {}, []
    if fused:
        bias_p, res_p = torch.from_numpy(bias_h).pin_memory(), torch.from_numpy(res_h).pin_memory()
        bias_d, res_d = epi_bufs[0]
        epi_copies = [(bias_d, bias_p), (res_d, res_p)]
        epi_kw = dict(bias=bias_d, residual=res_d, act=args.epilogue)
    with torch.cuda.stream(stream):
        for _ in range(2):  # warm-up
            Ad.copy_(Ap, non_blocking=True)
            Wd.copy_(Wp, non_blocking=True)
            Sd.copy_(Sp, non_blocking=True)
            for dst, src in epi_copies:
                dst.copy_(src, non_blocking=True)
            plan(Ad, Wd, Sd, out=Cd, stream=stream, **epi_kw)
            Cp.copy_(Cd, non_blocking=True)
    stream.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier(group)
    with torch.cuda.stream(stream):
        e_start.record(stream)
        for _ in range(e2e_steps):
            Ad.copy_(Ap, non_blocking=True)
            Wd.copy_(Wp, non_blocking=True)
            Sd.copy_(Sp, non_blocking=True)
            for dst, src in epi_copies:
                dst.copy_(src, non_blocking=True)
            plan(Ad, Wd, Sd, out=Cd, stream=stream, **epi_kw)
            Cp.copy_(Cd, non_blocking=True)
        e_end.record(stream)
    e_end.synchronize()
    e_ms = reduce_over_ranks(group, e_start.elapsed_time(e_end), "max", dev)
    e_bytes = reduce_over_ranks(group, float(bytes_per_call) * e2e_steps, "sum", dev)
    h2d = 4 * M * K + K * N + 4 * KB * N + ((4 * N + 4 * M * N) if fused else 0)
    e2e = {"value": round(e_bytes / (e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * M * N, "steps": e2e_steps,
           "what": "pinned host A, W, S" + (", bias, residual" if fused else "")
                   + " copied in, " + ("q8mv_run_fused" if fused else "q8mv_run") + ", C copied out, every step"}

    # the same workload with plain launches, for comparison with the overlapped headline
    plain = None
    if overlap:
        plan_plain = q8mv.Plan(K, N, device=local_rank, rows=M, transposed=args.transposed, overlap=0, **plan_opts)
        us_plain = time_calls(plan_plain, ptrs, stream, min(args.steps, 20000), epis=epis)
        pinfo = plan_plain.info
        plain = {"us_per_call": round(us_plain, 3), "value": round(bytes_per_call / us_plain / 1e3, 2),
                 "unit": UNIT, "what": "same workload and timing, launched without programmatic dependent launch",
                 "plan": {k: pinfo[k] for k in ("vec_bytes", "threads_per_cta", "threads_n", "split_k", "cluster",
                                                "grid_x", "grid_y")}}
        plan_plain.close()

    table = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del bufs, ptrs, epis, launch, g_full, g_rest
        torch.cuda.empty_cache()
        have = (args.workload, (A, W, S)) if (M == 1 and not args.transposed) else None
        table = per_config(q8mv, dev, local_rank, stream, l2, peak, overlap, have)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(A, W, S, bytes_per_call, args.cpu_seconds, wl, M,
                           (bias_h, res_h, EPILOGUE_ACTS[args.epilogue]) if fused else None, args.transposed,
                           args.a_int8, all_core_seconds=args.all_core_seconds)

    if rank != 0:
        return None
    info = plan.info
    us = ms * 1e3 / max(args.steps, 1)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / max(args.steps, 1), 6),
        "us_per_call": round(us, 3), "pct_of_peak": round(100.0 * achieved / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.description}" + (f", batched decode of M={M} rows" if M > 1 else "")
                               + (f", fused epilogue act({args.epilogue})(x + bias) + residual" if fused else "")
                               + (", weights stored one output row per row" if args.transposed else "")
                               + (", int8 activations (dp4a)" if args.a_int8 else ""),
                   "K": K, "N": N, "KB": KB, "M": M, "epilogue": args.epilogue,
                   "layout": "Wt [N,K], St [N,KB]" if args.transposed else "W [K,N], S [KB,N]",
                   "weights": "Q8_0: int8 W [K,N], f32 scales [KB,N], f32 A [M,K] and C [M,N]",
                   "bytes_per_call": bytes_per_call,
                   "l2": f"inputs larger than L2: {copies} rotating input copies "
                         f"({copies * bytes_per_call / 1e6:.0f} MB) vs {l2 / 1e6:.0f} MB L2",
                   "timing": f"CUDA events around graph replays of {chunk} back-to-back calls"
                             + (", programmatic dependent launch (each call reads A and writes C only after the "
                                "previous call completes)" if overlap else ""),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "plan": {k: info[k] for k in ("kernel", "vec_bytes", "threads_per_cta", "threads_n",
                                                 "groups_k", "split_k",
                                                 "blocks_per_split", "stages", "overlap", "cluster",
                                                 "grid_x", "grid_y", "ctas_per_sm", "rows_per_pass",
                                                 "grid_z")}},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "plain_launch": plain,
        "clocks": clocks,
        "gpu_launches": args.steps * launches_per_call(plan.info),
        "wall_s_timed_region": round(wall, 4),
        "per_config": table,
    }


EPILOGUE_ACTS = {"none": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}

PAIR_UP, PAIR_DOWN = "ffn_up", "ffn_down"


def run_pair(args, rank, local_rank, world):
    """``--pair``: one step is the 7B FFN pair through q8mv_pair_run,
    H = silu(A . W_up + bias) then C = H . W_down + residual, in the default
    mode (two launches chained by programmatic dependent launch) and, for
    comparison, the one-launch pair kernel.  Bytes: both products' algorithmic
    bytes plus the bias and the residual."""
    import numpy as np
    import torch

    import q8_matrix_vector_gb300 as q8mv

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the q8mv arm")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    group = init_group(world, "nccl")
    up, down = workloads.WORKLOADS[PAIR_UP], workloads.WORKLOADS[PAIR_DOWN]
    K, Nm, No = up.K, up.N, down.N
    bytes_per_step = up.algorithmic_bytes() + down.algorithmic_bytes() + 4 * Nm + 4 * No
    A, Wu, Su = workloads.make_inputs(up)
    _, Wd, Sd = workloads.make_inputs(down)
    rng = np.random.Generator(np.random.PCG64(2024))
    bias = rng.standard_normal(Nm).astype(np.float32)
    residual = (20.0 * rng.standard_normal(No)).astype(np.float32)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 126 * 1024 * 1024
    copies = max(2, math.ceil(2 * l2 / bytes_per_step) + 1)
    host = [torch.from_numpy(x) for x in (A.reshape(1, K), Wu, Su, Wd, Sd, bias, residual.reshape(1, No))]
    bufs = [[t.to(dev) for t in host] + [torch.empty((1, Nm), device=dev), torch.empty((1, No), device=dev)]
            for _ in range(copies)]
    stream = torch.cuda.Stream(dev)

    def make(mode):
        pair = q8mv.Pair(K, Nm, No, device=local_rank, overlap=0 if args.no_overlap else 1, mode=mode)
        calls = []
        for Ad, Wud, Sud, Wdd, Sdd, bd, rd, Hd, Cd in bufs:
            eu = q8mv.Epilogue(1.0, 0.0, bd.data_ptr(), None, q8mv.ACT_SILU)
            ed = q8mv.Epilogue(1.0, 0.0, None, rd.data_ptr(), q8mv.ACT_NONE)
            calls.append((Ad.data_ptr(), Wud.data_ptr(), Sud.data_ptr(), Hd.data_ptr(), Wdd.data_ptr(),
                          Sdd.data_ptr(), Cd.data_ptr(), eu, ed))

        def launch(i, st):
            pair.run_ptr(*calls[i % copies][:7], calls[i % copies][7], calls[i % copies][8], st)
        return pair, launch

    def timed(launch, steps, sample_clocks):
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                launch(i, stream.cuda_stream)
        stream.synchronize()
        chunk = max(copies, (min(GRAPH_CALLS, max(steps, 1)) // copies) * copies)
        full, rest = divmod(steps, chunk)
        graphs = []
        for n in ([chunk] if full else []) + ([rest] if rest else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                cs = torch.cuda.current_stream().cuda_stream
                for i in range(n):
                    launch(i, cs)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(group)
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local_rank) if sample_clocks else None
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(full):
                graphs[0].replay()
            if rest:
                graphs[-1].replay()
            e1.record(stream)
        e1.synchronize()
        barrier(group)
        clocks = sampler.stop() if sampler else None
        return reduce_over_ranks(group, e0.elapsed_time(e1), "max", dev), chunk, clocks

    pair, launch = make(q8mv.PAIR_AUTO)
    ms, chunk, clocks = timed(launch, args.steps, True)
    pair1, launch1 = make(q8mv.PAIR_ONE_LAUNCH)
    ms1, _, _ = timed(launch1, args.steps, False)
    for p in (pair, pair1):
        if p.check() != 0:
            raise RuntimeError("pair kernel recorded a device error")
    if rank != 0:
        return None
    steps = max(args.steps, 1)
    us, us1 = ms * 1e3 / steps, ms1 * 1e3 / steps
    value = world * bytes_per_step * steps / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
    peak, peak_kind = read_hbm_peak()
    achieved = bytes_per_step / (us * 1e-6) / 1e9
    info1 = pair1.info
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / steps, 6),
        "us_per_call": round(us, 3), "pct_of_peak": round(100.0 * achieved / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"ffn_pair: {up.description} (SiLU + bias) then {down.description} (+ residual), "
                               "q8mv_pair_run",
                   "K": K, "N_mid": Nm, "N_out": No, "bytes_per_call": bytes_per_step,
                   "l2": f"inputs larger than L2: {copies} rotating input copies "
                         f"({copies * bytes_per_step / 1e6:.0f} MB) vs {l2 / 1e6:.0f} MB L2",
                   "timing": f"CUDA events around graph replays of {chunk} back-to-back pair calls"
                             + ("" if args.no_overlap else ", programmatic dependent launch"),
                   "mode": "two launches (the default)", "parallelism": "single GPU" if world == 1 else
                   f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} copy bandwidth",
                     "traffic": None, "algorithmic_bytes_per_launch": bytes_per_step},
        "one_launch": {"us_per_call": round(us1, 3), "value": round(bytes_per_step / us1 / 1e3, 2), "unit": UNIT,
                       "plan": {k: info1[k] for k in ("threads_per_cta", "grid", "ctas_per_sm", "split_up",
                                                      "split_down")}},
        "cpu_baseline": None, "e2e": None, "clocks": clocks,
        "gpu_launches": args.steps * 2,
    }


def epilogue_inputs(N, M):
    """Seeded bias [N] and residual [M, N] for a fused-epilogue run."""
    import numpy as np

    rng = np.random.Generator(np.random.PCG64(4242))
    return (rng.standard_normal(N).astype(np.float32),
            np.ascontiguousarray(rng.standard_normal((M, N)).astype(np.float32)))


def make_launcher(plan, ptrs, epis=None):
    """launch(i, stream): call i of the rotation, with its epilogue if any."""
    copies = len(ptrs)
    if epis is None:
        return lambda i, s: plan.run_ptr(*ptrs[i % copies], s)
    return lambda i, s: plan.run_fused_ptr(*ptrs[i % copies], epis[i % copies], s)


def time_calls(plan, ptrs, stream, calls, reps=3, epis=None):
    """Microseconds per call of back-to-back graph-captured calls (best of reps)."""
    import torch

    copies = len(ptrs)
    launch = make_launcher(plan, ptrs, epis)
    chunk = max(copies, (min(GRAPH_CALLS, calls) // copies) * copies)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        s = torch.cuda.current_stream().cuda_stream
        for i in range(chunk):
            launch(i, s)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    replays = max(1, calls // chunk)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (replays * chunk)
        best = us if best is None else min(best, us)
    return best


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def affinity_cores():
    """The cores this process may run on."""
    if hasattr(os, "sched_getaffinity"):
        return sorted(os.sched_getaffinity(0))
    return list(range(os.cpu_count() or 1))


def oracle_product(orc, M=1, transposed=False, a_int8=False):
    """The oracle function of the path being timed: (A, W, S) -> (C, bound)."""
    if a_int8:
        return lambda A, W, S: orc.i8(*orc.quantize(A.reshape(-1)), W, S)
    if transposed:
        return orc.transposed
    return orc.factored if M == 1 else orc.batched


def cpu_baseline(A, W, S, bytes_per_call, seconds, wl, M=1, epilogue=None, transposed=False, a_int8=False,
                 all_core_seconds=CPU_ALL_CORES_SECONDS):
    """The fp64 oracle, as it stands, on the host cores: full calls on one
    core for ~seconds, then the same workload split by output columns over one
    process per core of the affinity mask (``cores`` counts those processes)."""
    import oracle

    orc = oracle.load()
    product = oracle_product(orc, M, transposed, a_int8)
    if epilogue is None:
        def run():
            product(A, W, S)
    else:
        bias, residual, act = epilogue

        def run():
            orc.epilogue(product(A, W, S)[0], bias=bias, residual=residual, act=act)
    run()  # page in
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    rows = "" if M == 1 else f" of M={M} rows"
    single = {"value": round(reps * bytes_per_call / dt / 1e9, 4), "unit": UNIT, "cores": 1,
              "sample": f"{reps} full {wl.name} calls{rows} (K={wl.K}, N={wl.N}) in {dt:.1f} s, fp64"}
    model = cpu_model()
    multi = None
    if all_core_seconds > 0 and epilogue is None:
        try:
            multi = cpu_all_cores(A, W, S, wl, M, all_core_seconds, transposed, a_int8)
        except Exception as exc:  # noqa: BLE001  (report, do not lose the run)
            multi = {"error": f"{type(exc).__name__}: {exc}"}
    if multi and "value" in multi:
        return {"value": multi["value"], "unit": UNIT, "cores": multi["cores"], "kind": "oracle",
                "cpu_model": model,
                "sample": multi["sample"], "single_thread": single}
    out = dict(single)
    out.update({"kind": "oracle", "cpu_model": model})
    if multi:
        out["all_cores"] = multi
    return out


def _oracle_chunk_worker(chunk, M, transposed, a_int8, seconds, core, barrier, out_q):
    """One core's share of the all-core oracle run: the columns in ``chunk``
    (A, W columns, S columns, bytes per call), repeated for ``seconds`` after
    every worker is ready."""
    try:
        if hasattr(os, "sched_setaffinity"):
            os.sched_setaffinity(0, {core})
        import oracle

        A, Wc, Sc, nbytes = chunk
        product = oracle_product(oracle.load(), M, transposed, a_int8)
        product(A, Wc, Sc)  # page in
        barrier.wait(timeout=600)
        reps, t0 = 0, time.perf_counter()
        while True:
            product(A, Wc, Sc)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= seconds:
                break
        out_q.put((reps * nbytes, dt, reps))
    except Exception as exc:  # noqa: BLE001
        out_q.put(("error", repr(exc), 0))
        try:
            barrier.abort()
        except Exception:  # noqa: BLE001
            pass


def cpu_all_cores(A, W, S, wl, M, seconds, transposed=False, a_int8=False):
    """The unchanged single-thread oracle in one spawned process per core of
    the affinity mask, each on its own contiguous range of output columns;
    throughput = the bytes all processes finished / the longest run."""
    import multiprocessing as mp

    import numpy as np

    cores = affinity_cores()
    P = len(cores)
    N = W.shape[0] if transposed else W.shape[1]
    K = wl.K
    KB = wl.KB
    P = max(1, min(P, N))
    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    barrier = ctx.Barrier(P)
    out_q = ctx.Queue()
    procs = []
    for i in range(P):
        c0, c1 = N * i // P, N * (i + 1) // P
        if transposed:
            Wc, Sc = np.ascontiguousarray(W[c0:c1]), np.ascontiguousarray(S[c0:c1])
        else:
            Wc, Sc = np.ascontiguousarray(W[:, c0:c1]), np.ascontiguousarray(S[:, c0:c1])
        nc = c1 - c0
        # this process's columns of W, S and C, and its share of A
        nbytes = K * nc + 4 * KB * nc + 4 * M * nc + 4 * M * K * nc / N
        proc = ctx.Process(target=_oracle_chunk_worker,
                           args=((A, Wc, Sc, nbytes), M, transposed, a_int8, seconds, cores[i], barrier, out_q))
        proc.start()
        procs.append(proc)
        del Wc, Sc
    import queue

    results = []
    deadline = time.monotonic() + seconds + 600
    try:
        while len(results) < P:
            try:
                results.append(out_q.get(timeout=1.0))
            except queue.Empty:
                dead = [proc for proc in procs if proc.exitcode not in (None, 0)]
                if dead:
                    raise RuntimeError(f"oracle worker exited with code {dead[0].exitcode}")
                if time.monotonic() > deadline:
                    raise RuntimeError("oracle workers did not finish in time")
    finally:
        for proc in procs:
            proc.join(timeout=60)
            if proc.is_alive():
                proc.kill()
    errors = [r for r in results if r[0] == "error"]
    if errors:
        raise RuntimeError(errors[0][1])
    total = sum(r[0] for r in results)
    longest = max(r[1] for r in results)
    calls = sum(r[2] for r in results) / P
    return {"value": round(total / longest / 1e9, 4), "unit": UNIT, "cores": P,
            "sample": f"{wl.name} (K={wl.K}, N={wl.N}" + (f", M={M} rows" if M > 1 else "")
                      + f") split by output columns over {P} processes, one per core, "
                      f"about {calls:.1f} passes over its columns each in {longest:.1f} s, fp64"}


def oracle_sample_gbs(A, W, S, wl, seconds):
    """The oracle on one core over a column sample of workload ``wl`` for
    about ``seconds``: (GB/s, columns in the sample)."""
    import numpy as np

    import oracle

    orc = oracle.load()
    n_s = wl.N
    t0 = time.perf_counter()
    orc.factored(A, np.ascontiguousarray(W[:, :min(n_s, 256)]), np.ascontiguousarray(S[:, :min(n_s, 256)]))
    t_256 = max(time.perf_counter() - t0, 1e-6)
    # about a fifth of the budget per call
    n_s = int(max(16, min(wl.N, 256 * (seconds / 5) / t_256)))
    Ws, Ss = np.ascontiguousarray(W[:, :n_s]), np.ascontiguousarray(S[:, :n_s])
    orc.factored(A, Ws, Ss)
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.factored(A, Ws, Ss)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return reps * workloads.batched_bytes(wl.K, n_s, 1) / dt / 1e9, n_s


def per_config(q8mv, dev, local_rank, stream, l2, peak, overlap, have=None, oracle_seconds=PER_CONFIG_ORACLE_SECONDS):
    """Every decode shape of ``workloads.ORDER`` with its default plan, timed
    like the headline (back-to-back graph replays over rotating input copies
    beyond twice the L2, best of three repetitions), with the oracle on one
    core over a column sample of the same inputs next to it."""
    import torch

    table = {}
    for name in workloads.ORDER:
        wl = workloads.WORKLOADS[name]
        if have is not None and have[0] == name:
            A, W, S = have[1]
        else:
            A, W, S = workloads.make_inputs(wl)
        nbytes = wl.algorithmic_bytes()
        plan = q8mv.Plan(wl.K, wl.N, device=local_rank, overlap=int(overlap))
        copies = max(2, math.ceil(2 * l2 / nbytes) + 1)
        Ah, Wh, Sh = torch.from_numpy(A), torch.from_numpy(W), torch.from_numpy(S)
        bufs = [(Ah.to(dev), Wh.to(dev), Sh.to(dev), torch.empty((1, wl.N), dtype=torch.float32, device=dev))
                for _ in range(copies)]
        ptrs = [(a.data_ptr(), w.data_ptr(), s.data_ptr(), c.data_ptr()) for a, w, s, c in bufs]
        # about PER_CONFIG_TARGET_S of device time per repetition (launch-bound
        # shapes counted at 3 us a call)
        est = max(nbytes / (0.8 * peak * 1e9), 3e-6)
        calls = int(min(20000, max(200, PER_CONFIG_TARGET_S / est)))
        us = time_calls(plan, ptrs, stream, calls)
        info = plan.info
        plan.close()
        del bufs, ptrs
        gbs = nbytes / us / 1e3
        cpu_gbs, n_s = oracle_sample_gbs(A, W, S, wl, oracle_seconds)
        table[name] = {
            "K": wl.K, "N": wl.N, "bytes_per_call": nbytes, "us_per_call": round(us, 3),
            "gb_s": round(gbs, 1), "frac": round(gbs / peak, 4), "calls_timed": calls,
            "plan": {k: info[k] for k in ("kernel", "vec_bytes", "threads_per_cta", "threads_n", "split_k",
                                          "cluster", "grid_x", "grid_y", "stages")},
            "oracle_1core_gb_s": round(cpu_gbs, 4),
            "oracle_sample": f"first {n_s} of {wl.N} columns, one core, fp64",
        }
        torch.cuda.empty_cache()
    return table


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle on the same workload and metric
# ----------------------------------------------------------------------------
def run_reference(args, rank, world):
    import numpy as np

    import oracle

    if rank != 0:
        return None  # rank 0 alone runs the reference arm
    wl = workloads.WORKLOADS[args.workload]
    M = args.rows
    A, W, S = workloads.make_inputs(wl)
    orc = oracle.load()
    if M > 1:
        A = workloads.make_rows(wl, M)
        product = orc.batched
    else:
        product = orc.factored
    if args.transposed:
        W, S = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
        product = orc.transposed
    if args.a_int8:
        def product(A, W, S):
            return orc.i8(*orc.quantize(A.reshape(-1)), W, S)
    fused = args.epilogue != "none"
    bias_h, res_h = epilogue_inputs(wl.N, M) if fused else (None, None)
    act = EPILOGUE_ACTS[args.epilogue]

    def call(A, W, S):
        x = product(A, W, S)[0]
        if fused:
            n = W.shape[0] if args.transposed else W.shape[1]
            orc.epilogue(x, bias=bias_h[:n], residual=np.ascontiguousarray(res_h[:, :n]), act=act)

    t0 = time.perf_counter()
    call(A, W, S)
    t_full = time.perf_counter() - t0
    # each step is a bounded sample of the workload: the first n_s columns
    budget = args.reference_seconds
    total_steps = args.steps + args.warmup
    n_s = wl.N
    if total_steps * t_full > budget:
        n_s = max(1, int(wl.N * budget / (total_steps * t_full)))
    if args.transposed:
        Ws, Ss = np.ascontiguousarray(W[:n_s]), np.ascontiguousarray(S[:n_s])
    else:
        Ws, Ss = np.ascontiguousarray(W[:, :n_s]), np.ascontiguousarray(S[:, :n_s])
    step_bytes = workloads.batched_bytes(wl.K, n_s, M) + ((4 * n_s + 4 * M * n_s) if fused else 0)
    for _ in range(args.warmup):
        call(A, Ws, Ss)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        call(A, Ws, Ss)
    dt = time.perf_counter() - t0
    value = args.steps * step_bytes / dt / 1e9 if dt > 0 else 0.0
    sample = (f"first {n_s} of {wl.N} columns of {wl.name} (K={wl.K}"
              + (f", M={M} rows" if M > 1 else "") + (f", epilogue {args.epilogue}" if fused else "")
              + ") per step, fp64 oracle, single thread")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.description}" + (f", batched decode of M={M} rows" if M > 1 else "")
                               + (f", fused epilogue act({args.epilogue})(x + bias) + residual" if fused else "")
                               + (", weights stored one output row per row" if args.transposed else "")
                               + (", int8 activations (dp4a)" if args.a_int8 else ""),
                   "K": wl.K, "N": wl.N, "KB": wl.KB, "M": M, "epilogue": args.epilogue},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default=workloads.HEADLINE)
    ap.add_argument("--rows", type=int, default=1,
                    help="activation rows per call (batched decode; 1 = the single-row matvec)")
    ap.add_argument("--epilogue", choices=sorted(EPILOGUE_ACTS), default="none",
                    help="fused epilogue: C = act(product + bias) + residual as C is written")
    ap.add_argument("--transposed", action="store_true",
                    help="weights stored one output row per row: Wt [N, K], St [N, KB] (dot_t layout)")
    ap.add_argument("--a-int8", action="store_true",
                    help="with --transposed: int8 activations per 32-element block, dp4a products")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=CPU_BASELINE_SECONDS)
    ap.add_argument("--reference-seconds", type=float, default=60.0,
                    help="CPU budget of the reference arm's timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-core-seconds", type=float, default=CPU_ALL_CORES_SECONDS,
                    help="seconds of the all-core oracle run in the CPU baseline (0 = single thread only)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config table (every decode shape with its default plan)")
    ap.add_argument("--kernel", choices=["auto", "regs", "stream", "mma", "tc"], default="auto",
                    help="plan override: kernel family (default: the plan's choice)")
    ap.add_argument("--split", type=int, default=0, help="plan override: K ranges per column tile")
    ap.add_argument("--stages", type=int, default=0, help="plan override: streaming kernel ring depth")
    ap.add_argument("--threads-n", type=int, default=0, help="plan override: threads along N per CTA")
    ap.add_argument("--cta-threads", type=int, default=0, help="plan override: threads per CTA (128 or 256)")
    ap.add_argument("--vec-bytes", type=int, default=0, help="plan override: widest weight load per thread and row")
    ap.add_argument("--limit-k", type=int, default=0,
                    help="draw the workload at K = LIMIT_K instead (a smaller case of the same recipe, for profiling)")
    ap.add_argument("--pair", action="store_true",
                    help="time the 7B FFN pair (up with SiLU + bias, down with residual) through q8mv_pair_run")
    ap.add_argument("--no-overlap", action="store_true",
                    help="plain launches instead of programmatic dependent launch (the plan's overlap option, "
                         "on by default: decode weights are constant across calls)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.limit_k < 0:
        ap.error("--limit-k must be positive")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if not 1 <= args.rows <= 1 << 19:
        ap.error("--rows must be in 1 .. 2^19")
    if args.transposed and args.rows != 1:
        ap.error("--transposed takes one activation row")
    if args.a_int8 and not args.transposed:
        ap.error("--a-int8 needs --transposed (weights stored one output row per row)")
    return args


def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if world != args.gpus and args.gpus != 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.pair:
        line = run_pair(args, rank, local_rank, world)
    else:
        line = run_ours(args, rank, local_rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
