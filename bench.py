#!/usr/bin/env python3
"""Throughput of the CP ring-attention hot path on GB300 GPUs.

One step = one pass of the hot path over one packed THD micro-batch: the
dynamic-CP plan (``cpattn_plan``, host) and the ring-attention forward with the
online-softmax merge fused (``cpattn_fwd``), on the 16,384-token packed batch
(lognormal lengths, world 4, per-rank limit 4096, CP sizes from {1, 2, 4},
H=32, D=128, causal).  ``value`` is attention TFLOP/s (4 * H * D per visible
query/key pair) over all GPUs; every GPU runs its own independent batch
(seed + rank), so scaling is weak and there is no collective on the data path.

The same JSON line also reports: ``e2e`` (host buffers, copies in the timed
region), the attention kernel's roofline, the float64 CPU oracle timed on a
bounded sample (``cpu_baseline``), GPU clocks during the timed regions, and
sub-measurements of the 131,072-token CP=4 sequence, the unfused path and the
CP=8 merge of stored partials.

``--impl reference`` times the oracle itself on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("causal ring-attn fwd TFLOP/s (% bf16 peak) on THD batches; "
          "merge GB/s (% HBM)")
WORKLOAD = "packed16k"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cpattn", choices=["cpattn", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the 128K, unfused and merge sub-measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nvtx", action="store_true",
                    help="NVTX ranges around the library calls and each measurement "
                         "(for profilers that filter by range)")
    ap.add_argument("--small", action="store_true",
                    help="profiling aid: the long-sequence forward and backward (one "
                         "32768-token sequence), merge, dcp, decode and ulysses measurements on "
                         "smaller inputs (each array still larger than L2); not a benchmark "
                         "configuration")
    ap.add_argument("--only", default=None,
                    choices=[None, "main", "long128k", "merge8", "backward", "dcp", "decode",
                             "ulysses", "sweep256", "seeds", "dcp_sweep256"],
                    help="run one measurement only (for profiling)")
    return ap.parse_args()


def attention_flops(lengths, H, D, causal=True):
    pairs = sum((L * (L + 1) // 2) if causal else L * L for L in lengths)
    return 4.0 * H * D * pairs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def profiled_traffic(name, source_file):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since it was taken (the summary records the source hash)."""
    prof = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "long_context_gb300", "csrc", source_file)
    try:
        text = open(prof).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != digest:
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while timed work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index
        self.windows = []
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, begin):
        now = time.time()
        if begin:
            self.t0 = now
        else:
            self.windows.append((self.t0, now))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names[1:], r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)]
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def aggregate(dist, torch, ms, flops, device):
    """Across ranks: the slowest rank's step time and the sum of all ranks'
    FLOPs (each rank runs its own batch).  Returns (ms_max, flops_total)."""
    t = torch.tensor([ms, flops], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(t[1])


def whole_job_tflops(total_flops, ms_max):
    """Whole-job throughput: all ranks' work over the slowest rank's time."""
    return total_flops / (ms_max * 1e-3) / 1e12


def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------ reference --

def _oracle_head_batch(lengths, H, D, seed):
    """The batch's Q, K, V (bf16 bytes the GPU sees, seeded) and cu_seqlens;
    the oracle takes them one head at a time."""
    from long_context_gb300 import workloads
    T = sum(lengths)
    q, k, v = workloads.qkv(T, H, D, seed)
    return q, k, v, workloads.cu_seqlens(lengths)


def cpu_oracle_sample(lengths, H, D, seed, budget_s):
    """Time the float64 oracle's full attention over every sample of the
    batch, one head at a time, until about ``budget_s`` seconds of work (each
    head is the batch's whole length mix); returns (TFLOP/s, desc, cores,
    seconds)."""
    import numpy as np
    from long_context_gb300 import workloads
    from oracle import attention as oa
    q, k, v, cu = _oracle_head_batch(lengths, H, D, seed)
    scale = 1.0 / np.sqrt(D)
    flops, t_total, heads = 0.0, 0.0, 0
    for h in range(H):
        sl = slice(h, h + 1)
        qf, kf, vf = (workloads.to_f64(x[:, sl]) for x in (q, k, v))
        t0 = time.perf_counter()
        oa.full_attention(qf, kf, vf, cu, scale)
        t_total += time.perf_counter() - t0
        flops += attention_flops(lengths, 1, D)
        heads += 1
        if t_total >= budget_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = ("float64 oracle full attention (NumPy/BLAS) over every sample of the batch "
            "(lengths %s), %d of its %d heads, D=%d; %.1f s" % (list(lengths), heads, H, D,
                                                              t_total))
    return flops / t_total / 1e12, desc, cores, t_total


def main_config(lengths, cp_sizes, H, D, seed):
    """The `config` of the packed16k line (both arms report it)."""
    T = sum(lengths)
    return {
        "workload": "packed THD micro-batch, 16384-token budget, lognormal(7.5,1) lengths "
                    "clipped to [64,16384], DPxCP world 4, max_seqlen_per_dp_cp_rank 4096, "
                    "CP from {1,2,4}, H=32, D=128, causal, bf16 N(0,1)",
        "lengths": [int(x) for x in lengths], "cp_sizes": [int(x) for x in cp_sizes],
        "tokens_per_gpu": T, "H": H, "D": D, "seed": seed,
        "parallelism": "one independent micro-batch per GPU (seed + rank), no collective",
        "l2": "inputs larger than L2 (Q/K/V %.0f MB per GPU)" % (3 * T * H * D * 2 / 1e6),
        "step": "cpattn_plan (host) + cp_size upload + cpattn_fwd fused",
    }


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from long_context_gb300 import workloads
    w = workloads.WORKLOADS[WORKLOAD]
    lengths = workloads.packed_lengths(args.seed, w["budget"])
    H, D = w["H"], w["D"]
    import numpy as np
    from oracle import attention as oa
    from oracle import planner as op
    plan = op.plan(lengths, w["world"], w["limit"], w["max_cp"])
    # One step = the oracle's full attention over every sample of the batch
    # for one head (the next head each step): the batch's whole length mix
    # at 1/H of its work.
    q, k, v, cu = _oracle_head_batch(lengths, H, D, args.seed)
    scale = 1.0 / np.sqrt(D)

    def one_step(i):
        sl = slice(i % H, i % H + 1)
        qf, kf, vf = (workloads.to_f64(x[:, sl]) for x in (q, k, v))
        t0 = time.perf_counter()
        oa.full_attention(qf, kf, vf, cu, scale)
        return time.perf_counter() - t0

    for i in range(args.warmup):
        one_step(i)
    dt = sum(one_step(args.warmup + i) for i in range(args.steps)) / max(args.steps, 1)
    value = attention_flops(lengths, 1, D) / dt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = ("float64 oracle full attention over every sample of the batch (lengths %s), "
              "one of its %d heads per step, D=%d, causal; rate = that head's FLOPs over "
              "the oracle's time" % (list(lengths), H, D))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": main_config(lengths, plan["cp_size"], H, D, args.seed),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- measured --

def time_loop(torch, fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / max(steps, 1)


def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    args.rank = rank
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch
    import torch.distributed as dist

    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn, workloads
    if args.nvtx:
        cpattn.set_tracing(True)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    hbm_peak, bf16_peak, bf16_sustained, peak_src = load_peaks()

    w = workloads.WORKLOADS[WORKLOAD]
    H, D, W, limit, max_cp = w["H"], w["D"], w["world"], w["limit"], w["max_cp"]
    seed = args.seed + rank
    lengths = workloads.packed_lengths(seed, w["budget"])
    T = sum(lengths)
    B = len(lengths)
    scale = 1.0 / np.sqrt(D)
    q, k, v = workloads.qkv_device(T, H, D, seed, device=dev)
    cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = cpattn.alloc_workspace(T, B, H, D, max_cp, cpattn.MODE_FUSED, device=dev)
    flops = attention_flops(lengths, H, D)
    # The plan goes up the way a caller streaming micro-batches sends it:
    # two pinned host / device buffer pairs and a copy stream, so that step
    # i's CP sizes are uploaded while step i-1's kernels run (the forward
    # waits on an event for its own upload; an upload waits until the forward
    # two steps back has finished reading that buffer).
    NP = 2
    cp_pinned = [torch.zeros(B, dtype=torch.int32).pin_memory() for _ in range(NP)]
    cp_bufs = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(NP)]
    cp_dev = cp_bufs[0]
    s_plan = torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(NP)]
    ev_read = [torch.cuda.Event() for _ in range(NP)]
    n_step = [0]

    def step():
        b_ = n_step[0] % NP
        n_step[0] += 1
        plan = cpattn.plan(lengths, W, limit, max_cp)           # dynamic-CP plan (host)
        ev_up[b_].synchronize()          # this pinned buffer's last upload is done
        cp_pinned[b_].numpy()[:] = plan["cp_size"]
        with torch.cuda.stream(s_plan):
            s_plan.wait_event(ev_read[b_])
            cp_bufs[b_].copy_(cp_pinned[b_], non_blocking=True)
            ev_up[b_].record(s_plan)
        stream.wait_event(ev_up[b_])
        cpattn.fwd(q, k, v, cu, cp_bufs[b_], max_seqlen=max(lengths), max_cp=max_cp,
                   softmax_scale=scale, out=out, lse=lse, workspace=ws)
        ev_read[b_].record(stream)

    def kernel_only():
        cpattn.fwd(q, k, v, cu, cp_dev, max_seqlen=max(lengths), max_cp=max_cp,
                   softmax_scale=scale, out=out, lse=lse, workspace=ws)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if args.only in ("long128k", "merge8", "backward", "dcp", "decode", "ulysses", "sweep256",
                     "seeds", "dcp_sweep256"):
        fn = {"long128k": run_long128k, "merge8": run_merge8, "backward": run_backward,
              "dcp": run_dcp_permute, "decode": run_decode, "ulysses": run_ulysses,
              "sweep256": run_sweep256, "seeds": run_packed16k_seeds,
              "dcp_sweep256": run_dcp_sweep256}[args.only]
        res = fn(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                 bf16_sustained, hbm_peak)
        clk = clocks.stop()
        if rank == 0:
            print(json.dumps({"only": args.only, **res, "clocks": clk}), flush=True)
        return 0

    # --- main timed region: exactly K steps, barrier + sync on both sides.
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    if world > 1:
        dist.barrier()
    status = cpattn.poll_error(ws)
    if status != cpattn.OK:
        raise RuntimeError("device status after timed steps: %s" % cpattn.status_string(status))
    ms_max, total_flops = ms, flops
    if world > 1:
        ms_max, total_flops = aggregate(dist, torch, ms, flops, dev)
    value = whole_job_tflops(total_flops, ms_max)

    # --- the attention kernel alone (roofline): average launch duration.
    k_ms = time_loop(torch, kernel_only, args.steps, 3, stream)
    achieved = flops / (k_ms * 1e-3) / 1e12
    traffic = profiled_traffic("attn_fwd_packed16k.md", "attn_fwd.cu")

    if args.only == "main":
        clk = clocks.stop()
        if rank == 0:
            print(json.dumps({"only": "main", "value": value, "ms_per_step": ms_max,
                              "kernel_ms": k_ms, "achieved": achieved, "clocks": clk}),
                  flush=True)
        return 0

    # --- end to end through the public API with host buffers.  Every step
    # copies its Q/K/V/cu_seqlens/cp_size from pinned host memory and its
    # O/LSE back; steps are pipelined over two device buffer sets and three
    # streams, so the copies of one step overlap the forward of its neighbour.
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    hcu = cu.cpu().pin_memory()
    NB = 2
    bufs = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                 cu=torch.empty_like(cu), cp=torch.empty_like(cp_dev),
                 out=torch.empty_like(out), lse=torch.empty_like(lse)) for _ in range(NB)]
    cp_host = [torch.zeros(B, dtype=torch.int32).pin_memory() for _ in range(NB)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NB)]
    h_lse = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(NB)]
    s_in, s_c, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = {key: [torch.cuda.Event() for _ in range(NB)] for key in ("cp", "in", "comp", "out")}
    used = {key: [False] * NB for key in ev}

    def e2e_run(nsteps):
        for i in range(nsteps):
            b_ = i % NB
            bf = bufs[b_]
            plan_i = cpattn.plan(lengths, W, limit, max_cp)          # host planner
            if used["cp"][b_]:
                ev["cp"][b_].synchronize()   # the upload from this host buffer is done
            cp_host[b_].numpy()[:] = plan_i["cp_size"]
            with torch.cuda.stream(s_in):
                if used["comp"][b_]:
                    s_in.wait_event(ev["comp"][b_])   # buffer set free again
                for key, host in (("q", hq), ("k", hk), ("v", hv), ("cu", hcu)):
                    bf[key].copy_(host, non_blocking=True)
                bf["cp"].copy_(cp_host[b_], non_blocking=True)
                ev["cp"][b_].record(s_in)
                ev["in"][b_].record(s_in)
            used["cp"][b_] = True
            with torch.cuda.stream(s_c):
                s_c.wait_event(ev["in"][b_])
                if used["out"][b_]:
                    s_c.wait_event(ev["out"][b_])     # previous outputs copied out
                cpattn.fwd(bf["q"], bf["k"], bf["v"], bf["cu"], bf["cp"],
                           max_seqlen=max(lengths), max_cp=max_cp, softmax_scale=scale,
                           out=bf["out"], lse=bf["lse"], workspace=ws)
                ev["comp"][b_].record(s_c)
            used["comp"][b_] = True
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["comp"][b_])
                h_out[b_].copy_(bf["out"], non_blocking=True)
                h_lse[b_].copy_(bf["lse"], non_blocking=True)
                ev["out"][b_].record(s_out)
            used["out"][b_] = True

    e2e_run(max(args.warmup, 3))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks.mark(True)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for s_ in (s_in, s_c, s_out):
        s_.wait_event(e_start)
    e2e_run(args.steps)
    for s_ in (s_in, s_c, s_out):
        mark = torch.cuda.Event()
        mark.record(s_)
        stream.wait_event(mark)
    e_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    e2e_ms = e_start.elapsed_time(e_end) / max(args.steps, 1)
    if cpattn.poll_error(ws) != cpattn.OK:
        raise RuntimeError("device status after the end-to-end steps")
    h2d = 3 * T * H * D * 2 + (B + 1) * 4 + B * 4
    d2h = T * H * D * 2 + T * H * 4
    e2e_ms_max = e2e_ms
    if world > 1:
        e2e_ms_max, _ = aggregate(dist, torch, e2e_ms, flops, dev)
    e2e_value = whole_job_tflops(total_flops, e2e_ms_max)
    del hq, hk, hv, bufs, h_out, h_lse

    extras = {}
    # The sub-measurements and the CPU baselines belong to the one-GPU line;
    # with N ranks only the main step is measured, so the N GPUs are held
    # for as short a time as possible.
    if not args.no_extras and world == 1:
        for fn in (run_packed16k_seeds, run_long128k, run_merge8, run_backward,
                   run_dcp_permute, run_decode, run_ulysses, run_sweep256, run_dcp_sweep256):
            if args.nvtx:
                torch.cuda.nvtx.range_push("bench:" + fn.__name__[4:])
            extras.update(fn(torch, cpattn, workloads, dev, stream, args, clocks,
                             bf16_peak, bf16_sustained, hbm_peak))
            if args.nvtx:
                torch.cuda.nvtx.range_pop()
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops, desc, cores, _ = cpu_oracle_sample(lengths, H, D, seed, budget_s=12.0)
        cpu = {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc}

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return 0
    plan = cpattn.plan(lengths, W, limit, max_cp)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": main_config(lengths, plan["cp_size"], H, D, args.seed),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel<128,false> + schedule_kernel",
                     "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": achieved / bf16_peak, "traffic": traffic,
                     "peak_source": "%s bf16_tflops (burst)" % peak_src,
                     "kernel_ms": k_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max,
                "pipeline": "2 buffer sets, copy-in / forward / copy-out streams"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    line.update(extras)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_packed16k_seeds(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                        bf16_sustained, hbm_peak):
    """The packed 16K forward (plan + cpattn_fwd fused) on seeds 0, 1 and 2 of
    the workload: seed 0 plans every sample at CP 1, seed 1 two samples at
    CP 2, seed 2 one at CP 4.  Each seed's attention kernel timed alone (CUDA
    events over the launches), as the headline roofline is."""
    import numpy as np
    w = workloads.WORKLOADS[WORKLOAD]
    H, D = w["H"], w["D"]
    res = {}
    steps = max(5, min(args.steps, 20))
    for seed in (0, 1, 2):
        lengths = workloads.packed_lengths(seed, w["budget"])
        plan = cpattn.plan(lengths, w["world"], w["limit"], w["max_cp"])
        cps_l = [int(c) for c in plan["cp_size"]]
        T = sum(lengths)
        q, k, v = workloads.qkv_device(T, H, D, seed, device=dev)
        cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
        cps = torch.tensor(cps_l, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        ws = cpattn.alloc_workspace(T, len(lengths), H, D, w["max_cp"], cpattn.MODE_FUSED,
                                    device=dev)
        fn = lambda: cpattn.fwd(q, k, v, cu, cps, max_seqlen=max(lengths),  # noqa: E731
                                max_cp=w["max_cp"], softmax_scale=1.0 / np.sqrt(D), out=out,
                                lse=lse, workspace=ws)
        clocks.mark(True)
        ms = time_loop(torch, fn, steps, 3, stream)
        clocks.mark(False)
        assert cpattn.poll_error(ws) == cpattn.OK
        flops = attention_flops(lengths, H, D)
        tf = flops / (ms * 1e-3) / 1e12
        res[str(seed)] = {"lengths": lengths, "cp_sizes": cps_l, "flops": flops,
                          "kernel_ms": ms, "tflops": tf, "frac": tf / bf16_peak}
        del q, k, v, out, lse, ws
    torch.cuda.empty_cache()
    return {"packed16k_seeds": {"what": "attention kernel (+ schedule kernel) alone per seed "
                                        "of the packed 16K workload; seed 0 is the headline",
                                **res}}


def cpu_oracle_long128k(budget_rows=4096):
    """The float64 oracle's full attention on the first ``budget_rows`` rows of
    the 131,072-token causal sequence (H=16, D=128, N(0, 0.5^2)): under
    causality those rows see only keys among themselves, so this is the
    oracle's computation for that labelled subset of the workload; the rate
    (TFLOP/s over the subset's visible pairs) is what the whole sequence would
    run at on these cores, and the time for the whole is extrapolated."""
    import numpy as np
    from long_context_gb300 import workloads
    from oracle import attention as oa
    w = workloads.WORKLOADS["long128k"]
    H, D, L = w["H"], w["D"], w["lengths"][0]
    n = budget_rows
    q, k, v = workloads.qkv(n, H, D, 0, std=w["std"])
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    cu = np.array([0, n], dtype=np.int64)
    t0 = time.perf_counter()
    oa.full_attention(qf, kf, vf, cu, 1.0 / np.sqrt(D))
    dt = time.perf_counter() - t0
    tf = attention_flops([n], H, D) / dt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "float64 oracle full attention over rows 0..%d of the causal %d-token "
                      "sequence (they see only each other), H=%d, D=%d: %.1f s; the whole "
                      "sequence at this rate: %.0f s" % (n - 1, L, H, D, dt,
                                                          attention_flops([L], H, D) / tf / 1e12)}


def cpu_oracle_merge8(rows=65536):
    """The float64 oracle's step-by-step merge on ``rows`` (token, head) rows of
    the CP=8 merge workload (S=8, D=128 fp32 partials); rate in GB/s of the
    merge's algorithmic bytes, extrapolated to the whole 4.9 GB."""
    import numpy as np
    from long_context_gb300 import workloads
    from oracle import attention as oa
    w = workloads.WORKLOADS["merge8"]
    S, D = w["S"], w["D"]
    o, m, l = workloads.merge_partials(S, rows, 1, D, seed=0)
    o, m, l = (x.numpy() for x in (o, m, l))
    t0 = time.perf_counter()
    oa.merge_partials(o, m, l)
    dt = time.perf_counter() - t0
    nbytes = S * rows * (D + 2) * 4 + rows * (D + 2) * 4
    gbs = nbytes / dt / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    total = S * w["T"] * w["H"] * (D + 2) * 4 + w["T"] * w["H"] * (D + 2) * 4
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "float64 oracle merge (step-by-step fold) of %d rows of the CP=8 "
                      "partials, D=%d: %.2f s; the whole %.1f GB at this rate: %.0f s"
                      % (rows, D, dt, total / 1e9, total / gbs / 1e9)}


def run_long128k(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                 bf16_sustained, hbm_peak):
    import numpy as np
    res = {}
    steps = max(3, min(args.steps, 10))
    # 131,072-token causal sequence at CP=4, fused and unfused.
    w = workloads.WORKLOADS["long128k"]
    H, D, L, c = w["H"], w["D"], w["lengths"][0], w["cp"]
    if args.small:
        L = 32768  # Q/K/V 134 MB each, still larger than L2
    q, k, v = workloads.qkv_device(L, H, D, args.seed, std=w["std"], device=dev)
    cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
    cps = torch.tensor([c], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((L, H), dtype=torch.float32, device=dev)
    flops = attention_flops([L], H, D)
    sub = {}
    for mode, name in ((cpattn.MODE_FUSED, "fused"), (cpattn.MODE_UNFUSED, "unfused")):
        ws = cpattn.alloc_workspace(L, 1, H, D, c, mode, device=dev)
        fn = lambda: cpattn.fwd(q, k, v, cu, cps, max_seqlen=L, max_cp=c,  # noqa: E731
                                softmax_scale=1.0 / np.sqrt(D), mode=mode, out=out, lse=lse,
                                workspace=ws)
        clocks.mark(True)
        ms = time_loop(torch, fn, steps, 2, stream)
        clocks.mark(False)
        assert cpattn.poll_error(ws) == cpattn.OK
        tf = flops / (ms * 1e-3) / 1e12
        sub[name] = {"ms": ms, "tflops": tf, "frac_of_burst": tf / bf16_peak,
                     "frac_of_sustained": tf / bf16_sustained}
        del ws
    res["long128k"] = {"workload": "one causal %d-token sequence, CP=4 (%d-token chunks), "
                                   "H=16, D=128, bf16 N(0,0.5^2)" % (L, L // c),
                       "flops": flops, "steps": steps, **sub}
    if args.rank == 0 and not args.no_cpu_baseline:
        res["long128k"]["cpu_baseline"] = cpu_oracle_long128k()
    del q, k, v, out, lse
    torch.cuda.empty_cache()
    return res


def run_backward(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                 bf16_sustained, hbm_peak):
    """cpattn_bwd (dQ, dK, dV) after a forward, on the packed 16K batch and on
    the 131,072-token sequence.  FLOPs: 2.5 x the forward's (five matmuls over
    the visible pairs: S recomputed, dP, dV, dK, dQ)."""
    import numpy as np
    sub = {}
    for name in ("packed16k", "long128k"):
        w = workloads.WORKLOADS[name]
        H, D = w["H"], w["D"]
        if name == "packed16k":
            lengths = workloads.packed_lengths(args.seed, w["budget"])
            plan = cpattn.plan(lengths, w["world"], w["limit"], w["max_cp"])
            cps_l = [int(x) for x in plan["cp_size"]]
            std, steps = 1.0, max(3, min(args.steps, 20))
        else:
            lengths, cps_l, std = list(w["lengths"]), [w["cp"]], w["std"]
            if args.small:
                lengths = [32768]  # profiling aid, as in run_long128k
            steps = max(3, min(args.steps, 5))
        T, max_cp = sum(lengths), max(cps_l)
        q, k, v = workloads.qkv_device(T, H, D, args.seed, std=std, device=dev)
        g = torch.Generator(device=dev).manual_seed(args.seed + 1)
        dout = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
        cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
        cps = torch.tensor(cps_l, dtype=torch.int32, device=dev)
        out, lse = cpattn.fwd(q, k, v, cu, cps, max_seqlen=max(lengths), max_cp=max_cp)
        ws = cpattn.alloc_bwd_workspace(T, len(lengths), H, D, max_cp, dev)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        fn = lambda: cpattn.bwd(q, k, v, out, dout, lse, cu, cps,  # noqa: E731
                                max_seqlen=max(lengths), max_cp=max_cp, dq=dq, dk=dk, dv=dv,
                                workspace=ws)
        clocks.mark(True)
        ms = time_loop(torch, fn, steps, 2, stream)
        clocks.mark(False)
        assert cpattn.poll_error(ws) == cpattn.OK
        flops = 2.5 * attention_flops(lengths, H, D)
        tf = flops / (ms * 1e-3) / 1e12
        sub[name] = {"tokens": T, "ms": ms, "tflops": tf, "frac_of_burst": tf / bf16_peak,
                     "frac_of_sustained": tf / bf16_sustained, "flops": flops, "steps": steps}
        del q, k, v, dout, out, lse, ws, dq, dk, dv
        torch.cuda.empty_cache()
    return {"backward": {"what": "cpattn_bwd (delta + dK/dV + dQ kernels), inputs resident; "
                                 "FLOPs = 2.5 x forward (5 matmuls over visible pairs)", **sub}}


def run_dcp_permute(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                    bf16_sustained, hbm_peak):
    """cpattn_permute_samples (select of every sample in reversed order, then
    restore) on a 65,536-token packed batch, H=32, D=128 bf16: HBM bound,
    bytes = rows x row bytes read + written per call."""
    H, D = 32, 128
    lengths = workloads.packed_lengths(args.seed, 32768 if args.small else 65536)
    T = sum(lengths)
    g = torch.Generator(device=dev).manual_seed(args.seed)
    x = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
    ids = torch.arange(len(lengths) - 1, -1, -1, dtype=torch.int32, device=dev)
    pack_cu, status = cpattn.select_cu(cu, ids)
    packed = torch.empty_like(x)
    back = torch.empty_like(x)
    steps = max(10, min(args.steps, 50))
    res = {}
    for name, fn in (("select", lambda: cpattn.permute_samples(x, cu, pack_cu, ids, status,
                                                               gather=True, dst=packed)),
                     ("restore", lambda: cpattn.permute_samples(packed, cu, pack_cu, ids, status,
                                                                gather=False, dst=back))):
        clocks.mark(True)
        ms = time_loop(torch, fn, steps, 3, stream)
        clocks.mark(False)
        nbytes = 2 * T * H * D * 2
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm_peak, "bytes": nbytes}
    assert torch.equal(back, x)
    del x, packed, back
    torch.cuda.empty_cache()
    return {"dcp_permute": {"workload": "%d-token packed batch (%d samples), H=32, D=128 bf16, "
                                        "every sample moved (reversed order)" % (T, len(lengths)),
                            **res}}


def run_decode(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
               bf16_sustained, hbm_peak):
    """Decode-time CP (cpattn_decode: shard partials + LSE-form merge): 64
    sequences with KV caches of uniform length in [4096, 32768], H=32, D=128,
    decode CP 4.  HBM bound: bytes = the KV cache read once + q + O, LSE and
    the partials written and read back."""
    import numpy as np
    B, H, D, c = (8 if args.small else 64), 32, 128, 4
    lengths = [int(x) for x in np.random.default_rng(args.seed).integers(4096, 32769, B)]
    T = sum(lengths)
    g = torch.Generator(device=dev).manual_seed(args.seed)
    k = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((B, H, D), generator=g, device=dev).to(torch.bfloat16)
    cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(cpattn._lib.cpattn_decode_workspace_size(B, H, D, c), dtype=torch.uint8,
                     device=dev)
    fn = lambda: cpattn.decode(q, k, v, cu, cp=c, out=out, lse=lse, workspace=ws)  # noqa: E731
    steps = max(10, min(args.steps, 50))
    clocks.mark(True)
    ms = time_loop(torch, fn, steps, 3, stream)
    clocks.mark(False)
    kv_bytes = 2 * T * H * D * 2
    other = B * H * D * 2 * 2 + B * H * 4 + 2 * c * B * H * (D + 1) * 4
    gbs = (kv_bytes + other) / (ms * 1e-3) / 1e9
    del k, v, q, out, lse, ws
    torch.cuda.empty_cache()
    return {"decode": {"workload": "%d sequences, KV cache lengths uniform in [4096, 32768] "
                                   "(%d tokens), H=32, D=128 bf16, decode CP 4" % (B, T),
                       "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm_peak,
                       "bytes": kv_bytes + other}}


def run_ulysses(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                bf16_sustained, hbm_peak):
    """Ulysses layout (cpattn_ulysses_layout) on 131,072 tokens, H=32, D=128
    bf16, SP 8: bytes = the tensor read once and written once.  And Ulysses
    attention (Q, K, V to head groups, one forward over the 8 groups of 4
    heads at the planned CP sizes, O and LSE back) on the packed 16K batch,
    FLOPs as the forward's."""
    import numpy as np
    T_lay, H, D, P = (65536 if args.small else 131072), 32, 128, 8
    T = T_lay
    g = torch.Generator(device=dev).manual_seed(args.seed)
    x = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((P, T, H // P, D), dtype=torch.bfloat16, device=dev)
    back = torch.empty_like(x)
    steps = max(10, min(args.steps, 50))
    res = {}
    nbytes = 2 * T * H * D * 2
    for name, fn in (("to_head_groups",
                      lambda: cpattn.ulysses_layout(x, P, to_head_groups=True, dst=y)),
                     ("from_head_groups",
                      lambda: cpattn.ulysses_layout(y, P, to_head_groups=False, dst=back))):
        clocks.mark(True)
        ms = time_loop(torch, fn, steps, 3, stream)
        clocks.mark(False)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm_peak, "bytes": nbytes}
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    del x, y, back
    torch.cuda.empty_cache()

    w = workloads.WORKLOADS["packed16k"]
    lengths = workloads.packed_lengths(args.seed, w["budget"])
    plan = cpattn.plan(lengths, w["world"], w["limit"], w["max_cp"])
    cps_l = [int(c) for c in plan["cp_size"]]
    Tp, Hp, Dp = sum(lengths), w["H"], w["D"]
    q, k, v = workloads.qkv_device(Tp, Hp, Dp, args.seed, device=dev)
    cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
    cps = torch.tensor(cps_l, dtype=torch.int32, device=dev)
    fn = lambda: cpattn.ulysses_fwd(q, k, v, cu, P, cps, max_seqlen=max(lengths),  # noqa: E731
                                    max_cp=max(cps_l), softmax_scale=1.0 / np.sqrt(Dp))
    clocks.mark(True)
    ms = time_loop(torch, fn, max(3, min(args.steps, 20)), 3, stream)
    clocks.mark(False)
    tf = attention_flops(lengths, Hp, Dp) / (ms * 1e-3) / 1e12
    res["attention_packed16k"] = {"ms": ms, "tflops": tf, "frac_of_burst": tf / bf16_peak,
                                  "sp": P}
    del q, k, v
    torch.cuda.empty_cache()
    return {"ulysses": {"workload": "layout: %d tokens, H=32, D=128 bf16, SP 8; attention: "
                                    "packed 16K batch (%d tokens), H=32 as 8 groups of 4 heads, "
                                    "planned CP sizes inside each group" % (T_lay, Tp), **res}}


def run_sweep256(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                 bf16_sustained, hbm_peak):
    """The 256-sample sweep: lengths uniform in [256, 32768], planned with
    cpattn_plan (world 8, limit 4096, CP up to 8); each micro-batch's samples
    form their own packed THD batch (inputs of every micro-batch resident,
    distinct data), and one step is the forward of every micro-batch at its
    planned CP sizes, back to back.  FLOPs as the forward's (4 H D per visible
    pair)."""
    import numpy as np
    w = workloads.WORKLOADS["sweep256"]
    H, D = w["H"], w["D"]
    lengths = workloads.uniform_lengths(args.seed, w["n"], w["lo"], w["hi"])
    plan = cpattn.plan(lengths, w["world"], w["limit"], w["max_cp"])
    mb = np.asarray(plan["micro_batch"])
    order = [int(b) for b in plan["order"]]
    cps_all = np.asarray(plan["cp_size"])
    g = torch.Generator(device=dev).manual_seed(args.seed)
    batches = []
    for m in range(int(plan["num_micro_batches"])):
        ids = [b for b in order if mb[b] == m]
        lens_m = [lengths[b] for b in ids]
        T = sum(lens_m)
        q, k, v = (torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
                   for _ in range(3))
        cu = torch.from_numpy(workloads.cu_seqlens(lens_m)).to(dev)
        cp_m = [int(cps_all[b]) for b in ids]
        cps = torch.tensor(cp_m, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        ws = cpattn.alloc_workspace(T, len(ids), H, D, max(cp_m), cpattn.MODE_FUSED, device=dev)
        batches.append((q, k, v, cu, cps, max(lens_m), max(cp_m), out, lse, ws))
    scale = 1.0 / np.sqrt(D)

    def step():
        for (q, k, v, cu, cps, max_L, max_c, out, lse, ws) in batches:
            cpattn.fwd(q, k, v, cu, cps, max_seqlen=max_L, max_cp=max_c, softmax_scale=scale,
                       out=out, lse=lse, workspace=ws)

    clocks.mark(True)
    ms = time_loop(torch, step, max(2, min(args.steps, 3)), 2, stream)
    clocks.mark(False)
    for b in batches:
        assert cpattn.poll_error(b[9]) == cpattn.OK
    flops = attention_flops(lengths, H, D)
    tf = flops / (ms * 1e-3) / 1e12
    n_mb = len(batches)
    del batches
    torch.cuda.empty_cache()
    return {"sweep256": {"workload": "256 lengths uniform in [256, 32768] (%d tokens), world 8, "
                                     "limit 4096, CP up to 8, %d micro-batches from cpattn_plan, "
                                     "H=32, D=128, causal, bf16 N(0,1)" % (sum(lengths), n_mb),
                         "ms": ms, "tflops": tf, "frac_of_burst": tf / bf16_peak,
                         "frac_of_sustained": tf / bf16_sustained, "flops": flops,
                         "launches_per_step": 2 * n_mb}}


def run_dcp_sweep256(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
                     bf16_sustained, hbm_peak):
    """The 256-sample sweep run the dynamic-CP way (cpattn.DcpForward): the
    whole mini-batch resident in original order, and per planned micro-batch
    select Q/K/V into packed arrays, the forward at the planned CP sizes, and O
    and LSE restored to the original rows -- no host synchronisation inside
    the step.  Compare with ``sweep256`` (the same forwards on inputs already
    packed per micro-batch): the difference is the DCP data movement."""
    import numpy as np
    w = workloads.WORKLOADS["sweep256"]
    H, D = w["H"], w["D"]
    lengths = workloads.uniform_lengths(args.seed, w["n"], w["lo"], w["hi"])
    plan = cpattn.plan(lengths, w["world"], w["limit"], w["max_cp"])
    T = sum(lengths)
    q, k, v = workloads.qkv_device(T, H, D, args.seed, device=dev)
    cu = torch.from_numpy(workloads.cu_seqlens(lengths)).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    run = cpattn.DcpForward(lengths, plan, num_heads=H, head_dim=D, max_cp=w["max_cp"],
                            device=dev)
    fn = lambda: run(q, k, v, cu, softmax_scale=1.0 / np.sqrt(D), out=out,  # noqa: E731
                     lse=lse)
    clocks.mark(True)
    ms = time_loop(torch, fn, max(2, min(args.steps, 3)), 1, stream)
    clocks.mark(False)
    assert cpattn.poll_error(run.workspace) == cpattn.OK
    assert int(run.status.item()) == 0
    flops = attention_flops(lengths, H, D)
    tf = flops / (ms * 1e-3) / 1e12
    moved = 2 * (3 * T * H * D * 2) + 2 * (T * H * D * 2 + T * H * 4)
    n_mb = len(run.micro)
    del q, k, v, out, lse, run
    torch.cuda.empty_cache()
    return {"dcp_sweep256": {"workload": "the 256-sample sweep (%d tokens) through "
                                         "cpattn.DcpForward: select, forward, restore per "
                                         "micro-batch (%d), H=32, D=128" % (T, n_mb),
                             "ms": ms, "tflops": tf, "frac_of_burst": tf / bf16_peak,
                             "permute_bytes": moved,
                             "launches_per_step": 7 * n_mb}}


def run_merge8(torch, cpattn, workloads, dev, stream, args, clocks, bf16_peak,
               bf16_sustained, hbm_peak):
    res = {}
    steps = max(3, min(args.steps, 10))
    # Merge of CP=8 stored partials, T=32768, H=32, D=128.
    w = workloads.WORKLOADS["merge8"]
    S, T, H, D = w["S"], w["T"], w["H"], w["D"]
    if args.small:
        T = 4096  # profiling aid: 0.54 GB of partials, still larger than L2
    g = torch.Generator(device=dev).manual_seed(args.seed)
    o = torch.randn((S, T, H, D), generator=g, device=dev, dtype=torch.float32)
    m = torch.rand((S, T, H), generator=g, device=dev, dtype=torch.float32) * 10 - 5
    l = torch.rand((S, T, H), generator=g, device=dev, dtype=torch.float32) * 1023 + 1
    oo = torch.empty((T, H, D), device=dev, dtype=torch.float32)
    om = torch.empty((T, H), device=dev, dtype=torch.float32)
    ol = torch.empty((T, H), device=dev, dtype=torch.float32)
    nbytes = S * T * H * (D + 2) * 4 + T * H * (D + 2) * 4
    fn = lambda: cpattn.merge(o, m, l, out_o=oo, out_m=om, out_l=ol)  # noqa: E731
    clocks.mark(True)
    ms = time_loop(torch, fn, max(steps, 10), 3, stream)
    clocks.mark(False)
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["merge8"] = {"workload": "CP=8 partials, T=%d, H=32, D=128 fp32 (inputs %.1f GB > L2)"
                                 % (T, S * T * H * (D + 2) * 4 / 1e9),
                     "bytes": nbytes, "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm_peak,
                     "traffic": profiled_traffic("merge_merge8.md", "merge.cu")}
    if args.rank == 0 and not args.no_cpu_baseline:
        res["merge8"]["cpu_baseline"] = cpu_oracle_merge8()
    del o, m, l, oo, om, ol
    torch.cuda.empty_cache()
    return res


if __name__ == "__main__":
    sys.exit(main())
