#!/usr/bin/env python3
"""Benchmark of MLA speculative-verify attention on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2] [--impl reference]

Prints ONE JSON line.  A step is one verify call (split kernel + combine) over
one synthetic batch of the named workload (default c2: 1 stream, q_len 9, H 64,
prefix 4096, contiguous slots, causal chain -- the pages' microbenchmark shape).
`value` is effective KV bandwidth (KV-row bytes / time) with inputs resident in
HBM, timed with CUDA events per step on the launching stream; L2 is flushed
(256 MiB written) before every step, outside the events.  `e2e` is the same
metric with the step's inputs copied from pinned host memory and the outputs
copied back inside the timed region.  `--impl reference` times the fp64 CPU
oracle on this host's cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as w  # noqa: E402

METRIC = "µs/call and effective KV GB/s for MLA verify attn; % of per-config roofline"
UNIT = "GB/s (effective KV)"
KV_ROW_BYTES = 576 * 2          # one bf16 latent KV row
IDX_BYTES = 4
L2_FLUSH_BYTES = 256 << 20      # > 2x the 129 MB L2
# The pages' own figure for the c2 shape (1 stream, q_len 9, H 64, prefix 4096,
# contiguous KV): 2887.8 us for their fastest kernel at that prefix, on an RTX PRO 6000.
PAGES_C2_US = 2887.8

WORKLOAD_TEXT = {
    "c1": "MLA verify B1 q_len9 H8 prefix256 contiguous chain-mask bf16",
    "c2": "MLA verify B1 q_len9 H64 prefix4096 contiguous chain-mask bf16",
    "c3-16k": "MLA verify B1 q_len9 H8 prefix16384 scattered 2^20-row pool tree-mask bf16",
    "c3-64k": "MLA verify B1 q_len9 H8 prefix65536 scattered 2^20-row pool tree-mask bf16",
    "c4": "MLA verify B8 q_len9 H8 prefixes U{1024..46080} scattered 2^20-row pool tree-masks bf16",
}


# --------------------------------------------------------------------------
# algorithmic work of one verify call (counts only what the method must move)
# --------------------------------------------------------------------------
def visible_keys(inp) -> int:
    """Sum over query rows of the number of keys each row attends to."""
    total = 0
    for b in range(inp.B):
        p = int(inp.seq_lens[b]) - inp.q_len
        for t in range(inp.q_len):
            nd = (t + 1) if inp.mask is None else int(inp.mask[b, t].astype(bool).sum())
            total += (p + nd) * inp.H
    return total


def flops_per_row_key() -> int:
    """2 * (576 + 512): one 576-d dot product for the score, one 512-d axpy for P V."""
    return 2 * (576 + 512)


def algorithmic(inp) -> dict:
    keys = int(np.sum(inp.seq_lens))
    rows = inp.B * inp.q_len * inp.H
    kv = keys * KV_ROW_BYTES
    total = kv + keys * IDX_BYTES + rows * 576 * 2 + rows * (512 + 1) * 4
    return {"kv_bytes": kv, "bytes": total, "flops": flops_per_row_key() * visible_keys(inp), "keys": keys,
            "rows": rows}


def roofline_us(work: dict, hbm_gbs: float, tflops: float) -> tuple:
    t_mem = work["bytes"] / (hbm_gbs * 1e9) * 1e6
    t_mma = work["flops"] / (tflops * 1e12) * 1e6
    return (max(t_mem, t_mma), "hbm" if t_mem >= t_mma else "tensor", t_mem, t_mma)


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback (no MEASURED_PEAKS.json)"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_speculative_verify_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(config: str):
    """DRAM bytes per launch of the split kernel from a committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(config)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# replicas: aggregation over ranks (no collective in the data path)
# --------------------------------------------------------------------------
def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over the default process group (identity
    when torch.distributed is not initialised).  Works with gloo (CPU) and nccl."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_throughput(bytes_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job GB/s of N replicas that each process `bytes_per_rank` per step, timed by
    the slowest rank."""
    return world * bytes_per_rank / (ms_per_step_max * 1e-3) / 1e9


# --------------------------------------------------------------------------
# clocks sampler
# --------------------------------------------------------------------------
class Clocks:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            os.makedirs(os.path.join(ROOT, "gpurun_out"), exist_ok=True)
            self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{self.index}.csv")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------
def time_oracle(inp, seconds: float, max_reps: int = 1000) -> dict:
    import oracle
    threads = os.cpu_count() or 1
    oracle.lib()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_inputs(inp, nthreads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            break
    per_call = el / reps
    return {"seconds_per_call": per_call, "reps": reps, "threads": threads}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = w.config(args.config)
    work = algorithmic(inp)
    steps = max(1, args.steps)
    # each step is one full oracle call on this workload (bounded: a few seconds each)
    import oracle
    threads = os.cpu_count() or 1
    oracle.lib()
    for _ in range(min(args.warmup, 1)):
        oracle.verify_inputs(inp, nthreads=threads)
    times = []
    budget = args.ref_seconds
    t_all = time.perf_counter()
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.verify_inputs(inp, nthreads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget:
            break
    per = statistics.mean(times)
    gbs = work["kv_bytes"] / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64 inputs)",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config},
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{len(times)} full oracle calls on the whole {args.config} workload"},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "us_per_call": per * 1e6,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from mla_speculative_verify_attention_gb300 import build as mvbuild
    if rank == 0 or world == 1:
        mvbuild.build()
    if world > 1:
        dist.barrier()
    import mla_speculative_verify_attention_gb300 as mv
    mv.load()

    inp = w.config(args.config)
    work = algorithmic(inp)
    peaks = load_peaks()
    rl_us, bound, t_mem, t_mma = roofline_us(work, peaks["hbm_gbs"], peaks["bf16_tflops"])

    def dev_tensor(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.to(dev)

    q = dev_tensor(inp.q_bits.view(np.int16)).view(torch.bfloat16)
    kv = dev_tensor(inp.kv_bits.view(np.int16)).view(torch.bfloat16)
    st = dev_tensor(inp.slot_table)
    sl = dev_tensor(inp.seq_lens)
    mk = None if inp.mask is None else dev_tensor(inp.mask)
    ns = args.nsplit or mv.auto_nsplit(inp.B, inp.q_len, inp.H, inp.slot_stride, mv.num_sms(dev), 1 << 62)
    ws = torch.empty(max(mv.workspace_bytes(inp.B, inp.q_len, inp.H, ns), 256), dtype=torch.uint8, device=dev)
    out = torch.empty((inp.B, inp.q_len, inp.H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((inp.B, inp.q_len, inp.H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 1 + (1 if ns > 1 else 0)

    def step(e0=None, e1=None, e2=None):
        if e0 is not None:
            e0.record(stream)
        if ns > 1:
            po, pl = mv.verify_partials(q, kv, st, sl, mk, inp.scale, nsplit=ns, workspace=ws, out=out, lse=lse,
                                        stream=stream)
            if e1 is not None:
                e1.record(stream)
            mv.verify_combine(po, pl, inp.B, inp.q_len, inp.H, out=out, lse=lse, stream=stream)
        else:
            mv.verify_partials(q, kv, st, sl, mk, inp.scale, nsplit=1, workspace=ws, out=out, lse=lse, stream=stream)
            if e1 is not None:
                e1.record(stream)
        if e2 is not None:
            e2.record(stream)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.25)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i))
        step(*ev[i])
    torch.cuda.synchronize(dev)
    wall_dev = time.perf_counter() - wall0
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    kern_ms = [a.elapsed_time(b) for a, b, c in ev]
    status = mv.device_status(stream)

    # end to end through the C ABI with host buffers: H2D of this step's inputs
    # (queries, slot table, lengths, mask, the q_len new draft KV rows per stream)
    # from pinned memory, the call, and D2H of out and lse, all inside the events.
    h_q = torch.from_numpy(inp.q_bits.view(np.int16)).pin_memory()
    h_st = torch.from_numpy(np.ascontiguousarray(inp.slot_table)).pin_memory()
    h_sl = torch.from_numpy(np.ascontiguousarray(inp.seq_lens)).pin_memory()
    h_mk = None if inp.mask is None else torch.from_numpy(np.ascontiguousarray(inp.mask)).pin_memory()
    draft_slots = [inp.slot_table[b, inp.seq_lens[b] - inp.q_len:inp.seq_lens[b]] for b in range(inp.B)]
    h_draft = torch.from_numpy(np.concatenate([inp.kv_bits[s] for s in draft_slots]).view(np.int16)).pin_memory()
    h_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    q_i16 = q.view(torch.int16)
    kv_i16 = kv.view(torch.int16)
    draft_runs = []          # (host row offset, first pool row, count) of contiguous slot runs
    off = 0
    for s in draft_slots:
        start = 0
        for k in range(1, len(s) + 1):
            if k == len(s) or s[k] != s[k - 1] + 1:
                draft_runs.append((off + start, int(s[start]), k - start))
                start = k
        off += len(s)
    h2d = h_q.numel() * 2 + h_st.numel() * 4 + h_sl.numel() * 4 + (0 if h_mk is None else h_mk.numel()) + \
        h_draft.numel() * 2
    d2h = h_out.numel() * 4 + h_lse.numel() * 4

    def e2e_step():
        q_i16.copy_(h_q, non_blocking=True)
        st.copy_(h_st, non_blocking=True)
        sl.copy_(h_sl, non_blocking=True)
        if mk is not None:
            mk.copy_(h_mk, non_blocking=True)
        for ho, row, cnt in draft_runs:
            kv_i16[row:row + cnt].copy_(h_draft[ho:ho + cnt], non_blocking=True)
        mv.verify_attn(q, kv, st, sl, mk, inp.scale, out=out, lse=lse, nsplit=ns, workspace=ws, stream=stream)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    Ke = max(1, min(K, 200))
    ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    torch.cuda.synchronize(dev)
    for i in range(Ke):
        flush.fill_(float(i))
        ee[i][0].record(stream)
        e2e_step()
        ee[i][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = [a.elapsed_time(b) for a, b in ee]
    clk = clocks.stop()

    # aggregate over ranks: max time, summed work
    mean_step = statistics.mean(step_ms)
    mean_kern = statistics.mean(kern_ms)
    mean_e2e = statistics.mean(e2e_ms)
    mean_step, mean_kern, mean_e2e = max_over_ranks([mean_step, mean_kern, mean_e2e], device=dev)
    value = aggregate_throughput(work["kv_bytes"], mean_step, world)
    e2e_value = aggregate_throughput(work["kv_bytes"], mean_e2e, world)

    if bound == "tensor":
        achieved = work["flops"] / (mean_kern * 1e-3) / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = work["bytes"] / (mean_kern * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r = time_oracle(inp, args.cpu_seconds)
        cpu = {"value": work["kv_bytes"] / r["seconds_per_call"] / 1e9, "unit": UNIT, "cores": r["threads"],
               "kind": "oracle",
               "sample": f"{r['reps']} full fp64 oracle calls on the whole {args.config} workload "
                         f"({r['seconds_per_call'] * 1e3:.1f} ms/call)"}

    srt = sorted(step_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": mean_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (PAGES_C2_US / (mean_step * 1e3)) if args.config == "c2" and world == 1 else None,
        "dtype": "bf16", "data": "synthetic (seeded SplitMix64 / Box-Muller inputs, shapes of the pages' workloads)",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config, "B": inp.B, "q_len": inp.q_len,
                   "H": inp.H, "keys": work["keys"], "n_pool": inp.n_pool, "nsplit": ns,
                   "l2": "flushed before every step (256 MiB write, outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_call": mean_step * 1e3,
        "us_per_call_p10_p50_p90": [srt[int(0.1 * (K - 1))] * 1e3, srt[(K - 1) // 2] * 1e3, srt[int(0.9 * (K - 1))] * 1e3],
        "roofline_us": rl_us, "roofline_pct": 100.0 * rl_us / (mean_step * 1e3),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": traffic_from_profiles(args.config), "kernel": "split (attention) kernel",
                     "kernel_us": mean_kern * 1e3, "peak_source": peaks["source"] + ", burst"},
        "algorithmic": work,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "us_per_call": mean_e2e * 1e3},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "device_status": status,
        "wall_s_timed_region": wall_dev,
        "cpu_baseline": cpu,
    }
    if world > 1:
        dist.barrier()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c2", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
