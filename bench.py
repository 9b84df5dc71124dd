#!/usr/bin/env python3
"""Benchmark of MLA speculative-verify attention on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--impl reference]

Prints ONE JSON line.  A step is one verify call through the C ABI
(mla_verify_attn: split kernel + combine) over one synthetic batch of the named
workload (default c4: 8 streams, q_len 9, H 8, prefixes U{1024..46080}, slots
scattered over a 2^20-row pool, random draft trees -- the serving shape of long
contexts at H 8 per rank).  `value` is effective KV bandwidth (KV-row bytes /
time) with inputs resident in HBM, timed with CUDA events per step on the
launching stream; L2 is flushed before every step, outside the events: 256 MiB
are written and then another 256 MiB buffer is read, so none of the call's inputs
is in L2 and the flush leaves no dirty line whose write-back would fall inside the
timed call (a write-only flush is timed too and reported beside it).  The split
kernel alone is timed the same way in a second loop (its duration is the
roofline's denominator), and a warm-L2 loop (no flush; a device-side spin covers
the host's submission instead) is reported beside it.  `e2e` is the same metric
end to end: the step's inputs (queries, slot table, lengths, mask and the new
draft KV rows) copied from one pinned host buffer in one copy, the KV append
kernel, the verify call and the outputs (out and lse, one buffer) copied back,
all inside the timed region.  `--impl reference` times the fp64 CPU oracle on
this host's cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
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
    "c5": "MLA fp8-e4m3 sparse decode B32 q_len1 H64 top-k 2048 of 65536 (per-token fp32 scale, bf16 rope)",
}
FP8_ROW_BYTES = 512 + 4 + 128          # e4m3 latent + fp32 scale + bf16 rope


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


def algorithmic_fp8(f) -> dict:
    """fp8 sparse decode: every (row, listed key) pair is visible; 644 B per key row."""
    keys = f.B * f.topk
    rows = f.B * f.H
    kv = keys * FP8_ROW_BYTES
    total = kv + keys * IDX_BYTES + rows * 576 * 2 + rows * (512 + 1) * 4
    return {"kv_bytes": kv, "bytes": total, "flops": flops_per_row_key() * rows * f.topk, "keys": keys, "rows": rows}


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


def _code_only(text: str) -> str:
    """CUDA source without comments, trailing spaces and blank lines: the hash below
    then changes with the code, not with its commentary."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_speculative_verify_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
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

    def __init__(self, index: int, csv_path: str | None = None):
        """Samples nvidia-smi every 100 ms into csv_path (a temporary file when None)."""
        self.index = index
        self.proc = None
        self.path = csv_path
        self.temporary = csv_path is None

    def start(self):
        try:
            if self.path is None:
                import tempfile
                fd, self.path = tempfile.mkstemp(prefix=f"clocks_gpu{self.index}_", suffix=".csv")
                os.close(fd)
            else:
                os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
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
        if self.temporary:
            os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------
def time_oracle(wl, seconds: float, max_reps: int = 1000, threads: int = 0) -> dict:
    import oracle
    threads = threads or os.cpu_count() or 1
    oracle.lib()
    reps, t0 = 0, time.perf_counter()
    while True:
        wl.oracle_call(threads)
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
    import oracle
    if args.config == "c5":
        f = w.config_fp8(args.config)
        work = algorithmic_fp8(f)
        call = lambda th: oracle.sparse_fp8_inputs(f, nthreads=th)
    else:
        inp = w.config(args.config)
        work = algorithmic(inp)
        call = lambda th: oracle.verify_inputs(inp, nthreads=th)
    # each step is one full oracle call on this workload (bounded by --ref-seconds overall)
    threads = os.cpu_count() or 1
    oracle.lib()
    for _ in range(min(args.warmup, 1)):
        call(threads)
    times = []
    t_all = time.perf_counter()
    for _ in range(max(1, args.steps)):
        t0 = time.perf_counter()
        call(threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > args.ref_seconds:
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
# workloads as seen by the GPU arm: device inputs, the split stage, the full call,
# and the per-step host -> device inputs of the end-to-end measurement
# --------------------------------------------------------------------------
def stage_inputs(named, dev):
    """[(name, pinned host tensor)] -> (pinned host buffer, device buffer, {name: device
    view}): every input in its own 256-byte-aligned section of one buffer, so a step's
    inputs cross in one copy (as a serving runtime stages them) instead of one copy each."""
    import torch
    offs, total = [], 0
    for _, h in named:
        offs.append(total)
        total += (h.numel() * h.element_size() + 255) // 256 * 256
    hbuf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for (name, h), off in zip(named, offs):
        n = h.numel() * h.element_size()
        hbuf[off:off + n].copy_(h.contiguous().view(-1).view(torch.uint8))
        views[name] = dbuf[off:off + n].view(h.dtype).view(h.shape)
    return hbuf, dbuf, views


class VerifyWorkload:
    def __init__(self, inp, mv, dev):
        import torch
        self.inp, self.mv, self.dev = inp, mv, dev
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.q = t(inp.q_bits.view(np.int16)).view(torch.bfloat16)
        self.kv = t(inp.kv_bits.view(np.int16)).view(torch.bfloat16)
        self.st, self.sl = t(inp.slot_table), t(inp.seq_lens)
        self.mk = None if inp.mask is None else t(inp.mask)
        self.B, self.q_len, self.H = inp.B, inp.q_len, inp.H
        self.work = algorithmic(inp)
        self.max_seq = inp.slot_stride

    def partials(self, ns, ws, out, lse, stream):
        return self.mv.verify_partials(self.q, self.kv, self.st, self.sl, self.mk, self.inp.scale, nsplit=ns,
                                       workspace=ws, out=out, lse=lse, stream=stream)

    def full(self, ns, ws, out, lse, stream):
        self.mv.verify_attn(self.q, self.kv, self.st, self.sl, self.mk, self.inp.scale, out=out, lse=lse,
                            nsplit=ns, workspace=ws, stream=stream)

    def stage(self):
        """A step's inputs in one pinned buffer and one device buffer: queries, slot table,
        lengths, mask and the q_len new draft KV rows of every stream ([B, q_len, 576],
        staged for the KV append kernel, which writes them into their pool slots).  The
        call's tensors are rebound to views of the device buffer.  Returns (host, device)."""
        import torch
        inp = self.inp
        named = [("q", torch.from_numpy(inp.q_bits.view(np.int16))),
                 ("st", torch.from_numpy(np.ascontiguousarray(inp.slot_table))),
                 ("sl", torch.from_numpy(np.ascontiguousarray(inp.seq_lens)))]
        if self.mk is not None:
            named.append(("mk", torch.from_numpy(np.ascontiguousarray(inp.mask))))
        rows = np.empty((inp.B, inp.q_len, 576), np.uint16)
        for b in range(inp.B):
            n = int(inp.seq_lens[b])
            rows[b] = inp.kv_bits[inp.slot_table[b, n - inp.q_len:n]]
        named.append(("new_rows", torch.from_numpy(rows.view(np.int16))))
        hbuf, dbuf, v = stage_inputs(named, self.dev)
        self.q, self.st, self.sl = v["q"].view(torch.bfloat16), v["st"], v["sl"]
        if self.mk is not None:
            self.mk = v["mk"]
        self.new_rows = v["new_rows"].view(torch.bfloat16)
        return hbuf, dbuf

    def before_call(self, stream):
        """KV append of the staged draft rows (end-to-end step only); returns launches."""
        self.mv.kv_append(self.kv, self.st, self.sl, self.new_rows, stream=stream)
        return 1

    def oracle_call(self, threads):
        import oracle
        oracle.verify_inputs(self.inp, nthreads=threads)


class Fp8Workload:
    def __init__(self, f, mv, dev):
        import torch
        self.f, self.mv, self.dev = f, mv, dev
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.q = t(f.q_bits.view(np.int16)).view(torch.bfloat16)
        self.lat, self.sc = t(f.kv_lat), t(f.kv_scale)
        self.rope = t(f.kv_rope.view(np.int16)).view(torch.bfloat16)
        self.ts = t(f.topk_slots)
        self.B, self.q_len, self.H = f.B, 1, f.H
        self.work = algorithmic_fp8(f)
        self.max_seq = f.topk

    def partials(self, ns, ws, out, lse, stream):
        return self.mv.sparse_fp8_decode(self.q, self.lat, self.sc, self.rope, self.ts, self.f.scale, out=out.view(self.B, self.H, 512),
                                         lse=lse.view(self.B, self.H), nsplit=ns, workspace=ws, stream=stream,
                                         partials_only=True)

    def full(self, ns, ws, out, lse, stream):
        self.mv.sparse_fp8_decode(self.q, self.lat, self.sc, self.rope, self.ts, self.f.scale, out=out.view(self.B, self.H, 512),
                                  lse=lse.view(self.B, self.H), nsplit=ns, workspace=ws, stream=stream)

    def stage(self):
        """A step's inputs in one pinned buffer and one device buffer: queries, top-k lists
        and the one new token row per stream (latent codes, scale, rope; written into the
        pool by the fp8 append kernel).  Returns (host, device)."""
        import torch
        f = self.f
        rows = np.ascontiguousarray(f.topk_slots[:, 0])
        named = [("q", torch.from_numpy(f.q_bits.view(np.int16))),
                 ("ts", torch.from_numpy(np.ascontiguousarray(f.topk_slots))),
                 ("new_slots", torch.from_numpy(rows)),
                 ("new_lat", torch.from_numpy(f.kv_lat[rows].copy())),
                 ("new_sc", torch.from_numpy(f.kv_scale[rows].copy())),
                 ("new_rope", torch.from_numpy(f.kv_rope[rows].view(np.int16).copy()))]
        hbuf, dbuf, v = stage_inputs(named, self.dev)
        self.q, self.ts = v["q"].view(torch.bfloat16), v["ts"]
        self.new_slots, self.new_lat, self.new_sc = v["new_slots"], v["new_lat"], v["new_sc"]
        self.new_rope = v["new_rope"].view(torch.bfloat16)
        return hbuf, dbuf

    def before_call(self, stream):
        """fp8 KV append of the staged new rows (end-to-end step only); returns launches."""
        self.mv.kv_append_fp8(self.lat, self.sc, self.rope, self.new_slots, self.new_lat, self.new_sc, self.new_rope,
                              stream=stream)
        return 1

    def oracle_call(self, threads):
        import oracle
        oracle.sparse_fp8_inputs(self.f, nthreads=threads)


def make_workload(name, mv, dev):
    if name == "c5":
        return Fp8Workload(w.config_fp8(name), mv, dev)
    return VerifyWorkload(w.config(name), mv, dev)


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

    wl = make_workload(args.config, mv, dev)
    work = wl.work
    peaks = load_peaks()
    rl_us, bound, t_mem, t_mma = roofline_us(work, peaks["hbm_gbs"], peaks["bf16_tflops"])
    B, q_len, H = wl.B, wl.q_len, wl.H
    # workspace for the automatic split count; the calls pass --nsplit (0 = automatic, which
    # for 2..64 streams is the balanced split over one wave of CTAs when it fits)
    ns = args.nsplit or mv.auto_nsplit(B, q_len, H, wl.max_seq, mv.num_sms(dev), 1 << 62)
    ws = torch.empty(max(mv.workspace_bytes(B, q_len, H, ns), 256), dtype=torch.uint8, device=dev)
    call_ns = args.nsplit
    split_desc = f"uniform, {ns} per stream"
    if call_ns == 0 and isinstance(wl, Fp8Workload):
        # the fp8 call's automatic count: one wave (equal-length streams), >= 128 keys per split
        tiles = -(-H // 80)
        ns = max(1, min(mv.num_sms(dev) // (B * tiles), -(-wl.max_seq // 128)))
        split_desc = f"uniform, {ns} per stream (one wave)"
    if call_ns == 0 and not isinstance(wl, Fp8Workload) and 2 <= B <= 64:
        tiles = -(-(q_len * H) // 96)
        slots = mv.num_sms(dev) // tiles
        need = -(-(slots * q_len * H * 512 * 4) // 256) * 256 + -(-(slots * q_len * H * 4) // 256) * 256
        if slots - B >= B and need <= ws.numel():
            split_desc = f"balanced, {slots} slots over all streams (one wave)"
            ns = slots
    out = torch.empty((B, q_len, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2_lines(i, clean=True):
        """Evict L2: write 256 MiB (> 2x L2); then, unless clean is False, read another
        256 MiB, which writes the dirty flush lines back and leaves L2 holding clean lines
        of a buffer the call never touches."""
        flush.fill_(float(i))
        if clean:
            torch.sum(flush_rd, dim=0, out=flush_sum)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 1 + (1 if ns > 1 else 0)

    def timed_loop(n, fn, flush_l2=True, clean=True):
        """n calls of fn(), each bracketed by CUDA events on the launching stream; L2 flushed
        before each call (outside the events) unless flush_l2 is False (clean=False: the
        write-only flush, whose dirty lines are written back during the call).  Returns ms
        per call.
        Each step ends with a synchronize, and the GPU is kept busy while the host submits
        the next call -- by the flush, or without one by a ~100 us device-side spin that
        touches no memory -- so the events never time the GPU waiting for the host (a loop
        that queued every step at once measured c4 at 222 us per call against 72 us once the
        host fell behind)."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        torch.cuda.synchronize(dev)
        for i in range(n):
            if flush_l2:
                flush_l2_lines(i, clean)
            else:
                torch.cuda._sleep(200_000)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
            torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    def full_call():
        wl.full(call_ns, ws, out, lse, stream)

    def split_kernel():
        wl.partials(call_ns, ws, out, lse, stream)

    for _ in range(max(args.warmup, 3)):
        flush_l2_lines(1)
        full_call()
        split_kernel()
    torch.cuda.synchronize(dev)

    clocks = Clocks(local, None if args.clocks_csv is None else args.clocks_csv.replace("{gpu}", str(local)))
    clocks.start()
    time.sleep(0.25)
    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    step_ms = timed_loop(K, full_call)                     # the timed region: K whole verify calls
    wall_dev = time.perf_counter() - wall0
    kern_ms = timed_loop(min(K, 500), split_kernel)        # the split (attention) kernel alone
    warm_ms = timed_loop(min(K, 200), full_call, flush_l2=False)
    dirty_ms = timed_loop(min(K, 200), full_call, clean=False)
    status = mv.device_status(stream)

    # end to end through the C ABI with host buffers: this step's inputs copied from
    # pinned memory (one staged buffer), the KV append (verify path), the call
    # (mla_verify_attn / mla_sparse_fp8_decode), and D2H of out and lse (one buffer), all
    # inside the events
    h_in, d_in = wl.stage()
    d_res = torch.empty(out.numel() + lse.numel(), dtype=torch.float32, device=dev)
    out_e, lse_e = d_res[:out.numel()].view(out.shape), d_res[out.numel():].view(lse.shape)
    h_res = torch.empty(d_res.numel(), dtype=torch.float32).pin_memory()
    h2d = h_in.numel()
    d2h = h_res.numel() * 4

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        wl.before_call(stream)
        wl.full(call_ns, ws, out_e, lse_e, stream)
        h_res.copy_(d_res, non_blocking=True)

    for _ in range(3):
        e2e_step()
    e2e_ms = timed_loop(max(1, min(K, 200)), e2e_step)
    clk = clocks.stop()

    # aggregate over ranks: max time, summed work
    mean_step = statistics.mean(step_ms)
    mean_kern = statistics.mean(kern_ms)
    mean_e2e = statistics.mean(e2e_ms)
    mean_warm = statistics.mean(warm_ms)
    mean_dirty = statistics.mean(dirty_ms)
    mean_step, mean_kern, mean_e2e, mean_warm, mean_dirty = max_over_ranks(
        [mean_step, mean_kern, mean_e2e, mean_warm, mean_dirty], device=dev)
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
        r = time_oracle(wl, args.cpu_seconds)
        # one core: a single call (or a few) of the same oracle, bounded by a quarter of the budget;
        # skipped when one call would take over 20 s on one core
        r1 = None
        if r["seconds_per_call"] * r["threads"] <= 20.0:
            r1 = time_oracle(wl, args.cpu_seconds / 4, max_reps=3, threads=1)
        cpu = {"value": work["kv_bytes"] / r["seconds_per_call"] / 1e9, "unit": UNIT, "cores": r["threads"],
               "kind": "oracle",
               "sample": f"{r['reps']} full fp64 oracle calls on the whole {args.config} workload "
                         f"({r['seconds_per_call'] * 1e3:.1f} ms/call)",
               "single_core": None if r1 is None else
               {"value": work["kv_bytes"] / r1["seconds_per_call"] / 1e9, "unit": UNIT,
                "sample": f"{r1['reps']} call(s) on one thread ({r1['seconds_per_call'] * 1e3:.1f} ms/call)"}}

    srt = sorted(step_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": mean_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (PAGES_C2_US / (mean_step * 1e3)) if args.config == "c2" and world == 1 else None,
        "dtype": "bf16", "data": "synthetic (seeded SplitMix64 / Box-Muller inputs, shapes of the pages' workloads)",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config, "B": B, "q_len": q_len,
                   "H": H, "keys": work["keys"], "nsplit": ns, "split": split_desc,
                   "l2": "flushed before every step, outside the timed events: 256 MiB written, then "
                         "another 256 MiB read (no dirty flush line left to write back inside the call)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_call": mean_step * 1e3,
        "us_per_call_p10_p50_p90": [srt[int(0.1 * (K - 1))] * 1e3, srt[(K - 1) // 2] * 1e3, srt[int(0.9 * (K - 1))] * 1e3],
        "us_per_call_warm_l2": mean_warm * 1e3,
        "us_per_call_write_only_flush": mean_dirty * 1e3,
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
    ap.add_argument("--config", default="c4", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi clock samples of the timed region in this file ({gpu} = GPU index)")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
