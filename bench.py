#!/usr/bin/env python3
"""Bench of paged-KV decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 1..5]

One step is one pass of the decode hot path over one batch of the seeded
synthetic workload (default: the Llama-3-8B-shaped GQA decode, 256 sequences,
32 q / 8 kv heads, D=128, block 16, L~U[1024,8192], 4.8 GB of KV -- larger than
L2, so no flush is needed between steps).  Rank 0 prints one JSON line with
the whole-job HBM GB/s (algorithmic bytes: valid K/V + q + fp32 out + table
entries + lengths), the roofline of the dominant kernel, an end-to-end figure
through the public API with host buffers, the CPU oracle as a reference
baseline, the SM clocks seen during the timed region, and the other named
workloads measured the same way.

With torchrun (N > 1) every rank runs its own replica of the batch (weak
scaling, no collective on the data path); timing is bracketed by barriers and
the slowest rank counts.  --impl reference times the CPU oracle instead (rank 0
only) on a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s (% of 8 TB/s) and seq-steps/s, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
DECODE_SOURCES = ["paged_kv_decode_pf_gb300/csrc/pf_decode.cuh", "paged_kv_decode_pf_gb300/csrc/pf_device.cuh",
                  "paged_kv_decode_pf_gb300/csrc/pf_internal.h",
                  "paged_kv_decode_pf_gb300/csrc/pf_decode_d128.cu", "paged_kv_decode_pf_gb300/csrc/pf_decode_d64.cu"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-extras", action="store_true", help="skip the other named workloads")
    ap.add_argument("--oracle-seconds", type=float, default=15.0, help="CPU work of the oracle baseline sample")
    ap.add_argument("--seqs", type=int, default=0,
                    help="profiling aid: keep only the first N sequences of the workload (0 = all)")
    ap.add_argument("--multi-query", type=int, default=0, metavar="Q",
                    help="profiling aid: time only pf_paged_attention_multi_query with Q new tokens per "
                         "sequence on the workload's cache and print a short line (0 = the normal bench)")
    ap.add_argument("--decode-variant", default="decode", choices=["decode", "split", "auto"],
                    help="headline path: single-pass decode, partition+merge, or the auto decode's own plan")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor peak for a kernel timed alone: MEASURED_PEAKS.json's burst figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured burst, MEASURED_PEAKS.json bf16_tflops"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


def decode_source_sha() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch recorded by an ncu capture of the current decode sources, if any."""
    sha = decode_source_sha()
    pat = re.compile(r"traffic-record:\s+workload=(\S+)\s+kernel=(\S+)\s+bytes_per_launch=(\d+)\s+source_sha=(\w+)")
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for m in pat.finditer(f.read()):
                if m.group(1) == workload and m.group(4) == sha:
                    return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons around the timed region."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.t_start = self.t_end = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def start(self):
        self.t_start = time.time()

    def stop(self):
        self.t_end = time.time()

    def close(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        win = [p for t, p in self.samples if self.t_start is not None and self.t_start <= t <= (self.t_end or t)]
        src = "timed region"
        if not win:
            win = [p for _, p in self.samples]
            src = "whole run (timed region shorter than the sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        smax = [num(p[1]) for p in win if num(p[1]) is not None]
        pw = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in win for n, v in zip(names, p[4:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(win), "window": src}


# -------------------------------------------------------------- GPU runner

class Runner:
    """Device-resident inputs of one workload and the launches of one step."""

    def __init__(self, pf, wl, dev, variant="decode"):
        import torch
        self.pf, self.wl, self.dev = pf, wl, dev

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.q, self.kc, self.vc = bf(wl.q), bf(wl.k_cache), bf(wl.v_cache)
        self.bt = torch.from_numpy(wl.block_tables).to(dev)
        self.cl = torch.from_numpy(wl.context_lens).to(dev)
        self.out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
        self.append = wl.slot_mapping is not None
        if self.append:
            self.nk, self.nv = bf(wl.new_k), bf(wl.new_v)
            self.sm = torch.from_numpy(wl.slot_mapping).to(dev)
        self.auto = variant == "auto"  # pf_paged_attention_decode_auto with the true longest context
        self.split = not self.auto and (variant == "split" or wl.partition_size is not None)
        self.cluster = False
        if self.auto:
            self.max_ctx = wl.max_context_len
            self.P, need = pf.decode_auto_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                               self.max_ctx, dev)
            self.ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
        # the cluster split: a chunk size and no workspace (one launch)
        self.cluster = self.auto and self.P > 0 and not need
        if self.split:
            self.P = wl.partition_size or 512
            self.max_ctx = wl.max_context_len
            self.ws = pf.alloc_workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, self.max_ctx, self.P, dev)
        self.fused = self.append and not self.split and variant == "fused"
        self.bf16 = variant == "bf16" and not self.split and not self.append  # the bf16-output single pass
        if self.bf16:
            self.out_bf16 = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16,
                                        device=dev)
        self.kernels_per_step = 1 if self.fused else (1 if self.append else 0) + (
            2 if self.split or (self.auto and self.P and not self.cluster) else 1)
        self.dominant = "partition" if self.split else ("decode_append" if self.fused else "decode")

    def step(self, ev=None):
        """One pass; when `ev` is a pair of CUDA events they bracket the dominant kernel."""
        pf = self.pf
        if self.fused:   # append and attend in one launch
            if ev is not None:
                ev[0].record()
            pf.paged_attention_decode_append(self.q, self.nk, self.nv, self.sm, self.kc, self.vc, self.bt, self.cl,
                                             self.wl.scale, self.out)
            if ev is not None:
                ev[1].record()
            return
        if self.append:
            pf.reshape_and_cache(self.nk, self.nv, self.sm, self.kc, self.vc)
        if ev is not None:
            ev[0].record()
        if self.auto:    # the whole call (single pass, or partition + merge) is the dominant region
            pf.paged_attention_decode_auto(self.q, self.kc, self.vc, self.bt, self.cl, self.max_ctx, self.wl.scale,
                                           self.ws, self.out)
            if ev is not None:
                ev[1].record()
            return
        if self.split:
            pf.paged_attention_decode_partition(self.q, self.kc, self.vc, self.bt, self.cl, self.P, self.max_ctx,
                                                self.ws, self.wl.scale)
            if ev is not None:
                ev[1].record()
            pf.paged_attention_merge(self.ws, self.cl, self.wl.num_q_heads, self.wl.head_dim, self.P, self.max_ctx,
                                     self.out)
        elif self.bf16:
            pf.paged_attention_decode_bf16(self.q, self.kc, self.vc, self.bt, self.cl, self.wl.scale, self.out_bf16)
            if ev is not None:
                ev[1].record()
        else:
            pf.paged_attention_decode(self.q, self.kc, self.vc, self.bt, self.cl, self.wl.scale, self.out)
            if ev is not None:
                ev[1].record()

    def step_bytes(self):
        b = self.wl.algorithmic_bytes(with_append=self.append)
        if self.bf16:      # the output is written as bf16: 2 bytes per element instead of 4
            b -= self.wl.num_seqs * self.wl.num_q_heads * self.wl.head_dim * 2
        return b

    def dominant_bytes(self):
        """Algorithmic bytes of the dominant kernel alone."""
        wl = self.wl
        b = wl.algorithmic_bytes(with_append=False)
        if self.bf16:
            b -= wl.num_seqs * wl.num_q_heads * wl.head_dim * 2
        if self.split:     # the partition pass reads everything but writes partials, not out
            b -= wl.num_seqs * wl.num_q_heads * wl.head_dim * 4
        return b


def host_seconds_per_step(runner, flush=None, n=10):
    """Host time to enqueue one step (the Python binding's argument checks and launches)."""
    import torch
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(n):
        runner.step()
        if flush is not None:
            flush.zero_()
    host = (time.perf_counter() - t) / n
    torch.cuda.synchronize()
    return host


def hold_gpu(seconds):
    """Queue a spin kernel so that everything enqueued after it runs back to back on the
    GPU, even when the host takes longer to enqueue a step than the GPU takes to run it."""
    import torch
    if seconds > 0:
        torch.cuda._sleep(int(min(seconds, 2.0) * 2.2e9))


def time_steps(runner, steps, warmup, flush=None, dist=None, sampler=None):
    """(ms per step over the timed region, mean ms of the dominant kernel, per-launch ms list).

    A spin kernel queued first covers the host's enqueue time of the whole loop, so
    the events measure the GPU back to back rather than the host's launch rate."""
    import torch
    for _ in range(warmup):
        runner.step()
        if flush is not None:
            flush.zero_()
    host = host_seconds_per_step(runner, flush)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    hold_gpu(1.5 * host * steps + 0.005)
    if sampler is not None:
        sampler.start()
    t0.record()
    for k in range(steps):
        runner.step(evs[k])
        if flush is not None:
            flush.zero_()
    t1.record()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.stop()
    if dist is not None:
        dist.barrier()
    total = t0.elapsed_time(t1)
    per = [a.elapsed_time(b) for a, b in evs]
    return total / steps, statistics.fmean(per), per


def max_over_ranks(value, dist, device):
    """The largest `value` over all ranks (the slowest rank decides the job's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_step_per_rank, ms_per_step):
    """Whole-job GB/s: every rank processes its own batch (weak scaling) in the slowest rank's time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


class MultiQueryRunner:
    """pf_paged_attention_multi_query over a resident workload: the last q_len tokens of
    every sequence are its new tokens (draft tokens under verification)."""

    def __init__(self, pf, runner, q_len, kernel="auto"):
        import torch
        from workloads import multi_query
        self.pf, self.r, self.q_len, self.kernel = pf, runner, q_len, kernel
        wl = runner.wl
        q = multi_query(wl, q_len)
        self.q = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).to(runner.dev)
        self.out = torch.empty((wl.num_seqs, q_len, wl.num_q_heads, wl.head_dim), dtype=torch.float32,
                               device=runner.dev)

    def step(self, ev=None):
        r = self.r
        if ev is not None:
            ev[0].record()
        self.pf.paged_attention_multi_query(self.q, r.kc, r.vc, r.bt, r.cl, r.wl.scale, self.out, kernel=self.kernel)
        if ev is not None:
            ev[1].record()

    def step_bytes(self):
        wl = self.r.wl
        rows = wl.num_seqs * self.q_len * wl.num_q_heads * wl.head_dim
        return wl.algorithmic_bytes() - wl.num_seqs * wl.num_q_heads * wl.head_dim * 6 + rows * 6

    def step_flops(self):
        """Useful flops: 4 D per (query row, visible token) -- Q.K and P.V, causal limits applied."""
        wl = self.r.wl
        L = wl.context_lens.astype(np.int64)
        vis = sum(np.clip(L - self.q_len + j + 1, 0, None).sum() for j in range(self.q_len))
        return int(4 * wl.head_dim * wl.num_q_heads * vis)


class CopyRunner:
    """pf_copy_blocks over `pairs` random (src, dst) pairs of Llama-3-8B-shaped blocks
    (8 kv heads x 16 tokens x 128 dims, bf16): a pure read + write stream."""

    def __init__(self, pf, dev, pairs=4096, num_blocks=8192, shape=(8, 16, 128)):
        import torch
        self.pf = pf
        g = torch.Generator(device=dev).manual_seed(11)
        self.kc = torch.empty((num_blocks,) + shape, dtype=torch.bfloat16, device=dev)
        self.vc = torch.empty_like(self.kc)
        perm = torch.randperm(num_blocks, device=dev, generator=g)
        self.mapping = torch.stack([perm[:pairs], perm[pairs:2 * pairs]], dim=1).contiguous()
        self.pairs = pairs
        self.block_bytes = int(np.prod(shape)) * 2

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.pf.copy_blocks(self.kc, self.vc, self.mapping)
        if ev is not None:
            ev[1].record()

    def step_bytes(self):
        return self.pairs * 2 * self.block_bytes * 2      # K and V, read and written


def time_e2e(runner, steps, warmup):
    """Same step through the public API with every step's inputs copied from pinned host memory
    and its output read back; the KV cache is the resident state the step reads in place.

    The loop is pipelined the usual way: two sets of device input/output buffers, host-to-device
    copies on one stream, device-to-host on another, so step k+1's inputs arrive and step k-1's
    output leaves while step k computes.  The timed region runs from the first copy in to the
    last copy out."""
    import torch
    wl = runner.wl
    names = ["q", "bt", "cl"] + (["nk", "nv", "sm"] if runner.append else [])
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    host = {"q": bf(wl.q), "bt": torch.from_numpy(wl.block_tables).pin_memory(),
            "cl": torch.from_numpy(wl.context_lens).pin_memory()}
    if runner.append:
        host.update(nk=bf(wl.new_k), nv=bf(wl.new_v), sm=torch.from_numpy(wl.slot_mapping).pin_memory())
    sets = [{n: getattr(runner, n) for n in names}, {n: getattr(runner, n).clone() for n in names}]
    sets[0]["out"], sets[1]["out"] = runner.out, torch.empty_like(runner.out)
    out_host = [torch.empty(runner.out.shape, dtype=runner.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_host[0].numel() * out_host[0].element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def one(k):
        b = k % 2
        cur = sets[b]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(done[b])          # step k-2 has finished reading this set
            for n in names:
                cur[n].copy_(host[n], non_blocking=True)
            ready[b].record(s_in)
        comp.wait_event(ready[b])
        if k >= 2:
            comp.wait_event(drained[b])           # step k-2's output has left this buffer
        for n in names:
            setattr(runner, n, cur[n])
        runner.out = cur["out"]
        runner.step()
        done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            out_host[b].copy_(cur["out"], non_blocking=True)
            drained[b].record(s_out)

    for k in range(warmup):
        one(k)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_in)
    for k in range(steps):
        one(k)
    t1.record(s_out)
    torch.cuda.synchronize()
    for n in names:
        setattr(runner, n, sets[0][n])
    runner.out = sets[0]["out"]
    return t0.elapsed_time(t1) / steps, h2d, d2h


def workload_description(wl, index):
    from workloads import CONFIGS
    return f"{CONFIGS[index].name}: {CONFIGS[index].description} (seed {wl.seed})"


# ------------------------------------------------------------ CPU oracle

def oracle_sample_run(orc, wl, target_s, threads=0):
    """Time the oracle on the first n sequences, n calibrated to about target_s seconds.
    Returns (seconds, sample bytes, n, description)."""
    import dataclasses

    def sub(n):
        return dataclasses.replace(wl, num_seqs=n, q=wl.q[:n], block_tables=wl.block_tables[:n],
                                   context_lens=wl.context_lens[:n], slot_mapping=None, new_k=None, new_v=None)

    def run(w):
        t = time.perf_counter()
        orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, threads=threads)
        return time.perf_counter() - t
    t1 = run(sub(1))
    n = int(max(1, min(wl.num_seqs, math.floor(target_s / max(t1, 1e-6)))))
    w = sub(n)
    secs = run(w) if n > 1 else t1
    tokens = int(w.context_lens.astype(np.int64).sum())
    desc = f"first {n} of {wl.num_seqs} sequences, all {wl.num_q_heads} query heads ({tokens} tokens)"
    return secs, w.algorithmic_bytes(), n, desc


# ------------------------------------------------------------------- main

def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peak, peak_src = measured_peak()

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    import torch.distributed as tdist

    dist = None
    if world > 1:
        tdist.init_process_group(backend="nccl", init_method="env://")
        dist = tdist
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    from paged_kv_decode_pf_gb300 import _build
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    import paged_kv_decode_pf_gb300 as pf
    from workloads import CONFIGS, make_config

    wl = first_sequences(make_config(args.workload), args.seqs)
    runner = Runner(pf, wl, dev, args.decode_variant)
    if args.multi_query > 0:
        return profile_multi_query(pf, runner, args)
    flush = None
    if runner.step_bytes() < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    ms_step, ms_dom, per = time_steps(runner, args.steps, max(args.warmup, 3), flush, dist, sampler)
    pf.check_device_error()
    sampler.close()
    ms_step = max_over_ranks(ms_step, dist, dev)
    step_bytes = runner.step_bytes()
    value = job_throughput(world, step_bytes, ms_step)
    dom_bytes = runner.dominant_bytes()
    achieved = dom_bytes / (ms_dom * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_e2e(runner, min(args.steps, 500), 3)
    pf.check_device_error()
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9
    # what the line reports about the timed step (the extras below free the runner's cache)
    step_text, kernel_text, kernels_per_step = runner_step(runner), runner_kernel(runner), runner.kernels_per_step

    extras = {}
    if not args.no_extras and rank == 0:
        g = wl.num_q_heads // wl.num_kv_heads
        runs = [(q_len, "auto") for q_len in (4, 8, 12, 16)]
        if wl.head_dim == 128:
            runs += [(8, "tcgen05")]  # past 32 rows the default entry runs the tcgen05 kernel itself
        runs += [(64, "auto"), (128, "auto")]  # prompt chunks: past 64 rows per kv head, the chunk kernel
        bf16_peak = measured_bf16_peak()
        for q_len, kernel in runs:
            if runner.split or g * q_len > 65536:
                continue
            # the same resident cache, with the last q_len tokens of every sequence as new (draft) tokens
            mr = MultiQueryRunner(pf, runner, q_len, kernel)
            ms_s, ms_d, _ = time_steps(mr, 200, 10)
            pf.check_device_error()
            mb = mr.step_bytes()
            fl = mr.step_flops()
            name = "pf_paged_attention_multi_query" + ("_tcgen05" if kernel == "tcgen05" else "")
            chunk = g * q_len > 64
            extras[CONFIGS[args.workload].name + f"_multi_query_q{q_len}" + ("_tcgen05" if kernel == "tcgen05" else "")] = {
                "description": f"{name} on the same cache: {q_len} new tokens per "
                               f"sequence, causal among them ({g * q_len} query rows per kv head"
                               + (", prompt-chunk kernel)" if chunk else ")"),
                "step": "multi_query", "us_dominant_kernel": round(ms_d * 1e3, 2), "algorithmic_bytes": mb,
                "gbs_dominant_kernel": round(mb / (ms_d * 1e-3) / 1e9, 1),
                "pct_of_8tbs_dominant": round(100 * mb / (ms_d * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 1),
                "frac_of_measured_peak_dominant": round(mb / (ms_d * 1e-3) / 1e9 / peak, 3),
                "tflops_dominant_kernel": round(fl / (ms_d * 1e-3) / 1e12, 1),
                "frac_of_measured_bf16_peak": round(fl / (ms_d * 1e-3) / 1e12 / bf16_peak[0], 3),
                "bf16_peak": f"{bf16_peak[0]} TFLOP/s ({bf16_peak[1]})",
                "l2": "inputs larger than L2",
            }
            del mr
        del runner
        torch.cuda.empty_cache()
        for idx, variant in [(4, "bf16"), (1, "decode"), (1, "auto"), (2, "decode"), (2, "auto"), (3, "decode"),
                             (3, "fused"), (5, "decode"), (5, "auto")]:
            if idx == args.workload and variant == "decode":
                continue
            w = make_config(idx)
            r = Runner(pf, w, dev, variant)
            fl = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if r.step_bytes() < 2 * L2_BYTES \
                else None
            n = 200 if fl is None else 400
            ms_s, ms_d, _ = time_steps(r, n, 10, fl)
            pf.check_device_error()
            b = r.step_bytes()
            extras[CONFIGS[idx].name + ("_fused" if r.fused else "_auto" if r.auto else "_bf16_out" if r.bf16 else "")] = {
                "description": CONFIGS[idx].description,
                "step": "append and decode fused in one launch" if r.fused else
                        "decode with a bf16 output (pf_paged_attention_decode_bf16)" if r.bf16 else
                        (f"decode_auto ({('cluster split, chunk ' + str(r.P) + ' tokens per CTA, one launch') if r.cluster else ('partition + merge, P=' + str(r.P)) if r.P else 'single pass'}, "
                         f"max_context_len {r.max_ctx})") if r.auto else
                        ("append + " if r.append else "") + ("partition + merge" if r.split else "decode"),
                "us_per_step": round(ms_s * 1e3, 2) if fl is None else None,
                "us_dominant_kernel": round(ms_d * 1e3, 2),
                "algorithmic_bytes": b,
                "gbs_step": round(b / (ms_s * 1e-3) / 1e9, 1) if fl is None else None,
                "gbs_dominant_kernel": round(r.dominant_bytes() / (ms_d * 1e-3) / 1e9, 1),
                "pct_of_8tbs_dominant": round(100 * r.dominant_bytes() / (ms_d * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 1),
                "frac_of_measured_peak_dominant": round(r.dominant_bytes() / (ms_d * 1e-3) / 1e9 / peak, 3),
                "seq_steps_per_s": round(w.num_seqs / ((ms_s if fl is None else ms_d) * 1e-3), 1),
                "l2": "flushed between steps (kernel time only)" if fl is not None else "inputs larger than L2",
            }
            del r, fl
            torch.cuda.empty_cache()
        cr = CopyRunner(pf, dev)
        ms_s, ms_d, _ = time_steps(cr, 200, 10)
        pf.check_device_error()
        cb = cr.step_bytes()
        extras["copy_blocks"] = {
            "description": "pf_copy_blocks: 4096 (src, dst) pairs of 8x16x128 bf16 blocks, K and V "
                           "(268 MB read + 268 MB written)",
            "step": "copy_blocks", "us_dominant_kernel": round(ms_d * 1e3, 2), "algorithmic_bytes": cb,
            "gbs_dominant_kernel": round(cb / (ms_d * 1e-3) / 1e9, 1),
            "frac_of_measured_copy_peak": round(cb / (ms_d * 1e-3) / 1e9 / peak, 3),
            "l2": "inputs larger than L2",
        }
        del cr
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0:
        import oracle
        orc = oracle.load()
        secs, sb, n, desc = oracle_sample_run(orc, wl, args.oracle_seconds)
        cpu = {"value": round(sb / secs / 1e9, 4), "unit": "GB/s", "cores": orc.max_threads(), "kind": "oracle",
               "sample": desc, "seconds": round(secs, 3),
               "seq_steps_per_s": round(n / secs, 3)}
        secs1, sb1, n1, desc1 = oracle_sample_run(orc, wl, min(args.oracle_seconds, 5.0), threads=1)
        cpu["single_thread"] = {"value": round(sb1 / secs1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": desc1, "seconds": round(secs1, 3),
                                "seq_steps_per_s": round(n1 / secs1, 3)}

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32", "storage_dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(wl, args.workload),
                           step=step_text,
                           algorithmic_bytes_per_step=step_bytes,
                           l2="inputs larger than L2, no flush" if flush is None else "L2 flushed between steps",
                           parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "seq_steps_per_s": round(world * wl.num_seqs / (ms_step * 1e-3), 1),
            "us_per_call": round(ms_step * 1e3, 2),
            "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": profiled_traffic(CONFIGS[args.workload].name),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback 6.8 TB/s", "kernel": kernel_text,
                         "kernel_us_mean": round(ms_dom * 1e3, 2),
                         "kernel_us_p10_p90": [round(float(np.percentile(per, 10)) * 1e3, 2),
                                               round(float(np.percentile(per, 90)) * 1e3, 2)]},
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "us_per_step": round(e2e_ms * 1e3, 2),
                    "note": "every step copies its inputs (q, block tables, lengths) in from pinned host "
                            "memory and its output back, pipelined on two copy streams with double-buffered "
                            "device inputs and outputs; the KV cache stays resident"},
            "gpu_launches": args.steps * kernels_per_step,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def workload_config(wl, index):
    """The workload's name and shape keys, the same in both arms' `config`."""
    return {"workload": workload_description(wl, index), "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "total_tokens": int(wl.context_lens.astype(np.int64).sum())}


def profile_multi_query(pf, runner, args):
    """--multi-query Q: the multi-token query alone on the resident cache, for profilers."""
    mr = MultiQueryRunner(pf, runner, args.multi_query)
    ms_s, ms_d, per = time_steps(mr, args.steps, max(args.warmup, 3))
    pf.check_device_error()
    fl = mr.step_flops()
    print(json.dumps({"profile": "pf_paged_attention_multi_query", "q_len": args.multi_query,
                      "rows_per_kv_head": runner.wl.group * args.multi_query, "num_seqs": runner.wl.num_seqs,
                      "us_mean": round(ms_d * 1e3, 2), "useful_tflops": round(fl / (ms_d * 1e-3) / 1e12, 1),
                      "algorithmic_bytes": mr.step_bytes()}), flush=True)


def first_sequences(wl, n):
    """The workload restricted to its first n sequences, with the pool compacted to the
    blocks they use (kept in pool order) and the tables and slots renumbered."""
    import dataclasses
    if n <= 0 or n >= wl.num_seqs:
        return wl
    L = wl.context_lens[:n].astype(np.int64)
    nblk = (L + wl.block_size - 1) // wl.block_size
    tables = wl.block_tables[:n].copy()
    used = np.unique(np.concatenate([tables[i, :nblk[i]] for i in range(n)]))
    remap = np.full(wl.num_blocks, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    for i in range(n):
        tables[i, :nblk[i]] = remap[tables[i, :nblk[i]]]
    sm = None
    if wl.slot_mapping is not None:
        s = wl.slot_mapping[:n].copy()
        ok = s >= 0
        s[ok] = remap[s[ok] // wl.block_size] * wl.block_size + s[ok] % wl.block_size
        sm = s
    return dataclasses.replace(wl, num_seqs=n, num_blocks=int(used.size), q=wl.q[:n], block_tables=tables,
                               context_lens=wl.context_lens[:n], k_cache=np.ascontiguousarray(wl.k_cache[used]),
                               v_cache=np.ascontiguousarray(wl.v_cache[used]), slot_mapping=sm,
                               new_k=None if sm is None else wl.new_k[:n], new_v=None if sm is None else wl.new_v[:n])


def runner_step(runner):
    """The timed step's entry points, as the line's config.step names them."""
    if runner.auto:
        plan = ("cluster split, chunk %d tokens per CTA" % runner.P if runner.cluster else
                "partition + merge, P=%d" % runner.P if runner.P else "single pass")
        return f"pf_paged_attention_decode_auto ({plan})"
    if runner.split:
        return "pf_paged_attention_decode_partition + pf_paged_attention_merge"
    return ("pf_reshape_and_cache + " if runner.append else "") + "pf_paged_attention_decode"


def runner_kernel(runner):
    if runner.split or (runner.auto and runner.P and not runner.cluster):
        return "paged_decode_kernel (partition pass)"
    if runner.cluster:
        return "paged_decode_kernel (cluster split)"
    return "paged_decode_kernel"


def reference_arm(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 times it on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    from workloads import make_config
    wl = make_config(args.workload)
    orc = oracle.load()
    steps, warmup = args.steps, max(args.warmup, 3)
    per_step = max(0.02, min(args.oracle_seconds, 150.0 / (steps + warmup)))
    secs1, sb, n, desc = oracle_sample_run(orc, wl, per_step)
    import dataclasses
    w = dataclasses.replace(wl, num_seqs=n, q=wl.q[:n], block_tables=wl.block_tables[:n],
                            context_lens=wl.context_lens[:n], slot_mapping=None, new_k=None, new_v=None)
    for _ in range(warmup):
        orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    t = time.perf_counter()
    for _ in range(steps):
        orc.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    el = (time.perf_counter() - t) / steps
    value = round(sb / el / 1e9, 4)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(el * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(wl, args.workload), sample=desc),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": orc.max_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
