"""Benchmark of the exact-attention forward path on GB300.

One timed step is one forward pass of causal prefill attention over the workload the headline
metric is quoted on (B=4, Hq=Hkv=32, S=4096, d=128, bf16, synthetic N(0,1) inputs). The same run
also times, with the same step and warm-up counts, the other workloads of the hot path: long-context
GQA prefill (S=32768), paged ragged prefill (64 sequences), paged split-KV decode (128
sequences), the paged KV append that fills the prefill batch's cache, decode behind a shared
prefix (cascade), a batch mixing prefill, chunked prefill and decode, and multi-token verify;
their numbers go to the "extra" object of the single JSON line rank 0 prints.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this project has) on a bounded
sample of the same workload. Under torchrun every rank runs the same per-GPU work (weak scaling,
no collective on the data path); rank 0 reports the whole-job throughput over the slowest rank.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from io_aware_exact_flash_gb300.workloads import (  # noqa: E402
    WORKLOADS,
    CascadeWorkload,
    PagedWorkload,
    make_append,
    make_cascade,
    make_dense,
    make_paged,
    paged_allowed_scores,
)

METRIC = "attn fwd TFLOP/s (prefill) & decode HBM GB/s on 1 GB300, % of roofline"
HEADLINE = "causal_prefill_b4_h32_s4096_d128"
EXTRAS = ["gqa_causal_prefill_b1_hq32_hkv8_s32768_d128", "paged_prefill_64seq_512_8192_hq32_hkv8_d128_p16",
          "paged_decode_128seq_1024_16384_hq32_hkv8_d128_p16", "paged_append_64seq_512_8192_hkv8_d128_p16",
          "cascade_decode_128seq_prefix16384_suffix256_2048_hq32_hkv8_d128_p16",
          "mixed_paged_64seq_512_8192_hq32_hkv8_d128_p16", "verify_paged_128seq_q2_8_kv1024_16384_hq32_hkv8_d128_p16",
          "paged_decode_16seq_1024_16384_hq32_hkv8_d128_p16",
          "paged_decode_128seq_1024_16384_hq32_hkv8_d128_p16@splits=4"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) of one headline prefill launch from an ncu capture, and the kernel
# state it was taken on (the digest of its sources without comments); the bench reports it as
# roofline.traffic only while that code is unchanged.
PREFILL_TRAFFIC = {"bytes": 433830656 + 111355136,
                   "source_sha256": "b436afe8a8638ec6ab6946daf906fa2e835754f64960a86444021467a88257d4"}
L2_FLUSH_BYTES = 512 << 20


# ----------------------------------------------------------------------------- distributed glue
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself with one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def prefill_source_digest():
    """SHA-256 of the prefill kernel's sources with // comments and blank lines removed, so that
    only a change to the code (not to its comments) retires the recorded ncu traffic figure."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in ("prefill.cu", "ptx.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "io_aware_exact_flash_gb300", "csrc", f)) as fh:
            lines = (re.sub(r"//.*$", "", line).rstrip() for line in fh.read().splitlines())
            h.update("\n".join(line for line in lines if line).encode())
    return h.hexdigest()


# ----------------------------------------------------------------------------- peaks and clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                raw = json.load(f)

            def pick(*names):
                for n in names:
                    for k, v in raw.items():
                        if k == n and isinstance(v, (int, float)):
                            return float(v)
                return None

            peaks = {"hbm_gbs": pick("hbm_gbs"), "bf16_tflops": pick("bf16_tflops"),
                     "bf16_tflops_sustained": pick("bf16_tflops_sustained")}
            if all(v is not None for v in peaks.values()):
                peaks["source"] = "measured"
                return peaks
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(text)):
            if len(row) < len(self.FIELDS):
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            for n, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads on device
def to_dev(bits, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def i32(a, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class DenseCase:
    def __init__(self, name, device):
        import torch

        self.w = WORKLOADS[name]
        t = make_dense(self.w)
        self.host = t
        self.q, self.k, self.v = (to_dev(t[x], device) for x in ("q", "k", "v"))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=device)
        self.flops = self.w.flops()
        self.kind = "prefill"

    def run(self):
        import io_aware_exact_flash_gb300 as fa

        fa.fa_fwd(self.q, self.k, self.v, causal=self.w.causal, scale=self.w.scale, out=self.o, lse=self.lse)

    launches = 1


class PagedCase:
    """A paged workload through fa_paged_fwd; num_splits > 0 forces that many key splits (their
    partial states then go through the LSE merge), 0 lets the planner choose."""

    def __init__(self, name, device, num_splits=0):
        import torch

        import io_aware_exact_flash_gb300 as fa

        self.w = WORKLOADS[name]
        self.num_splits = num_splits
        t = make_paged(self.w)
        self.host = t
        self.q = to_dev(t["q"], device)
        self.kp, self.vp = to_dev(t["k_pages"], device), to_dev(t["v_pages"], device)
        self.pt, self.cu, self.kl = i32(t["page_table"], device), i32(t["cu_seqlens_q"], device), i32(t["kv_lens"], device)
        self.max_q = int(t["q_lens"].max())
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=device)
        need = fa.fa_paged_workspace_bytes(self.w.num_seqs, t["total_q"], self.max_q, self.w.page_size,
                                           t["page_table"].shape[1], t["num_pages"], self.w.Hq, self.w.Hkv, self.w.d,
                                           num_splits)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.scores = paged_allowed_scores(t, self.w.Hq, self.w.causal)
        self.flops = 4.0 * self.w.d * self.scores
        # verify batches (a few query rows per sequence) are bound by reading K/V, like decode
        self.kind = "decode" if self.w.decode else ("verify" if 0 < self.w.q_hi <= 16 else "prefill")
        # algorithmic bytes of decode: every K and V row read once, q read, o and lse written
        kv_rows = int(t["kv_lens"].astype(np.int64).sum())
        self.bytes = (2 * kv_rows * self.w.Hkv * self.w.d * 2 + t["total_q"] * self.w.Hq * self.w.d * 2 * 2
                      + t["total_q"] * self.w.Hq * 4)
        self.splits = num_splits if num_splits > 0 else fa.fa_paged_num_splits(
            self.w.num_seqs, t["total_q"], self.max_q, self.w.page_size, t["page_table"].shape[1], t["num_pages"],
            self.w.Hq, self.w.Hkv, self.w.d)
        max_tiles = (t["page_table"].shape[1] * self.w.page_size + 127) // 128
        self.splits = min(self.splits, max_tiles)
        g = self.w.Hq // self.w.Hkv
        # decode runs on the tensor cores unless FA_DECODE_TC=0 sends it to the CUDA-core kernel
        self.tensor_cores = not (self.w.decode and os.environ.get("FA_DECODE_TC") == "0" and g in (1, 2, 4, 8))

    def run(self):
        import io_aware_exact_flash_gb300 as fa

        fa.fa_paged_fwd(self.q, self.kp, self.vp, self.pt, self.cu, self.kl, self.max_q, causal=self.w.causal,
                        scale=self.w.scale, out=self.o, lse=self.lse, workspace=self.ws, num_splits=self.num_splits)

    @property
    def launches(self):
        # tensor-core path: the planning kernel, the attention kernel, and the merge when the keys
        # are split; CUDA-core decode: one kernel (its merge is fused; the counter reset is a
        # cudaMemsetAsync, not a kernel)
        if not self.tensor_cores:
            return 1
        return 2 + (self.splits > 1)


class AppendCase:
    """Paged KV append of a whole batch's K/V rows into their pages (the cache fill of the paged
    prefill batch). Algorithmic bytes: every new K and V row read once and written once."""

    def __init__(self, name, device):
        import torch

        self.w = WORKLOADS[name]
        t = make_append(self.w)
        self.k_new, self.v_new = to_dev(t["k_new"], device), to_dev(t["v_new"], device)
        shape = (t["num_pages"], self.w.page_size, self.w.Hkv, self.w.d)
        self.kp = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.vp = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.cu, self.before = i32(t["cu_seqlens_new"], device), i32(t["kv_lens_before"], device)
        self.pt = i32(t["page_table"], device)
        self.bytes = 2 * 2 * t["total_new"] * self.w.Hkv * self.w.d * 2
        self.kind = "append"

    def run(self):
        import io_aware_exact_flash_gb300 as fa

        fa.fa_paged_append(self.k_new, self.v_new, self.cu, self.before, self.pt, self.kp, self.vp)

    launches = 1


class CascadeCase:
    """Decode batch behind one shared prefix through fa_cascade_fwd (prefix attended once for all
    query rows, then each suffix, then the merge). Algorithmic bytes: the shared prefix's K/V and
    every suffix's K/V read once, q read and O, LSE written. The same batch is also timed through
    fa_paged_fwd with flat page tables (each sequence reading the shared pages itself)."""

    def __init__(self, name, device):
        import torch

        import io_aware_exact_flash_gb300 as fa

        self.w = w = WORKLOADS[name]
        t = make_cascade(w)
        self.q = to_dev(t["q"], device)
        self.kp, self.vp = to_dev(t["k_pages"], device), to_dev(t["v_pages"], device)
        self.cu_g, self.pre_t, self.pre_l = (i32(t[k], device) for k in ("cu_q_groups", "prefix_page_table",
                                                                          "prefix_lens"))
        self.cu, self.pt, self.kl = (i32(t[k], device) for k in ("cu_seqlens_q", "page_table", "kv_lens"))
        self.flat_pt, self.flat_kl = i32(t["flat_page_table"], device), i32(t["flat_kv_lens"], device)
        self.total_q = t["total_q"]
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=device)
        need = fa.fa_cascade_workspace_bytes(1, w.num_seqs, self.total_q, self.total_q, w.q_len, w.page_size,
                                             t["prefix_page_table"].shape[1], t["page_table"].shape[1],
                                             t["num_pages"], w.Hq, w.Hkv, w.d)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        need_flat = fa.fa_paged_workspace_bytes(w.num_seqs, self.total_q, w.q_len, w.page_size,
                                                t["flat_page_table"].shape[1], t["num_pages"], w.Hq, w.Hkv, w.d)
        self.ws_flat = torch.empty(max(need_flat, 256), dtype=torch.uint8, device=device)
        # launches: each pass is planning + attention, the suffix pass also a merge when its keys
        # are split; the prefix pass's key splits go straight into the final merge
        sp_pre = fa.fa_paged_num_splits(1, self.total_q, self.total_q, w.page_size, t["prefix_page_table"].shape[1],
                                        t["num_pages"], w.Hq, w.Hkv, w.d)
        sp_suf = fa.fa_paged_num_splits(w.num_seqs, self.total_q, w.q_len, w.page_size, t["page_table"].shape[1],
                                        t["num_pages"], w.Hq, w.Hkv, w.d)
        self.launches = 2 + (2 + (sp_suf > 1)) + 1
        self.prefix_splits = sp_pre
        kv_rows = w.prefix_len + int(t["kv_lens"].astype(np.int64).sum())
        self.bytes = (2 * kv_rows * w.Hkv * w.d * 2 + self.total_q * w.Hq * w.d * 2 * 2 + self.total_q * w.Hq * 4)
        self.kind = "cascade"

    def run(self):
        import io_aware_exact_flash_gb300 as fa

        fa.fa_cascade_fwd(self.q, self.kp, self.vp, self.cu_g, self.pre_t, self.pre_l, self.total_q, self.cu,
                          self.pt, self.kl, self.w.q_len, causal=True, scale=self.w.scale, out=self.o, lse=self.lse,
                          workspace=self.ws)

    def run_flat(self):
        import io_aware_exact_flash_gb300 as fa

        fa.fa_paged_fwd(self.q, self.kp, self.vp, self.flat_pt, self.cu, self.flat_kl, self.w.q_len, causal=True,
                        scale=self.w.scale, out=self.o, lse=self.lse, workspace=self.ws_flat)



class FlatView:
    """Times CascadeCase.run_flat with the harness of time_case."""

    def __init__(self, case):
        self.run = case.run_flat


def make_case(name, device):
    """name is a workload name, optionally followed by "@splits=N" to force N key splits."""
    if "@splits=" in name:
        base, n = name.split("@splits=")
        return PagedCase(base, device, num_splits=int(n))
    w = WORKLOADS[name]
    if isinstance(w, CascadeWorkload):
        return CascadeCase(name, device)
    if name.startswith("paged_append"):
        return AppendCase(name, device)
    return (PagedCase if isinstance(w, PagedWorkload) else DenseCase)(name, device)


def time_case(case, steps, warmup, flush):
    """Per-step device time (ms) of case.run() with CUDA events on the launching stream; L2 is
    flushed before every step, outside the timed interval."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        case.run()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        case.run()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def e2e_dense(case, steps, warmup, device):
    """Headline metric through the public API with host buffers: every step copies q, k, v from
    pinned host memory, runs the forward and copies O and LSE back to pinned host memory. The
    copies run on their own streams with two device buffer sets, so step i+1's upload overlaps
    step i's forward and download (the two copy directions use separate links); every step still
    moves all of its inputs and results. Returns (ms per step, h2d bytes, d2h bytes per step)."""
    import torch

    import io_aware_exact_flash_gb300 as fa

    hq, hk, hv = (case.q.cpu().pin_memory(), case.k.cpu().pin_memory(), case.v.cpu().pin_memory())
    ho = [torch.empty(case.o.shape, dtype=case.o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(case.lse.shape, dtype=case.lse.dtype).pin_memory() for _ in range(2)]
    dev_in = [tuple(torch.empty_like(t) for t in (case.q, case.k, case.v)) for _ in range(2)]
    dev_out = [(torch.empty_like(case.o), torch.empty_like(case.lse)) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_comp = torch.cuda.current_stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # every buffer starts free
        in_free[b].record(s_comp)
        out_free[b].record(s_out)

    def step(i):
        b = i & 1
        dq, dk, dv = dev_in[b]
        do, dl = dev_out[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])      # the forward that last read this buffer is done
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            in_ready[b].record(s_in)
        s_comp.wait_event(in_ready[b])
        s_comp.wait_event(out_free[b])       # the download that last read these outputs is done
        fa.fa_fwd(dq, dk, dv, causal=case.w.causal, scale=case.w.scale, out=do, lse=dl, stream=s_comp)
        in_free[b].record(s_comp)
        out_ready[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            ho[b].copy_(do, non_blocking=True)
            hl[b].copy_(dl, non_blocking=True)
            out_free[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_comp)
    s_in.wait_event(start)
    for i in range(steps):
        step(i)
    s_comp.wait_stream(s_out)
    end.record(s_comp)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    return ms, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, t, target_s=12.0, seed=0):
    """Times the fp64 oracle, as it stands, on a bounded random sample of query rows of the dense
    workload; returns (TFLOP/s, sample description, threads)."""
    import oracle

    orc = oracle.get()
    threads = oracle.default_threads()
    rng = np.random.default_rng(seed)

    def rows_for(n):
        b = rng.integers(0, w.B, n)
        i = rng.integers(0, w.S, n)
        h = rng.integers(0, w.Hq, n)
        return np.stack([b, i, h], axis=1).astype(np.int64)

    def flops_of(rows):
        n_keys = rows[:, 1] + 1 if w.causal else np.full(len(rows), w.S)
        return 4.0 * w.d * float(n_keys.sum())

    probe = rows_for(max(threads, 64))
    t0 = time.perf_counter()
    orc.dense_rows(t["q"], t["k"], t["v"], w.causal, w.scale, probe, threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(200000, max(threads, len(probe) * target_s / dt)))
    rows = rows_for(n)
    t0 = time.perf_counter()
    orc.dense_rows(t["q"], t["k"], t["v"], w.causal, w.scale, rows, threads)
    dt = time.perf_counter() - t0
    return flops_of(rows) / dt / 1e12, f"{n} random (b, i, h) query rows of {w.name}, {dt:.1f} s", threads


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle on the same workload, metric and unit."""
    if rank != 0:
        return 0
    w = WORKLOADS[HEADLINE]
    t = make_dense(w)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    desc, threads = "", 1
    for i in range(args.warmup + args.steps):
        v, desc, threads = oracle_sample(w, t, target_s=per_step, seed=i)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "causal": True},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "TFLOP/s", "cores": threads,
                             "sample": desc + " per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_only(args, device):
    """Time one workload by itself (for profiler runs); prints one line with its own metric."""
    import dataclasses

    import torch

    base = args.only.split("@")[0]
    w = WORKLOADS[base]
    if args.seqs is not None:
        if not hasattr(w, "num_seqs"):
            raise SystemExit("--seqs applies to paged workloads")
        WORKLOADS[base] = dataclasses.replace(w, num_seqs=args.seqs)
    case = make_case(args.only, device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    ms = statistics.mean(time_case(case, args.steps, args.warmup, flush))
    if case.kind in ("decode", "append", "cascade", "verify"):
        out = {"workload": args.only, "seqs": case.w.num_seqs, "ms": ms, "GB/s": case.bytes / (ms * 1e-3) / 1e9}
        if isinstance(case, PagedCase):
            out["splits"] = case.splits
        if case.kind == "cascade":
            out["flat_paged_fwd_ms"] = statistics.mean(time_case(FlatView(case), args.steps, args.warmup, flush))
    else:
        out = {"workload": args.only, "ms": ms, "TFLOP/s": case.flops / (ms * 1e-3) / 1e12}
    print(json.dumps(out), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--extras", default="all", help="comma list of extra workloads, 'all' or 'none'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="profiling aid: time only this workload (no headline line is printed)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="profiling aid: override the sequence count of a paged workload given with --only")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch

    dist_init(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import io_aware_exact_flash_gb300 as fa

    fa.load_library()
    if args.only is not None:
        return profile_only(args, device)
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    head = DenseCase(HEADLINE, device)
    extra_names = EXTRAS if args.extras == "all" else ([] if args.extras == "none" else args.extras.split(","))
    extras = [(n, make_case(n, device)) for n in extra_names]

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    head_ms = time_case(head, args.steps, args.warmup, flush)
    extra_ms = {n: time_case(c, args.steps, args.warmup, flush) for n, c in extras}
    flat_ms = {n: time_case(FlatView(c), args.steps, args.warmup, flush) for n, c in extras if c.kind == "cascade"}
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    barrier(world)
    clocks = sampler.stop()
    code, site = fa.fa_get_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} at site {site}")

    mean_ms = max_over_ranks(statistics.mean(head_ms), world, device)
    value = world * head.flops / (mean_ms * 1e-3) / 1e12
    e2e_ms, h2d, d2h = e2e_dense(head, max(3, args.steps // 2), 3, device)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = world * head.flops / (e2e_ms * 1e-3) / 1e12

    peak_t = peaks["bf16_tflops"]
    label = "of measured" if peaks["source"] == "measured" else "of fallback"
    roof = {"bound": "tensor", "achieved": head.flops / (statistics.mean(head_ms) * 1e-3) / 1e12, "peak": peak_t,
            "unit": "TFLOP/s", "frac": None, "traffic": None, "peak_source": label,
            "kernel": "prefill_kernel<128,false,true>", "per_launch_flops": head.flops}
    roof["frac"] = roof["achieved"] / peak_t
    if prefill_source_digest() == PREFILL_TRAFFIC["source_sha256"]:
        roof["traffic"] = PREFILL_TRAFFIC["bytes"]

    extra = {}
    for n, c in extras:
        ms = statistics.mean(extra_ms[n])
        if c.kind in ("decode", "append", "cascade", "verify"):
            gbs = c.bytes / (ms * 1e-3) / 1e9
            extra[n] = {"metric": f"{c.kind} HBM GB/s", "value": gbs, "unit": "GB/s", "ms": ms,
                        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": gbs / peaks["hbm_gbs"], "peak_source": label,
                                     "per_launch_bytes": c.bytes}}
            if isinstance(c, PagedCase):
                extra[n]["splits"] = c.splits
                extra[n]["path"] = "tensor cores" if c.tensor_cores else "cuda cores"
            if c.kind == "verify":
                extra[n]["tflops"] = c.flops / (ms * 1e-3) / 1e12
            if c.kind == "cascade":
                fm = statistics.mean(flat_ms[n])
                extra[n]["flat_paged_fwd_ms"] = fm
                extra[n]["speedup_vs_flat"] = fm / ms
        else:
            tf = c.flops / (ms * 1e-3) / 1e12
            extra[n] = {"metric": "prefill TFLOP/s", "value": tf, "unit": "TFLOP/s", "ms": ms,
                        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_t, "unit": "TFLOP/s",
                                     "frac": tf / peak_t, "peak_source": label, "per_launch_flops": c.flops}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, threads = oracle_sample(head.w, head.host, target_s=12.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    launches = args.steps * (head.launches + sum(c.launches for _, c in extras)
                             + sum(2 for _, c in extras if c.kind == "cascade"))  # the flat comparison
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": HEADLINE, "B": head.w.B, "S": head.w.S, "Hq": head.w.Hq, "Hkv": head.w.Hkv,
                           "d": head.w.d, "causal": True, "parallelism": f"replicas x{world}",
                           "l2": "flushed before every timed step (512 MB write)"},
                "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms},
                "gpu_launches": launches, "clocks": clocks, "timed_wall_s": wall, "extra": extra}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
