#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention hot path on GB300.

Default workload: batched decode, Llama-3-8B-shaped layer (32 query / 8 kv heads,
head_dim 128, block_size 16, 32768-block pool, batch 64, seq_len U[512, 4096]).  One
step = store the 64 new tokens' K/V through slot_mapping, then split-K paged decode
and the LSE combine (one pa_decode call with the fused store).  The metric is decode
KV-read GB/s: the K and V bytes the attention must read (sum over sequences of the
attended keys x num_kv_heads x head_dim x 2 tensors x 2 bytes) divided by the step
time.  A second leg times the varlen causal prefill workload (16 prompts of
U[128, 2048] tokens, store + prefill) in TFLOP/s (4 x head_dim x num_heads FLOP per
unmasked query/key pair).

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_attention_03_gb300.inputs import WORKLOADS, make_case, split_mixed  # noqa: E402

L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2


class L2Flush:
    """Untimed L2 flush before every timed step: write a buffer larger than L2, then read
    a second one. The write evicts the step's inputs; the read replaces the dirty lines the
    write leaves behind (about 126 MB) with clean ones, so their write-back happens here
    and not inside the next timed step, as after the weight-reading GEMMs that precede
    attention in a decode step. `write_only=True` skips the read: the timed step then also
    pays for writing those lines back."""

    def __init__(self, dev, write_only=False):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = (None if write_only else
                  torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev))

    def __call__(self):
        self.w.zero_()
        if self.r is not None:
            self.r.sum()

    def describe(self):
        if self.r is None:
            return f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write, untimed)"
        return (f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write, then a "
                f"{L2_FLUSH_BYTES >> 20} MiB read so no dirty line is written back inside "
                f"the step; untimed)")

# DRAM bytes (read + write) of one launch on the default workloads, from the ncu
# captures summarised in the named profiles/ files (commands there), with the commit of
# the kernel source they were taken on.  A changed kernel needs a new capture.
NCU_TRAFFIC = {
    "decode_split_kernel": {"bytes": 639.53e6 + 3.91e6,
                            "source": "profiles/decode_split_kernel_batched_decode.md",
                            "kernel_commit": "ec426f0"},
    "decode_split_kernel_long": {"bytes": 2934.95e6 + 3.64e6,
                                 "source": "profiles/decode_split_kernel_long_decode.md",
                                 "kernel_commit": "ec426f0"},
    "prefill_kernel": {"bytes": 318.28e6 + 104.80e6,
                       "source": "profiles/prefill_kernel_varlen_prefill.md",
                       "kernel_commit": "ec426f0"},
}


# ----------------------------------------------------------------- helpers ---

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, ws


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ work counting ---

def attended_keys(case, seqs=None):
    """Per query row, the number of visible keys (bottom-right causal + window)."""
    w = case.workload.sliding_window
    seqs = range(case.num_seqs) if seqs is None else seqs
    total = 0
    for i in seqs:
        sq, sk = int(case.query_lens[i]), int(case.seq_lens[i])
        p = np.arange(sk - sq, sk, dtype=np.int64)
        n = p + 1
        if w > 0:
            n = np.minimum(n, w)
        total += int(n.sum())
    return total


def decode_kv_bytes(case, seqs=None):
    """K+V bytes decode must read: attended keys x Hkv x D x 2 tensors x 2 bytes."""
    w = case.workload
    return attended_keys(case, seqs) * w.num_kv_heads * w.head_dim * 2 * 2


def prefill_flops(case, seqs=None):
    w = case.workload
    return attended_keys(case, seqs) * 4 * w.head_dim * w.num_heads


def cascade_bytes(case, prefix_len):
    """(logical, physical) K+V bytes of a shared-prefix decode batch: logical counts every
    request's keys (what plain decode reads), physical each cache row once (the prefix
    rows are shared by all requests, each suffix is its request's own)."""
    w = case.workload
    row = w.num_kv_heads * w.head_dim * 2 * 2  # K + V bytes of one key
    logical = int(case.seq_lens.sum()) * row
    physical = (prefix_len + int((case.seq_lens - prefix_len).sum())) * row
    return logical, physical


# ------------------------------------------------------------------ runners ---

class DecodeRunner:
    """One step: split-K decode with the store of the new tokens fused in (+ combine)."""

    def __init__(self, case, device, seqs=None):
        import paged_kv_attention_03_gb300 as pa

        self.pa = pa
        self.case = case
        w = case.workload
        self.seqs = np.arange(case.num_seqs) if seqs is None else np.asarray(seqs)
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)
        rows = torch.as_tensor(case.cu_seqlens_q[self.seqs], dtype=torch.long, device=device)
        self.q = case.q[rows].contiguous()
        self.key = case.key[rows].contiguous()
        self.value = case.value[rows].contiguous()
        self.slots = t(case.slot_mapping[case.cu_seqlens_q[self.seqs]])
        self.bt = t(case.block_table[self.seqs])
        self.seq_lens = t(case.seq_lens[self.seqs])
        self.max_len = int(case.seq_lens[self.seqs].max())
        self.window = w.sliding_window
        self.scale = w.final_scale
        self.out = torch.empty_like(self.q)
        self.splits = pa.pa_decode_num_splits(len(self.seqs), w.num_heads, w.num_kv_heads,
                                              w.head_dim, self.max_len, self.window, 0)
        need = pa.pa_decode_workspace_size(len(self.seqs), w.num_heads, w.num_kv_heads,
                                           w.head_dim, self.max_len, self.window, 0)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        # The store of the new tokens runs inside the split kernel.
        self.launches = 1 + (1 if self.splits > 1 else 0)
        self.work = decode_kv_bytes(case, self.seqs)

    def step(self):
        self.pa.pa_decode(self.q, self.case.k_cache, self.case.v_cache, self.bt, self.seq_lens,
                          self.max_len, self.scale, self.window, 0, key=self.key,
                          value=self.value, slot_mapping=self.slots, out=self.out,
                          workspace=self.ws)

    def attention_only(self):
        self.pa.pa_decode(self.q, self.case.k_cache, self.case.v_cache, self.bt, self.seq_lens,
                          self.max_len, self.scale, self.window, 0, out=self.out,
                          workspace=self.ws)

    # End-to-end: the step's inputs are staged in one pinned host buffer and copied to the
    # device in one transfer (as a serving loop stages a step); the output goes back.
    def host_buffers(self):
        srcs = (self.q, self.key, self.value, self.slots, self.bt, self.seq_lens)
        sizes = [x.numel() * x.element_size() for x in srcs]
        offs, total = [], 0
        for n in sizes:
            offs.append(total)
            total += (n + 255) // 256 * 256
        self.h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_stage = torch.empty(total, dtype=torch.uint8, device=self.q.device)
        self.d_in = []
        for x, o, n in zip(srcs, offs, sizes):
            self.h_stage[o:o + n].copy_(x.contiguous().view(torch.uint8).reshape(-1).cpu())
            self.d_in.append(self.d_stage[o:o + n].view(x.dtype).view(x.shape))
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d = sum(sizes)
        self.d2h = self.h_out.numel() * self.h_out.element_size()

    def e2e_step(self):
        self.d_stage.copy_(self.h_stage, non_blocking=True)
        q, key, value, slots, bt, sl = self.d_in
        self.pa.pa_decode(q, self.case.k_cache, self.case.v_cache, bt, sl, self.max_len,
                          self.scale, self.window, 0, key=key, value=value, slot_mapping=slots,
                          out=self.out, workspace=self.ws)
        self.h_out.copy_(self.out, non_blocking=True)

    def capture_e2e(self):
        """Capture e2e_step (the H2D copy, the pa_decode call, the D2H copy) once as a CUDA
        graph, as a serving loop captures its decode step; each replay issues the same two
        copies and kernel launches, so every step still moves its inputs and output."""
        dev = self.q.device
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            self.e2e_step()  # the library's one-time set-up runs outside the capture
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.e2e_step()
        torch.cuda.synchronize()


class PrefillRunner:
    """One step: store of the prompt tokens + varlen causal prefill (one call, two launches)."""

    def __init__(self, case, device):
        import paged_kv_attention_03_gb300 as pa

        self.pa = pa
        self.case = case
        w = case.workload
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)
        self.cu = t(case.cu_seqlens_q)
        self.seq_lens = t(case.seq_lens)
        self.bt = t(case.block_table)
        self.slots = t(case.slot_mapping)
        self.out = torch.empty_like(case.q)
        self.launches = 3  # the store of the prompt tokens, the prefill, the single-row decode
        self.work = prefill_flops(case)

    def step(self):
        c = self.case
        self.pa.pa_varlen_prefill(c.q, c.k_cache, c.v_cache, self.cu, self.seq_lens, self.bt,
                                  c.max_query_len, c.max_seq_len, c.workload.final_scale,
                                  c.workload.sliding_window, key=c.key, value=c.value,
                                  slot_mapping=self.slots, out=self.out)

    def attention_only(self):
        c = self.case
        self.pa.pa_varlen_prefill(c.q, c.k_cache, c.v_cache, self.cu, self.seq_lens, self.bt,
                                  c.max_query_len, c.max_seq_len, c.workload.final_scale,
                                  c.workload.sliding_window, out=self.out)


class MixedRunner:
    """The mixed-window workload (chunked prefill + decodes, window 4096) two ways:
    `single` = one pa_varlen_prefill call over the whole packed batch (store + prefill);
    `split` = pa_varlen_prefill on the chunks, then pa_decode on the decode rows."""

    def __init__(self, case, device):
        import paged_kv_attention_03_gb300 as pa

        self.pa = pa
        self.case = case
        pre, dec = split_mixed(case)
        self.full = PrefillRunner(case, device)
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)
        cu = case.cu_seqlens_q
        rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in pre])
        r = torch.as_tensor(rows, dtype=torch.long, device=device)
        self.pq, self.pkey, self.pval = case.q[r].contiguous(), case.key[r].contiguous(), \
            case.value[r].contiguous()
        ql = case.query_lens[pre]
        sub_cu = np.zeros(len(pre) + 1, np.int32)
        sub_cu[1:] = np.cumsum(ql)
        self.pcu, self.psl = t(sub_cu), t(case.seq_lens[pre])
        self.pbt, self.pslots = t(case.block_table[pre]), t(case.slot_mapping[rows])
        self.pmax_q, self.pmax_k = int(ql.max()), int(case.seq_lens[pre].max())
        self.pout = torch.empty_like(self.pq)
        self.dec = DecodeRunner(case, device, dec)
        self.chunk_flops = prefill_flops(case, pre)
        self.decode_bytes = decode_kv_bytes(case, dec)
        self.n_chunks, self.n_decodes = len(pre), len(dec)

    def single(self):
        self.full.step()

    def chunks_only(self):
        w = self.case.workload
        self.pa.pa_varlen_prefill(self.pq, self.case.k_cache, self.case.v_cache, self.pcu,
                                  self.psl, self.pbt, self.pmax_q, self.pmax_k, w.final_scale,
                                  w.sliding_window, key=self.pkey, value=self.pval,
                                  slot_mapping=self.pslots, out=self.pout)

    def split(self):
        w = self.case.workload
        self.pa.pa_varlen_prefill(self.pq, self.case.k_cache, self.case.v_cache, self.pcu,
                                  self.psl, self.pbt, self.pmax_q, self.pmax_k, w.final_scale,
                                  w.sliding_window, key=self.pkey, value=self.pval,
                                  slot_mapping=self.pslots, out=self.pout)
        self.dec.step()


class CascadeRunner:
    """64 decode requests sharing a 4096-token cached prefix (one system prompt), each
    with its own suffix of U[128, 1024] tokens; 32/8 heads, D=128, bs=16."""

    PREFIX_BLOCKS = 256

    def __init__(self, device, seed):
        import paged_kv_attention_03_gb300 as pa
        from paged_kv_attention_03_gb300.inputs import Workload, make_shared_prefix_case

        self.pa = pa
        w = Workload("shared_prefix", 32, 8, 128, 16, ())
        rng = np.random.default_rng(seed)
        suffix = rng.integers(128, 1025, size=64)
        self.case = make_shared_prefix_case(w, self.PREFIX_BLOCKS, suffix, seed, device)
        c = self.case
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)
        self.bt, self.sl = t(c.block_table), t(c.seq_lens)
        self.max_len = int(c.seq_lens.max())
        self.prefix = self.PREFIX_BLOCKS * w.block_size
        self.out = torch.empty_like(c.q)
        self.ws = torch.empty(pa.pa_cascade_decode_workspace_size(64, 32, 8, 128, self.max_len,
                                                                  self.prefix, 0),
                              dtype=torch.uint8, device=device)
        need = pa.pa_decode_workspace_size(64, 32, 8, 128, self.max_len, 0, 0)
        self.dws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.logical_bytes, self.physical_bytes = cascade_bytes(c, self.prefix)

    def cascade(self):
        c = self.case
        self.pa.pa_cascade_decode(c.q, c.k_cache, c.v_cache, self.bt, self.sl, self.max_len,
                                  self.prefix, c.workload.final_scale, 0, out=self.out,
                                  workspace=self.ws)

    def plain(self):
        c = self.case
        self.pa.pa_decode(c.q, c.k_cache, c.v_cache, self.bt, self.sl, self.max_len,
                          c.workload.final_scale, 0, 0, out=self.out, workspace=self.dws)


def _time_steps(fn, steps, warmup, flush, stream):
    """Per-step device time (ms) with CUDA events on `stream`, L2 flushed (untimed) before
    each step."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


# ------------------------------------------------------------ CPU baseline ---

def oracle_decode_time(case, seqs, budget_s=12.0):
    """Time the fp64 oracle (store + attention) on the given decode sequences, repeating
    the sample until about `budget_s` seconds of CPU work; returns (s per sample, threads)."""
    import oracle
    from paged_kv_attention_03_gb300.inputs import bf16_bits

    w = case.workload
    seqs = np.asarray(seqs)
    cu = case.cu_seqlens_q
    rows = cu[seqs]
    q = bf16_bits(case.q)[rows]
    key = bf16_bits(case.key)[rows]
    value = bf16_bits(case.value)[rows]
    kc = bf16_bits(case.k_cache)
    vc = bf16_bits(case.v_cache)
    slots = np.ascontiguousarray(case.slot_mapping[rows])
    sub_cu = np.arange(len(seqs) + 1, dtype=np.int32)
    bt = np.ascontiguousarray(case.block_table[seqs])
    sl = np.ascontiguousarray(case.seq_lens[seqs])
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle.store_kvcache(key, value, kc, vc, slots, w.block_size)
        oracle.paged_attention(q, kc, vc, sub_cu, sl, bt, w.num_heads, w.num_kv_heads,
                               w.sliding_window, w.final_scale, threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 50:
            break
    return statistics.median(times), threads, len(times)


# -------------------------------------------------------------------- main ---

def run_reference(args, rank, ws):
    """The fp64 CPU oracle as the reference arm, on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    from paged_kv_attention_03_gb300.inputs import bf16_bits

    wl = WORKLOADS[args.workload]
    case = make_case(wl, seed=0, device="cpu")
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    order = np.argsort(case.seq_lens)
    # Sequences per step: sized so warmup + steps fit in about two minutes.
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    probe = [int(order[len(order) // 2])]
    t_probe, _, _ = oracle_decode_time(case, probe, budget_s=0.0)
    n = max(1, min(case.num_seqs, int(per_step_budget / max(t_probe, 1e-6))))
    rng = np.random.default_rng(0)
    q_bits, kc, vc = bf16_bits(case.q), bf16_bits(case.k_cache), bf16_bits(case.v_cache)
    key, value = bf16_bits(case.key), bf16_bits(case.value)
    w = case.workload
    times, work = [], []
    for it in range(args.warmup + args.steps):
        seqs = np.sort(rng.choice(case.num_seqs, size=n, replace=False))
        rows = case.cu_seqlens_q[seqs]
        t0 = time.perf_counter()
        oracle.store_kvcache(key[rows], value[rows], kc, vc,
                             np.ascontiguousarray(case.slot_mapping[rows]), w.block_size)
        oracle.paged_attention(np.ascontiguousarray(q_bits[rows]), kc, vc,
                               np.arange(n + 1, dtype=np.int32),
                               np.ascontiguousarray(case.seq_lens[seqs]),
                               np.ascontiguousarray(case.block_table[seqs]), w.num_heads,
                               w.num_kv_heads, w.sliding_window, w.final_scale, threads)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt)
            work.append(decode_kv_bytes(case, seqs))
    total_t = sum(times)
    value_gbs = sum(work) / total_t / 1e9
    line = {
        "impl": "reference", "metric": "decode KV-read GB/s", "value": round(value_gbs, 4),
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {_describe(wl)}", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value_gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n} of {case.num_seqs} sequences per step (random), "
                                   f"store + fp64 attention"},
        "e2e": {"value": round(value_gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _describe(wl):
    return (f"H={wl.num_heads} Hkv={wl.num_kv_heads} D={wl.head_dim} bs={wl.block_size} "
            f"groups={wl.groups} window={wl.sliding_window}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="batched_decode",
                    choices=["batched_decode", "long_decode", "tiny_decode", "mixed_window"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-mixed", action="store_true")
    ap.add_argument("--no-cascade", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-long", action="store_true")
    ap.add_argument("--no-tiny", action="store_true")
    ap.add_argument("--leg", default="both",
                    choices=["both", "decode", "prefill", "fp8_decode", "fp8_prefill", "cascade",
                             "mixed"],
                    help="one leg alone, printing its JSON object (profiling runs): decode, "
                         "prefill, fp8_decode, fp8_prefill, cascade or mixed; both: the full "
                         "JSON line")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    rank, local, ws = _dist()
    if args.impl == "reference":
        run_reference(args, rank, ws)
        return

    import paged_kv_attention_03_gb300 as pa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pa.build()
    pa.load()
    peaks = _peaks()
    if args.leg in ("prefill", "fp8_prefill", "cascade", "mixed", "fp8_decode"):
        flush = L2Flush(dev)
        stream = torch.cuda.current_stream(dev)
        if args.leg == "fp8_decode":
            # The batched-decode batch over an E4M3 cache, as in the full line.
            case = make_case(WORKLOADS["batched_decode"], seed=rank, device=dev)
            res = _fp8_leg(pa, dev, rank, peaks, flush, stream, args, case,
                           DecodeRunner(case, dev))
        else:
            leg = {"prefill": _prefill_leg, "fp8_prefill": _fp8_prefill_leg,
                   "cascade": _cascade_leg, "mixed": _mixed_leg}[args.leg]
            res = leg(pa, dev, rank, peaks, flush, stream, args)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    wl = WORKLOADS[args.workload]
    # Weak scaling: every rank runs its own replica (own seed), no data-path collective.
    case = make_case(wl, seed=rank, device=dev)
    seqs = None
    if args.workload == "mixed_window":
        seqs = split_mixed(case)[1]
    runner = DecodeRunner(case, dev, seqs)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        flush()
        runner.step()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    _barrier(ws)
    torch.cuda.synchronize()
    step_ms = _time_steps(runner.step, args.steps, 0, flush, stream)
    torch.cuda.synchronize()
    _barrier(ws)
    # Attention call alone (split kernel + combine, no store): the roofline numerator.
    attn_ms = _time_steps(runner.attention_only, max(20, args.steps // 4), 3, flush, stream)
    # The same call after a write-only flush, whose dirty lines are written back in the step.
    attn_wo_ms = _time_steps(runner.attention_only, max(20, args.steps // 4), 3,
                             L2Flush(dev, write_only=True), stream)
    clocks = sampler.stop() if sampler else None

    total_ms = _max_over_ranks(sum(step_ms), ws, dev)
    units = _sum_over_ranks(runner.work * args.steps, ws, dev)
    value = units / (total_ms / 1e3) / 1e9
    ms_per_step = total_ms / args.steps
    attn_mean = statistics.mean(attn_ms)
    achieved = runner.work / (attn_mean / 1e3) / 1e9

    if args.leg == "decode":
        if rank == 0:
            print(json.dumps({"decode_gbs": round(value, 2), "attention_gbs": round(achieved, 2),
                              "ms_per_step": ms_per_step}), flush=True)
        return

    e2e = None
    if not args.no_e2e:
        # Host wall clock around one step at a time (synchronised before and after), L2
        # flushed before each: the step replayed as a CUDA graph, and issued eagerly through
        # the Python binding for comparison.
        runner.host_buffers()
        runner.capture_e2e()

        def wall(fn):
            ms = []
            for _ in range(3):
                flush()
                fn()
            torch.cuda.synchronize()
            for _ in range(max(20, args.steps // 4)):
                flush()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ms.append((time.perf_counter() - t0) * 1e3)
            return _max_over_ranks(statistics.mean(ms), ws, dev)

        e2e_t = wall(runner.graph.replay)
        eager_t = wall(runner.e2e_step)
        units_step = _sum_over_ranks(runner.work, ws, dev)
        e2e = {"value": round(units_step / (e2e_t / 1e3) / 1e9, 3),
               "unit": "GB/s", "h2d_bytes_per_step": runner.h2d,
               "d2h_bytes_per_step": runner.d2h, "ms_per_step": round(e2e_t, 4),
               "mode": "CUDA graph of (pinned H2D of the step's inputs, pa_decode, D2H of the "
                       "output), replayed per step",
               "eager": {"value": round(units_step / (eager_t / 1e3) / 1e9, 3),
                         "ms_per_step": round(eager_t, 4),
                         "mode": "the same three calls issued through the Python binding"}}

    prefill = None
    if not args.no_prefill:
        prefill = _prefill_leg(pa, dev, rank, peaks, flush, stream, args)
    mixed = None
    if not args.no_mixed:
        mixed = _mixed_leg(pa, dev, rank, peaks, flush, stream, args)
    cascade = None
    if not args.no_cascade:
        cascade = _cascade_leg(pa, dev, rank, peaks, flush, stream, args)
    fp8 = None
    fp8_prefill = None
    if not args.no_fp8:
        fp8 = _fp8_leg(pa, dev, rank, peaks, flush, stream, args, case, runner)
        fp8_prefill = _fp8_prefill_leg(pa, dev, rank, peaks, flush, stream, args)

    long_dec = None
    if not args.no_long and args.workload != "long_decode":
        long_dec = _long_decode_leg(pa, dev, rank, peaks, flush, stream, args)
    tiny = None
    if not args.no_tiny and args.workload != "tiny_decode":
        tiny = _tiny_decode_leg(pa, dev, rank, peaks, flush, stream, args)

    cpu = None
    if rank == 0 and ws >= 1 and not args.no_cpu_baseline and args.gpus == 1:
        t_s, threads, reps = oracle_decode_time(case, runner.seqs)
        cpu = {"value": round(runner.work / t_s / 1e9, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"the whole step ({len(runner.seqs)} sequences: store + fp64 "
                         f"attention), median of {reps} runs"}

    if rank != 0:
        return
    line = {
        "metric": "decode KV-read GB/s", "value": round(value, 3), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {_describe(wl)}",
                   "batch": len(runner.seqs), "kv_bytes_per_step": runner.work,
                   "num_splits": runner.splits,
                   "l2": flush.describe(),
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "kernel": "pa_decode (decode_split_kernel + combine)",
                     "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"],
                     "traffic": (NCU_TRAFFIC["decode_split_kernel"]["bytes"]
                                 if args.workload == "batched_decode" else None),
                     "traffic_kernel": "decode_split_kernel",
                     "traffic_source": (NCU_TRAFFIC["decode_split_kernel"]
                                        if args.workload == "batched_decode" else None),
                     "algorithmic_bytes": runner.work,
                     "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                     "achieved_after_write_only_flush": round(
                         runner.work / (statistics.mean(attn_wo_ms) / 1e3) / 1e9, 2)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": runner.launches * args.steps,
        "clocks": clocks,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if mixed is not None:
        line["mixed"] = mixed
    if cascade is not None:
        line["cascade"] = cascade
    if fp8 is not None:
        line["fp8_decode"] = fp8
    if fp8_prefill is not None:
        line["fp8_prefill"] = fp8_prefill
    if long_dec is not None:
        line["long_decode"] = long_dec
    if tiny is not None:
        line["tiny_decode"] = tiny
    print(json.dumps(line), flush=True)


def _fp8_leg(pa, dev, rank, peaks, flush, stream, args, case, runner):
    """The decode workload over an FP8 E4M3 cache (codes of the bf16 cache / 0.02): the
    bytes actually read (one per element) and the tokens per second against bf16."""
    kv_scale = 0.02
    k8 = (case.k_cache.float() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (case.v_cache.float() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    w = case.workload
    need = pa.pa_decode_workspace_size(len(runner.seqs), w.num_heads, w.num_kv_heads,
                                       w.head_dim, runner.max_len, runner.window, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out = torch.empty_like(runner.q)

    def step():
        pa.pa_decode_fp8(runner.q, k8, v8, runner.bt, runner.seq_lens, runner.max_len,
                         runner.scale, kv_scale, runner.window, 0, key=runner.key,
                         value=runner.value, slot_mapping=runner.slots, out=out, workspace=ws)

    steps = max(20, args.steps // 10)
    t = statistics.mean(_time_steps(step, steps, 3, flush, stream))
    bytes8 = runner.work // 2  # one byte per element instead of two
    return {"kv_bytes_per_step": bytes8, "ms_per_step": round(t, 5),
            "gbs": round(bytes8 / (t / 1e3) / 1e9, 2),
            "frac_of_hbm": round(bytes8 / (t / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "bf16_equivalent_gbs": round(runner.work / (t / 1e3) / 1e9, 2),
            "kv_scale": kv_scale}


def _cascade_leg(pa, dev, rank, peaks, flush, stream, args):
    """Shared-prefix decode: cascade vs plain decode on the same batch.  Logical bytes
    count the prefix once per request (what plain decode reads); physical bytes once."""
    r = CascadeRunner(dev, 300 + rank)
    steps = max(20, args.steps // 10)
    tc = statistics.mean(_time_steps(r.cascade, steps, 3, flush, stream))
    tp = statistics.mean(_time_steps(r.plain, steps, 3, flush, stream))
    return {"workload": "shared_prefix: 64 requests, prefix 4096 + own suffix U[128,1024], "
                        "32/8 heads, D=128, bs=16",
            "logical_bytes": r.logical_bytes, "physical_bytes": r.physical_bytes,
            "cascade": {"ms_per_step": round(tc, 4), "launches": 3,
                        "effective_gbs": round(r.logical_bytes / (tc / 1e3) / 1e9, 1),
                        "physical_gbs": round(r.physical_bytes / (tc / 1e3) / 1e9, 1),
                        "physical_frac_of_hbm": round(r.physical_bytes / (tc / 1e3) / 1e9 /
                                                      peaks["hbm_gbs"], 4)},
            "plain_decode": {"ms_per_step": round(tp, 4),
                             "gbs": round(r.logical_bytes / (tp / 1e3) / 1e9, 1)},
            "speedup": round(tp / tc, 2)}


def _mixed_leg(pa, dev, rank, peaks, flush, stream, args):
    """The mixed-window workload (chunked prefill + decodes, window 4096): the one-call
    step, the two-call step, and each part alone against its own roofline.  The step is
    reported against two bounds: the serial sum (decode bytes / HBM peak + chunk FLOPs /
    bf16 peak) and the overlapped max() of the two, which the one-call design aims at
    because its decode CTAs run beside the prefill kernel."""
    case = make_case(WORKLOADS["mixed_window"], seed=200 + rank, device=dev)
    runner = MixedRunner(case, dev)
    steps = max(20, args.steps // 10)
    single = statistics.mean(_time_steps(runner.single, steps, 3, flush, stream))
    split = statistics.mean(_time_steps(runner.split, steps, 3, flush, stream))
    chunks = statistics.mean(_time_steps(runner.chunks_only, steps, 3, flush, stream))
    decodes = statistics.mean(_time_steps(runner.dec.step, steps, 3, flush, stream))
    dec_ms = 1e3 * runner.decode_bytes / (peaks["hbm_gbs"] * 1e9)
    chunk_ms = 1e3 * runner.chunk_flops / (peaks["bf16_tflops"] * 1e12)
    serial_ms, overlap_ms = dec_ms + chunk_ms, max(dec_ms, chunk_ms)
    return {"workload": f"mixed_window: {runner.n_chunks} chunks of 512 + "
                        f"{runner.n_decodes} decodes, ctx U[1024,8192], window 4096",
            "chunk_flops": runner.chunk_flops, "decode_bytes": runner.decode_bytes,
            "roofline_ms": round(serial_ms, 4),
            "roofline_ms_overlapped": round(overlap_ms, 4),
            "single_call": {"ms_per_step": round(single, 4), "launches": 3,
                            "frac_of_roofline": round(serial_ms / single, 4),
                            "frac_of_overlapped_bound": round(overlap_ms / single, 4)},
            "two_calls": {"ms_per_step": round(split, 4), "launches": 2 + runner.dec.launches,
                          "frac_of_roofline": round(serial_ms / split, 4),
                          "frac_of_overlapped_bound": round(overlap_ms / split, 4)},
            "chunks_alone": {"ms_per_step": round(chunks, 4),
                             "tflops": round(runner.chunk_flops / (chunks / 1e3) / 1e12, 2),
                             "frac_of_bf16_peak": round(chunk_ms / chunks, 4),
                             "note": "store of the chunk tokens + prefill, one call"},
            "decodes_alone": {"ms_per_step": round(decodes, 4),
                              "gbs": round(runner.decode_bytes / (decodes / 1e3) / 1e9, 2),
                              "frac_of_hbm": round(dec_ms / decodes, 4),
                              "note": "pa_decode with the fused store, + combine"}}


def _long_decode_leg(pa, dev, rank, peaks, flush, stream, args):
    """Long-context decode (split-K stress): batch 8, 40/8 heads, seq_len U[32768, 131072];
    store fused + split kernel + combine, with its own clock record."""
    case = make_case(WORKLOADS["long_decode"], seed=rank, device=dev)
    runner = DecodeRunner(case, dev)
    steps = max(20, args.steps // 10)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(3):
        flush()
        runner.step()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    step = statistics.mean(_time_steps(runner.step, steps, 0, flush, stream))
    attn = statistics.mean(_time_steps(runner.attention_only, steps, 3, flush, stream))
    clocks = sampler.stop() if sampler else None
    ach = runner.work / (attn / 1e3) / 1e9
    del case
    return {"workload": f"long_decode: {_describe(WORKLOADS['long_decode'])}, batch 8, "
                        f"seq_len U[32768,131072]",
            "kv_bytes_per_step": runner.work, "num_splits": runner.splits,
            "ms_per_step": round(step, 4),
            "gbs": round(runner.work / (step / 1e3) / 1e9, 2),
            "roofline": {"bound": "hbm", "kernel": "pa_decode (decode_split_kernel + combine)",
                         "achieved": round(ach, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(ach / peaks["hbm_gbs"], 4),
                         "peak_source": peaks["source"],
                         "traffic": NCU_TRAFFIC["decode_split_kernel_long"]["bytes"],
                         "traffic_kernel": "decode_split_kernel",
                         "traffic_source": NCU_TRAFFIC["decode_split_kernel_long"],
                         "algorithmic_bytes": runner.work},
            "clocks": clocks}


def _tiny_decode_leg(pa, dev, rank, peaks, flush, stream, args):
    """Tiny decode (4 sequences of {17, 33, 64, 100} keys, 8/2 heads, D=64): a latency
    figure, microseconds per call, after an L2 flush (cold) and with the data left in L2
    (warm).  Before each warm step a ~20 us spin kernel keeps the GPU busy while the host
    queues the call, so the figure is device time, not host launch time."""
    case = make_case(WORKLOADS["tiny_decode"], seed=0, device=dev)
    runner = DecodeRunner(case, dev)
    steps = max(50, args.steps // 5)
    cold = statistics.median(_time_steps(runner.step, steps, 5, flush, stream))
    warm = statistics.median(_time_steps(runner.step, steps, 5,
                                         lambda: torch.cuda._sleep(40000), stream))
    return {"workload": f"tiny_decode: {_describe(WORKLOADS['tiny_decode'])}, seq_lens "
                        f"{{17,33,64,100}}",
            "kv_bytes_per_step": runner.work,
            "us_per_call_cold": round(cold * 1e3, 2), "us_per_call_warm": round(warm * 1e3, 2),
            "launches": runner.launches,
            "note": "median device time of one pa_decode call (store fused); the data fit "
                    "in L2, so a roofline fraction is not meaningful"}


def _fp8_prefill_leg(pa, dev, rank, peaks, flush, stream, args):
    """The varlen-prefill workload over an FP8 E4M3 cache (codes of the bf16 pool / 0.02;
    the prompt tokens quantised into it by the call), TFLOP/s as the bf16 leg counts them."""
    case = make_case(WORKLOADS["varlen_prefill"], seed=100 + rank, device=dev)
    kv_scale = 0.02
    k8 = (case.k_cache.float() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (case.v_cache.float() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    runner = PrefillRunner(case, dev)
    c, w = case, case.workload

    def step(store=True):
        kw = dict(key=c.key, value=c.value, slot_mapping=runner.slots) if store else {}
        pa.pa_varlen_prefill_fp8(c.q, k8, v8, runner.cu, runner.seq_lens, runner.bt,
                                 c.max_query_len, c.max_seq_len, w.final_scale, kv_scale,
                                 w.sliding_window, out=runner.out, **kw)

    steps = max(20, args.steps // 10)
    ms = statistics.mean(_time_steps(step, steps, 3, flush, stream))
    attn = statistics.mean(_time_steps(lambda: step(False), steps, 3, flush, stream))
    return {"workload": "varlen_prefill over an E4M3 cache (kv_scale 0.02)",
            "ms_per_step": round(ms, 4), "tflops": round(runner.work / (ms / 1e3) / 1e12, 2),
            "attention_ms": round(attn, 4),
            "attention_tflops": round(runner.work / (attn / 1e3) / 1e12, 2),
            "frac_of_bf16_peak": round(runner.work / (attn / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
            "note": "f16 products on codes expanded in shared memory; FLOPs of the bf16 leg"}


def _prefill_leg(pa, dev, rank, peaks, flush, stream, args):
    """TFLOP/s of the varlen causal prefill workload (store + prefill), or a status entry
    if the library's prefill entry point returns an error."""
    case = make_case(WORKLOADS["varlen_prefill"], seed=100 + rank, device=dev)
    runner = PrefillRunner(case, dev)
    try:
        runner.step()
        torch.cuda.synchronize()
    except pa.PAError as e:
        return {"status": f"unavailable: {e}"}
    steps = max(20, args.steps // 10)
    ms = _time_steps(runner.step, steps, 3, flush, stream)
    attn = _time_steps(runner.attention_only, steps, 3, flush, stream)
    tf = runner.work / (statistics.mean(ms) / 1e3) / 1e12
    ach = runner.work / (statistics.mean(attn) / 1e3) / 1e12
    return {"metric": "varlen prefill TFLOP/s", "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(statistics.mean(ms), 4), "flops_per_step": runner.work,
            "workload": "varlen_prefill: 16 prompts U[128,2048], 32/8 heads, D=128, bs=16",
            "roofline": {"bound": "tensor", "kernel": "pa_varlen_prefill (prefill_kernel)",
                         "achieved": round(ach, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                         "peak_source": peaks["source"],
                         "traffic": NCU_TRAFFIC["prefill_kernel"]["bytes"],
                         "traffic_source": NCU_TRAFFIC["prefill_kernel"],
                         "algorithmic_flops": runner.work}}


if __name__ == "__main__":
    main()
