"""Benchmark of the decode hot path on synthetic workloads.

Default workload (N = 1): paged Full-attention decode, batch 64, 32 query /
8 KV heads, head_dim 128, pages of 16 tokens, lengths uniform in [1K, 32K]
(about 1.08 M cached tokens, 4.43 GB of K/V per step).  One step = append of
the new token of every request + split-KV decode + cross-split merge,
through the C ABI of libphs.so.

Prints one JSON line with the throughput in algorithmic HBM GB/s (the K/V
bytes the step must read, plus query, output and append bytes), attended KV
tokens/s, the roofline of the dominant kernel, an end-to-end number through
the public API with host buffers, and the CPU oracle timed on a bounded
sample on the host cores.  --impl reference times the CPU oracle alone.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no exchange step); the timed region is bracketed by barriers and
the slowest rank's time is used.
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
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attention HBM GB/s (% of GB300 peak) and attended KV tokens/s, 1 GPU"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------- helpers --
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


SPLIT_KERNEL_SOURCES = ("phs_decode.cu", "phs_attn.cuh", "phs_common.cuh", "phs_internal.h")


def kernel_source_hash(files=SPLIT_KERNEL_SOURCES):
    """Hash of the sources the split-KV decode kernel is compiled from."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_hybrid_sliding_gb300", "csrc")
    for name in files:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(kernel, {})
    if e.get("workload") != workload or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------- config 2 workload --
class PagedFullWorkload:
    """Paged Full-attention decode, batch 64 (one step = append + decode)."""

    def __init__(self, device, seed=2, batch=64):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.w = w = synth.paged_full(seed=seed, B=batch)
        self.name = f"paged_full_b{batch}_hq32_hkv8_d128_p16_seqU[1K,32K]"
        self.device = device
        B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
        self.k = synth.normal_bf16((w.num_pages, Hkv, 16, D), seed * 100 + 1, device=device)
        self.v = synth.normal_bf16((w.num_pages, Hkv, 16, D), seed * 100 + 2, device=device)
        self.pool = phs.PagedPool(self.k, self.v)
        self.q = synth.normal_bf16((B, Hq, D), seed * 100 + 3, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), seed * 100 + 4, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), seed * 100 + 5, device=device)
        self.bt = torch.from_numpy(w.block_table).to(device)
        self.sl = torch.from_numpy(w.n_after).to(device)
        self.max_seq = int(w.n_after.max())
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps),
                              dtype=torch.uint8, device=device)
        tokens = int(w.n_after.sum())
        self.tokens_per_step = tokens
        kv = tokens * Hkv * D * 2 * 2
        qo = 2 * B * Hq * D * 2
        app = 2 * B * Hkv * D * 2 * 2
        tables = int(synth.pages_needed(w.n_after).sum()) * 4 + B * 4
        self.bytes_per_step = kv + qo + app + tables
        self.split_bytes = kv + B * Hq * D * 2 + tables
        self.launches_per_step = 3
        # pinned host copies of the per-step inputs for the end-to-end leg
        self.h_q = self.q.cpu().pin_memory()
        self.h_kn = self.kn.cpu().pin_memory()
        self.h_vn = self.vn.cpu().pin_memory()
        self.h_bt = self.bt.cpu().pin_memory()
        self.h_sl = self.sl.cpu().pin_memory()
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size()
                             for t in (self.h_q, self.h_kn, self.h_vn, self.h_bt, self.h_sl))
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()

    def step(self, ev=None):
        phs = self.phs
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        if ev is not None:
            ev[0].record()
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                         self.ws, self.out, tokens_per_split=self.tps)
        if ev is not None:
            ev[1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, self.sl, self.max_seq, self.ws,
                              tokens_per_split=self.tps)

    def e2e_step(self):
        """Public API from host buffers: inputs in, output out, every step."""
        phs = self.phs
        self.q.copy_(self.h_q, non_blocking=True)
        self.kn.copy_(self.h_kn, non_blocking=True)
        self.vn.copy_(self.h_vn, non_blocking=True)
        self.bt.copy_(self.h_bt, non_blocking=True)
        self.sl.copy_(self.h_sl, non_blocking=True)
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                   out=self.out, tokens_per_split=self.tps, workspace=self.ws)
        self.h_out.copy_(self.out, non_blocking=True)

    def cpu_baseline(self, budget_s=12.0):
        """The oracle as it stands on a sample of requests of this step."""
        import oracle
        w = self.w
        order = list(range(w.B))
        # one request first to size the sample to the time budget
        t_one, _ = self._oracle_time([order[0]])
        per_tok = t_one / float(w.n_after[order[0]])
        rows, acc = [], 0.0
        for b in order:
            rows.append(b)
            acc += per_tok * float(w.n_after[b])
            if acc >= budget_s:
                break
        t, toks = self._oracle_time(rows)
        kv_bytes = toks * w.Hkv * w.D * 2 * 2
        return {"value": kv_bytes / t / 1e9, "unit": "GB/s", "tokens_per_s": toks / t,
                "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests of one decode step "
                          f"({toks} tokens, all 32 query heads), fp64 oracle, {t:.2f} s"}

    def _oracle_time(self, rows):
        import oracle
        w = self.w
        pages = [w.block_table[b, :int(synth.pages_needed(w.n_after[b]))] for b in rows]
        idx = torch.from_numpy(np.concatenate(pages).astype(np.int64)).to(self.device)
        hk = synth.bits(self.k.index_select(0, idx))
        hv = synth.bits(self.v.index_select(0, idx))
        bt = np.full((len(rows), max(len(p) for p in pages)), -1, np.int32)
        o = 0
        for i, p in enumerate(pages):
            bt[i, :len(p)] = np.arange(o, o + len(p))
            o += len(p)
        qh = synth.bits(self.q)[rows]
        sl = w.n_after[rows]
        t0 = time.perf_counter()
        oracle.decode_full_paged(qh, hk, hv, bt, sl, w.softmax_scale)
        return time.perf_counter() - t0, int(sl.sum())


# ------------------------------------------------------------------ arms --
def time_copy(device, nbytes=4 << 30, reps=10):
    import paged_hybrid_sliding_gb300 as phs
    a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    b = torch.empty_like(a)
    a.fill_(1)
    for _ in range(3):
        phs.copy_d2d(b, a)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        s.record()
        phs.copy_d2d(b, a)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del a, b
    return 2 * nbytes / best / 1e9


def run_gpu(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import paged_hybrid_sliding_gb300 as phs
    phs.lib()
    wl = PagedFullWorkload(device, batch=args.batch)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        start.record()
        for i in range(args.steps):
            wl.step(evs[i])
        stop.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = start.elapsed_time(stop) / 1e3
    split_t = statistics.fmean(a.elapsed_time(b) for a, b in evs) / 1e3
    if world > 1:
        tt = torch.tensor([t], device=device)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        t = float(tt.item())

    # end-to-end through the public API with host buffers
    for _ in range(3):
        wl.e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(10, args.steps // 4)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        wl.e2e_step()
    torch.cuda.synchronize()
    t_e2e = time.perf_counter() - t0
    copy_gbs = time_copy(device)

    peak, peak_kind = peaks()
    ms = t / args.steps * 1e3
    value = wl.bytes_per_step * args.steps * world / t / 1e9
    achieved = wl.split_bytes / split_t / 1e9
    traffic = recorded_traffic("phs_split_decode_kernel", wl.name)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.w.B, "kv_tokens_per_step": wl.tokens_per_step,
                   "bytes_per_step": wl.bytes_per_step, "tokens_per_split": wl.tps,
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": round(wl.tokens_per_step * args.steps * world / t, 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "copy_gbs": round(copy_gbs, 1),
        "pct_of_copy": round(100 * value / world / copy_gbs, 2),
        "roofline": {"bound": "hbm", "kernel": "phs_split_decode_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "bytes_per_launch": wl.split_bytes,
                     "avg_launch_ms": round(split_t * 1e3, 4), "traffic": traffic},
        "e2e": {"value": round(wl.bytes_per_step * e2e_steps * world / t_e2e / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": wl.h2d_bytes,
                "d2h_bytes_per_step": wl.d2h_bytes, "steps": e2e_steps},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = wl.cpu_baseline()
    return line


def run_reference(args, rank, budget_s=40.0):
    """The CPU oracle as the reference arm: each step is the oracle over a
    bounded sample of the same workload's requests, sized so that all
    warm-up and timed steps together take about budget_s seconds."""
    if rank != 0:
        return None
    import oracle
    w = synth.paged_full()
    order = [int(b) for b in np.argsort(w.n_after)]  # shortest first

    def inputs(rows):
        pages = [int(synth.pages_needed(w.n_after[b])) for b in rows]
        npg = sum(pages)
        kp = synth.bits(synth.normal_bf16((npg, w.Hkv, 16, w.D), 201))
        vp = synth.bits(synth.normal_bf16((npg, w.Hkv, 16, w.D), 202))
        q = synth.bits(synth.normal_bf16((len(rows), w.Hq, w.D), 203))
        bt = np.full((len(rows), max(pages)), -1, np.int32)
        o = 0
        for i, p in enumerate(pages):
            bt[i, :p] = np.arange(o, o + p)
            o += p
        return q, kp, vp, bt, w.n_after[rows]

    q, kp, vp, bt, sl = inputs(order[:1])
    t0 = time.perf_counter()
    oracle.decode_full_paged(q, kp, vp, bt, sl, w.softmax_scale)
    per_tok = (time.perf_counter() - t0) / float(sl.sum())
    per_step = budget_s / max(1, args.steps + args.warmup)
    rows, acc = [], 0.0
    for b in order:
        if rows and acc + per_tok * float(w.n_after[b]) > per_step:
            break
        rows.append(b)
        acc += per_tok * float(w.n_after[b])
    q, kp, vp, bt, sl = inputs(rows)
    toks = int(sl.sum())
    for _ in range(args.warmup):
        oracle.decode_full_paged(q, kp, vp, bt, sl, w.softmax_scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_full_paged(q, kp, vp, bt, sl, w.softmax_scale)
    t = time.perf_counter() - t0
    gbs = toks * w.Hkv * w.D * 4 * args.steps / t / 1e9
    sample = (f"{len(rows)} of {w.B} requests ({toks} tokens, all 32 query heads) of the "
              f"batch-64 paged workload per step, fp64 oracle")
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "paged_full_b64_hq32_hkv8_d128_p16_seqU[1K,32K]",
                       "sample": sample},
            "tokens_per_s": round(toks * args.steps / t, 1),
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.max_threads(), "sample": sample},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="phs", choices=["phs", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=64,
                    help="requests in the paged workload (64 = the benchmark case)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
