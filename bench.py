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


SPLIT_KERNEL_SOURCES = ("phs_decode.cu", "phs_attn.cuh", "phs_common.cuh", "phs_internal.h",
                        "phs_merge.cuh")


def peak_tflops():
    """Measured dense bf16 tensor peak (burst), TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def kernel_source_hash(files=SPLIT_KERNEL_SOURCES):
    """Hash of the kernel sources a traffic record was taken on."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_hybrid_sliding_gb300", "csrc")
    for name in files:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu records (profiles/
    traffic.json), if one was taken for this kernel and workload on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    for e in rec.get("entries", []):
        if e.get("kernel") == kernel and e.get("workload") == workload:
            if e.get("source_hash") != kernel_source_hash(e.get("sources", SPLIT_KERNEL_SOURCES)):
                return None
            return e.get("dram_bytes_per_launch")
    return None


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


# --------------------------------------------------------------- workloads --
def host_pages(pool_t, block_table, rows, n_after):
    """Host bit copy of the pages the selected requests reference, with a
    block table remapped onto that compact copy."""
    pages = [block_table[b, :int(synth.pages_needed(n_after[b]))] for b in rows]
    idx = torch.from_numpy(np.concatenate(pages).astype(np.int64)).to(pool_t.device)
    host = synth.bits(pool_t.index_select(0, idx))
    bt = np.full((len(rows), max(len(p) for p in pages)), -1, np.int32)
    o = 0
    for i, p in enumerate(pages):
        bt[i, :len(p)] = np.arange(o, o + len(p))
        o += len(p)
    return host, bt


def pinned(t):
    return t.cpu().pin_memory()


def nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


class Arena:
    """Tensors carved from one device buffer (256-byte aligned slots) and
    mirrored by one pinned host buffer, so that a step's inputs (or outputs)
    cross the host link in a single copy instead of one per tensor."""

    def __init__(self, device, tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = off
        self.dev = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        self.host = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()

        def view(buf, o, t):
            n = t.numel() * t.element_size()
            return buf[o:o + n].view(t.dtype).view(t.shape)
        self.views = [view(self.dev, o, t) for o, t in zip(offs, tensors)]
        self.host_views = [view(self.host, o, t) for o, t in zip(offs, tensors)]
        for v, t in zip(self.views, tensors):
            v.copy_(t)
        self.host.copy_(self.dev)



def rows_for_budget(n_after, order, per_token_s, budget_s):
    rows, acc = [], 0.0
    for b in order:
        if rows and acc + per_token_s * float(n_after[b]) > budget_s:
            break
        rows.append(int(b))
        acc += per_token_s * float(n_after[b])
    return rows


class Workload:
    """One decode step of a synthetic workload on the device.  Subclasses
    set the byte / token accounting and implement step() (inputs resident),
    e2e_io() / e2e_compute() (public API from pinned host buffers) and
    cpu_baseline()."""
    kernel = "phs_split_decode_kernel"
    l2 = "inputs larger than L2 (K/V read per step >> 129 MB)"
    e2e_pipelined = True

    def kernel_seconds(self, evs):
        return statistics.fmean(a.elapsed_time(b) for a, b in evs) / 1e3 if evs else None

    def new_events(self, steps):
        return [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(self.kernel_launches_per_step)] for _ in range(steps)]

    # ---- end to end through the public API, from and to pinned host memory.
    # Subclasses give e2e_io(k) -> (inputs [(host, device)], outputs
    # [(device, host)]) and e2e_compute(k) (the API calls of step k, inputs
    # resident in the device tensors).
    def e2e_run(self, steps):
        """Serving-style loop: step k+1's inputs go up on one copy stream and
        step k's outputs come down on another while step k computes.  The
        host copies land in double-buffered device staging; a step moves its
        staged inputs onto its working tensors (device copy) before its API
        calls and its outputs onto a staging slot after them.  Every step's
        host copies happen inside the loop.  A latency-bound step (where the
        staging would cost more than it hides) copies in and out directly."""
        if not self.e2e_pipelined:
            for k in range(steps):
                ins, outs = self.e2e_io(k)
                for h, d in ins:
                    d.copy_(h, non_blocking=True)
                self.e2e_compute(k)
                for src, h in outs:
                    h.copy_(src, non_blocking=True)
            return
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        comp = torch.cuda.current_stream()
        ins0, outs0 = self.e2e_io(0)
        st_in = [[torch.empty_like(d) for _, d in ins0] for _ in range(2)]
        st_out = [[torch.empty_like(src) for src, _ in outs0] for _ in range(2)]
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        h2d_done, in_free, out_ready, out_free = ev(), ev(), ev(), ev()

        def upload(k):
            b = k % 2
            ins, _ = self.e2e_io(k)
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(in_free[b])  # step k-2 has taken its inputs off slot b
                for (h, _), sbuf in zip(ins, st_in[b]):
                    sbuf.copy_(h, non_blocking=True)
                h2d_done[b].record(up)

        upload(0)
        for k in range(steps):
            b = k % 2
            if k + 1 < steps:
                upload(k + 1)
            ins, outs = self.e2e_io(k)
            comp.wait_event(h2d_done[b])
            for sbuf, (_, d) in zip(st_in[b], ins):
                d.copy_(sbuf, non_blocking=True)
            in_free[b].record(comp)
            self.e2e_compute(k)
            if k >= 2:
                comp.wait_event(out_free[b])  # step k-2's outputs have left slot b
            for (src, _), obuf in zip(outs, st_out[b]):
                obuf.copy_(src, non_blocking=True)
            out_ready[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                for obuf, (_, h) in zip(st_out[b], outs):
                    h.copy_(obuf, non_blocking=True)
                out_free[b].record(down)


class PagedFullWorkload(Workload):
    """Paged Full-attention decode, batch 64 (one step = append + decode)."""

    kernel_launches_per_step = 1

    def __init__(self, device, seed=2, batch=64, tokens_per_split=0):
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
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq, tokens_per_split)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps),
                              dtype=torch.uint8, device=device)
        tokens = int(w.n_after.sum())
        self.tokens_per_step = tokens
        kv = tokens * Hkv * D * 2 * 2
        qo = 2 * B * Hq * D * 2
        app = 2 * B * Hkv * D * 2 * 2
        tables = int(synth.pages_needed(w.n_after).sum()) * 4 + B * 4
        self.bytes_per_step = kv + qo + app + tables
        self.kernel_bytes = kv + B * Hq * D * 2 + tables
        self.launches_per_step = 3
        self.extra = {"batch": B, "tokens_per_split": self.tps}
        # the step's inputs in one staged buffer: one host->device copy per step
        self.inp = Arena(device, [self.q, self.kn, self.vn, self.bt, self.sl])
        self.q, self.kn, self.vn, self.bt, self.sl = self.inp.views
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = nbytes(self.h_out)

    def step(self, ev=None):
        phs = self.phs
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        if ev is not None:
            ev[0][0].record()
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                         self.ws, self.out, tokens_per_split=self.tps)
        if ev is not None:
            ev[0][1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, self.sl, self.max_seq, self.ws,
                              tokens_per_split=self.tps)

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.out, self.h_out)]

    def e2e_compute(self, k):
        phs = self.phs
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                   out=self.out, tokens_per_split=self.tps, workspace=self.ws)

    def cpu_baseline(self, budget_s=12.0):
        """The oracle as it stands on a sample of requests of this step."""
        import oracle
        w = self.w
        t1, _ = self._oracle_time([0])
        rows = rows_for_budget(w.n_after, range(w.B), t1 / float(w.n_after[0]), budget_s)
        t, toks = self._oracle_time(rows)
        kv_bytes = toks * w.Hkv * w.D * 2 * 2
        return {"value": kv_bytes / t / 1e9, "unit": "GB/s", "tokens_per_s": toks / t,
                "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests of one decode step "
                          f"({toks} tokens, all {w.Hq} query heads), fp64 oracle, {t:.2f} s"}

    def _oracle_time(self, rows):
        import oracle
        w = self.w
        hk, bt = host_pages(self.k, w.block_table, rows, w.n_after)
        hv, _ = host_pages(self.v, w.block_table, rows, w.n_after)
        qh = synth.bits(self.q)[rows]
        sl = w.n_after[rows]
        t0 = time.perf_counter()
        oracle.decode_full_paged(qh, hk, hv, bt, sl, w.softmax_scale)
        return time.perf_counter() - t0, int(sl.sum())


class TinyHybridWorkload(Workload):
    """Batch 2, 4 q / 2 KV heads, D 64: one Full (paged) + one SWA (ring)
    layer, append + attend through the hybrid-stack call.  Latency-bound."""

    kernel_launches_per_step = 0
    l2 = "latency-bound case: ~0.2 MB per step, resident in L2"
    e2e_pipelined = False  # 13 us steps: staging costs more than it hides

    def __init__(self, device, seed=1, fused=True):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.fused = fused
        self.w = w = synth.tiny_hybrid(seed=seed)
        self.name = "tiny_hybrid_b2_hq4_hkv2_d64_full+swa_w128"
        B, Hq, Hkv, D, W = w.B, w.Hq, w.Hkv, w.D, w.W
        g = seed * 100
        self.kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 1, device=device)
        self.vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 2, device=device)
        self.kr = synth.normal_bf16((B, Hkv, W, D), g + 3, device=device)
        self.vr = synth.normal_bf16((B, Hkv, W, D), g + 4, device=device)
        self.qf = synth.normal_bf16((B, Hq, D), g + 5, device=device)
        self.qs = synth.normal_bf16((B, Hq, D), g + 6, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), g + 7, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), g + 8, device=device)
        self.of = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
        self.os = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
        self.bt = torch.from_numpy(w.block_table).to(device)
        self.sl = torch.from_numpy(w.n_after).to(device)
        self.rp = torch.from_numpy(w.ring_pos).to(device)
        # the step's inputs and outputs each in one staged buffer
        self.inp = Arena(device, [self.qf, self.qs, self.kn, self.vn, self.sl, self.rp, self.bt])
        self.qf, self.qs, self.kn, self.vn, self.sl, self.rp, self.bt = self.inp.views
        self.outp = Arena(device, [self.of, self.os])
        self.of, self.os = self.outp.views
        self.layers = [
            phs.Layer(q=self.qf, out=self.of, paged=phs.PagedPool(self.kp, self.vp),
                      k_new=self.kn, v_new=self.vn),
            phs.Layer(q=self.qs, out=self.os, ring=phs.RingPool(self.kr, self.vr),
                      k_new=self.kn, v_new=self.vn)]
        self.max_seq = int(w.n_after.max())
        ws_bytes = (phs.hybrid_stack_fused_workspace_bytes(B, Hq, Hkv, D, self.max_seq, 1)
                    if fused else phs.hybrid_stack_workspace_bytes(B, Hq, Hkv, D, self.max_seq))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        full_tok = int(w.n_after.sum())
        swa_tok = int(np.minimum(w.n_after, W).sum())
        self.tokens_per_step = full_tok + swa_tok
        tok_bytes = Hkv * D * 2 * 2
        self.bytes_per_step = (full_tok + swa_tok) * tok_bytes + 2 * 2 * B * Hq * D * 2 + \
            2 * 2 * B * Hkv * D * 2
        self.kernel_bytes = None
        # fused: Full split (append fused, one split: no merge) + SWA decode;
        # else 2 appends, SWA decode, split
        self.launches_per_step = 2 if fused else 4
        self.extra = {"batch": B, "layers": "1 Full + 1 SWA(W=128)",
                      "append_fused_into_attention": fused}
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = self.outp.nbytes

    def step(self, ev=None):
        if self.fused:
            self.phs.attn_decode_hybrid_stack_fused(self.layers, self.w.Hq, self.sl, self.max_seq,
                                                    block_table=self.bt, ring_pos=self.rp,
                                                    workspace=self.ws)
            return
        self.phs.attn_decode_hybrid_stack(self.layers, self.w.Hq, self.sl, self.max_seq,
                                          block_table=self.bt, ring_pos=self.rp,
                                          workspace=self.ws)

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.outp.dev, self.outp.host)]

    def e2e_compute(self, k):
        self.step()

    def cpu_baseline(self):
        import oracle
        w = self.w
        hk, hv = synth.bits(self.kp), synth.bits(self.vp)
        hkr, hvr = synth.bits(self.kr), synth.bits(self.vr)
        kn, vn = synth.bits(self.kn), synth.bits(self.vn)
        qf, qs = synth.bits(self.qf), synth.bits(self.qs)
        reps = 200
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.append_paged(hk, hv, kn, vn, w.block_table, w.n_after)
            oracle.append_ring(hkr, hvr, kn, vn, None, w.ring_pos)
            oracle.decode_full_paged(qf, hk, hv, w.block_table, w.n_after, w.softmax_scale)
            oracle.decode_swa_ring(qs, hkr, hvr, None, w.ring_pos, w.n_after, w.softmax_scale)
        t = (time.perf_counter() - t0) / reps
        return {"value": self.bytes_per_step / t / 1e9, "unit": "GB/s",
                "us_per_step": t * 1e6, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"the whole step (2 appends + 2 decodes), mean of {reps} repetitions"}


class HybridStackWorkload(Workload):
    """70 layers (Full iff layer % 7 == 6: 10 Full, 60 SWA W=128), batch 256,
    32 q / 8 KV heads, D 128, lengths log-uniform in [4K, 128K]; one step =
    append into every layer + attend every layer, one hybrid-stack call.
    Ten distinct 37.6 GB Full pools do not fit one GPU: `distinct` pools are
    allocated and the Full layers use them round-robin (each layer still
    streams its whole pool, far above L2, so no layer reads another's data
    from cache)."""

    kernel_launches_per_step = 0

    def __init__(self, device, seed=3, distinct=4, batch=256, swa_only=False, fused=True):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.fused = fused
        self.w = w = synth.hybrid_stack(seed=seed, B=batch)
        B, Hq, Hkv, D, W = w.B, w.Hq, w.Hkv, w.D, w.W
        lf = w.extra["layer_is_full"]
        if swa_only:
            lf = np.zeros_like(lf)[:60]
            distinct = 0
        self.swa_only = swa_only
        self.name = (f"hybrid_stack_70l_10full_60swa_w128_b{B}_hq32_hkv8_d128_seqlogU[4K,128K]"
                     if not swa_only else f"swa_60l_w128_b{B}_hq32_hkv8_d128")
        g = seed * 1000
        self.pools = [phs.PagedPool(
            synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 10 * i + 1, device=device),
            synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 10 * i + 2, device=device))
            for i in range(distinct)]
        self.layers, nf = [], 0
        self.dev_in, self.outs = [], []
        for l, full in enumerate(lf):
            q = synth.normal_bf16((B, Hq, D), g + 500 + 3 * l, device=device)
            kn = synth.normal_bf16((B, Hkv, D), g + 501 + 3 * l, device=device)
            vn = synth.normal_bf16((B, Hkv, D), g + 502 + 3 * l, device=device)
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
            if full:
                L = phs.Layer(q=q, out=out, paged=self.pools[nf % distinct], k_new=kn, v_new=vn)
                nf += 1
            else:
                ring = phs.RingPool(synth.normal_bf16((B, Hkv, W, D), g + 800 + 2 * l,
                                                      device=device),
                                    synth.normal_bf16((B, Hkv, W, D), g + 801 + 2 * l,
                                                      device=device))
                L = phs.Layer(q=q, out=out, ring=ring, k_new=kn, v_new=vn)
            self.layers.append(L)
            self.dev_in += [q, kn, vn]
            self.outs.append(out)
        self.bt = torch.from_numpy(w.block_table).to(device)
        self.sl = torch.from_numpy(w.n_after).to(device)
        self.rp = torch.from_numpy(w.ring_pos).to(device)
        self.dev_in += [self.bt, self.sl, self.rp]
        # every layer's q / k_new / v_new and the tables in one staged buffer,
        # every layer's output in another: one copy each way per step
        self.inp = Arena(device, self.dev_in)
        v = self.inp.views
        for l, L in enumerate(self.layers):
            L.q, L.k_new, L.v_new = v[3 * l], v[3 * l + 1], v[3 * l + 2]
        self.bt, self.sl, self.rp = v[-3], v[-2], v[-1]
        self.outp = Arena(device, self.outs)
        for L, o in zip(self.layers, self.outp.views):
            L.out = o
        self.outs = self.outp.views
        del self.dev_in
        self.max_seq = int(w.n_after.max())
        nfull, nswa = int(lf.sum()), int(len(lf) - lf.sum())
        ws_bytes = (phs.hybrid_stack_fused_workspace_bytes(B, Hq, Hkv, D, self.max_seq, nfull)
                    if fused else phs.hybrid_stack_workspace_bytes(B, Hq, Hkv, D, self.max_seq))
        self.ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
        full_tok = int(w.n_after.sum())
        swa_tok = int(np.minimum(w.n_after, W).sum())
        tok_bytes = Hkv * D * 2 * 2
        self.tokens_per_step = nfull * full_tok + nswa * swa_tok
        small = len(lf) * (2 * B * Hq * D * 2 + 2 * B * Hkv * D * 2 * 2)
        tables = nfull * (int(synth.pages_needed(w.n_after).sum()) * 4)
        self.bytes_per_step = self.tokens_per_step * tok_bytes + small + tables
        self.full_layer_bytes = full_tok * tok_bytes + B * Hq * D * 2 + \
            int(synth.pages_needed(w.n_after).sum()) * 4
        self.swa_bytes = nswa * (swa_tok * tok_bytes + B * Hq * D * 2)
        self.kernel_bytes = self.full_layer_bytes if nfull else self.swa_bytes
        if not nfull:
            self.kernel = "phs_swa_decode_kernel"
        elif fused:
            self.kernel = ("phs_stack_full_kernel + merges (all Full layers in one launch, "
                           "append fused; per-layer average)")
        if fused:
            # Full split launch + SWA launch (which also runs the Full merges)
            self.launches_per_step = (1 if nfull else 0) + (1 if nswa else 0) + \
                (1 if nfull and not nswa else 0)
        else:
            self.launches_per_step = (2 if nfull else 1) + 1 + 2 * nfull
        self.extra = {"batch": B, "layers": f"{nfull} Full + {nswa} SWA(W=128)",
                      "distinct_full_pools": distinct, "full_layers_aliased_onto": distinct,
                      "full_bytes_per_step": nfull * self.full_layer_bytes,
                      "swa_bytes_per_step": self.swa_bytes,
                      "append_fused_into_attention": fused}
        if nfull:
            self.extra["kv_tokens_stored_ratio_vs_all_full"] = round(
                (nfull * full_tok + nswa * swa_tok) / (len(lf) * full_tok), 4)
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = self.outp.nbytes

    def step(self, ev=None):
        if self.fused:
            self.phs.attn_decode_hybrid_stack_fused(self.layers, self.w.Hq, self.sl, self.max_seq,
                                                    block_table=self.bt, ring_pos=self.rp,
                                                    workspace=self.ws)
            return
        self.phs.attn_decode_hybrid_stack(self.layers, self.w.Hq, self.sl, self.max_seq,
                                          block_table=self.bt, ring_pos=self.rp,
                                          workspace=self.ws)

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.outp.dev, self.outp.host)]

    def e2e_compute(self, k):
        self.step()

    def kernel_times(self, reps=3):
        """Average launch time of the split kernel on the Full layers and of
        the SWA kernel on all SWA layers (separate timed loops)."""
        phs = self.phs
        w = self.w
        full = [L for L in self.layers if L.paged is not None]
        if not full:
            return None, self._swa_time(reps)
        if self.fused:
            # the step's Full part: one multi-layer split launch (append fused)
            # plus its merges (a merge launch, as the layers run without the
            # SWA launch here); per-layer average reported
            def run():
                phs.attn_decode_hybrid_stack_fused(full, w.Hq, self.sl, self.max_seq,
                                                   block_table=self.bt, workspace=self.ws)
            run()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                run()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / 1e3 / reps / len(full), self._swa_time(reps)
        ts = []
        for _ in range(reps):
            for L in full:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                phs.attn_decode_full_paged_split(L.q, L.paged, self.bt, self.sl, self.max_seq,
                                                 self.ws, L.out)
                b.record()
                ts.append((a, b))
        torch.cuda.synchronize()
        split_s = statistics.fmean(a.elapsed_time(b) for a, b in ts) / 1e3
        return split_s, self._swa_time(reps)

    def _swa_time(self, reps):
        w = self.w
        swa = [self.phs.Layer(q=L.q, out=L.out, ring=L.ring) for L in self.layers
               if L.ring is not None]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.phs.attn_decode_hybrid_stack(swa, w.Hq, self.sl, self.max_seq, ring_pos=self.rp,
                                          do_append=False)
        a.record()
        for _ in range(reps):
            self.phs.attn_decode_hybrid_stack(swa, w.Hq, self.sl, self.max_seq, ring_pos=self.rp,
                                              do_append=False)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / reps

    def cpu_baseline(self, budget_s=12.0):
        import oracle
        w = self.w
        if self.swa_only:
            return self._cpu_baseline_swa()
        L = next(L for L in self.layers if L.paged is not None)
        order = [int(b) for b in np.argsort(w.n_after)]
        hk, bt = host_pages(L.paged.k, w.block_table, order[:1], w.n_after)
        hv, _ = host_pages(L.paged.v, w.block_table, order[:1], w.n_after)
        t0 = time.perf_counter()
        oracle.decode_full_paged(synth.bits(L.q)[order[:1]], hk, hv, bt, w.n_after[order[:1]],
                                 w.softmax_scale)
        per_tok = (time.perf_counter() - t0) / float(w.n_after[order[0]])
        rows = rows_for_budget(w.n_after, order, per_tok, budget_s)
        hk, bt = host_pages(L.paged.k, w.block_table, rows, w.n_after)
        hv, _ = host_pages(L.paged.v, w.block_table, rows, w.n_after)
        t0 = time.perf_counter()
        oracle.decode_full_paged(synth.bits(L.q)[rows], hk, hv, bt, w.n_after[rows],
                                 w.softmax_scale)
        t = time.perf_counter() - t0
        toks = int(w.n_after[rows].sum())
        return {"value": toks * w.Hkv * w.D * 4 / t / 1e9, "unit": "GB/s",
                "tokens_per_s": toks / t, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests of one Full layer ({toks} tokens), "
                          f"fp64 oracle, {t:.2f} s"}


    def _cpu_baseline_swa(self):
        import oracle
        w = self.w
        L = next(L for L in self.layers if L.ring is not None)
        kr, vr, q = synth.bits(L.ring.k), synth.bits(L.ring.v), synth.bits(L.q)
        t0 = time.perf_counter()
        oracle.decode_swa_ring(q, kr, vr, None, w.ring_pos, w.n_after, w.softmax_scale)
        t = time.perf_counter() - t0
        toks = int(np.minimum(w.n_after, w.W).sum())
        return {"value": toks * w.Hkv * w.D * 4 / t / 1e9, "unit": "GB/s",
                "tokens_per_s": toks / t, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"one SWA layer, all {w.B} requests ({toks} tokens), fp64 oracle, "
                          f"{t:.2f} s"}


class Int8Workload(Workload):
    """Batch 32, 65,536 cached tokens: tokens [0, 64512) as INT8 (one fp32
    absmax/127 scale per 32 tokens per KV head, quantised on the GPU at set
    up), the last 1025 in bf16; K/V N(0,1) with 1% N(0, 8^2) outliers.  One
    step = append into the bf16 tail + split-KV decode + merge."""

    kernel_launches_per_step = 1

    def __init__(self, device, seed=4, batch=32, tokens_per_split=0):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.w = w = synth.int8_block32(seed=seed, B=batch)
        B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
        self.name = f"int8_block32_b{B}_n65536_hot1024_hq32_hkv8_d128"
        g = seed * 100
        self.k = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 1, device=device,
                                   outlier_p=0.01)
        self.v = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 2, device=device,
                                   outlier_p=0.01)
        self.pool = phs.PagedPool(self.k, self.v)
        self.qlen = w.extra["qlen"]
        self.qt = torch.from_numpy(w.extra["qtable"]).to(device)
        self.i8 = phs.Int8Pool.empty(w.extra["num_qpages"], Hkv, D, device=device)
        self.bt = torch.from_numpy(w.block_table).to(device)
        nqb = (self.qlen // 32).astype(np.int32)
        zeros = torch.zeros(B, dtype=torch.int32, device=device)
        nqb_d = torch.from_numpy(nqb).to(device)

        def quantise():
            phs.kv_quant_int8_block32(self.pool, self.bt, self.i8, self.qt, zeros, nqb_d,
                                      int(nqb.max()))
        quantise()  # set-up (also loads the module); then time warm repeats
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        a.record()
        for _ in range(reps):
            quantise()
        b.record()
        torch.cuda.synchronize()
        q_s = a.elapsed_time(b) / 1e3 / reps
        # algorithmic bytes: read the bf16 group, write codes + one scale
        qbytes = int(nqb.sum()) * Hkv * 2 * (32 * D * 2 + 32 * D + 4)
        self.quant_setup = {"kernel": "phs_quant_kernel", "ms": round(q_s * 1e3, 3),
                            "GB/s": round(qbytes / q_s / 1e9, 1), "bytes": qbytes}
        self.q = synth.normal_bf16((B, Hq, D), g + 3, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), g + 4, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), g + 5, device=device)
        self.sl = torch.from_numpy(w.n_after).to(device)
        self.ql = torch.from_numpy(self.qlen).to(device)
        self.max_seq = int(w.n_after.max())
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq, tokens_per_split)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps,
                                                         has_int8=True),
                              dtype=torch.uint8, device=device)
        i8_tok = int(self.qlen.sum())
        bf_tok = int((w.n_after - self.qlen).sum())
        self.tokens_per_step = i8_tok + bf_tok
        codes = i8_tok * Hkv * D * 2
        scales = i8_tok // 32 * Hkv * 4 * 2
        tail = bf_tok * Hkv * D * 2 * 2
        tables = int(synth.pages_needed(w.n_after - self.qlen).sum()) * 4 + i8_tok // 32 * 4
        self.kernel_bytes = codes + scales + tail + B * Hq * D * 2 + tables
        self.bytes_per_step = self.kernel_bytes + B * Hq * D * 2 + 2 * B * Hkv * D * 2 * 2
        self.launches_per_step = 3
        self.extra = {"batch": B, "int8_tokens": i8_tok, "bf16_tokens": bf_tok,
                      "codes_bytes": codes, "scale_bytes": scales, "bf16_tail_bytes": tail,
                      "tokens_per_split": self.tps, "quantiser_setup": self.quant_setup}
        self.inp = Arena(device, [self.q, self.kn, self.vn, self.sl])
        self.q, self.kn, self.vn, self.sl = self.inp.views
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = nbytes(self.h_out)

    def _decode(self, split_only=False):
        phs = self.phs
        if split_only:
            phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                             self.ws, self.out, int8=self.i8, qtable=self.qt,
                                             qlens=self.ql, tokens_per_split=self.tps)
        else:
            phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                       int8=self.i8, qtable=self.qt, qlens=self.ql,
                                       tokens_per_split=self.tps, out=self.out,
                                       workspace=self.ws)

    def step(self, ev=None):
        self.phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        if ev is not None:
            ev[0][0].record()
        self._decode(split_only=True)
        if ev is not None:
            ev[0][1].record()
        self.phs.attn_merge_splits(self.out, self.w.Hkv, self.sl, self.max_seq, self.ws,
                                   qlens=self.ql, has_int8=True, tokens_per_split=self.tps)

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.out, self.h_out)]

    def e2e_compute(self, k):
        self.phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl)
        self._decode()

    def cpu_baseline(self):
        import oracle
        w = self.w
        rows = [0]
        hk, bt = host_pages(self.k, w.block_table, rows, w.n_after)
        hv, _ = host_pages(self.v, w.block_table, rows, w.n_after)
        nq = int(self.qlen[0] // 32)
        ids = self.qt[0, :nq].long()
        i8 = dict(k_codes=self.i8.k.index_select(0, ids).cpu().numpy(),
                  v_codes=self.i8.v.index_select(0, ids).cpu().numpy(),
                  k_scale=self.i8.k_scale.index_select(0, ids).cpu().numpy(),
                  v_scale=self.i8.v_scale.index_select(0, ids).cpu().numpy(),
                  qtable=np.arange(nq, dtype=np.int32)[None], qlens=self.qlen[rows])
        t0 = time.perf_counter()
        oracle.decode_full_paged(synth.bits(self.q)[rows], hk, hv, bt, w.n_after[rows],
                                 w.softmax_scale, int8=i8)
        t = time.perf_counter() - t0
        b = self.kernel_bytes / w.B
        return {"value": b / t / 1e9, "unit": "GB/s", "tokens_per_s": float(w.n_after[0]) / t,
                "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"1 of {w.B} requests ({int(w.n_after[0])} tokens, INT8 + bf16 tail),"
                          f" fp64 oracle, {t:.2f} s"}


class SharedPrefixWorkload(Workload):
    """64 requests sharing one 250,000-token prefix (15,625 pages, refcount
    64) + a unique 512-token suffix each; 128 decode steps with append.  One
    bench step = one decode step; the timed loop walks the 128 steps."""

    kernel_launches_per_step = 1
    l2 = "logical K/V bytes per step 65.7 GB >> L2; the shared prefix is reused through L2"

    def __init__(self, device, seed=5, prefix_kernel=True, prefix_len=250_000):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.w = w = synth.shared_prefix(seed=seed, prefix=prefix_len)
        B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
        self.name = f"shared_prefix_{prefix_len}_b64_suffix512_128steps_hq32_hkv8_d128"
        g = seed * 100
        self.k = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 1, device=device)
        self.v = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 2, device=device)
        self.pool = phs.PagedPool(self.k, self.v)
        self.bt = torch.from_numpy(w.block_table).to(device)
        self.rc = torch.from_numpy(w.extra["refcount"]).to(device)
        self.nsteps = w.extra["steps"]
        self.sls = [torch.from_numpy((w.n_pre + 1 + k).astype(np.int32)).to(device)
                    for k in range(self.nsteps)]
        self.q = synth.normal_bf16((B, Hq, D), g + 3, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), g + 4, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), g + 5, device=device)
        self.max_seq = int(w.n_pre.max()) + self.nsteps
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps),
                              dtype=torch.uint8, device=device)
        self.k_idx = 0
        # tensor-core pass over the shared prefix (whole 64-token tiles)
        self.prefix_kernel = prefix_kernel
        self.shared_len = (w.extra["prefix_pages"] * 16 // 64) * 64
        if prefix_kernel:
            self.ws = torch.empty(phs.shared_prefix_workspace_bytes(B, Hq, Hkv, D, self.max_seq,
                                                                    self.shared_len),
                                  dtype=torch.uint8, device=device)
            self.kernel = "phs_attn_decode_shared_prefix (prefix tcgen05 + suffix split + merge)"
            self.l2 = "prefix read once per KV head for all 64 requests (tensor-core pass)"
        mean_n = float(w.n_pre.mean()) + (self.nsteps + 1) / 2
        tok_bytes = Hkv * D * 2 * 2
        self.tokens_per_step = int(round(B * mean_n))
        self.bytes_per_step = self.tokens_per_step * tok_bytes + 2 * B * Hq * D * 2 + \
            2 * B * Hkv * D * 2 * 2
        self.kernel_bytes = self.tokens_per_step * tok_bytes + B * Hq * D * 2
        npref = w.extra["prefix_pages"]
        unique_tok = npref * 16 + B * (float(w.n_pre.mean()) - npref * 16 + (self.nsteps + 1) / 2)
        self.unique_bytes = int(unique_tok * tok_bytes)
        self.launches_per_step = 4 if prefix_kernel else 3
        # tensor work of the prefix pass: QK and PV over B*G rows x D per token
        self.prefix_flops = 4 * B * Hq * D * self.shared_len
        self.extra = {"batch": B, "logical_bytes_per_step": self.bytes_per_step,
                      "unique_kv_bytes_per_step": self.unique_bytes,
                      "tokens_per_split": self.tps, "shared_prefix_kernel": prefix_kernel,
                      "shared_len_tensor_pass": self.shared_len if prefix_kernel else 0}
        # q / k_new / v_new in one staged buffer; the step's lengths (a
        # different vector every step) travel in a second copy
        self.inp = Arena(device, [self.q, self.kn, self.vn])
        self.q, self.kn, self.vn = self.inp.views
        self.h_sls = [pinned(s) for s in self.sls]
        self.sl_in = torch.empty_like(self.sls[0])
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = self.inp.nbytes + nbytes(self.h_sls[0])
        self.d2h_bytes = nbytes(self.h_out)

    def step(self, ev=None):
        phs = self.phs
        sl = self.sls[self.k_idx % self.nsteps]
        self.k_idx += 1
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, sl, page_refcount=self.rc)
        if ev is not None:
            ev[0][0].record()
        if self.prefix_kernel:
            phs.attn_decode_shared_prefix(self.q, self.pool, self.bt, sl, self.max_seq,
                                          self.shared_len, out=self.out, workspace=self.ws)
            if ev is not None:
                ev[0][1].record()
            return
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, sl, self.max_seq, self.ws,
                                         self.out, tokens_per_split=self.tps)
        if ev is not None:
            ev[0][1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, sl, self.max_seq, self.ws,
                              tokens_per_split=self.tps)

    def e2e_io(self, k):
        return ([(self.inp.host, self.inp.dev), (self.h_sls[k % self.nsteps], self.sl_in)],
                [(self.out, self.h_out)])

    def e2e_compute(self, k):
        self.phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl_in,
                                 page_refcount=self.rc)
        if self.prefix_kernel:
            self.phs.attn_decode_shared_prefix(self.q, self.pool, self.bt, self.sl_in,
                                               self.max_seq, self.shared_len, out=self.out,
                                               workspace=self.ws)
        else:
            self.phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl_in, self.max_seq,
                                            out=self.out, tokens_per_split=self.tps,
                                            workspace=self.ws)

    def cpu_baseline(self):
        import oracle
        w = self.w
        rows = [0]
        n = w.n_pre + 1
        hk, bt = host_pages(self.k, w.block_table, rows, n)
        hv, _ = host_pages(self.v, w.block_table, rows, n)
        t0 = time.perf_counter()
        oracle.decode_full_paged(synth.bits(self.q)[rows], hk, hv, bt, n[rows], w.softmax_scale)
        t = time.perf_counter() - t0
        toks = int(n[0])
        return {"value": toks * w.Hkv * w.D * 4 / t / 1e9, "unit": "GB/s",
                "tokens_per_s": toks / t, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"1 of {w.B} requests of one step ({toks} tokens), fp64 oracle, "
                          f"{t:.2f} s"}


def make_workload(config, device, args):
    if config == 1:
        return TinyHybridWorkload(device, fused=not args.no_fused)
    if config == 2:
        return PagedFullWorkload(device, batch=args.batch or 64,
                                 tokens_per_split=args.tokens_per_split)
    if config == 3:
        return HybridStackWorkload(device, distinct=args.distinct_pools,
                                   batch=args.batch or 256, swa_only=args.swa_only,
                                   fused=not args.no_fused)
    if config == 4:
        return Int8Workload(device, batch=args.batch or 32,
                            tokens_per_split=args.tokens_per_split)
    if config == 5:
        return SharedPrefixWorkload(device, prefix_kernel=not args.no_prefix_kernel,
                                    prefix_len=args.prefix_len)
    raise ValueError(config)


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


def slowest_rank_time(t, world, device=None):
    """Timed-region length of the slowest rank (the job's time).  Replicas
    exchange nothing else: this MAX is the only collective."""
    if world <= 1:
        return t
    tt = torch.tensor([float(t)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(bytes_per_step, steps, world, t):
    """Whole-job throughput: every rank processes its own replica."""
    return bytes_per_step * steps * world / t / 1e9


def run_gpu(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import paged_hybrid_sliding_gb300 as phs
    phs.lib()
    wl = make_workload(args.config, device, args)
    use_graph = args.graph if args.graph is not None else args.config == 1
    if use_graph and isinstance(wl, SharedPrefixWorkload):
        raise SystemExit("--graph: the shared-prefix steps change lengths every step")
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        # one step recorded as a CUDA graph and replayed: the library's
        # launches are captured as they are issued on the current stream
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wl.step()
        graph.replay()
        torch.cuda.synchronize()
    # the dominant kernel is timed with CUDA events around its launch on every
    # `stride`-th step of the timed loop: an event between two launches ends
    # the programmatic overlap of the second with the first, so events on
    # every step would slow the step they measure
    stride = max(1, args.steps // 200)
    evs = [] if graph is not None else wl.new_events((args.steps + stride - 1) // stride)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        start.record()
        for i in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                wl.step(evs[i // stride] if evs and i % stride == 0 else None)
        stop.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = start.elapsed_time(stop) / 1e3
    flat = [p for e in evs for p in e]
    kernel_s = wl.kernel_seconds(flat)
    t = slowest_rank_time(t, world, device)
    extra_kernels = {}
    if isinstance(wl, HybridStackWorkload):
        kernel_s, swa_s = wl.kernel_times()
        if kernel_s is None:
            kernel_s = swa_s
        else:
            extra_kernels["phs_swa_decode_kernel"] = {
                "bytes_per_launch": wl.swa_bytes, "avg_launch_ms": round(swa_s * 1e3, 4),
                "achieved_gbs": round(wl.swa_bytes / swa_s / 1e9, 1),
                "frac": round(wl.swa_bytes / swa_s / 1e9 / peaks()[0], 4)}

    # end-to-end through the public API with host buffers (copies overlapped
    # with compute, as a serving loop would)
    wl.e2e_run(3)
    torch.cuda.synchronize()
    e2e_steps = max(3, args.steps // 4)
    t0 = time.perf_counter()
    wl.e2e_run(e2e_steps)
    torch.cuda.synchronize()
    t_e2e = time.perf_counter() - t0
    copy_gbs = time_copy(device)

    peak, peak_kind = peaks()
    ms = t / args.steps * 1e3
    value = job_throughput(wl.bytes_per_step, args.steps, world, t)
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
        "config": {"workload": wl.name, "kv_tokens_per_step": wl.tokens_per_step,
                   "bytes_per_step": wl.bytes_per_step, "l2": wl.l2,
                   "parallelism": "replicas" if world > 1 else "single", **wl.extra},
        "tokens_per_s": round(wl.tokens_per_step * args.steps * world / t, 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "copy_gbs": round(copy_gbs, 1),
        "pct_of_copy": round(100 * value / world / copy_gbs, 2),
        "e2e": {"value": round(wl.bytes_per_step * e2e_steps * world / t_e2e / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": wl.h2d_bytes,
                "d2h_bytes_per_step": wl.d2h_bytes, "steps": e2e_steps,
                "copies": ("every step's inputs up and outputs down through pinned host "
                           "buffers, overlapped with the previous/next step's compute (two "
                           "copy streams, double-buffered device staging)"
                           if wl.e2e_pipelined else
                           "every step's inputs up and outputs down through pinned host "
                           "buffers, in line with the step")},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    line["config"]["cuda_graph"] = graph is not None
    if isinstance(wl, TinyHybridWorkload):
        line["us_per_step"] = round(ms * 1e3, 2)
    if kernel_s is not None and wl.kernel_bytes:
        achieved = wl.kernel_bytes / kernel_s / 1e9
        line["roofline"] = {
            "bound": "hbm", "kernel": wl.kernel, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "bytes_per_launch": wl.kernel_bytes, "avg_launch_ms": round(kernel_s * 1e3, 4),
            "traffic": recorded_traffic(wl.kernel, wl.name)}
        if flat:
            line["roofline"]["timed_launches"] = (
                f"{len(flat)} launches inside the timed loop (CUDA events around the launch, "
                f"on its stream, in 1 of every {stride} steps)")
        if isinstance(wl, SharedPrefixWorkload):
            if wl.prefix_kernel:
                # the decode call reads each prefix page once: its HBM bound is
                # the unique bytes; its tensor work is the prefix contraction
                uniq = wl.unique_bytes / kernel_s / 1e9
                tflops = wl.prefix_flops / kernel_s / 1e12
                line["roofline"].update({
                    "achieved": round(uniq, 1), "frac": round(uniq / peak, 4),
                    "bytes_per_launch": wl.unique_bytes,
                    "bytes_are": "unique K/V bytes (prefix read once per KV head)",
                    "logical_gbs": round(achieved, 1),
                    "tensor_tflops": round(tflops, 1),
                    "tensor_frac_of_bf16_peak": round(tflops / peak_tflops()[0], 4)})
            else:
                line["roofline"]["bytes_are"] = "logical (prefix pages reused through L2)"
                line["roofline"]["unique_kv_gbs"] = round(wl.unique_bytes / kernel_s / 1e9, 1)
    if extra_kernels:
        line["other_kernels"] = extra_kernels
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
    ap.add_argument("--batch", type=int, default=0,
                    help="requests (0 = the workload's own batch: 64 / 256 / 32 for configs "
                         "2 / 3 / 4); smaller batches are for profiler captures")
    ap.add_argument("--tokens-per-split", type=int, default=0,
                    help="configs 2 and 4: split length (0 = the library's choice for the "
                         "batch); profiler captures of a smaller batch pass the full-size one")
    ap.add_argument("--graph", dest="graph", action="store_true", default=None,
                    help="replay each step as a CUDA graph (default: only for config 1)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--no-prefix-kernel", action="store_true",
                    help="config 5: decode each request separately (no shared-prefix pass)")
    ap.add_argument("--prefix-len", type=int, default=250_000,
                    help="config 5: shared prefix tokens (a multiple of 16; smaller for "
                         "profiler captures)")
    ap.add_argument("--swa-only", action="store_true",
                    help="config 3: only the 60 SWA layers (profiler captures)")
    ap.add_argument("--no-fused", action="store_true",
                    help="configs 1 and 3: separate append launches and one split + merge per "
                         "Full layer instead of the fused step (appends inside the attention "
                         "launches, all Full layers in one launch)")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5],
                    help="1 tiny hybrid, 2 paged Full batch 64 (default), 3 70-layer hybrid "
                         "stack, 4 INT8 block-32, 5 shared 250K prefix")
    ap.add_argument("--distinct-pools", type=int, default=4,
                    help="config 3: distinct 37.6 GB Full pools allocated (layers alias them)")
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
