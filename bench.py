"""Benchmark of the decode hot path on synthetic workloads.

Default run (no --config): every workload in one invocation.  The headline
line is the 70-layer hybrid stack (10 Full paged layers + 60 SWA ring layers
of W = 128, batch 256, 32 query / 8 KV heads, head_dim 128, lengths
log-uniform in [4K, 128K]): one step appends every layer's new token and
attends every layer, through the fused hybrid-stack call (two launches).
The tiny hybrid case, the batch-64 paged Full decode, the INT8 block-32
decode (with the rolling hot-to-warm hand-off) and the shared 250K-token
prefix decode are measured in the same run, each with its own roofline,
end-to-end number and CPU-oracle baseline, under the line's "configs" key.
--config N measures one workload alone.

Each line gives the throughput in algorithmic HBM GB/s (the K/V bytes the
step must read, plus query, output, table and append bytes), attended KV
tokens/s, the roofline of the dominant kernel (CUDA events around its
launch on its stream inside the timed loop), an end-to-end number through
the public API with host buffers, and the CPU oracle timed on a bounded
sample on the host cores.  --impl reference times the CPU oracle alone.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no exchange step); the timed region is bracketed by barriers and
the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import gc
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



def repeat_for(fn, min_s):
    """Run fn until at least min_s seconds have passed (once at least);
    returns (mean seconds per call, calls)."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        t = time.perf_counter() - t0
        if t >= min_s:
            return t / n, n


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
    cpu_baseline().  A workload whose steps differ (a walk of `cycle`
    steps: lengths that grow, INT8 blocks that age out) keeps the index of
    its next step in `idx` and accounts bytes per step index."""
    kernel = "phs_split_decode_kernel"
    l2 = "inputs larger than L2 (K/V read per step >> 129 MB)"
    e2e_pipelined = True
    graphable = True
    cycle = 1
    idx = 0
    us_per_step = False

    def step_bytes(self, i):
        return self.bytes_per_step

    def step_tokens(self, i):
        return self.tokens_per_step

    def step_kernel_bytes(self, i):
        return self.kernel_bytes

    def advance(self):
        i = self.idx
        self.idx = (self.idx + 1) % self.cycle
        return i

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
            if getattr(self, "e2e_graph", False):
                # the step as the timed loop replays it: one CUDA graph
                # holding the host-to-device copy, the API call and the
                # device-to-host copy (pinned host buffers, every step)
                if getattr(self, "_e2e_g", None) is None:
                    ins, outs = self.e2e_io(0)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for h, d in ins:
                            d.copy_(h, non_blocking=True)
                        self.e2e_compute(0)
                        for src, h in outs:
                            h.copy_(src, non_blocking=True)
                    self._e2e_g = g
                for _ in range(steps):
                    self._e2e_g.replay()
                return
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
    """Paged Full-attention decode, batch 64 (one step = append + decode,
    the append fused into the split launch)."""

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
        self.launches_per_step = 2  # split (with the append) + merge
        self.extra = {"batch": B, "tokens_per_split": self.tps}
        # the step's inputs in one staged buffer: one host->device copy per step
        self.inp = Arena(device, [self.q, self.kn, self.vn, self.bt, self.sl])
        self.q, self.kn, self.vn, self.bt, self.sl = self.inp.views
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = nbytes(self.h_out)

    def step(self, ev=None):
        phs = self.phs
        self.advance()
        if ev is not None:
            ev[0].record()
        # the append fused into the split launch
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                         self.ws, self.out, tokens_per_split=self.tps,
                                         k_new=self.kn, v_new=self.vn)
        if ev is not None:
            ev[1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, self.sl, self.max_seq, self.ws,
                              tokens_per_split=self.tps)

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.out, self.h_out)]

    def e2e_compute(self, k):
        self.phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl, self.max_seq,
                                        out=self.out, tokens_per_split=self.tps,
                                        workspace=self.ws, k_new=self.kn, v_new=self.vn)

    def cpu_baseline(self, budget_s=2.0, min_s=8.0):
        """The oracle as it stands on a sample of requests of this step,
        repeated for at least min_s seconds."""
        import oracle
        w = self.w
        t1, _, _ = self._oracle_time([0])
        rows = rows_for_budget(w.n_after, range(w.B), t1 / float(w.n_after[0]), budget_s)
        t, toks, reps = self._oracle_time(rows, min_s)
        kv_bytes = toks * w.Hkv * w.D * 2 * 2
        return {"value": kv_bytes / t / 1e9, "unit": "GB/s", "tokens_per_s": toks / t,
                "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests of one decode step "
                          f"({toks} tokens, all {w.Hq} query heads), fp64 oracle, "
                          f"{t:.3f} s per call, mean of {reps} calls"}

    def _oracle_time(self, rows, min_s=0.0):
        import oracle
        w = self.w
        hk, bt = host_pages(self.k, w.block_table, rows, w.n_after)
        hv, _ = host_pages(self.v, w.block_table, rows, w.n_after)
        qh = synth.bits(self.q)[rows]
        sl = w.n_after[rows]
        t, reps = repeat_for(lambda: oracle.decode_full_paged(qh, hk, hv, bt, sl,
                                                              w.softmax_scale), min_s)
        return t, int(sl.sum()), reps


class TinyHybridWorkload(Workload):
    """Batch 2, 4 q / 2 KV heads, D 64: one Full (paged) + one SWA (ring)
    layer, append + attend through the hybrid-stack call.  Latency-bound:
    replayed as a CUDA graph, the whole step timed."""

    l2 = "latency-bound case: ~0.2 MB per step, resident in L2"
    e2e_pipelined = False  # 13 us steps: staging costs more than it hides
    us_per_step = True

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
        self.kernel_bytes = self.bytes_per_step
        self.kernel = ("the whole step (" + ("one launch: Full splits + SWA units, append fused"
                                             if fused else "2 appends, SWA, split") + ")")
        # fused: one launch for the whole step (every request in one split,
        # so no merge, and the Full and SWA work in one wave); else 2 appends,
        # SWA decode, split
        self.launches_per_step = 1 if fused else 4
        self.extra = {"batch": B, "layers": "1 Full + 1 SWA(W=128)",
                      "append_fused_into_attention": fused}
        self.h2d_bytes = self.inp.nbytes
        self.d2h_bytes = self.outp.nbytes

    def step(self, ev=None):
        self.advance()
        if ev is not None:
            ev[0].record()
        if self.fused:
            self.phs.attn_decode_hybrid_stack_fused(self.layers, self.w.Hq, self.sl, self.max_seq,
                                                    block_table=self.bt, ring_pos=self.rp,
                                                    workspace=self.ws)
        else:
            self.phs.attn_decode_hybrid_stack(self.layers, self.w.Hq, self.sl, self.max_seq,
                                              block_table=self.bt, ring_pos=self.rp,
                                              workspace=self.ws)
        if ev is not None:
            ev[1].record()

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
        def one():
            oracle.append_paged(hk, hv, kn, vn, w.block_table, w.n_after)
            oracle.append_ring(hkr, hvr, kn, vn, None, w.ring_pos)
            oracle.decode_full_paged(qf, hk, hv, w.block_table, w.n_after, w.softmax_scale)
            oracle.decode_swa_ring(qs, hkr, hvr, None, w.ring_pos, w.n_after, w.softmax_scale)
        t, reps = repeat_for(one, 5.0)
        return {"value": self.bytes_per_step / t / 1e9, "unit": "GB/s",
                "us_per_step": t * 1e6, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"the whole step (2 appends + 2 decodes), mean of {reps} repetitions"}


class HybridStackWorkload(Workload):
    """70 layers (Full iff layer % 7 == 6: 10 Full, 60 SWA W=128), batch 256,
    32 q / 8 KV heads, D 128, lengths log-uniform in [4K, 128K]; one step =
    append into every layer + attend every layer, one hybrid-stack call.
    Ten distinct 44 GB Full pools do not fit one GPU: `distinct` pools are
    allocated and the Full layers use them round-robin (each layer still
    streams its whole pool, far above L2, so no layer reads another's data
    from cache)."""

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
        self.nfull, self.nswa = nfull, nswa
        # the step is the two launches of the fused call (the Full layers'
        # split launch and the SWA launch that also runs their merges), timed
        # together by events around the call; separately timed parts are
        # reported as a breakdown
        self.kernel_bytes = self.bytes_per_step
        if not nfull:
            self.kernel = "phs_swa_decode_kernel"
        elif fused:
            self.kernel = ("phs_stack_full_kernel + phs_swa_decode_kernel (the fused step's two "
                           "launches: all Full layers, then all SWA layers and the Full merges)")
        else:
            self.kernel = "the whole unfused step (appends, SWA launch, split + merge per layer)"
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

    def _call(self, layers, **kw):
        if self.fused:
            self.phs.attn_decode_hybrid_stack_fused(layers, self.w.Hq, self.sl, self.max_seq,
                                                    block_table=self.bt, ring_pos=self.rp,
                                                    workspace=self.ws, **kw)
        else:
            self.phs.attn_decode_hybrid_stack(layers, self.w.Hq, self.sl, self.max_seq,
                                              block_table=self.bt, ring_pos=self.rp,
                                              workspace=self.ws, **kw)

    def step(self, ev=None):
        self.advance()
        if ev is not None:
            ev[0].record()
        self._call(self.layers)
        if ev is not None:
            ev[1].record()

    def e2e_io(self, k):
        return [(self.inp.host, self.inp.dev)], [(self.outp.dev, self.outp.host)]

    def e2e_compute(self, k):
        self._call(self.layers)

    def breakdown(self, reps=3):
        """The step's two parts timed in loops of their own (after the timed
        region): the Full layers alone (their split launch, append fused, and
        a merge launch) and the SWA layers alone (one launch, no append)."""
        out = {}
        peak = peaks()[0]

        def timed(fn):
            fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / 1e3 / reps

        full = [L for L in self.layers if L.paged is not None]
        swa = [self.phs.Layer(q=L.q, out=L.out, ring=L.ring) for L in self.layers
               if L.ring is not None]
        if full and self.fused:
            t = timed(lambda: self._call(full))
            b = self.nfull * self.full_layer_bytes
            out["phs_stack_full_kernel + merge (10 Full layers)"] = {
                "bytes": b, "ms": round(t * 1e3, 4), "achieved_gbs": round(b / t / 1e9, 1),
                "frac": round(b / t / 1e9 / peak, 4)}
        if swa:
            t = timed(lambda: self.phs.attn_decode_hybrid_stack(
                swa, self.w.Hq, self.sl, self.max_seq, ring_pos=self.rp, do_append=False))
            out["phs_swa_decode_kernel (60 SWA layers)"] = {
                "bytes": self.swa_bytes, "ms": round(t * 1e3, 4),
                "achieved_gbs": round(self.swa_bytes / t / 1e9, 1),
                "frac": round(self.swa_bytes / t / 1e9 / peak, 4)}
        return out

    def cpu_baseline(self, pass_s=1.5, min_s=10.0):
        """The oracle on a sample of the step: requests of one Full layer and
        the same requests in six SWA layers (the stack's 1 : 6 mix), chosen
        so that one pass takes about pass_s seconds, repeated for at least
        min_s seconds."""
        import oracle
        w = self.w
        full = [L for L in self.layers if L.paged is not None]
        swa = [L for L in self.layers if L.ring is not None][:6]
        order = [int(b) for b in np.random.default_rng(11).permutation(w.B)]

        def gather(rows):
            x = {"sl": w.n_after[rows], "rp": w.ring_pos[rows], "swa": []}
            if full:
                L = full[0]
                x["hk"], x["bt"] = host_pages(L.paged.k, w.block_table, rows, w.n_after)
                x["hv"], _ = host_pages(L.paged.v, w.block_table, rows, w.n_after)
                x["qf"] = synth.bits(L.q)[rows]
            for L in swa:
                x["swa"].append((synth.bits(L.ring.k[rows]), synth.bits(L.ring.v[rows]),
                                 synth.bits(L.q)[rows]))
            return x

        def run(x):
            if full:
                oracle.decode_full_paged(x["qf"], x["hk"], x["hv"], x["bt"], x["sl"],
                                         w.softmax_scale)
            for kr, vr, qh in x["swa"]:
                oracle.decode_swa_ring(qh, kr, vr, None, x["rp"], x["sl"], w.softmax_scale)

        def tokens(rows):
            fb = int(w.n_after[rows].sum()) if full else 0
            return fb, int(np.minimum(w.n_after[rows], w.W).sum()) * len(swa)

        t1, _ = repeat_for(lambda x=gather(order[:1]): run(x), 0.0)
        per_tok = t1 / max(1, sum(tokens(order[:1])))
        rows, acc = [], 0.0
        for b in order:
            e = per_tok * sum(tokens([b]))
            if rows and acc + e > pass_s:
                break
            rows.append(b)
            acc += e
        x = gather(rows)
        t, reps = repeat_for(lambda: run(x), min_s)
        fb, sb = tokens(rows)
        toks = fb + sb
        return {"value": toks * w.Hkv * w.D * 4 / t / 1e9, "unit": "GB/s",
                "tokens_per_s": toks / t, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests in {1 if full else 0} Full and "
                          f"{len(swa)} SWA layers ({fb} + {sb} attended tokens), fp64 oracle, "
                          f"{t:.2f} s per pass, mean of {reps} passes"}


class Int8Workload(Workload):
    """Batch 32, 65,536 cached tokens: tokens [0, qlen) as INT8 (one fp32
    absmax/127 scale per 32 tokens per KV head, quantised on the GPU at set
    up), the rest bf16; K/V N(0,1) with 1% N(0, 8^2) outliers.  One step =
    (when a tail reaches 1056 tokens) the quantisation of its oldest bf16
    block + split-KV decode with the append into the bf16 tail fused in +
    merge.  The
    steps walk 64 decode positions (lengths 65,537 .. 65,600, each request's
    INT8 length growing by 32 at steps 31 and 63), then start over."""

    cycle = 64
    hot = 1024
    graphable = False  # each step decodes other lengths

    def __init__(self, device, seed=4, batch=32, tokens_per_split=0):
        import paged_hybrid_sliding_gb300 as phs
        self.phs = phs
        self.w = w = synth.int8_block32(seed=seed, B=batch, steps=self.cycle)
        B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
        self.name = f"int8_block32_b{B}_n65536_hot1024_hq32_hkv8_d128"
        g = seed * 100
        self.k = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 1, device=device,
                                   outlier_p=0.01)
        self.v = synth.normal_bf16((w.num_pages, Hkv, 16, D), g + 2, device=device,
                                   outlier_p=0.01)
        self.pool = phs.PagedPool(self.k, self.v)
        self.qlen0 = w.extra["qlen"]
        self.qt = torch.from_numpy(w.extra["qtable"]).to(device)
        self.i8 = phs.Int8Pool.empty(w.extra["num_qpages"], Hkv, D, device=device)
        self.bt = torch.from_numpy(w.block_table).to(device)
        nqb = (self.qlen0 // 32).astype(np.int32)
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
        self.group_bytes = Hkv * 2 * (32 * D * 2 + 32 * D + 4)
        qbytes = int(nqb.sum()) * self.group_bytes
        self.quant_setup = {"kernel": "phs_quant_kernel", "ms": round(q_s * 1e3, 3),
                            "GB/s": round(qbytes / q_s / 1e9, 1), "bytes": qbytes}
        self.q = synth.normal_bf16((B, Hq, D), g + 3, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), g + 4, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), g + 5, device=device)
        # the walk: lengths after each step's append, the INT8 length each
        # step decodes with, and the blocks that age out at that step
        n0 = w.n_after.astype(np.int64)
        self.n_walk = [(n0 + k).astype(np.int32) for k in range(self.cycle)]
        self.q_walk = [(((n - self.hot) // 32) * 32).astype(np.int32) for n in self.n_walk]
        assert np.array_equal(self.q_walk[0], self.qlen0)
        self.sls = [torch.from_numpy(n).to(device) for n in self.n_walk]
        self.qls = [torch.from_numpy(q).to(device) for q in self.q_walk]
        self.ages = {}
        for k in range(1, self.cycle):
            grown = (self.q_walk[k] > self.q_walk[k - 1]).astype(np.int32)
            if grown.any():
                first = (self.q_walk[k - 1] // 32).astype(np.int32)
                self.ages[k] = (torch.from_numpy(first).to(device),
                                torch.from_numpy(grown).to(device), int(grown.sum()))
        self.max_seq = int(self.n_walk[-1].max())
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq, tokens_per_split)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps,
                                                         has_int8=True),
                              dtype=torch.uint8, device=device)
        self.tokens_per_step = int(self.n_walk[0].sum())
        self.kernel_bytes = self.step_kernel_bytes(0)
        self.bytes_per_step = self.step_bytes(0)
        self.launches_per_step = 2  # split (with the append) + merge; + one quantiser launch at steps 31 and 63
        i8_tok = int(self.qlen0.sum())
        bf_tok = int((w.n_after - self.qlen0).sum())
        self.extra = {"batch": B, "int8_tokens_step0": i8_tok, "bf16_tokens_step0": bf_tok,
                      "walk": f"{self.cycle} steps, lengths {int(n0.min())}..{self.max_seq}; "
                              f"one 32-token block per request quantised at steps "
                              f"{sorted(self.ages)} of the walk",
                      "tokens_per_split": self.tps, "quantiser_setup": self.quant_setup}
        self.inp = Arena(device, [self.q, self.kn, self.vn])
        self.q, self.kn, self.vn = self.inp.views
        self.h_sls = [pinned(s) for s in self.sls]
        self.h_qls = [pinned(s) for s in self.qls]
        self.sl_in = torch.empty_like(self.sls[0])
        self.ql_in = torch.empty_like(self.qls[0])
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d_bytes = self.inp.nbytes + nbytes(self.h_sls[0]) + nbytes(self.h_qls[0])
        self.d2h_bytes = nbytes(self.h_out)

    def step_tokens(self, i):
        return int(self.n_walk[i % self.cycle].sum())

    def step_kernel_bytes(self, i):
        w = self.w
        n, ql = self.n_walk[i % self.cycle].astype(np.int64), self.q_walk[i % self.cycle]
        i8_tok, bf_tok = int(ql.sum()), int((n - ql).sum())
        codes = i8_tok * w.Hkv * w.D * 2
        scales = i8_tok // 32 * w.Hkv * 4 * 2
        tail = bf_tok * w.Hkv * w.D * 2 * 2
        tables = int(synth.pages_needed(n - ql).sum()) * 4 + i8_tok // 32 * 4
        return codes + scales + tail + w.B * w.Hq * w.D * 2 + tables

    def step_bytes(self, i):
        w = self.w
        k = i % self.cycle
        aged = self.ages[k][2] if k in self.ages else 0
        return (self.step_kernel_bytes(i) + w.B * w.Hq * w.D * 2 + 2 * w.B * w.Hkv * w.D * 2 * 2
                + aged * self.group_bytes)

    def _age(self, k):
        if k in self.ages:
            first, num, _ = self.ages[k]
            self.phs.kv_quant_int8_block32(self.pool, self.bt, self.i8, self.qt, first, num, 1)

    def step(self, ev=None):
        k = self.advance()
        phs = self.phs
        sl, ql = self.sls[k], self.qls[k]
        self._age(k)  # reads the oldest bf16 block, far behind the new token
        if ev is not None:
            ev[0].record()
        # the append fused into the split launch (the new token is in the bf16 tail)
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, sl, self.max_seq,
                                         self.ws, self.out, int8=self.i8, qtable=self.qt,
                                         qlens=ql, tokens_per_split=self.tps, k_new=self.kn,
                                         v_new=self.vn)
        if ev is not None:
            ev[1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, sl, self.max_seq, self.ws, qlens=ql,
                              has_int8=True, tokens_per_split=self.tps)

    def e2e_io(self, k):
        c = k % self.cycle
        return ([(self.inp.host, self.inp.dev), (self.h_sls[c], self.sl_in),
                 (self.h_qls[c], self.ql_in)], [(self.out, self.h_out)])

    def e2e_compute(self, k):
        self._age(k % self.cycle)
        self.phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl_in, self.max_seq,
                                        int8=self.i8, qtable=self.qt, qlens=self.ql_in,
                                        tokens_per_split=self.tps, out=self.out,
                                        workspace=self.ws, k_new=self.kn, v_new=self.vn)

    def cpu_baseline(self, nrows=8, min_s=8.0):
        """The oracle on the first nrows requests of step 0 (INT8 codes and
        scales from the GPU quantiser, which the parity tests pin to the
        oracle's), repeated for at least min_s seconds."""
        import oracle
        w = self.w
        rows = list(range(min(nrows, w.B)))
        n = self.n_walk[0]
        hk, bt = host_pages(self.k, w.block_table, rows, n)
        hv, _ = host_pages(self.v, w.block_table, rows, n)
        nq = [int(self.qlen0[b] // 32) for b in rows]
        ids = torch.cat([self.qt[b, :nq[i]].long() for i, b in enumerate(rows)])
        qt = np.full((len(rows), max(nq)), -1, np.int32)
        o = 0
        for i, k in enumerate(nq):
            qt[i, :k] = np.arange(o, o + k)
            o += k
        gk, gv = self.i8.codes(ids)
        i8 = dict(k_codes=gk.cpu().numpy(), v_codes=gv.cpu().numpy(),
                  k_scale=self.i8.k_scale.index_select(0, ids).cpu().numpy(),
                  v_scale=self.i8.v_scale.index_select(0, ids).cpu().numpy(),
                  qtable=qt, qlens=self.qlen0[rows])
        qh = synth.bits(self.q)[rows]
        t, reps = repeat_for(lambda: oracle.decode_full_paged(qh, hk, hv, bt, n[rows],
                                                              w.softmax_scale, int8=i8), min_s)
        b = self.step_kernel_bytes(0) / w.B * len(rows)
        toks = int(n[rows].sum())
        return {"value": b / t / 1e9, "unit": "GB/s", "tokens_per_s": toks / t,
                "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests ({toks} tokens, INT8 + bf16 tail),"
                          f" fp64 oracle, {t:.3f} s per call, mean of {reps} calls"}


class SharedPrefixWorkload(Workload):
    """64 requests sharing one 250,000-token prefix (15,625 pages, refcount
    64) + a unique 512-token suffix each; 128 decode steps with append.  One
    bench step = one decode step; the steps walk the 128 positions."""

    l2 = "logical K/V bytes per step 65.7 GB >> L2; the shared prefix is reused through L2"
    graphable = False  # each step decodes other lengths

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
        self.cycle = w.extra["steps"]
        self.sls = [torch.from_numpy((w.n_pre + 1 + k).astype(np.int32)).to(device)
                    for k in range(self.cycle)]
        self.q = synth.normal_bf16((B, Hq, D), g + 3, device=device)
        self.kn = synth.normal_bf16((B, Hkv, D), g + 4, device=device)
        self.vn = synth.normal_bf16((B, Hkv, D), g + 5, device=device)
        self.max_seq = int(w.n_pre.max()) + self.cycle
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
        self.tps = phs.decode_tokens_per_split(B, Hkv, self.max_seq)
        self.ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, self.max_seq, self.tps),
                              dtype=torch.uint8, device=device)
        # tensor-core pass over the shared prefix (whole 64-token tiles)
        self.prefix_kernel = prefix_kernel
        self.npref = w.extra["prefix_pages"]
        self.shared_len = (self.npref * 16 // 64) * 64
        if prefix_kernel:
            self.ws = torch.empty(phs.shared_prefix_workspace_bytes(B, Hq, Hkv, D, self.max_seq,
                                                                    self.shared_len),
                                  dtype=torch.uint8, device=device)
            self.kernel = "phs_attn_decode_shared_prefix (prefix tcgen05 + suffix split + merge)"
            self.l2 = "prefix read once per KV head for all 64 requests (tensor-core pass)"
        self.tok_bytes = Hkv * D * 2 * 2
        self.tokens_per_step = self.step_tokens(0)
        self.bytes_per_step = self.step_bytes(0)
        self.kernel_bytes = self.step_kernel_bytes(0)
        self.launches_per_step = 3  # prefix: tensor pass, own-token split (+ append), merge
        # tensor work of the prefix pass: QK and PV over B*G rows x D per token
        self.prefix_flops = 4 * B * Hq * D * self.shared_len
        self.extra = {"batch": B, "logical_bytes_step0": self.bytes_per_step,
                      "unique_kv_bytes_step0": self.step_unique_bytes(0),
                      "walk": f"{self.cycle} decode steps (lengths {int(w.n_pre[0]) + 1}.."
                              f"{self.max_seq})",
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

    def step_tokens(self, i):
        return int((self.w.n_pre + 1 + i % self.cycle).sum())

    def step_unique_bytes(self, i):
        w = self.w
        own = int((w.n_pre + 1 + i % self.cycle - self.npref * 16).sum())
        return (self.npref * 16 + own) * self.tok_bytes + w.B * w.Hq * w.D * 2

    def step_kernel_bytes(self, i):
        w = self.w
        return self.step_tokens(i) * self.tok_bytes + w.B * w.Hq * w.D * 2

    def step_bytes(self, i):
        w = self.w
        return (self.step_tokens(i) * self.tok_bytes + 2 * w.B * w.Hq * w.D * 2
                + 2 * w.B * w.Hkv * w.D * 2 * 2)

    def step(self, ev=None):
        phs = self.phs
        sl = self.sls[self.advance()]
        if self.prefix_kernel:  # one call: the append is fused into the own-token split
            if ev is not None:
                ev[0].record()
            phs.attn_decode_shared_prefix(self.q, self.pool, self.bt, sl, self.max_seq,
                                          self.shared_len, out=self.out, workspace=self.ws,
                                          k_new=self.kn, v_new=self.vn, page_refcount=self.rc)
            if ev is not None:
                ev[1].record()
            return
        phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, sl, page_refcount=self.rc)
        if ev is not None:
            ev[0].record()
        phs.attn_decode_full_paged_split(self.q, self.pool, self.bt, sl, self.max_seq, self.ws,
                                         self.out, tokens_per_split=self.tps)
        if ev is not None:
            ev[1].record()
        phs.attn_merge_splits(self.out, self.w.Hkv, sl, self.max_seq, self.ws,
                              tokens_per_split=self.tps)

    def e2e_io(self, k):
        return ([(self.inp.host, self.inp.dev), (self.h_sls[k % self.cycle], self.sl_in)],
                [(self.out, self.h_out)])

    def e2e_compute(self, k):
        if self.prefix_kernel:
            self.phs.attn_decode_shared_prefix(self.q, self.pool, self.bt, self.sl_in,
                                               self.max_seq, self.shared_len, out=self.out,
                                               workspace=self.ws, k_new=self.kn, v_new=self.vn,
                                               page_refcount=self.rc)
        else:
            self.phs.kv_append_paged(self.pool, self.kn, self.vn, self.bt, self.sl_in,
                                     page_refcount=self.rc)
            self.phs.attn_decode_full_paged(self.q, self.pool, self.bt, self.sl_in, self.max_seq,
                                            out=self.out, tokens_per_split=self.tps,
                                            workspace=self.ws)

    def cpu_baseline(self, nrows=4, min_s=8.0):
        """The oracle on nrows requests of step 0 (the oracle reads every
        request's prefix from its own gathered copy), repeated for at least
        min_s seconds."""
        import oracle
        w = self.w
        rows = list(range(min(nrows, w.B)))
        n = w.n_pre + 1
        hk, bt = host_pages(self.k, w.block_table, rows, n)
        hv, _ = host_pages(self.v, w.block_table, rows, n)
        qh = synth.bits(self.q)[rows]
        t, reps = repeat_for(lambda: oracle.decode_full_paged(qh, hk, hv, bt, n[rows],
                                                              w.softmax_scale), min_s)
        toks = int(n[rows].sum())
        return {"value": toks * w.Hkv * w.D * 4 / t / 1e9, "unit": "GB/s",
                "tokens_per_s": toks / t, "cores": oracle.max_threads(), "kind": "oracle",
                "sample": f"{len(rows)} of {w.B} requests of one step ({toks} tokens), fp64 "
                          f"oracle, {t:.3f} s per call, mean of {reps} calls"}


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


def time_read(device, nbytes=4 << 30, reps=10):
    """Read-side yardstick: the streaming read-checksum kernel over a buffer
    larger than L2 (GB/s of bytes read)."""
    import paged_hybrid_sliding_gb300 as phs
    a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    a.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    for _ in range(3):
        phs.read_checksum(a, sink)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        s.record()
        phs.read_checksum(a, sink)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del a
    return nbytes / best / 1e9


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


def measure(wl, steps, warmup, world, device, use_graph, copy_gbs, with_cpu, read_gbs=None):
    """Warm-up, then exactly `steps` steps timed with CUDA events between
    barriers (max over ranks); the dominant kernel timed by events around
    its launch on its stream on every `stride`-th step; then the same number
    of steps end to end through the public API from pinned host buffers."""
    warmup = max(3, warmup)
    for _ in range(warmup):
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
    # an event between two launches ends the programmatic overlap of the
    # second with the first, so the events go on every `stride`-th step only
    stride = max(1, steps // 200)
    evs = []
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    idx0 = wl.idx
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device.index or 0) as clk:
        start.record()
        for i in range(steps):
            pair = None
            if i % stride == 0:
                pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                evs.append((pair, (idx0 + i) % wl.cycle))
            if graph is not None:
                if pair is not None:
                    pair[0].record()
                graph.replay()
                if pair is not None:
                    pair[1].record()
            else:
                wl.step(pair)
        stop.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = slowest_rank_time(start.elapsed_time(stop) / 1e3, world, device)
    step_ids = [(idx0 + i) % wl.cycle for i in range(steps)] if graph is None else [0] * steps
    total_bytes = sum(wl.step_bytes(i) for i in step_ids)
    total_tokens = sum(wl.step_tokens(i) for i in step_ids)
    k_time = sum(a.elapsed_time(b) for (a, b), _ in evs) / 1e3
    k_bytes = sum(wl.step_kernel_bytes(i) for _, i in evs)
    breakdown = wl.breakdown() if hasattr(wl, "breakdown") else None

    # end to end through the public API with host buffers, the same number
    # of steps as the timed loop (copies overlapped with compute, as a
    # serving loop would; a graph-replayed step replays its copies with it)
    wl.e2e_graph = graph is not None and wl.graphable and not wl.e2e_pipelined
    wl.e2e_run(3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    wl.e2e_run(steps)
    torch.cuda.synchronize()
    t_e2e = slowest_rank_time(time.perf_counter() - t0, world, device)
    e2e_bytes = sum(wl.step_bytes(k % wl.cycle) for k in range(steps))

    peak, peak_kind = peaks()
    ms = t / steps * 1e3
    value = total_bytes * world / t / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "kv_tokens_per_step": round(total_tokens / steps),
                   "bytes_per_step": round(total_bytes / steps), "l2": wl.l2,
                   "parallelism": "replicas" if world > 1 else "single", **wl.extra,
                   "cuda_graph": graph is not None},
        "tokens_per_s": round(total_tokens * world / t, 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "copy_gbs": round(copy_gbs, 1),
        "pct_of_copy": round(100 * value / world / copy_gbs, 2),
        **({"read_gbs": round(read_gbs, 1),
            "pct_of_read": round(100 * value / world / read_gbs, 2)} if read_gbs else {}),
        "e2e": {"value": round(e2e_bytes * world / t_e2e / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": wl.h2d_bytes,
                "d2h_bytes_per_step": wl.d2h_bytes, "steps": steps,
                "copies": ("every step's inputs up and outputs down through pinned host "
                           "buffers, overlapped with the previous/next step's compute (two "
                           "copy streams, double-buffered device staging)"
                           if wl.e2e_pipelined else
                           "every step's inputs up and outputs down through pinned host "
                           "buffers, in line with the step" + (
                               " (the copies and the API call replayed as one CUDA graph)"
                               if getattr(wl, "e2e_graph", False) else ""))},
        "gpu_launches": wl.launches_per_step * steps + sum(
            1 for i in step_ids if i in getattr(wl, "ages", {})),
        "clocks": clk.summary(),
    }
    if wl.us_per_step:
        line["us_per_step"] = round(ms * 1e3, 2)
    if evs and k_time > 0:
        achieved = k_bytes / k_time / 1e9
        line["roofline"] = {
            "bound": "hbm", "kernel": wl.kernel, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "bytes_per_launch": round(k_bytes / len(evs)),
            "avg_launch_ms": round(k_time / len(evs) * 1e3, 4),
            "traffic": recorded_traffic(wl.kernel, wl.name),
            "timed_launches": (f"{len(evs)} launches inside the timed loop (CUDA events around "
                               f"the launch, on its stream, in 1 of every {stride} steps)")}
        if wl.us_per_step:
            line["roofline"]["note"] = ("latency-bound: the step moves ~0.2 MB, so its launch "
                                        "latency, not HBM bandwidth, sets its time")
        if isinstance(wl, SharedPrefixWorkload):
            if wl.prefix_kernel:
                # the decode call reads each prefix page once: its HBM bound is
                # the unique bytes; its tensor work is the prefix contraction
                ub = sum(wl.step_unique_bytes(i) for _, i in evs)
                uniq = ub / k_time / 1e9
                tflops = wl.prefix_flops * len(evs) / k_time / 1e12
                line["roofline"].update({
                    "achieved": round(uniq, 1), "frac": round(uniq / peak, 4),
                    "bytes_per_launch": round(ub / len(evs)),
                    "bytes_are": "unique K/V bytes (prefix read once per KV head)",
                    "logical_gbs": round(achieved, 1),
                    "tensor_tflops": round(tflops, 1),
                    "tensor_frac_of_bf16_peak": round(tflops / peak_tflops()[0], 4)})
            else:
                ub = sum(wl.step_unique_bytes(i) for _, i in evs)
                line["roofline"]["bytes_are"] = "logical (prefix pages reused through L2)"
                line["roofline"]["unique_kv_gbs"] = round(ub / k_time / 1e9, 1)
    if breakdown:
        line["breakdown"] = breakdown
    if with_cpu:
        line["cpu_baseline"] = wl.cpu_baseline()
    return line


SUITE = (3, 1, 2, 4, 5)          # headline first (the largest workload)
# at least ~0.25 s of timed loop per workload, so that the clock samples
# (every 100 ms) see it; walks in whole cycles (64 INT8 steps, 128 prefix steps)
SUITE_MIN_STEPS = {1: 20000, 2: 500, 3: 0, 4: 512, 5: 1280}


def run_gpu(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import paged_hybrid_sliding_gb300 as phs
    phs.lib()
    copy_gbs = time_copy(device)
    read_gbs = time_read(device)
    run_list = [args.config] if args.config else list(SUITE)
    lines = {}
    for c in run_list:
        wl = make_workload(c, device, args)
        use_graph = args.graph if args.graph is not None else c == 1
        if use_graph and not wl.graphable:
            raise SystemExit("--graph: this workload's steps differ")
        steps = args.steps if (args.config or c == SUITE[0]) else max(args.steps,
                                                                      SUITE_MIN_STEPS[c])
        lines[c] = measure(wl, steps, args.warmup, world, device, use_graph, copy_gbs,
                           with_cpu=rank == 0 and not args.no_cpu_baseline, read_gbs=read_gbs)
        del wl
        gc.collect()
        torch.cuda.empty_cache()
    head = lines[run_list[0]]
    if len(run_list) > 1:
        head["configs"] = {str(c): lines[c] for c in run_list[1:]}
        head["suite"] = ("the headline is the 70-layer hybrid stack (the largest workload); "
                         "the other workloads were measured in the same run, each line with "
                         "its own steps, roofline, e2e and CPU-oracle baseline")
    return head


def run_reference(args, rank, budget_s=40.0):
    """The CPU oracle as the reference arm, on the headline workload (the
    70-layer hybrid stack): each step is the oracle over a bounded sample
    of the step -- a few requests, appended and attended in one Full layer
    and in six SWA layers (the stack's 1 : 6 mix) -- sized so that all
    warm-up and timed steps together take about budget_s seconds.  Inputs
    are drawn on the host; nothing runs on the GPU."""
    if rank != 0:
        return None
    import oracle
    if args.config not in (None, 3):
        raise SystemExit("--impl reference times the hybrid-stack workload (config 3)")
    w = synth.hybrid_stack()
    name = HYBRID_STACK_NAME
    W, Hkv, D, Hq = w.W, w.Hkv, w.D, w.Hq
    order = [int(b) for b in np.random.default_rng(11).permutation(w.B)]
    n_swa = 6

    def inputs(rows):
        pages = [int(synth.pages_needed(w.n_after[b])) for b in rows]
        npg = sum(pages)
        kp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), 201))
        vp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), 202))
        bt = np.full((len(rows), max(pages)), -1, np.int32)
        o = 0
        for i, p in enumerate(pages):
            bt[i, :p] = np.arange(o, o + p)
            o += p
        nr = len(rows)
        rings = [(synth.bits(synth.normal_bf16((nr, Hkv, W, D), 300 + 2 * l)),
                  synth.bits(synth.normal_bf16((nr, Hkv, W, D), 301 + 2 * l)))
                 for l in range(n_swa)]
        qs = [synth.bits(synth.normal_bf16((nr, Hq, D), 400 + l)) for l in range(1 + n_swa)]
        kn = synth.bits(synth.normal_bf16((nr, Hkv, D), 500))
        vn = synth.bits(synth.normal_bf16((nr, Hkv, D), 501))
        return kp, vp, bt, rings, qs, kn, vn, w.n_after[rows], w.ring_pos[rows]

    def step(x):
        kp, vp, bt, rings, qs, kn, vn, sl, rp = x
        oracle.append_paged(kp, vp, kn, vn, bt, sl)
        oracle.decode_full_paged(qs[0], kp, vp, bt, sl, w.softmax_scale)
        for l, (kr, vr) in enumerate(rings):
            oracle.append_ring(kr, vr, kn, vn, None, rp)
            oracle.decode_swa_ring(qs[1 + l], kr, vr, None, rp, sl, w.softmax_scale)

    def tokens(rows):
        sl = w.n_after[rows]
        return int(sl.sum()), int(np.minimum(sl, W).sum()) * n_swa

    x = inputs(order[:1])
    t0 = time.perf_counter()
    step(x)
    f1, s1 = tokens(order[:1])
    per_tok = (time.perf_counter() - t0) / (f1 + s1)
    per_step = budget_s / max(1, args.steps + args.warmup)
    rows, acc = [], 0.0
    for b in order:
        e = per_tok * (float(w.n_after[b]) + n_swa * min(float(w.n_after[b]), W))
        if rows and acc + e > per_step:
            break
        rows.append(b)
        acc += e
    x = inputs(rows)
    ft, st = tokens(rows)
    step_bytes = (ft + st) * Hkv * D * 4
    for _ in range(args.warmup):
        step(x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(x)
    t = time.perf_counter() - t0
    gbs = step_bytes * args.steps / t / 1e9
    sample = (f"{len(rows)} of {w.B} requests of the 70-layer stack step, appended and attended "
              f"in 1 Full and {n_swa} SWA layers ({ft} + {st} attended tokens, all {Hq} query "
              f"heads), fp64 oracle")
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "sample": sample},
            "tokens_per_s": round((ft + st) * args.steps / t, 1),
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.max_threads(), "sample": sample},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


HYBRID_STACK_NAME = "hybrid_stack_70l_10full_60swa_w128_b256_hq32_hkv8_d128_seqlogU[4K,128K]"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
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
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="one workload alone: 1 tiny hybrid, 2 paged Full batch 64, 3 70-layer "
                         "hybrid stack, 4 INT8 block-32, 5 shared 250K prefix (default: all, "
                         "config 3 as the headline)")
    ap.add_argument("--distinct-pools", type=int, default=4,
                    help="config 3: distinct 44 GB Full pools allocated (layers alias them)")
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
