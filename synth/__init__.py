"""Seeded synthetic inputs for paged hybrid sliding-window decode.

This module only draws inputs: sequence lengths, page and ring
assignments and random bf16 values.  It holds none of the attention,
append or quantisation arithmetic, so both the CPU oracle side and the CUDA
side of a test (and the benchmark) can take their inputs from it.

Workload shapes follow the decode cases described for hybrid-SWA serving:
a 10 Full + 60 SWA (W=128) layer stack ("Xiaomi MiMo-V2.5 inference system"
page, section 1), paged KV with refcounted shared prefixes ("Kimi K3 context
caching" page, sections 1 and 4: a 250,000-token shared prefix) and INT8
block-32 warm-zone KV with a bf16 hot window ("Kimi K2.5 architecture deep
dive" page, sections 2.2 and 2.3).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 16          # tokens per Full-pool page
QBLOCK = 32        # tokens per INT8 scale group / INT8 page


# --------------------------------------------------------------------------
# value generators
# --------------------------------------------------------------------------
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal_bf16(shape, seed: int, device="cpu", outlier_p: float = 0.0,
                outlier_sigma: float = 8.0, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """bf16 tensor of N(0,1) values; with probability outlier_p each element
    is replaced by an N(0, outlier_sigma^2) draw.  Drawn in chunks so that
    very large pools do not need a full fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = _gen(seed, device)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if outlier_p > 0.0:
            m = torch.rand(e - s, generator=g, device=device) < outlier_p
            o = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
            x = torch.where(m, o * outlier_sigma, x)
        flat[s:e].copy_(x.to(torch.bfloat16))
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a bf16 tensor (bit pattern, no conversion)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """bf16 tensor from a uint16 bit-pattern array."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


# --------------------------------------------------------------------------
# index generators
# --------------------------------------------------------------------------
def seq_lens_uniform(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)


def seq_lens_loguniform(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """exp(U[ln lo, ln hi]) rounded down, clipped to [lo, hi]."""
    rng = np.random.default_rng(seed)
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=B))
    return np.clip(np.floor(x), lo, hi).astype(np.int32)


def pages_needed(n_tokens, page=PAGE):
    return (np.asarray(n_tokens, dtype=np.int64) + page - 1) // page


def block_tables_from_permutation(pages_per_req, seed: int, num_pages: int | None = None,
                                  width: int | None = None):
    """Each request gets pages_per_req[b] physical page ids taken, without
    replacement, from a seeded random permutation of [0, num_pages).
    Returns (block_table [B, width] int32 padded with -1, num_pages)."""
    ppr = np.asarray(pages_per_req, dtype=np.int64)
    total = int(ppr.sum())
    num_pages = total if num_pages is None else int(num_pages)
    assert num_pages >= total
    width = int(ppr.max()) if width is None else int(width)
    perm = np.random.default_rng(seed).permutation(num_pages).astype(np.int32)
    bt = np.full((len(ppr), max(width, 1)), -1, dtype=np.int32)
    off = 0
    for b, k in enumerate(ppr):
        bt[b, :k] = perm[off:off + k]
        off += k
    return bt, num_pages


def ring_positions(B: int, W: int, seed: int) -> np.ndarray:
    """Slot of the newest token of each request's ring: any slot is a valid
    ring state, so it is drawn uniformly from [0, W)."""
    return np.random.default_rng(seed).integers(0, W, size=B).astype(np.int32)


# --------------------------------------------------------------------------
# workload configurations
# --------------------------------------------------------------------------
@dataclass
class Workload:
    """Index structure of one decode step.  Values are drawn separately
    (``normal_bf16``) on whatever device the caller wants."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    n_pre: np.ndarray                      # context length before this step
    seed: int
    P: int = PAGE
    W: int = 128
    num_pages: int = 0
    block_table: np.ndarray | None = None  # [B, max_pages]
    ring_pos: np.ndarray | None = None     # [B]
    extra: dict = field(default_factory=dict)

    @property
    def n_after(self) -> np.ndarray:
        return (self.n_pre + 1).astype(np.int32)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def tiny_hybrid(seed: int = 1) -> Workload:
    """Batch 2, 4 q / 2 KV heads, head_dim 64, pages of 16, lengths 37 and
    200; pages are a seeded random permutation of a 64-page pool; one SWA
    ring of W = 128 per request."""
    n_pre = np.array([37, 200], dtype=np.int32)
    w = Workload("tiny_hybrid_b2_d64", B=2, Hq=4, Hkv=2, D=64, n_pre=n_pre, seed=seed)
    w.block_table, w.num_pages = block_tables_from_permutation(
        pages_needed(w.n_after), seed + 11, num_pages=64)
    w.ring_pos = ring_positions(2, w.W, seed + 12)
    return w


def paged_full(seed: int = 2, B: int = 64, lo: int = 1024, hi: int = 32768) -> Workload:
    """Batch 64, 32 q / 8 KV heads, head_dim 128, pages of 16, lengths
    uniform in [1K, 32K]; block tables drawn without replacement from a pool
    sized to the total page count."""
    n_pre = seq_lens_uniform(B, lo, hi, seed + 1)
    w = Workload(f"paged_full_b{B}_d128", B=B, Hq=32, Hkv=8, D=128, n_pre=n_pre, seed=seed)
    w.block_table, w.num_pages = block_tables_from_permutation(pages_needed(w.n_after), seed + 2)
    return w


def hybrid_stack(seed: int = 3, B: int = 256, lo: int = 4096, hi: int = 131072,
                 num_layers: int = 70) -> Workload:
    """70 layers, Full iff layer % 7 == 6 (10 Full, 60 SWA W=128), batch 256,
    32 q / 8 KV heads, head_dim 128, lengths log-uniform in [4K, 128K].  All
    Full layers share one block table (one page id per logical page, each
    layer in its own pool); each request owns ring b in every SWA layer."""
    n_pre = seq_lens_loguniform(B, lo, hi, seed + 1)
    w = Workload(f"hybrid_stack_{num_layers}l_b{B}", B=B, Hq=32, Hkv=8, D=128, n_pre=n_pre,
                 seed=seed)
    w.block_table, w.num_pages = block_tables_from_permutation(pages_needed(w.n_after), seed + 2)
    w.ring_pos = ring_positions(B, w.W, seed + 3)
    w.extra["layer_is_full"] = np.array([1 if l % 7 == 6 else 0 for l in range(num_layers)],
                                        dtype=np.int32)
    return w


def int8_block32(seed: int = 4, B: int = 32, n_pre: int = 65536, hot: int = 1024,
                 steps: int = 1) -> Workload:
    """Batch 32, length 65536, 32 q / 8 KV heads, head_dim 128.  Tokens
    [0, qlen) are held as INT8 in 32-token pages, qlen the largest multiple
    of 32 leaving at least `hot` tokens (the new one included) in bf16.
    K/V values: N(0,1) with 1% outliers N(0, 8^2).  The tables have room for
    `steps` decode steps (lengths n_pre + 1 .. n_pre + steps, the INT8
    length following the same rule)."""
    npre = np.full(B, n_pre, dtype=np.int32)
    w = Workload(f"int8_block32_b{B}_n{n_pre}", B=B, Hq=32, Hkv=8, D=128, n_pre=npre, seed=seed)
    n_after = npre + 1
    qlen = ((n_after - hot) // QBLOCK) * QBLOCK
    qlen = np.maximum(qlen, 0).astype(np.int32)
    n_last = npre + max(int(steps), 1)
    # bf16 pages cover the whole logical range at setup (the quantiser reads
    # them); only pages at or past qlen stay referenced by decode.
    w.block_table, w.num_pages = block_tables_from_permutation(pages_needed(n_last), seed + 2)
    nq = ((np.maximum(n_last - hot, 0) // QBLOCK)).astype(np.int64)
    qt, nqp = block_tables_from_permutation(np.maximum(nq, 1), seed + 3)
    w.extra.update(qlen=qlen, qtable=qt, num_qpages=nqp, outlier_p=0.01, outlier_sigma=8.0)
    return w


def shared_prefix(seed: int = 5, B: int = 64, prefix: int = 250_000, suffix: int = 512,
                  steps: int = 128) -> Workload:
    """64 requests sharing one 250,000-token prefix (15,625 pages of 16 with
    refcount 64) plus a unique 512-token suffix each, with room for `steps`
    more decode tokens.  Page ids: one seeded permutation over all pages."""
    assert prefix % PAGE == 0
    n_pre = np.full(B, prefix + suffix, dtype=np.int32)
    w = Workload(f"shared_prefix_{prefix}_b{B}", B=B, Hq=32, Hkv=8, D=128, n_pre=n_pre,
                 seed=seed)
    npref = prefix // PAGE
    nown = (suffix + steps + PAGE - 1) // PAGE
    total = npref + B * nown
    perm = np.random.default_rng(seed + 2).permutation(total).astype(np.int32)
    bt = np.empty((B, npref + nown), dtype=np.int32)
    bt[:, :npref] = perm[:npref][None, :]
    for b in range(B):
        s = npref + b * nown
        bt[b, npref:] = perm[s:s + nown]
    refcount = np.ones(total, dtype=np.int32)
    refcount[perm[:npref]] = B
    w.block_table, w.num_pages = bt, total
    w.extra.update(refcount=refcount, prefix_pages=npref, steps=steps)
    return w


CONFIGS = {
    1: tiny_hybrid,
    2: paged_full,
    3: hybrid_stack,
    4: int8_block32,
    5: shared_prefix,
}
