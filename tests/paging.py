"""Test-side layout helpers: scatter a dense logical K/V sequence into the
paged pool, the SWA ring or INT8 pages, and a dense reference through a
library routine.  Independent of both the oracle and the CUDA library; used
to pin the oracle and to build GPU parity inputs."""
from __future__ import annotations

import numpy as np
import torch


def dense_to_paged(dense, block_table, num_pages, P=16, fill=None, rng=None):
    """dense: list over requests of uint16 [Hkv, n_b, D].  Returns a pool
    uint16 [num_pages, Hkv, P, D] where token t of request b lives at
    (block_table[b][t // P], :, t % P).  Unused slots get random bits (so
    that reading them would show up) unless `fill` is given."""
    Hkv, _, D = dense[0].shape
    if fill is None:
        rng = rng or np.random.default_rng(1234)
        pool = rng.integers(0, 1 << 16, size=(num_pages, Hkv, P, D), dtype=np.uint16)
        # keep garbage finite: clear the exponent's top bit (|x| < 2)
        pool &= np.uint16(0xBFFF)
    else:
        pool = np.full((num_pages, Hkv, P, D), fill, dtype=np.uint16)
    for b, kv in enumerate(dense):
        n = kv.shape[1]
        for t in range(n):
            pool[block_table[b][t // P], :, t % P, :] = kv[:, t, :]
    return pool


def dense_to_ring(dense, ring_pos, W, num_rings=None, ring_ids=None, rng=None):
    """Ring layout [num_rings, Hkv, W, D]: the newest token (index n-1) sits
    at slot ring_pos[b] and token t at (ring_pos[b] - (n-1-t)) mod W, for the
    last min(n, W) tokens.  Other slots hold random finite bits."""
    B = len(dense)
    Hkv, _, D = dense[0].shape
    num_rings = B if num_rings is None else num_rings
    rng = rng or np.random.default_rng(4321)
    ring = rng.integers(0, 1 << 16, size=(num_rings, Hkv, W, D), dtype=np.uint16)
    ring &= np.uint16(0xBFFF)
    for b, kv in enumerate(dense):
        n = kv.shape[1]
        r = b if ring_ids is None else ring_ids[b]
        for t in range(max(0, n - W), n):
            ring[r, :, (ring_pos[b] - (n - 1 - t)) % W, :] = kv[:, t, :]
    return ring


def bf16_bits_to_f64(a):
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def random_bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def sdpa_reference(q_bits, k_dense, v_dense, scale):
    """Library reference: torch scaled_dot_product_attention in float64 on
    the CPU, one query per request, GQA by repeating each KV head over its
    contiguous group of query heads.  q_bits: uint16 [B, Hq, D];
    k_dense/v_dense: lists of float64 arrays [Hkv, n_b, D]."""
    B, Hq, D = q_bits.shape
    q = torch.from_numpy(bf16_bits_to_f64(q_bits))
    out = np.zeros((B, Hq, D))
    for b in range(B):
        k = torch.from_numpy(np.asarray(k_dense[b], dtype=np.float64))
        v = torch.from_numpy(np.asarray(v_dense[b], dtype=np.float64))
        Hkv = k.shape[0]
        G = Hq // Hkv
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b][:, None, :], k, v, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out
