"""Helpers for the GPU parity tests: seeded inputs moved between host bit
patterns and device tensors, sub-pool extraction for sampled parity at full
size, and the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Decode outputs: |gpu - oracle| <= ATOL + RTOL * |oracle|, element by element
# (the stated max-abs 1e-2 / max-rel 2e-2 bar read as one combined bound).
ATOL, RTOL = 1e-2, 2e-2


def assert_close(got, ref, what="", atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    ok = err <= atol + rtol * np.abs(ref)
    if not ok.all():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(
            f"{what}: {int((~ok).sum())}/{ok.size} elements outside tolerance; worst at {idx}: "
            f"got {got[idx]:.6g} ref {ref[idx]:.6g}; max abs err {err.max():.3e}")
    return float(err.max())


def dev(a, device="cuda"):
    """numpy int array -> device int32 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_dev(bits, device="cuda"):
    return synth.from_bits(bits, device)


def out_np(t):
    return t.double().cpu().numpy()


def sub_pool(pool_t, block_table, rows, n_after, page=16):
    """Host copy of just the pages the selected requests reference, and a
    block table remapped onto the compact copy (layout bookkeeping only)."""
    tables = []
    pages = []
    off = 0
    for b in rows:
        k = (int(n_after[b]) + page - 1) // page
        ids = block_table[b, :k]
        pages.append(ids)
        tables.append(np.arange(off, off + k, dtype=np.int32))
        off += k
    width = max(len(t) for t in tables)
    bt = np.full((len(rows), width), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    idx = torch.from_numpy(np.concatenate(pages).astype(np.int64)).to(pool_t.device)
    host = synth.bits(pool_t.index_select(0, idx))
    return host, bt
