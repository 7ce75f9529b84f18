"""GPU parity of the shared-prefix decode (tensor-core pass over the shared
prefix for all requests + split-KV over each request's own tokens + merge)
against the fp64 oracle and against the per-request decode path."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, dev, out_np

pytestmark = pytest.mark.gpu


def _shared_case(B, Hq, Hkv, shared_len, suffixes, seed, D=128):
    """Block tables: the same shared_len/16 prefix pages first, then each
    request's own pages; page ids from one seeded permutation."""
    npref = shared_len // 16
    own = [(s + 15) // 16 for s in suffixes]
    total = npref + sum(own) + 2
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    width = npref + max(max(own), 1)
    bt = np.full((B, width), -1, np.int32)
    o = npref
    for b in range(B):
        bt[b, :npref] = perm[:npref]
        bt[b, npref:npref + own[b]] = perm[o:o + own[b]]
        o += own[b]
    lens = np.array([shared_len + s for s in suffixes], np.int32)
    pool = phs.PagedPool(synth.normal_bf16((total, Hkv, 16, D), seed + 1, device="cuda"),
                         synth.normal_bf16((total, Hkv, 16, D), seed + 2, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), seed + 3, device="cuda")
    return pool, q, bt, lens


def _oracle_rows(pool, q, bt, lens, rows, D=128):
    used = np.unique(bt[rows][bt[rows] >= 0])
    remap = np.full(bt.max() + 1, -1, np.int64)
    remap[used] = np.arange(len(used))
    bt_s = np.where(bt[rows] >= 0, remap[np.maximum(bt[rows], 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    hk, hv = synth.bits(pool.k.index_select(0, idx)), synth.bits(pool.v.index_select(0, idx))
    ref, st = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, lens[rows],
                                       1 / math.sqrt(D))
    assert st == 0
    return ref


@pytest.mark.parametrize("B,Hq,Hkv,shared_len,seed,max_suffix", [
    (2, 32, 8, 64, 1, 700),        # one tile, 8 rows per head
    (8, 32, 8, 1024, 2, 700),      # 16 tiles, 32 rows
    (64, 32, 8, 4096, 3, 700),     # 256 rows: both 128-row tiles full
    (5, 16, 2, 2048, 4, 700),      # G = 8, 40 rows
    (33, 32, 8, 640, 5, 700),      # rows 132: second tile partly used
    (16, 32, 2, 512, 6, 700),      # G = 16, 256 rows
    (6, 32, 8, 256, 7, 5000),      # own tokens over several splits: merged with the prefix
    (64, 8, 8, 1024, 8, 700),      # G = 1: one row per request and KV head, 64 rows
])
def test_shared_prefix_matches_oracle_and_paged_path(B, Hq, Hkv, shared_len, seed, max_suffix):
    rng = np.random.default_rng(seed)
    suffixes = [int(x) for x in rng.integers(0, max_suffix, size=B)]
    suffixes[0] = 0                  # a request with no tokens of its own
    pool, q, bt, lens = _shared_case(B, Hq, Hkv, shared_len, suffixes, seed)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), shared_len,
                                        out_dtype=torch.float32, status=st)
    ref_gpu = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), int(lens.max()),
                                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out_np(out)
    rows = sorted(set([0, B - 1, B // 2]))
    assert_close(got[rows], _oracle_rows(pool, q, bt, lens, rows), f"B={B} shared={shared_len}")
    assert_close(got, out_np(ref_gpu), "vs per-request decode")


def test_shared_prefix_rejects_bad_shapes():
    pool, q, bt, lens = _shared_case(2, 32, 8, 128, [5, 9], 7)
    with pytest.raises(phs.PhsError) as e:          # not a multiple of 64
        phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), 96)
    assert e.value.code == -7
    big_q = synth.normal_bf16((65, 32, 128), 1, device="cuda")   # 260 rows > 256
    bt65 = np.tile(bt[:1], (65, 1))
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_shared_prefix(big_q, pool, dev(bt65), dev(np.full(65, 133, np.int32)),
                                      133, 128)
    assert e.value.code == -7


@pytest.mark.slow
def test_shared_prefix_full_size_sampled():
    """The 250,000-token shared prefix of 64 requests (+512-token suffixes):
    the tensor-core pass covers 249,984 tokens, the split kernel the rest."""
    w = synth.shared_prefix()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    pool = phs.PagedPool(synth.normal_bf16((w.num_pages, Hkv, 16, D), 51, device="cuda"),
                         synth.normal_bf16((w.num_pages, Hkv, 16, D), 52, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), 53, device="cuda")
    n = (w.n_pre + 1).astype(np.int32)
    shared = (250_000 // 64) * 64
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_shared_prefix(q, pool, dev(w.block_table), dev(n), int(n.max()), shared,
                                        out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = [0, B - 1]
    assert_close(out_np(out)[rows], _oracle_rows(pool, q, w.block_table, n, rows), "config 5")
