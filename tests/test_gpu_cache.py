"""GPU side of the cache bookkeeping: block tables built through the radix
tree and page allocator feed the decode kernels; copy on write with the page
copy kernel; the append's shared-page check driven by the allocator's
reference counts."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np

pytestmark = pytest.mark.gpu
P = 16


def test_copy_pages_bitexact():
    pool = phs.PagedPool(synth.normal_bf16((12, 8, 16, 128), 1, device="cuda"),
                         synth.normal_bf16((12, 8, 16, 128), 2, device="cuda"))
    k0, v0 = pool.k.clone(), pool.v.clone()
    src = np.array([3, 0, 7], np.int32)
    dst = np.array([10, 5, 1], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.copy_pages(pool, dev(src), dev(dst), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s, d in zip(src, dst):
        assert torch.equal(pool.k[d], k0[s]) and torch.equal(pool.v[d], v0[s])
    untouched = [i for i in range(12) if i not in dst]
    assert torch.equal(pool.k[untouched], k0[untouched])


def test_radix_shared_prefix_decode_and_cow_append():
    """Eight requests share a 1024-token prompt through the radix tree, each
    with its own 40-token continuation; decode must equal the oracle and be
    bit-identical across requests with equal continuations.  An append into
    a shared page is refused until the page is copied on write."""
    B, Hq, Hkv, D = 8, 32, 8, 128
    npg = 512
    alloc = phs.PageAllocator(npg)
    tree = phs.RadixTree(alloc, P)
    pool = phs.PagedPool(synth.normal_bf16((npg, Hkv, 16, D), 5, device="cuda"),
                         synth.normal_bf16((npg, Hkv, 16, D), 6, device="cuda"))
    prompt = list(range(1000, 1000 + 1024))
    # request 0 "prefills" the prompt into fresh pages and caches them
    p0 = alloc.alloc(1024 // P)
    tree.insert(prompt, p0)
    alloc.decref(p0)
    tables, lens = [], []
    for b in range(B):
        hit = tree.match(prompt)                 # 64 shared pages, +1 reference each
        assert hit.tolist() == p0.tolist()
        own = alloc.alloc(3)                     # 40-token continuation (+ room)
        tables.append(np.concatenate([hit, own]))
        lens.append(1024 + 40)
    bt = np.stack(tables).astype(np.int32)
    n = np.array(lens, np.int32)
    # continuation K/V: requests 2b and 2b+1 get identical contents
    for b in range(B):
        for j in range(3):
            src = bt[b - (b % 2), 64 + j]
            if b % 2:
                pool.k[bt[b, 64 + j]] = pool.k[src]
                pool.v[bt[b, 64 + j]] = pool.v[src]
    q1 = synth.normal_bf16((B // 2, Hq, D), 7, device="cuda")
    q = q1.repeat_interleave(2, dim=0).contiguous()
    out = phs.attn_decode_full_paged(q, pool, dev(bt), dev(n), int(n.max()),
                                     out_dtype=torch.float32, tokens_per_split=256)
    torch.cuda.synchronize()
    got = out_np(out)
    for b in range(0, B, 2):
        assert np.array_equal(got[b], got[b + 1])
    rows = [0, 5]
    used = np.unique(bt[rows].ravel())
    remap = {int(p): i for i, p in enumerate(used)}
    bt_s = np.vectorize(remap.get)(bt[rows]).astype(np.int32)
    hk = synth.bits(pool.k[dev(used).long()])
    hv = synth.bits(pool.v[dev(used).long()])
    ref, s = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, n[rows], 1 / math.sqrt(D))
    assert s == 0
    assert_close(got[rows], ref, "radix-shared prefix")

    # append at position 1064 goes to each request's own page: allowed
    rc = dev(alloc.refcounts())
    kn = synth.normal_bf16((B, Hkv, D), 8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_append_paged(pool, kn, kn, dev(bt), dev(n + 1), page_refcount=rc, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # rewriting token 1000 (inside a shared prompt page) is refused ...
    shared_page = int(bt[3, 1000 // P])
    n_bad = np.full(B, 1001, np.int32)
    phs.kv_append_paged(pool, kn, kn, dev(bt), dev(n_bad), page_refcount=rc, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -4
    # ... until request 3 copies the page on write
    fresh = alloc.cow(shared_page)
    assert fresh != shared_page
    phs.copy_pages(pool, dev([shared_page]), dev([fresh]))
    bt3 = bt[3:4].copy()
    bt3[0, 1000 // P] = fresh
    st.zero_()
    before = pool.k[shared_page].clone()
    phs.kv_append_paged(pool, kn[3:4].contiguous(), kn[3:4].contiguous(), dev(bt3),
                        dev([1001]), page_refcount=dev(alloc.refcounts()), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pool.k[shared_page], before)          # the shared copy is intact
    assert torch.equal(pool.k[fresh, :, 1000 % P], kn[3])     # the private copy took the token
    assert torch.equal(pool.k[fresh, :, :1000 % P], before[:, :1000 % P])
