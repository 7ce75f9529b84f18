"""A cached prefix resumed by a new request of a hybrid stack ("Xiaomi
MiMo-V2.5 inference system" page, section 2: the prefix tree's nodes carry
the Full pages and the SWA mapping; a hit is usable only at a window-safe
length).  A finished request saves the whole pages of its SWA window into
segment pages (phs_swa_ring_save) and is inserted into the radix tree with
them; a new request sharing the prefix matches it window-safely, seeds its
ring from the returned segment pages (phs_swa_ring_seed) and decodes on.
Save and seed are checked byte for byte against the oracle; the decode step
after the hit against the oracle over the dense sequence."""
import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np
from paging import dense_to_paged, dense_to_ring, random_bf16

pytestmark = pytest.mark.gpu
P = 16


def test_swa_save_and_seed_bitexact_against_oracle():
    rng = np.random.default_rng(21)
    L, R, W, Hkv, D, NSEG = 3, 5, 128, 8, 128, 40
    rings = [(random_bf16(rng, (R, Hkv, W, D)), random_bf16(rng, (R, Hkv, W, D)))
             for _ in range(L)]
    segs = [(random_bf16(rng, (NSEG, Hkv, P, D)), random_bf16(rng, (NSEG, Hkv, P, D)))
            for _ in range(L)]
    drings = [phs.RingPool(bf16_dev(k), bf16_dev(v)) for k, v in rings]
    dsegs = [phs.PagedPool(bf16_dev(k), bf16_dev(v)) for k, v in segs]
    # save: pages inside each request's window, plus one that is not
    ring_ids = np.array([0, 0, 3, 3, 1, 2], np.int32)
    ring_pos = np.array([17, 17, 127, 127, 0, 64], np.int32)
    lens = np.array([400, 400, 1024, 1024, 128, 300], np.int32)
    page_index = np.array([17, 24, 56, 63, 0, 10], np.int32)   # 300: window [172,300)
    seg_pages = np.array([3, 9, 11, 0, 39, 20], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.swa_ring_save(drings, dsegs, dev(ring_ids), dev(ring_pos), dev(lens), dev(page_index),
                      dev(seg_pages), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3          # the last entry starts before its window
    for (kr, vr), (ks, vs), dr, ds in zip(rings, segs, drings, dsegs):
        assert oracle.swa_ring_save(kr, vr, ks, vs, ring_ids, ring_pos, lens, page_index,
                                    seg_pages) == oracle.ORC_ERANGE
        assert np.array_equal(synth.bits(ds.k), ks) and np.array_equal(synth.bits(ds.v), vs)
    # seed: requests of several lengths (below W, page-aligned, not aligned)
    B = 4
    s_lens = np.array([5, 128, 131, 1000], np.int32)
    s_ids = np.array([4, 1, 0, 2], np.int32)
    s_pos = np.array([9, 127, 0, 55], np.int32)
    width = W // P + 1
    table = np.full((B, width), -1, np.int32)
    for b, n in enumerate(s_lens):
        k = (n + P - 1) // P - (n - min(n, W)) // P
        table[b, :k] = rng.choice(NSEG, size=k, replace=False)
    st.zero_()
    phs.swa_ring_seed(drings, dsegs, dev(s_pos), dev(s_lens), dev(table), ring_ids=dev(s_ids),
                      status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for (kr, vr), (ks, vs), dr in zip(rings, segs, drings):
        assert oracle.swa_ring_seed(kr, vr, ks, vs, s_ids, s_pos, s_lens, table) == 0
        assert np.array_equal(synth.bits(dr.k), kr) and np.array_equal(synth.bits(dr.v), vr)


@pytest.mark.parametrize("fused", [False, True])
def test_window_safe_hit_seeds_ring_and_decodes(fused):
    """Request A (1,024 tokens) finishes: its Full pages and the segment
    pages of its last window go into the tree.  Request B shares A's first
    1,024 tokens: the window-safe match returns A's 64 Full pages and 8
    segment pages, B's ring (another ring id, another newest slot) is seeded
    from them, and one decode step of the 2 Full + 3 SWA stack appends B's
    token 1,024 and attends.  Outputs against the oracle over B's dense
    sequence (Full: all 1,025 tokens; SWA: the last 128), the prefix pages
    untouched, B's ring equal to the oracle's seed + append."""
    rng = np.random.default_rng(7 + fused)
    Hq, Hkv, D, W = 32, 8, 128, 128
    lf = [1, 0, 0, 1, 0]
    nA = 1024
    NP, NSEG, NR = 80, 16, 3
    fa, sa = phs.PageAllocator(NP), phs.PageAllocator(NSEG)
    tree = phs.RadixTree(fa, P, swa_alloc=sa)
    tokens_a = rng.integers(0, 50_000, size=nA).astype(np.int32)
    pages_a = fa.alloc(nA // P)
    rp_a = 93
    dense = []                 # per layer: A's dense K, V [Hkv, nA, D]
    layers = []
    for l, full in enumerate(lf):
        k = random_bf16(rng, (Hkv, nA, D))
        v = random_bf16(rng, (Hkv, nA, D))
        dense.append((k, v))
        if full:
            bt_a = pages_a[None].astype(np.int32)
            pool = phs.PagedPool(bf16_dev(dense_to_paged([k], bt_a, NP)),
                                 bf16_dev(dense_to_paged([v], bt_a, NP)))
            layers.append(dict(full=True, pool=pool))
        else:
            ring = phs.RingPool(bf16_dev(dense_to_ring([k], [rp_a], W, num_rings=NR)),
                                bf16_dev(dense_to_ring([v], [rp_a], W, num_rings=NR)))
            seg = phs.PagedPool.empty(NSEG, Hkv, D)
            layers.append(dict(full=False, ring=ring, seg=seg))
    swa_layers = [x for x in layers if not x["full"]]
    rings = [x["ring"] for x in swa_layers]
    segs = [x["seg"] for x in swa_layers]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # A finishes: snapshot the whole pages of its window, insert, release
    wpages = np.arange((nA - W) // P, nA // P, dtype=np.int32)
    seg_a = sa.alloc(len(wpages))
    m = len(wpages)
    phs.swa_ring_save(rings, segs, dev(np.zeros(m, np.int32)), dev(np.full(m, rp_a, np.int32)),
                      dev(np.full(m, nA, np.int32)), dev(wpages), dev(seg_a), status=st)
    swa_map = np.full(nA // P, -1, np.int32)
    swa_map[wpages] = seg_a
    tree.insert(tokens_a, pages_a, swa_pages=swa_map)
    fa.decref(pages_a)
    sa.decref(seg_a)
    # B: shares A's 1,024 tokens, then goes on
    tokens_b = np.concatenate([tokens_a, rng.integers(0, 50_000, size=37).astype(np.int32)])
    got_pages, got_seg = tree.match_window_safe(tokens_b, W)
    assert got_pages.tolist() == pages_a.tolist() and got_seg.tolist() == seg_a.tolist()
    L = len(got_pages) * P
    rid_b, rp_b0 = 2, 40
    phs.swa_ring_seed(rings, segs, dev(np.array([rp_b0], np.int32)), dev(np.array([L], np.int32)),
                      dev(got_seg[None]), ring_ids=dev(np.array([rid_b], np.int32)), status=st)
    sa.decref(got_seg)                       # copied: B lets go of the snapshots
    fresh = fa.alloc(1)                      # B's own page for token 1,024
    bt_b = np.concatenate([got_pages, fresh])[None].astype(np.int32)
    prefix_before = [synth.bits(x["pool"].k)[pages_a].copy() for x in layers if x["full"]]
    # one decode step of B: append token L, attend
    n_after = np.array([L + 1], np.int32)
    rp_b = np.array([(rp_b0 + 1) % W], np.int32)
    dl, host = [], []
    for l, x in enumerate(layers):
        q = random_bf16(rng, (1, Hq, D))
        kn, vn = random_bf16(rng, (1, Hkv, D)), random_bf16(rng, (1, Hkv, D))
        out = torch.empty((1, Hq, D), dtype=torch.float32, device="cuda")
        kw = dict(q=bf16_dev(q), out=out, k_new=bf16_dev(kn), v_new=bf16_dev(vn))
        if x["full"]:
            dl.append(phs.Layer(paged=x["pool"], **kw))
        else:
            dl.append(phs.Layer(ring=x["ring"], **kw))
        host.append((q, kn, vn))
    call = phs.attn_decode_hybrid_stack_fused if fused else phs.attn_decode_hybrid_stack
    call(dl, Hq, dev(n_after), L + 1, block_table=dev(bt_b), ring_pos=dev(rp_b),
         ring_ids=dev(np.array([rid_b], np.int32)), page_refcount=dev(fa.refcounts()), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    scale = 1.0 / np.sqrt(D)
    for l, (x, L_, (q, kn, vn)) in enumerate(zip(layers, dl, host)):
        k_seq = np.concatenate([dense[l][0], kn[0][:, None]], axis=1)   # B's dense sequence
        v_seq = np.concatenate([dense[l][1], vn[0][:, None]], axis=1)
        if not x["full"]:
            k_seq, v_seq = k_seq[:, -W:], v_seq[:, -W:]                 # its last window
        n = k_seq.shape[1]
        bt = np.arange((n + P - 1) // P, dtype=np.int32)[None]
        ref, s = oracle.decode_full_paged(q, dense_to_paged([k_seq], bt, bt.shape[1]),
                                          dense_to_paged([v_seq], bt, bt.shape[1]), bt, [n],
                                          scale)
        assert s == 0
        assert_close(out_np(L_.out), ref, f"layer {l} ({'Full' if x['full'] else 'SWA'})")
        if not x["full"]:
            # B's ring: the oracle's seed from A's window pages, then the append
            kr = dense_to_ring([dense[l][0]], [rp_a], W, num_rings=NR)
            vr = dense_to_ring([dense[l][1]], [rp_a], W, num_rings=NR)
            ks = np.zeros((NSEG, Hkv, P, D), np.uint16)
            vs = np.zeros_like(ks)
            assert oracle.swa_ring_save(kr, vr, ks, vs, np.zeros(m), np.full(m, rp_a),
                                        np.full(m, nA), wpages, seg_a) == 0
            assert oracle.swa_ring_seed(kr, vr, ks, vs, [rid_b], [rp_b0], [L], got_seg[None]) == 0
            assert oracle.append_ring(kr, vr, kn, vn, [rid_b], rp_b) == 0
            assert np.array_equal(synth.bits(x["ring"].k)[rid_b], kr[rid_b])
            assert np.array_equal(synth.bits(x["ring"].v)[rid_b], vr[rid_b])
    # the shared prefix pages were not written (B's token went to its own page)
    after = [synth.bits(x["pool"].k)[pages_a] for x in layers if x["full"]]
    assert all(np.array_equal(a_, b_) for a_, b_ in zip(prefix_before, after))
    tree.close()
