"""GPU parity on the five workload configurations: the tiny hybrid case
completely, a reduced hybrid stack completely, and the full-size paged,
INT8 and shared-prefix cases on sampled requests (the oracle computes the
sampled requests one by one from a compact host copy of their pages)."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np, sub_pool

pytestmark = pytest.mark.gpu


def test_config1_tiny_hybrid():
    w = synth.tiny_hybrid()
    B, Hq, Hkv, D, W = w.B, w.Hq, w.Hkv, w.D, w.W
    kp = synth.bits(synth.normal_bf16((w.num_pages, Hkv, 16, D), 1))
    vp = synth.bits(synth.normal_bf16((w.num_pages, Hkv, 16, D), 2))
    kr = synth.bits(synth.normal_bf16((B, Hkv, W, D), 3))
    vr = synth.bits(synth.normal_bf16((B, Hkv, W, D), 4))
    qf = synth.bits(synth.normal_bf16((B, Hq, D), 5))
    qs = synth.bits(synth.normal_bf16((B, Hq, D), 6))
    kn = synth.bits(synth.normal_bf16((B, Hkv, D), 7))
    vn = synth.bits(synth.normal_bf16((B, Hkv, D), 8))
    pool = phs.PagedPool(bf16_dev(kp), bf16_dev(vp))
    ring = phs.RingPool(bf16_dev(kr), bf16_dev(vr))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl, bt, rp = dev(w.n_after), dev(w.block_table), dev(w.ring_pos)
    phs.kv_append_paged(pool, bf16_dev(kn), bf16_dev(vn), bt, sl, status=st)
    phs.kv_append_ring(ring, bf16_dev(kn), bf16_dev(vn), rp, status=st)
    of = phs.attn_decode_full_paged(bf16_dev(qf), pool, bt, sl, int(w.n_after.max()),
                                    softmax_scale=w.softmax_scale, out_dtype=torch.float32,
                                    status=st)
    os_ = phs.attn_decode_swa_ring(bf16_dev(qs), ring, rp, sl, softmax_scale=w.softmax_scale,
                                   out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    hk, hv, hkr, hvr = kp.copy(), vp.copy(), kr.copy(), vr.copy()
    oracle.append_paged(hk, hv, kn, vn, w.block_table, w.n_after)
    oracle.append_ring(hkr, hvr, kn, vn, None, w.ring_pos)
    assert np.array_equal(synth.bits(pool.k), hk) and np.array_equal(synth.bits(pool.v), hv)
    assert np.array_equal(synth.bits(ring.k), hkr) and np.array_equal(synth.bits(ring.v), hvr)
    rf, _ = oracle.decode_full_paged(qf, hk, hv, w.block_table, w.n_after, w.softmax_scale)
    rs, _ = oracle.decode_swa_ring(qs, hkr, hvr, None, w.ring_pos, w.n_after, w.softmax_scale)
    assert_close(out_np(of), rf, "config 1 full layer")
    assert_close(out_np(os_), rs, "config 1 SWA layer")
    # request 0 (38 tokens <= W): the SWA layer on the same KV equals Full
    # attention; checked through the oracle's own invariant tests.


def test_config3_reduced_hybrid_stack():
    """14-layer stack (Full iff l % 7 == 6), batch 8, lengths log-uniform in
    [4K, 8K], distinct pools per layer, append + attend in one call."""
    w = synth.hybrid_stack(seed=33, B=8, lo=4096, hi=8192, num_layers=14)
    B, Hq, Hkv, D, W = w.B, w.Hq, w.Hkv, w.D, w.W
    lf = w.extra["layer_is_full"]
    dev_layers, host = [], []
    for l, full in enumerate(lf):
        s = 1000 + 10 * l
        q = synth.bits(synth.normal_bf16((B, Hq, D), s))
        kn = synth.bits(synth.normal_bf16((B, Hkv, D), s + 1))
        vn = synth.bits(synth.normal_bf16((B, Hkv, D), s + 2))
        if full:
            k = synth.bits(synth.normal_bf16((w.num_pages, Hkv, 16, D), s + 3))
            v = synth.bits(synth.normal_bf16((w.num_pages, Hkv, 16, D), s + 4))
            L = phs.Layer(q=bf16_dev(q), out=torch.empty((B, Hq, D), device="cuda"),
                          paged=phs.PagedPool(bf16_dev(k), bf16_dev(v)), k_new=bf16_dev(kn),
                          v_new=bf16_dev(vn))
        else:
            k = synth.bits(synth.normal_bf16((B, Hkv, W, D), s + 3))
            v = synth.bits(synth.normal_bf16((B, Hkv, W, D), s + 4))
            L = phs.Layer(q=bf16_dev(q), out=torch.empty((B, Hq, D), device="cuda"),
                          ring=phs.RingPool(bf16_dev(k), bf16_dev(v)), k_new=bf16_dev(kn),
                          v_new=bf16_dev(vn))
        dev_layers.append(L)
        host.append((full, q, kn, vn, k.copy(), v.copy()))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_hybrid_stack(dev_layers, Hq, dev(w.n_after), int(w.n_after.max()),
                                 block_table=dev(w.block_table), ring_pos=dev(w.ring_pos),
                                 softmax_scale=w.softmax_scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for l, (L, (full, q, kn, vn, k, v)) in enumerate(zip(dev_layers, host)):
        if full:
            oracle.append_paged(k, v, kn, vn, w.block_table, w.n_after)
            ref, s = oracle.decode_full_paged(q, k, v, w.block_table, w.n_after, w.softmax_scale)
            pk, pv = L.paged.k, L.paged.v
        else:
            oracle.append_ring(k, v, kn, vn, None, w.ring_pos)
            ref, s = oracle.decode_swa_ring(q, k, v, None, w.ring_pos, w.n_after, w.softmax_scale)
            pk, pv = L.ring.k, L.ring.v
        assert s == 0
        assert np.array_equal(synth.bits(pk), k) and np.array_equal(synth.bits(pv), v), l
        assert_close(out_np(L.out), ref, f"layer {l} ({'Full' if full else 'SWA'})")


@pytest.mark.slow
def test_config2_full_size_sampled():
    w = synth.paged_full()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 21, device="cuda")
    vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 22, device="cuda")
    q = synth.normal_bf16((B, Hq, D), 23, device="cuda")
    kn = synth.normal_bf16((B, Hkv, D), 24, device="cuda")
    vn = synth.normal_bf16((B, Hkv, D), 25, device="cuda")
    rows = [0, 9, int(np.argmax(w.n_pre)), int(np.argmin(w.n_pre)), B - 1]
    hk, bt_s = sub_pool(kp, w.block_table, rows, w.n_after)
    hv, _ = sub_pool(vp, w.block_table, rows, w.n_after)
    pool = phs.PagedPool(kp, vp)
    sl, bt = dev(w.n_after), dev(w.block_table)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_append_paged(pool, kn, vn, bt, sl, status=st)
    out = phs.attn_decode_full_paged(q, pool, bt, sl, int(w.n_after.max()),
                                     softmax_scale=w.softmax_scale, out_dtype=torch.bfloat16,
                                     status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qh, knh, vnh = synth.bits(q)[rows], synth.bits(kn)[rows], synth.bits(vn)[rows]
    oracle.append_paged(hk, hv, knh, vnh, bt_s, w.n_after[rows])
    ref, s = oracle.decode_full_paged(qh, hk, hv, bt_s, w.n_after[rows], w.softmax_scale)
    assert s == 0
    assert_close(out_np(out)[rows], ref, "config 2 sampled")
    # the appended token is in place for every request (bit-exact)
    last = (w.n_after - 1)
    pages = w.block_table[np.arange(B), last // 16]
    got_k = pool.k[dev(pages).long(), :, dev(last % 16).long()]
    assert torch.equal(got_k, kn)


@pytest.mark.slow
def test_config4_full_size_sampled():
    w = synth.int8_block32()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    qlen, qt, nq = w.extra["qlen"], w.extra["qtable"], w.extra["num_qpages"]
    kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 41, device="cuda", outlier_p=0.01)
    vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 42, device="cuda", outlier_p=0.01)
    q = synth.normal_bf16((B, Hq, D), 43, device="cuda")
    kn = synth.normal_bf16((B, Hkv, D), 44, device="cuda")
    vn = synth.normal_bf16((B, Hkv, D), 45, device="cuda")
    rows = [0, 13, B - 1]
    hk, bt_s = sub_pool(kp, w.block_table, rows, w.n_after)
    hv, _ = sub_pool(vp, w.block_table, rows, w.n_after)
    src = phs.PagedPool(kp, vp)
    i8 = phs.Int8Pool.empty(nq, Hkv, D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqb = (qlen // 32).astype(np.int32)
    phs.kv_quant_int8_block32(src, dev(w.block_table), i8, dev(qt), dev(np.zeros(B, np.int32)),
                              dev(nqb), int(nqb.max()), status=st)
    sl, bt = dev(w.n_after), dev(w.block_table)
    phs.kv_append_paged(src, kn, vn, bt, sl, status=st)
    out = phs.attn_decode_full_paged(q, src, bt, sl, int(w.n_after.max()),
                                     softmax_scale=w.softmax_scale, int8=i8, qtable=dev(qt),
                                     qlens=dev(qlen), out_dtype=torch.bfloat16, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # oracle: quantise the sampled requests itself, compare codes bit for bit
    ns = len(rows)
    nqs = int(nqb[rows].sum())
    qt_s = np.full((ns, int(nqb.max())), -1, np.int32)
    o = 0
    for i, b in enumerate(rows):
        qt_s[i, :nqb[b]] = np.arange(o, o + nqb[b])
        o += nqb[b]
    kc = np.zeros((nqs, Hkv, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nqs, Hkv), np.float32)
    vs = np.zeros_like(ks)
    assert oracle.quant_int8_block32(hk, hv, bt_s, kc, vc, ks, vs, qt_s, np.zeros(ns, np.int32),
                                     nqb[rows]) == 0
    gpu_ids = torch.from_numpy(np.concatenate([qt[b, :nqb[b]] for b in rows]).astype(np.int64))
    gpu_ids = gpu_ids.cuda()
    gk, gv = i8.codes(gpu_ids)
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)
    assert np.array_equal(i8.k_scale.index_select(0, gpu_ids).cpu().numpy(), ks)
    assert np.array_equal(i8.v_scale.index_select(0, gpu_ids).cpu().numpy(), vs)
    qh, knh, vnh = synth.bits(q)[rows], synth.bits(kn)[rows], synth.bits(vn)[rows]
    oracle.append_paged(hk, hv, knh, vnh, bt_s, w.n_after[rows])
    ref, s = oracle.decode_full_paged(
        qh, hk, hv, bt_s, w.n_after[rows], w.softmax_scale,
        int8=dict(k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs, qtable=qt_s,
                  qlens=qlen[rows]))
    assert s == 0
    assert_close(out_np(out)[rows], ref, "config 4 sampled")


@pytest.mark.slow
def test_config5_shared_prefix_steps_sampled():
    w = synth.shared_prefix()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    rc = w.extra["refcount"]
    kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 51, device="cuda")
    vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 52, device="cuda")
    pool = phs.PagedPool(kp, vp)
    steps = 3
    rows = [0, B - 1]
    n_final = w.n_pre + steps
    hk, bt_s = sub_pool(kp, w.block_table, rows, n_final)
    hv, _ = sub_pool(vp, w.block_table, rows, n_final)
    bt, rcd = dev(w.block_table), dev(rc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in range(steps):
        n_after = (w.n_pre + 1 + k).astype(np.int32)
        q = synth.normal_bf16((B, Hq, D), 60 + 3 * k, device="cuda")
        kn = synth.normal_bf16((B, Hkv, D), 61 + 3 * k, device="cuda")
        vn = synth.normal_bf16((B, Hkv, D), 62 + 3 * k, device="cuda")
        sl = dev(n_after)
        phs.kv_append_paged(pool, kn, vn, bt, sl, page_refcount=rcd, status=st)
        out = phs.attn_decode_full_paged(q, pool, bt, sl, int(n_after.max()),
                                         softmax_scale=w.softmax_scale,
                                         out_dtype=torch.float32, status=st)
        oracle.append_paged(hk, hv, synth.bits(kn)[rows], synth.bits(vn)[rows], bt_s,
                            n_after[rows])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, s = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, n_after[rows],
                                      w.softmax_scale)
    assert s == 0
    assert_close(out_np(out)[rows], ref, "config 5 sampled")


@pytest.mark.slow
def test_config3_full_size_fused_sampled():
    """The 70-layer stack at full size (batch 256, lengths log-uniform in
    [4K, 128K]) through the fused step the bench times; the 10 Full layers
    share one pool, as the bench aliases them (each layer still attends to
    its own new token, taken from its input).  Sampled requests of two Full
    and two SWA layers against the oracle."""
    w = synth.hybrid_stack()
    B, Hq, Hkv, D, W = w.B, w.Hq, w.Hkv, w.D, w.W
    lf = w.extra["layer_is_full"]
    kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 71, device="cuda")
    vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 72, device="cuda")
    pool = phs.PagedPool(kp, vp)
    rows = [0, int(np.argmax(w.n_after)), int(np.argmin(w.n_after)), B - 1]
    check = {6, 69, 0, 35}  # Full, Full, SWA, SWA
    hk, bt_s = sub_pool(kp, w.block_table, rows, w.n_after)
    hv, _ = sub_pool(vp, w.block_table, rows, w.n_after)
    layers, host = [], {}
    for l, full in enumerate(lf):
        q = synth.normal_bf16((B, Hq, D), 3000 + 3 * l, device="cuda")
        kn = synth.normal_bf16((B, Hkv, D), 3001 + 3 * l, device="cuda")
        vn = synth.normal_bf16((B, Hkv, D), 3002 + 3 * l, device="cuda")
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        if full:
            L = phs.Layer(q=q, out=out, paged=pool, k_new=kn, v_new=vn)
        else:
            ring = phs.RingPool(synth.normal_bf16((B, Hkv, W, D), 4000 + 2 * l, device="cuda"),
                                synth.normal_bf16((B, Hkv, W, D), 4001 + 2 * l, device="cuda"))
            L = phs.Layer(q=q, out=out, ring=ring, k_new=kn, v_new=vn)
            if l in check:
                host[l] = (synth.bits(ring.k)[rows], synth.bits(ring.v)[rows])
        layers.append(L)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_hybrid_stack_fused(layers, Hq, dev(w.n_after), int(w.n_after.max()),
                                       block_table=dev(w.block_table), ring_pos=dev(w.ring_pos),
                                       status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n_s, rp_s = w.n_after[rows], w.ring_pos[rows]
    for l in sorted(check):
        L = layers[l]
        qh = synth.bits(L.q)[rows]
        knh, vnh = synth.bits(L.k_new)[rows], synth.bits(L.v_new)[rows]
        if lf[l]:
            k, v = hk.copy(), hv.copy()
            oracle.append_paged(k, v, knh, vnh, bt_s, n_s)
            ref, s = oracle.decode_full_paged(qh, k, v, bt_s, n_s, w.softmax_scale)
        else:
            k, v = (x.copy() for x in host[l])
            oracle.append_ring(k, v, knh, vnh, None, rp_s)
            ref, s = oracle.decode_swa_ring(qh, k, v, None, rp_s, n_s, w.softmax_scale)
            # the ring now holds the new token (bit-exact)
            assert np.array_equal(synth.bits(L.ring.k)[rows], k), l
        assert s == 0
        assert_close(out_np(L.out)[rows], ref, f"config 3 fused, layer {l}")
