"""GPU parity, bit-exact: KV append (paged and ring) and the block-32 INT8
quantiser against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import bf16_dev, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hkv,D", [(8, 128), (2, 64)])
def test_append_paged_bitexact(Hkv, D):
    lens = np.array([1, 15, 16, 17, 33, 200, 2048, 4097], np.int32)  # after append
    B = len(lens)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(lens), 7, num_pages=None)
    npg += 3
    kp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), 1))
    vp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), 2))
    kn = synth.bits(synth.normal_bf16((B, Hkv, D), 3))
    vn = synth.bits(synth.normal_bf16((B, Hkv, D), 4))
    pool = phs.PagedPool(bf16_dev(kp), bf16_dev(vp))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_append_paged(pool, bf16_dev(kn), bf16_dev(vn), dev(bt), dev(lens), status=st)
    hk, hv = kp.copy(), vp.copy()
    assert oracle.append_paged(hk, hv, kn, vn, bt, lens) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(synth.bits(pool.k), hk)
    assert np.array_equal(synth.bits(pool.v), hv)


def test_append_paged_refuses_shared_page():
    Hkv, D = 2, 64
    kp = synth.bits(synth.normal_bf16((4, Hkv, 16, D), 5))
    vp = synth.bits(synth.normal_bf16((4, Hkv, 16, D), 6))
    kn = synth.bits(synth.normal_bf16((2, Hkv, D), 7))
    vn = synth.bits(synth.normal_bf16((2, Hkv, D), 8))
    bt = np.array([[0, 1], [0, 2]], np.int32)
    rc = np.array([2, 1, 1, 1], np.int32)
    lens = np.array([5, 20], np.int32)
    pool = phs.PagedPool(bf16_dev(kp), bf16_dev(vp))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_append_paged(pool, bf16_dev(kn), bf16_dev(vn), dev(bt), dev(lens),
                        page_refcount=dev(rc), status=st)
    hk, hv = kp.copy(), vp.copy()
    assert oracle.append_paged(hk, hv, kn, vn, bt, lens, page_refcount=rc) == oracle.ORC_ESHARED
    torch.cuda.synchronize()
    assert int(st.item()) == -4
    assert np.array_equal(synth.bits(pool.k), hk)
    assert np.array_equal(synth.bits(pool.v), hv)


@pytest.mark.parametrize("W,D", [(128, 128), (16, 64), (1024, 128)])
def test_append_ring_bitexact(W, D):
    B, Hkv = 6, 4
    kr = synth.bits(synth.normal_bf16((B + 2, Hkv, W, D), 9))
    vr = synth.bits(synth.normal_bf16((B + 2, Hkv, W, D), 10))
    kn = synth.bits(synth.normal_bf16((B, Hkv, D), 11))
    vn = synth.bits(synth.normal_bf16((B, Hkv, D), 12))
    ids = np.random.default_rng(1).permutation(B + 2)[:B].astype(np.int32)
    pos = synth.ring_positions(B, W, 13)
    ring = phs.RingPool(bf16_dev(kr), bf16_dev(vr))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_append_ring(ring, bf16_dev(kn), bf16_dev(vn), dev(pos), ring_ids=dev(ids), status=st)
    hk, hv = kr.copy(), vr.copy()
    assert oracle.append_ring(hk, hv, kn, vn, ids, pos) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(synth.bits(ring.k), hk)
    assert np.array_equal(synth.bits(ring.v), hv)


def _quant_case(D, Hkv, nblocks_per_req, seed, outlier_p=0.01):
    B = len(nblocks_per_req)
    n_tok = [32 * (nb + 1) for nb in nblocks_per_req]
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(n_tok), seed)
    kp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), seed + 1, outlier_p=outlier_p))
    vp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), seed + 2, outlier_p=outlier_p))
    qt, nq = synth.block_tables_from_permutation(np.array(nblocks_per_req) + 1, seed + 3)
    first = np.array([1 if b % 2 else 0 for b in range(B)], np.int32)
    num = np.array(nblocks_per_req, np.int32)
    return kp, vp, bt, qt, nq, first, num


@pytest.mark.parametrize("D,Hkv", [(128, 8), (64, 2)])
def test_quant_int8_bitexact(D, Hkv):
    kp, vp, bt, qt, nq, first, num = _quant_case(D, Hkv, [3, 1, 5, 2], 20)
    # one all-zero group and one group of tiny (subnormal-range) values
    kp[bt[0, 0], 1] = 0
    kp[bt[0, 1], 1] = 0
    vp[bt[2, 2], 0] = synth.bits(torch.full((16, D), 3e-39, dtype=torch.float32).to(torch.bfloat16))
    kc = np.zeros((nq, Hkv, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nq, Hkv), np.float32)
    vs = np.zeros_like(ks)
    assert oracle.quant_int8_block32(kp, vp, bt, kc, vc, ks, vs, qt, first, num) == 0
    src = phs.PagedPool(bf16_dev(kp), bf16_dev(vp))
    dst = phs.Int8Pool.empty(nq, Hkv, D)
    for t in (dst.k, dst.v):
        t.fill_(128)  # the stored form of code 0
    dst.k_scale.zero_()
    dst.v_scale.zero_()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_quant_int8_block32(src, dev(bt), dst, dev(qt), dev(first), dev(num), int(num.max()),
                              status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gk, gv = dst.codes()
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)
    assert np.array_equal(dst.k_scale.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(dst.v_scale.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert (ks == 0).any()  # the zero group really was zero


def test_copy_kernel():
    x = torch.randint(0, 255, (1 << 22,), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    phs.copy_d2d(y, x)
    torch.cuda.synchronize()
    assert torch.equal(x, y)


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 1 << 24, (1 << 26) + 48])
def test_read_checksum_kernel(nbytes):
    """The read yardstick really reads every word: its XOR fold equals the
    host's, on sizes with ragged tails past whole 4-load rounds."""
    g = torch.Generator().manual_seed(nbytes)
    x = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)
    want = np.bitwise_xor.reduce(x.numpy().view(np.uint32))
    sink = torch.tensor([0x1234], dtype=torch.int32, device="cuda")
    phs.read_checksum(x.cuda(), sink)
    torch.cuda.synchronize()
    got = np.array([sink.item()], dtype=np.int32).view(np.uint32)[0]
    assert got == (want ^ np.uint32(0x1234))


@pytest.mark.parametrize("scale_pow", [0, -1, 1, -20])
def test_quant_int8_half_integer_quotients_bitexact(scale_pow):
    """Groups whose absmax is 127 * 2^p, so s = 2^p exactly and x / s lands
    on half-integers: every such element decides by round-half-even."""
    D, Hkv = 128, 2
    rng = np.random.default_rng(100 + scale_pow)
    vals = np.empty((4, Hkv, 16, D), np.float32)
    k = rng.integers(-63, 63, size=vals.shape)
    vals[:] = (k + 0.5) * np.float32(2.0 ** scale_pow)
    vals[:, :, 0, 0] = 127 * np.float32(2.0 ** scale_pow)   # absmax of each group
    from paging import f32_to_bf16_bits
    kp = f32_to_bf16_bits(vals)
    vp = f32_to_bf16_bits(-vals)
    bt = np.array([[0, 1, 2, 3]], np.int32)
    qt = np.array([[1, 0]], np.int32)
    kc = np.zeros((2, Hkv, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((2, Hkv), np.float32)
    vs = np.zeros_like(ks)
    assert oracle.quant_int8_block32(kp, vp, bt, kc, vc, ks, vs, qt, [0], [2]) == 0
    assert np.all(ks == np.float32(2.0 ** scale_pow))
    src = phs.PagedPool(bf16_dev(kp), bf16_dev(vp))
    dst = phs.Int8Pool.empty(2, Hkv, D)
    phs.kv_quant_int8_block32(src, dev(bt), dst, dev(qt), dev(np.zeros(1, np.int32)),
                              dev(np.array([2], np.int32)), 2)
    torch.cuda.synchronize()
    gk, gv = dst.codes()
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)
    assert np.array_equal(dst.k_scale.cpu().numpy(), ks)
