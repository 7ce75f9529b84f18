"""GPU tests of the hybrid-stack step with the appends fused into the
attention launches (phs_attn_decode_hybrid_stack_fused): outputs against the
oracle, pools bit-exact against the oracle's append, and outputs and pools
bit-identical to the unfused call on the same inputs.  Lengths are chosen so
the newest token lands on the first, a middle and the last slot of a page,
in single- and multi-split requests, with rings partly and fully filled."""
import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np

pytestmark = pytest.mark.gpu


def _stack(n_after, Hq, Hkv, D, layer_is_full, seed, W=128, out_dtype=torch.float32):
    """Host copies and device layers of a stack; every layer has its own
    pool and new token, the Full layers share one block table."""
    B = len(n_after)
    bt, num_pages = synth.block_tables_from_permutation(synth.pages_needed(n_after), seed + 1,
                                                        num_pages=int(synth.pages_needed(
                                                            n_after).sum()) + 7)
    ring_pos = synth.ring_positions(B, W, seed + 2)
    host, layers = [], []
    for l, full in enumerate(layer_is_full):
        s = seed * 1000 + 10 * l
        q = synth.bits(synth.normal_bf16((B, Hq, D), s))
        kn = synth.bits(synth.normal_bf16((B, Hkv, D), s + 1))
        vn = synth.bits(synth.normal_bf16((B, Hkv, D), s + 2))
        shape = (num_pages, Hkv, 16, D) if full else (B, Hkv, W, D)
        k = synth.bits(synth.normal_bf16(shape, s + 3))
        v = synth.bits(synth.normal_bf16(shape, s + 4))
        host.append((bool(full), q, kn, vn, k, v))
    return bt, ring_pos, host


def _device_layers(host, out_dtype):
    layers = []
    for full, q, kn, vn, k, v in host:
        B, Hq, D = q.shape
        kw = dict(q=bf16_dev(q), out=torch.empty((B, Hq, D), dtype=out_dtype, device="cuda"),
                  k_new=bf16_dev(kn), v_new=bf16_dev(vn))
        if full:
            kw["paged"] = phs.PagedPool(bf16_dev(k), bf16_dev(v))
        else:
            kw["ring"] = phs.RingPool(bf16_dev(k), bf16_dev(v))
        layers.append(phs.Layer(**kw))
    return layers


def _pools(L):
    p = L.paged if L.paged is not None else L.ring
    return p.k, p.v


CASES = [
    # (n_after per request, Hq, Hkv, D, layers)
    ([1, 16, 17, 130, 1025, 2048, 3001, 4096], 32, 8, 128, [0, 1, 0, 0, 1, 0, 1]),
    ([5, 128, 129, 700, 1040], 4, 2, 64, [1, 0, 1, 0]),
    ([33, 2049, 4000], 32, 2, 128, [1, 0]),  # G = 16: two row tiles per warp
    ([64, 300, 2500], 8, 8, 64, [1, 0, 1]),  # G = 1: one live row per tile
    ([17, 900, 3000, 48], 24, 4, 128, [0, 1, 1]),  # G = 6: rows 6 and 7 of the tile masked
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_stack_matches_oracle(case):
    n, Hq, Hkv, D, lf = CASES[case]
    n_after = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=40 + case)
    layers = _device_layers(host, torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_hybrid_stack_fused(layers, Hq, dev(n_after), int(n_after.max()),
                                       block_table=dev(bt), ring_pos=dev(rp), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    scale = 1.0 / np.sqrt(D)
    for l, (L, (full, q, kn, vn, k, v)) in enumerate(zip(layers, host)):
        k, v = k.copy(), v.copy()
        if full:
            oracle.append_paged(k, v, kn, vn, bt, n_after)
            ref, s = oracle.decode_full_paged(q, k, v, bt, n_after, scale)
        else:
            oracle.append_ring(k, v, kn, vn, None, rp)
            ref, s = oracle.decode_swa_ring(q, k, v, None, rp, n_after, scale)
        assert s == 0
        pk, pv = _pools(L)
        assert np.array_equal(synth.bits(pk), k) and np.array_equal(synth.bits(pv), v), l
        assert_close(out_np(L.out), ref, f"case {case} layer {l} ({'Full' if full else 'SWA'})")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fused_equals_unfused_bitexact(out_dtype):
    n, Hq, Hkv, D, lf = CASES[0]
    n_after = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=77)
    a = _device_layers(host, out_dtype)
    b = _device_layers(host, out_dtype)
    common = dict(block_table=dev(bt), ring_pos=dev(rp))
    phs.attn_decode_hybrid_stack(a, Hq, dev(n_after), int(n_after.max()), do_append=True, **common)
    phs.attn_decode_hybrid_stack_fused(b, Hq, dev(n_after), int(n_after.max()), **common)
    torch.cuda.synchronize()
    for l, (La, Lb) in enumerate(zip(a, b)):
        assert torch.equal(La.out, Lb.out), l
        for x, y in zip(_pools(La), _pools(Lb)):
            assert torch.equal(x, y), l


def test_fused_stack_two_steps():
    """Two consecutive steps: the second attends to the token the first
    appended (read back from the pool) plus its own new token."""
    n, Hq, Hkv, D, lf = CASES[1]
    n1 = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n1 + 1, Hq, Hkv, D, lf, seed=91)  # table covers both steps
    layers = _device_layers(host, torch.float32)
    scale = 1.0 / np.sqrt(D)
    rp2 = ((rp.astype(np.int64) + 1) % 128).astype(np.int32)
    for step, (nn, pos) in enumerate([(n1, rp), (n1 + 1, rp2)]):
        if step == 1:  # fresh new tokens and queries for the second step
            for L, hst in zip(layers, host):
                kn2 = synth.bits(synth.normal_bf16(hst[2].shape, 500 + step))
                vn2 = synth.bits(synth.normal_bf16(hst[3].shape, 600 + step))
                q2 = synth.bits(synth.normal_bf16(hst[1].shape, 700 + step))
                L.k_new.copy_(bf16_dev(kn2))
                L.v_new.copy_(bf16_dev(vn2))
                L.q.copy_(bf16_dev(q2))
        phs.attn_decode_hybrid_stack_fused(layers, Hq, dev(nn), int(nn.max()),
                                           block_table=dev(bt), ring_pos=dev(pos))
    torch.cuda.synchronize()
    for l, (L, (full, q, kn, vn, k, v)) in enumerate(zip(layers, host)):
        k, v = k.copy(), v.copy()
        kn2 = synth.bits(L.k_new)
        vn2 = synth.bits(L.v_new)
        q2 = synth.bits(L.q)
        if full:
            oracle.append_paged(k, v, kn, vn, bt, n1)
            oracle.append_paged(k, v, kn2, vn2, bt, n1 + 1)
            ref, _ = oracle.decode_full_paged(q2, k, v, bt, n1 + 1, scale)
        else:
            oracle.append_ring(k, v, kn, vn, None, rp)
            oracle.append_ring(k, v, kn2, vn2, None, rp2)
            ref, _ = oracle.decode_swa_ring(q2, k, v, None, rp2, n1 + 1, scale)
        pk, pv = _pools(L)
        assert np.array_equal(synth.bits(pk), k) and np.array_equal(synth.bits(pv), v), l
        assert_close(out_np(L.out), ref, f"second step, layer {l}")


def test_fused_stack_errors():
    n, Hq, Hkv, D, lf = CASES[1]
    n_after = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=5)
    layers = _device_layers(host, torch.float32)
    args = (layers, Hq, dev(n_after), int(n_after.max()))
    kw = dict(block_table=dev(bt), ring_pos=dev(rp))
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_hybrid_stack_fused(*args, workspace=small, **kw)
    assert e.value.code == -5  # PHS_EWORKSPACE
    layers[0].k_new = None
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_hybrid_stack_fused(*args, **kw)
    assert e.value.code == -1  # PHS_EINVAL: every layer needs its new token
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_hybrid_stack_fused(_device_layers(host, torch.float32), Hq, dev(n_after),
                                           int(n_after.max()), block_table=dev(bt))
    assert e.value.code == -1  # SWA layers without ring positions
    assert phs.hybrid_stack_fused_workspace_bytes(8, 32, 8, 128, 4096, 0) == 0
    one = phs.hybrid_stack_fused_workspace_bytes(8, 32, 8, 128, 4096, 1)
    assert phs.hybrid_stack_fused_workspace_bytes(8, 32, 8, 128, 4096, 10) == 10 * one


@pytest.mark.parametrize("D,Hq,Hkv,out_dtype", [(128, 8, 2, torch.float32),
                                                (64, 32, 2, torch.bfloat16),
                                                (128, 32, 8, torch.float32)])
def test_small_step_one_launch_equals_unfused(D, Hq, Hkv, out_dtype):
    """Short requests (one split each) and a few layers of each kind: the
    fused call runs the whole step in one launch (Full splits and SWA units
    side by side).  Outputs and pools equal the unfused call's bit for bit;
    the last layer of each kind matches the oracle."""
    n_after = np.array([1, 16, 17, 100, 200, 256], dtype=np.int32)
    lf = [1, 0, 0, 1, 0]  # 2 Full + 3 SWA layers
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=140 + D + Hq, out_dtype=out_dtype)
    a = _device_layers(host, out_dtype)
    b = _device_layers(host, out_dtype)
    common = dict(block_table=dev(bt), ring_pos=dev(rp))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_hybrid_stack(a, Hq, dev(n_after), int(n_after.max()), do_append=True, **common)
    phs.attn_decode_hybrid_stack_fused(b, Hq, dev(n_after), int(n_after.max()), status=st, **common)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for l, (La, Lb) in enumerate(zip(a, b)):
        assert torch.equal(La.out, Lb.out), l
        for x, y in zip(_pools(La), _pools(Lb)):
            assert torch.equal(x, y), l
    scale = 1.0 / np.sqrt(D)
    for l in (3, 4):  # the last Full and the last SWA layer
        full, q, kn, vn, k, v = host[l]
        k, v = k.copy(), v.copy()
        if full:
            oracle.append_paged(k, v, kn, vn, bt, n_after)
            ref, _ = oracle.decode_full_paged(q, k, v, bt, n_after, scale)
        else:
            oracle.append_ring(k, v, kn, vn, None, rp)
            ref, _ = oracle.decode_swa_ring(q, k, v, None, rp, n_after, scale)
        assert_close(out_np(b[l].out), ref, f"layer {l}")


@pytest.mark.parametrize("nfull,nswa", [(1, 66), (18, 2)])
def test_fused_stack_many_layers_equals_unfused(nfull, nswa):
    # more SWA layers than one launch carries (64: a second SWA launch, a
    # dependent of the first) and more Full layers than one split launch
    # carries (16: a second multi-layer launch, the first batch merged by a
    # merge launch, the last by the SWA launch); multi-split requests
    n = [40, 700, 3001, 5100]
    n_after = np.array(n, dtype=np.int32)
    Hq, Hkv, D = 4, 1, 64
    lf = [1] * nfull + [0] * nswa
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=130 + nfull, W=16)
    a = _device_layers(host, torch.float32)
    b = _device_layers(host, torch.float32)
    common = dict(block_table=dev(bt), ring_pos=dev(rp))
    phs.attn_decode_hybrid_stack(a, Hq, dev(n_after), int(n_after.max()), do_append=True, **common)
    phs.attn_decode_hybrid_stack_fused(b, Hq, dev(n_after), int(n_after.max()), **common)
    torch.cuda.synchronize()
    for l, (La, Lb) in enumerate(zip(a, b)):
        assert torch.equal(La.out, Lb.out), l
        for x, y in zip(_pools(La), _pools(Lb)):
            assert torch.equal(x, y), l
    # and the last layer of each kind against the oracle
    scale = 1.0 / np.sqrt(D)
    for l in (nfull - 1, nfull + nswa - 1):
        full, q, kn, vn, k, v = host[l]
        k, v = k.copy(), v.copy()
        if full:
            oracle.append_paged(k, v, kn, vn, bt, n_after)
            ref, _ = oracle.decode_full_paged(q, k, v, bt, n_after, scale)
        else:
            oracle.append_ring(k, v, kn, vn, None, rp)
            ref, _ = oracle.decode_swa_ring(q, k, v, None, rp, n_after, scale)
        assert_close(out_np(b[l].out), ref, f"layer {l}")


@pytest.mark.parametrize("fused", [False, True])
def test_stack_refuses_append_into_shared_page(fused):
    """Page reference counts in the stack calls ("Kimi K3 context caching"
    page, section 1: a request writes its new tokens only into blocks of its
    own).  Request 1's newest token falls in a page with count 2: that page
    stays byte-identical in every Full layer, the status is PHS_ESHARED, the
    other requests append as usual, and the outputs are those of the oracle
    on the pools as they stand (request 1 attends to the page unchanged)."""
    n, Hq, Hkv, D, lf = CASES[0]
    n_after = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=150)
    num_pages = host[next(i for i, x in enumerate(lf) if x)][4].shape[0]
    shared = int(bt[1, (n_after[1] - 1) // 16])
    rc = np.ones(num_pages, np.int32)
    rc[shared] = 2
    layers = _device_layers(host, torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    call = phs.attn_decode_hybrid_stack_fused if fused else phs.attn_decode_hybrid_stack
    call(layers, Hq, dev(n_after), int(n_after.max()), block_table=dev(bt), ring_pos=dev(rp),
         page_refcount=dev(rc), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -4  # PHS_ESHARED
    scale = 1.0 / np.sqrt(D)
    for l, (L, (full, q, kn, vn, k, v)) in enumerate(zip(layers, host)):
        k, v = k.copy(), v.copy()
        if full:
            assert oracle.append_paged(k, v, kn, vn, bt, n_after, page_refcount=rc) == -4
            ref, s = oracle.decode_full_paged(q, k, v, bt, n_after, scale)
            pk, pv = _pools(L)
            assert np.array_equal(synth.bits(pk)[shared], host[l][4][shared]), l
            assert np.array_equal(synth.bits(pv)[shared], host[l][5][shared]), l
        else:
            oracle.append_ring(k, v, kn, vn, None, rp)
            ref, s = oracle.decode_swa_ring(q, k, v, None, rp, n_after, scale)
        assert s == 0
        pk, pv = _pools(L)
        assert np.array_equal(synth.bits(pk), k) and np.array_equal(synth.bits(pv), v), l
        assert_close(out_np(L.out), ref, f"layer {l} ({'Full' if full else 'SWA'})")


def test_stack_fused_equals_unfused_with_shared_page():
    n, Hq, Hkv, D, lf = CASES[2]
    n_after = np.array(n, dtype=np.int32)
    bt, rp, host = _stack(n_after, Hq, Hkv, D, lf, seed=151)
    num_pages = host[0][4].shape[0]
    rc = np.ones(num_pages, np.int32)
    rc[int(bt[2, (n_after[2] - 1) // 16])] = 3
    a = _device_layers(host, torch.bfloat16)
    b = _device_layers(host, torch.bfloat16)
    common = dict(block_table=dev(bt), ring_pos=dev(rp), page_refcount=dev(rc))
    phs.attn_decode_hybrid_stack(a, Hq, dev(n_after), int(n_after.max()), **common)
    phs.attn_decode_hybrid_stack_fused(b, Hq, dev(n_after), int(n_after.max()), **common)
    torch.cuda.synchronize()
    for l, (La, Lb) in enumerate(zip(a, b)):
        assert torch.equal(La.out, Lb.out), l
        for x, y in zip(_pools(La), _pools(Lb)):
            assert torch.equal(x, y), l
