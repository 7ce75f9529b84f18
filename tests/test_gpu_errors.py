"""Error behaviour through the C ABI: host-side argument errors return a
status before anything is launched; data-dependent errors are recorded in
the device status word and the offending item is skipped (nothing traps)."""
import math

import numpy as np
import pytest
import torch

import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import bf16_dev, dev

pytestmark = pytest.mark.gpu


def _pool(npg=8, Hkv=2, D=64):
    return phs.PagedPool(synth.normal_bf16((npg, Hkv, 16, D), 1, device="cuda"),
                         synth.normal_bf16((npg, Hkv, 16, D), 2, device="cuda"))


def test_out_of_range_page_is_recorded_not_faulted():
    pool = _pool()
    q = synth.normal_bf16((2, 4, 64), 3, device="cuda")
    bt = dev(np.array([[0, 1, 99], [2, -5, 3]], np.int32))
    sl = dev(np.array([40, 40], np.int32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_full_paged(q, pool, bt, sl, 40, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3


def test_sequence_longer_than_table_is_recorded():
    pool = _pool()
    q = synth.normal_bf16((1, 4, 64), 3, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_full_paged(q, pool, dev(np.array([[0, 1]], np.int32)),
                               dev(np.array([50], np.int32)), 64, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3


def test_bad_int8_length_is_recorded():
    pool = _pool()
    i8 = phs.Int8Pool.empty(4, 2, 64)
    i8.k_scale.fill_(1.0)
    i8.v_scale.fill_(1.0)
    q = synth.normal_bf16((1, 4, 64), 3, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_full_paged(q, pool, dev(np.array([[0, 1, 2]], np.int32)),
                               dev(np.array([40], np.int32)), 48, int8=i8,
                               qtable=dev(np.array([[0, 1]], np.int32)),
                               qlens=dev(np.array([20], np.int32)), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3


def test_ring_bad_slot_is_recorded():
    ring = phs.RingPool(synth.normal_bf16((2, 2, 128, 64), 4, device="cuda"),
                        synth.normal_bf16((2, 2, 128, 64), 5, device="cuda"))
    q = synth.normal_bf16((2, 4, 64), 6, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_swa_ring(q, ring, dev(np.array([3, 128], np.int32)),
                             dev(np.array([10, 10], np.int32)), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3
    st.zero_()
    kn = synth.normal_bf16((2, 2, 64), 7, device="cuda")
    phs.kv_append_ring(ring, kn, kn, dev(np.array([0, 1], np.int32)),
                       ring_ids=dev(np.array([0, 7], np.int32)), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -3


def test_host_errors():
    pool = _pool()
    q = synth.normal_bf16((1, 4, 64), 3, device="cuda")
    bt = dev(np.array([[0, 1]], np.int32))
    sl = dev(np.array([20], np.int32))
    with pytest.raises(phs.PhsError) as e:   # workspace too small
        phs.attn_decode_full_paged(q, pool, bt, sl, 20,
                                   workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -5
    with pytest.raises(phs.PhsError) as e:   # Hq not a multiple of Hkv
        phs.attn_decode_full_paged(synth.normal_bf16((1, 3, 64), 3, device="cuda"), pool, bt, sl,
                                   20)
    assert e.value.code == -2
    odd = phs.PagedPool(torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(phs.PhsError) as e:   # head_dim 96
        phs.attn_decode_full_paged(synth.normal_bf16((1, 4, 96), 3, device="cuda"), odd, bt, sl,
                                   20)
    assert e.value.code == -7
    qbuf = torch.zeros(1 * 4 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(phs.PhsError) as e:   # q not 16-byte aligned
        phs.attn_decode_full_paged(qbuf[1:].view(1, 4, 64), pool, bt, sl, 20)
    assert e.value.code == -9
    with pytest.raises(phs.PhsError) as e:   # tokens_per_split not a multiple of 32
        phs.attn_decode_full_paged(q, pool, bt, sl, 20, tokens_per_split=48)
    assert e.value.code == -7
    with pytest.raises(phs.PhsError) as e:   # group of 34 query heads per KV head (max 16)
        phs.attn_decode_full_paged(synth.normal_bf16((1, 68, 64), 3, device="cuda"), pool, bt,
                                   sl, 20)
    assert e.value.code == -7


def test_stack_rejects_bad_scale_before_any_launch():
    """A rejected hybrid-stack call launches nothing: no append has happened
    when the scale is found to be invalid."""
    B, Hq, Hkv, D, W = 2, 4, 2, 64, 16
    pool = _pool()
    ring = phs.RingPool(synth.normal_bf16((B, Hkv, W, D), 4, device="cuda"),
                        synth.normal_bf16((B, Hkv, W, D), 5, device="cuda"))
    kn = synth.normal_bf16((B, Hkv, D), 6, device="cuda")
    layers = [phs.Layer(q=synth.normal_bf16((B, Hq, D), 7, device="cuda"),
                        out=torch.empty((B, Hq, D), device="cuda"), paged=pool, k_new=kn,
                        v_new=kn),
              phs.Layer(q=synth.normal_bf16((B, Hq, D), 8, device="cuda"),
                        out=torch.empty((B, Hq, D), device="cuda"), ring=ring, k_new=kn,
                        v_new=kn)]
    before = [t.clone() for t in (pool.k, pool.v, ring.k, ring.v)]
    bt = dev(np.array([[0, 1], [2, 3]], np.int32))
    sl = dev(np.array([20, 9], np.int32))
    rp = dev(np.array([3, 8], np.int32))
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        for call in (phs.attn_decode_hybrid_stack, phs.attn_decode_hybrid_stack_fused):
            with pytest.raises(phs.PhsError) as e:
                call(layers, Hq, sl, 20, block_table=bt, ring_pos=rp, softmax_scale=bad)
            assert e.value.code == -1
    torch.cuda.synchronize()
    for x, y in zip(before, (pool.k, pool.v, ring.k, ring.v)):
        assert torch.equal(x, y)


def test_too_many_kv_heads_for_one_append_cta_is_unsupported():
    # 72 KV heads of 128 dims: 1,152 16-byte pieces per token row, more than
    # one CTA of the append kernel covers
    pool = phs.PagedPool(torch.zeros((2, 72, 16, 128), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((2, 72, 16, 128), dtype=torch.bfloat16, device="cuda"))
    kn = torch.zeros((1, 72, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(phs.PhsError) as e:
        phs.kv_append_paged(pool, kn, kn, dev(np.array([[0]], np.int32)),
                            dev(np.array([1], np.int32)))
    assert e.value.code == -7
    ring = phs.RingPool(torch.zeros((1, 72, 16, 128), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((1, 72, 16, 128), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(phs.PhsError) as e:
        phs.kv_append_ring(ring, kn, kn, dev(np.array([0], np.int32)))
    assert e.value.code == -7
