"""The INT8 warm zone grows as decode proceeds ("Kimi K2.5 architecture deep
dive" page, sections 2.2-2.3: recent tokens stay in the bf16 hot window and
age into block-wise INT8 one 32-token group at a time).  Each step appends
every request's new token in bf16; a request whose bf16 tail reaches 1056
tokens has its oldest bf16 block quantised (first_qblock = qlen / 32) and
its INT8 length advanced by 32; then all requests decode.  Codes and scales
must be bit-exact and outputs within tolerance of the oracle at every
step, with requests crossing the boundary at different steps."""
import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, dev, out_np

pytestmark = pytest.mark.gpu

HOT = 1024       # bf16 tokens kept (the new one excluded)
QB = 32


def test_int8_hot_to_warm_handoff_over_steps():
    B, Hq, Hkv, D = 4, 32, 8, 128
    steps = 45
    qlen = np.full(B, 2048, np.int32)
    # bf16 tail before the first step's append: 1024, 1040, 1050, 1055
    n_pre = qlen + np.array([1024, 1040, 1050, 1055], np.int32)
    n_max = n_pre + steps
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(n_max), 401)
    nq_max = (n_max // QB).astype(np.int64)
    qt, nqp = synth.block_tables_from_permutation(nq_max, 402)
    kp = synth.normal_bf16((npg, Hkv, 16, D), 403, device="cuda", outlier_p=0.01)
    vp = synth.normal_bf16((npg, Hkv, 16, D), 404, device="cuda", outlier_p=0.01)
    pool = phs.PagedPool(kp, vp)
    i8 = phs.Int8Pool.empty(nqp, Hkv, D)
    hk, hv = synth.bits(kp), synth.bits(vp)
    hkc = np.zeros((nqp, Hkv, QB, D), np.int8)
    hvc = np.zeros_like(hkc)
    hks = np.zeros((nqp, Hkv), np.float32)
    hvs = np.zeros_like(hks)
    bt_d, qt_d = dev(bt), dev(qt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def quantise(first, num):
        phs.kv_quant_int8_block32(pool, bt_d, i8, qt_d, dev(first), dev(num), int(num.max()),
                                  status=st)
        assert oracle.quant_int8_block32(hk, hv, bt, hkc, hvc, hks, hvs, qt, first, num) == 0

    def same_int8():
        torch.cuda.synchronize()
        gk, gv = i8.codes()
        return (np.array_equal(gk.cpu().numpy(), hkc) and np.array_equal(gv.cpu().numpy(), hvc)
                and np.array_equal(i8.k_scale.cpu().numpy(), hks)
                and np.array_equal(i8.v_scale.cpu().numpy(), hvs))

    # set-up: the warm zone [0, qlen) quantised once
    i8.k.fill_(128)  # the stored form of code 0
    i8.v.fill_(128)
    i8.k_scale.zero_()
    i8.v_scale.zero_()
    quantise(np.zeros(B, np.int32), (qlen // QB).astype(np.int32))
    assert same_int8()
    crossings = np.zeros(B, np.int32)
    max_seq = int(n_max.max())
    ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, max_seq, has_int8=True),
                     dtype=torch.uint8, device="cuda")
    for k in range(steps):
        n_after = (n_pre + 1 + k).astype(np.int32)
        q = synth.normal_bf16((B, Hq, D), 500 + 3 * k, device="cuda")
        kn = synth.normal_bf16((B, Hkv, D), 501 + 3 * k, device="cuda")
        vn = synth.normal_bf16((B, Hkv, D), 502 + 3 * k, device="cuda")
        phs.kv_append_paged(pool, kn, vn, bt_d, dev(n_after), status=st)
        assert oracle.append_paged(hk, hv, synth.bits(kn), synth.bits(vn), bt, n_after) == 0
        # the oldest bf16 block of a tail that reached HOT + 32 tokens ages out
        cross = (n_after - qlen >= HOT + QB).astype(np.int32)
        if cross.any():
            quantise((qlen // QB).astype(np.int32), cross)
            qlen = qlen + QB * cross
            crossings += cross
            assert same_int8(), f"step {k}"
        assert np.all(n_after - qlen >= HOT) and np.all(n_after - qlen < HOT + QB)
        out = phs.attn_decode_full_paged(q, pool, bt_d, dev(n_after), max_seq, int8=i8,
                                         qtable=qt_d, qlens=dev(qlen), out_dtype=torch.float32,
                                         workspace=ws, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"step {k}"
        ref, s = oracle.decode_full_paged(
            synth.bits(q), hk, hv, bt, n_after, 1 / np.sqrt(D),
            int8=dict(k_codes=hkc, v_codes=hvc, k_scale=hks, v_scale=hvs, qtable=qt, qlens=qlen))
        assert s == 0
        assert_close(out_np(out), ref, f"step {k}")
    # every request crossed once or twice, at different steps
    assert np.all(crossings >= 1) and crossings.sum() > B
    # the bf16 pool (appends included) stayed byte-equal to the oracle's
    assert np.array_equal(synth.bits(pool.k), hk) and np.array_equal(synth.bits(pool.v), hv)
