"""The no-allocation decode entry point, for callers that cannot give the
library a workspace (a host framework that owns all device memory, an
engine that has reserved nearly all of HBM for its KV pool, a decode loop
that must not call cudaMalloc).  It must give the same results as the
workspace-taking entry point and as the oracle, call after call, and refuse
requests that do not fit its built-in scratch before launching anything.

This file is collected last so that a run stopping at the first failure
has already run every other test."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, dev, out_np, sub_pool

pytestmark = pytest.mark.gpu


def _case(seed, lens, Hq=32, Hkv=8, D=128):
    lens = np.asarray(lens, np.int32)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(lens), seed)
    pool = phs.PagedPool(synth.normal_bf16((npg, Hkv, 16, D), seed + 1, device="cuda"),
                         synth.normal_bf16((npg, Hkv, 16, D), seed + 2, device="cuda"))
    q = synth.normal_bf16((len(lens), Hq, D), seed + 3, device="cuda")
    return pool, q, bt, lens


def _oracle(pool, q, bt, lens, rows, int8=None):
    hk, bt_s = sub_pool(pool.k, bt, rows, lens)
    hv, _ = sub_pool(pool.v, bt, rows, lens)
    D = q.shape[2]
    ref, s = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, lens[rows],
                                      1 / math.sqrt(D), int8=int8)
    assert s == 0
    return ref


def test_noalloc_matches_workspace_entry_point_and_oracle_twice():
    cases = [_case(71, [1, 17, 900, 5000, 32769, 2048]), _case(72, [3000, 12, 7000])]
    for pool, q, bt, lens in cases:   # two calls in a row, different inputs
        ms = int(lens.max())
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), ms,
                                         out_dtype=torch.float32, status=st)
        out = torch.full_like(ref, float("nan"))
        phs.attn_decode_full_paged_noalloc(q, pool, dev(bt), dev(lens), ms, out, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_close(out_np(out), out_np(ref), "no-allocation vs workspace entry point")
        rows = list(range(len(lens)))
        assert_close(out_np(out), _oracle(pool, q, bt, lens, rows), "no-allocation vs oracle")


def test_noalloc_single_split_bf16_output():
    # every request fits one split of 512 tokens (no merge launch); bf16 output
    pool, q, bt, lens = _case(74, [1, 40, 333, 512], Hq=8, Hkv=2, D=64)
    ms = int(lens.max())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        ref = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), ms, tokens_per_split=512,
                                         status=st)
        out = torch.empty_like(ref)
        phs.attn_decode_full_paged_noalloc(q, pool, dev(bt), dev(lens), ms, out,
                                           tokens_per_split=512, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out, ref)
        assert_close(out_np(out), _oracle(pool, q, bt, lens, [0, 1, 2, 3]), "single split")


def test_noalloc_int8_region():
    """An INT8 warm zone below qlens (one more split per request) through
    the scratch: codes and scales from the library's quantiser."""
    B, Hq, Hkv, D = 3, 32, 8, 128
    lens = np.array([3000, 4097, 1200], np.int32)
    qlen = np.array([1024, 2048, 0], np.int32)
    pool, q, bt, _ = _case(76, lens, Hq, Hkv, D)
    nq = np.maximum(qlen // 32, 1).astype(np.int64)
    qt, nqp = synth.block_tables_from_permutation(nq, 77)
    i8 = phs.Int8Pool.empty(nqp, Hkv, D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqb = (qlen // 32).astype(np.int32)
    phs.kv_quant_int8_block32(pool, dev(bt), i8, dev(qt), dev(np.zeros(B, np.int32)), dev(nqb),
                              int(nqb.max()), status=st)
    ms = int(lens.max())
    kw = dict(int8=i8, qtable=dev(qt), qlens=dev(qlen), status=st)
    ref = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), ms, out_dtype=torch.float32,
                                     **kw)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        phs.attn_decode_full_paged_noalloc(q, pool, dev(bt), dev(lens), ms, out, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_close(out_np(out), out_np(ref), "INT8 no-allocation vs workspace entry point")
    gk, gv = i8.codes()
    codes = dict(k_codes=gk.cpu().numpy(), v_codes=gv.cpu().numpy(),
                 k_scale=i8.k_scale.cpu().numpy(), v_scale=i8.v_scale.cpu().numpy(),
                 qtable=qt, qlens=qlen)
    hk, hv = synth.bits(pool.k), synth.bits(pool.v)
    ref_o, s = oracle.decode_full_paged(synth.bits(q), hk, hv, bt, lens, 1 / math.sqrt(D),
                                        int8=codes)
    assert s == 0
    assert_close(out_np(out), ref_o, "INT8 no-allocation vs oracle")


def test_noalloc_lengthens_splits_to_fit_and_rejects_beyond_scratch():
    # two requests of one KV head with 16 query heads and a stated bound of
    # 600,000 tokens: for so small a grid the library's split length is short
    # (256 tokens on 152 SMs) and its partials (39 MB) do not fit the 32 MiB
    # scratch, so the call must lengthen its splits and still match the
    # workspace path and the oracle
    Hq, Hkv, D, bound = 16, 1, 128, 600_000
    pool, q, bt, lens = _case(73, [3000, 7001], Hq=Hq, Hkv=Hkv, D=D)
    assert phs.decode_workspace_bytes(2, Hq, Hkv, D, bound) > phs.NOALLOC_SCRATCH_BYTES
    out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_full_paged_noalloc(q, pool, dev(bt), dev(lens), bound, out, status=st)
    ref = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), bound, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out_np(out), out_np(ref), "lengthened splits")
    assert_close(out_np(out), _oracle(pool, q, bt, lens, [0, 1]), "lengthened splits vs oracle")
    # a request that cannot fit even with 4096-token splits is refused on
    # the host, before anything is launched
    bound = 131072
    pool, *_ = _case(75, [16])
    big_b = 512
    qb = torch.zeros((big_b, 32, 128), dtype=torch.bfloat16, device="cuda")
    btb = torch.zeros((big_b, 64), dtype=torch.int32, device="cuda")
    slb = torch.ones(big_b, dtype=torch.int32, device="cuda")
    outb = torch.empty((big_b, 32, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_full_paged_noalloc(qb, pool, btb, slb, bound, outb)
    assert e.value.code == -10
    with pytest.raises(phs.PhsError) as e:   # an explicit split length that does not fit
        phs.attn_decode_full_paged_noalloc(qb, pool, btb, slb, bound, outb,
                                           tokens_per_split=1024)
    assert e.value.code == -10
