"""GPU: the step's append fused into the Full decode calls.  The CTA that
attends a request's newest token writes it into its bf16 page and attends it
from the input; the result must equal kv_append_paged (same page reference
counts) followed by the same call, bit for bit, outputs and pools, for bf16
pools, INT8 regions, several splits, and the two-phase entry points."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np

pytestmark = pytest.mark.gpu


def _case(lens, Hq, Hkv, D, seed, qlens=None):
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(lens), seed)
    npg += 2
    c = dict(lens=lens, bt=bt, B=B, Hq=Hq, Hkv=Hkv, D=D,
             k=synth.normal_bf16((npg, Hkv, 16, D), seed + 1, device="cuda"),
             v=synth.normal_bf16((npg, Hkv, 16, D), seed + 2, device="cuda"),
             q=synth.normal_bf16((B, Hq, D), seed + 3, device="cuda"),
             kn=synth.normal_bf16((B, Hkv, D), seed + 4, device="cuda"),
             vn=synth.normal_bf16((B, Hkv, D), seed + 5, device="cuda"),
             rc=np.ones(npg, np.int32))
    if qlens is not None:
        qlens = np.asarray(qlens, np.int32)
        nqb = qlens // 32
        qt, nq = synth.block_tables_from_permutation(np.maximum(nqb, 1), seed + 6)
        i8 = phs.Int8Pool.empty(nq, Hkv, D)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        phs.kv_quant_int8_block32(phs.PagedPool(c["k"], c["v"]), dev(bt), i8, dev(qt),
                                  dev(np.zeros(B, np.int32)), dev(nqb), max(int(nqb.max()), 1),
                                  status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        c.update(qlens=qlens, qt=qt, i8=i8)
    return c


def _two_ways(c, tps=0, phases=False):
    """(outputs, statuses, pools) of append-then-decode and of the fused call."""
    outs, sts, pools = [], [], []
    int8 = dict(int8=c["i8"], qtable=dev(c["qt"]), qlens=dev(c["qlens"])) if "i8" in c else {}
    ms = int(c["lens"].max())
    for fused in (False, True):
        pool = phs.PagedPool(c["k"].clone(), c["v"].clone())
        bt, sl, rc = dev(c["bt"]), dev(c["lens"]), dev(c["rc"])
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            app = dict(k_new=c["kn"], v_new=c["vn"], page_refcount=rc)
        else:
            app = {}
            phs.kv_append_paged(pool, c["kn"], c["vn"], bt, sl, page_refcount=rc, status=st)
        scale = 1 / math.sqrt(c["D"])
        if phases:
            ws = torch.empty(phs.decode_workspace_bytes(c["B"], c["Hq"], c["Hkv"], c["D"], ms, tps,
                                                        bool(int8)),
                             dtype=torch.uint8, device="cuda")
            out = torch.empty((c["B"], c["Hq"], c["D"]), dtype=torch.float32, device="cuda")
            phs.attn_decode_full_paged_split(c["q"], pool, bt, sl, ms, ws, out, softmax_scale=scale,
                                             tokens_per_split=tps, status=st, **int8, **app)
            phs.attn_merge_splits(out, c["Hkv"], sl, ms, ws, qlens=int8.get("qlens"),
                                  has_int8=bool(int8), tokens_per_split=tps)
        else:
            out = phs.attn_decode_full_paged(c["q"], pool, bt, sl, ms, softmax_scale=scale,
                                             tokens_per_split=tps, out_dtype=torch.float32,
                                             status=st, **int8, **app)
        torch.cuda.synchronize()
        outs.append(out_np(out))
        sts.append(int(st.item()))
        pools.append(pool)
    return outs, sts, pools


def _same(outs, pools):
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(pools[0].k, pools[1].k) and torch.equal(pools[0].v, pools[1].v)


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 8, 1), (128, 24, 4), (128, 32, 2)])
@pytest.mark.parametrize("tps", [0, 256])
@pytest.mark.parametrize("phases", [False, True])
def test_fused_append_equals_append_then_decode(D, Hq, Hkv, tps, phases):
    # new tokens at the first and the last slot of a page, in between, and
    # in the last of several splits
    c = _case([1, 16, 17, 32, 100, 2048, 2049, 5000], Hq, Hkv, D, seed=70 + D + Hq + tps)
    outs, sts, pools = _two_ways(c, tps, phases)
    assert sts == [0, 0]
    _same(outs, pools)
    if not phases and tps == 0:
        kp, vp = synth.bits(pools[1].k), synth.bits(pools[1].v)
        ref, s = oracle.decode_full_paged(synth.bits(c["q"]), kp, vp, c["bt"], c["lens"],
                                          1 / math.sqrt(D))
        assert s == 0
        assert_close(outs[1], ref, "fused append vs oracle")


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 32, 2)])
def test_fused_append_single_wave(D, Hq, Hkv):
    # short requests: one split each, a grid of at most one CTA per SM (8
    # warps per CTA); the new token at the first, a middle and the last slot
    # of its page
    c = _case([1, 16, 17, 100, 200, 256], Hq, Hkv, D, seed=90 + D)
    outs, sts, pools = _two_ways(c)
    assert sts == [0, 0]
    _same(outs, pools)
    kp, vp = synth.bits(pools[1].k), synth.bits(pools[1].v)
    ref, s = oracle.decode_full_paged(synth.bits(c["q"]), kp, vp, c["bt"], c["lens"],
                                      1 / math.sqrt(D))
    assert s == 0
    assert_close(outs[1], ref, "single-wave fused append vs oracle")


@pytest.mark.parametrize("tps", [0, 512])
def test_fused_append_with_int8_region(tps):
    # INT8 below qlens, the new token in the bf16 tail
    c = _case([1100, 2100, 5000, 64], 32, 8, 128, seed=81, qlens=[64, 1024, 3968, 32])
    outs, sts, pools = _two_ways(c, tps)
    assert sts == [0, 0]
    _same(outs, pools)


def test_fused_append_refuses_shared_page_and_int8_region():
    """Request 1's newest page has a reference count of 2: not written,
    PHS_ESHARED both ways, same outputs and pools.  Request 2's new token
    lies inside its INT8 region (qlens = seq_lens): the fused call writes
    nothing and records PHS_ERANGE, and attends the token's INT8 code, as
    the unfused call does (which wrote the unread bf16 page)."""
    c = _case([700, 900, 1024, 300], 32, 8, 128, seed=85)
    page = int(c["bt"][1, (900 - 1) // 16])
    c["rc"][page] = 2
    outs, sts, pools = _two_ways(c)
    assert sts == [-4, -4]
    _same(outs, pools)
    c = _case([700, 900, 1024, 300], 32, 8, 128, seed=86, qlens=[64, 512, 1024, 0])
    page = int(c["bt"][2, (1024 - 1) // 16])
    before = c["k"][page].clone()
    outs, sts, pools = _two_ways(c)
    assert sts == [0, -3]
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(pools[1].k[page], before)
