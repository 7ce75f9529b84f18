"""The no-allocation decode entry point, for callers that cannot give the
library a workspace (a host framework that owns all device memory, an
engine that has reserved nearly all of HBM for its KV pool, a decode loop
that must not call cudaMalloc).  It must give the same results as the
workspace-taking entry point, call after call, and refuse requests that do
not fit its built-in scratch before launching anything.

This file is collected last so that a run stopping at the first failure
has already run every other test."""
import math

import numpy as np
import pytest
import torch

import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, dev, out_np

pytestmark = pytest.mark.gpu


def _case(seed, lens, Hq=32, Hkv=8, D=128):
    lens = np.asarray(lens, np.int32)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(lens), seed)
    pool = phs.PagedPool(synth.normal_bf16((npg, Hkv, 16, D), seed + 1, device="cuda"),
                         synth.normal_bf16((npg, Hkv, 16, D), seed + 2, device="cuda"))
    q = synth.normal_bf16((len(lens), Hq, D), seed + 3, device="cuda")
    return pool, q, dev(bt), dev(lens), int(lens.max())


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [_case(71, [1, 17, 900, 5000, 32769, 2048]), _case(72, [3000, 12, 7000])]
    for pool, q, bt, sl, ms in cases:   # two calls in a row, different inputs
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = phs.attn_decode_full_paged(q, pool, bt, sl, ms, out_dtype=torch.float32, status=st)
        out = torch.full_like(ref, float("nan"))
        phs.attn_decode_full_paged_noalloc(q, pool, bt, sl, ms, out, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_close(out_np(out), out_np(ref), "no-allocation vs workspace entry point")


def test_noalloc_lengthens_splits_to_fit_and_rejects_beyond_scratch():
    # two requests of one KV head with 16 query heads and a stated bound of
    # 600,000 tokens: for so small a grid the library's split length is short
    # (256 tokens on 152 SMs) and its partials (39 MB) do not fit the 32 MiB
    # scratch, so the call must lengthen its splits and still match the
    # workspace path
    Hq, Hkv, D, bound = 16, 1, 128, 600_000
    pool, q, bt, sl, _ = _case(73, [3000, 7001], Hq=Hq, Hkv=Hkv, D=D)
    assert phs.decode_workspace_bytes(2, Hq, Hkv, D, bound) > phs.NOALLOC_SCRATCH_BYTES
    out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.attn_decode_full_paged_noalloc(q, pool, bt, sl, bound, out, status=st)
    ref = phs.attn_decode_full_paged(q, pool, bt, sl, bound, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out_np(out), out_np(ref), "lengthened splits")
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
