"""GPU parity of the shared-prefix decode (tensor-core pass over the shared
prefix for all requests + split-KV over each request's own tokens + merge)
against the fp64 oracle and against the per-request decode path."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, dev, out_np, sub_pool

pytestmark = pytest.mark.gpu


def _shared_case(B, Hq, Hkv, shared_len, suffixes, seed, D=128):
    """Block tables: the same shared_len/16 prefix pages first, then each
    request's own pages; page ids from one seeded permutation."""
    npref = shared_len // 16
    own = [(s + 15) // 16 for s in suffixes]
    total = npref + sum(own) + 2
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    width = npref + max(max(own), 1)
    bt = np.full((B, width), -1, np.int32)
    o = npref
    for b in range(B):
        bt[b, :npref] = perm[:npref]
        bt[b, npref:npref + own[b]] = perm[o:o + own[b]]
        o += own[b]
    lens = np.array([shared_len + s for s in suffixes], np.int32)
    pool = phs.PagedPool(synth.normal_bf16((total, Hkv, 16, D), seed + 1, device="cuda"),
                         synth.normal_bf16((total, Hkv, 16, D), seed + 2, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), seed + 3, device="cuda")
    return pool, q, bt, lens


def _oracle_rows(pool, q, bt, lens, rows, D=128):
    used = np.unique(bt[rows][bt[rows] >= 0])
    remap = np.full(bt.max() + 1, -1, np.int64)
    remap[used] = np.arange(len(used))
    bt_s = np.where(bt[rows] >= 0, remap[np.maximum(bt[rows], 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    hk, hv = synth.bits(pool.k.index_select(0, idx)), synth.bits(pool.v.index_select(0, idx))
    ref, st = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, lens[rows],
                                       1 / math.sqrt(D))
    assert st == 0
    return ref


@pytest.mark.parametrize("B,Hq,Hkv,shared_len,seed,max_suffix", [
    (2, 32, 8, 64, 1, 700),        # one tile, 8 rows per head
    (8, 32, 8, 1024, 2, 700),      # 16 tiles, 32 rows
    (64, 32, 8, 4096, 3, 700),     # 256 rows: both 128-row tiles full
    (5, 16, 2, 2048, 4, 700),      # G = 8, 40 rows
    (33, 32, 8, 640, 5, 700),      # rows 132: second tile partly used
    (16, 32, 2, 512, 6, 700),      # G = 16, 256 rows
    (6, 32, 8, 256, 7, 5000),      # own tokens over several splits: merged with the prefix
    (64, 8, 8, 1024, 8, 700),      # G = 1: one row per request and KV head, 64 rows
    (40, 32, 8, 2368, 9, 700),     # 37 halves: a partial last S tile; rows 160
])
def test_shared_prefix_matches_oracle_and_paged_path(B, Hq, Hkv, shared_len, seed, max_suffix):
    rng = np.random.default_rng(seed)
    suffixes = [int(x) for x in rng.integers(0, max_suffix, size=B)]
    suffixes[0] = 0                  # a request with no tokens of its own
    pool, q, bt, lens = _shared_case(B, Hq, Hkv, shared_len, suffixes, seed)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), shared_len,
                                        out_dtype=torch.float32, status=st)
    ref_gpu = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), int(lens.max()),
                                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out_np(out)
    rows = sorted(set([0, B - 1, B // 2]))
    assert_close(got[rows], _oracle_rows(pool, q, bt, lens, rows), f"B={B} shared={shared_len}")
    assert_close(got, out_np(ref_gpu), "vs per-request decode")
    # bf16 output is the fp32 result rounded once: bit for bit
    out16 = phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), shared_len,
                                          out_dtype=torch.bfloat16, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out16, out.to(torch.bfloat16))


def test_shared_prefix_rejects_bad_shapes():
    pool, q, bt, lens = _shared_case(2, 32, 8, 128, [5, 9], 7)
    with pytest.raises(phs.PhsError) as e:          # not a multiple of 64
        phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), 96)
    assert e.value.code == -7
    big_q = synth.normal_bf16((65, 32, 128), 1, device="cuda")   # 260 rows > 256
    bt65 = np.tile(bt[:1], (65, 1))
    with pytest.raises(phs.PhsError) as e:
        phs.attn_decode_shared_prefix(big_q, pool, dev(bt65), dev(np.full(65, 133, np.int32)),
                                      133, 128)
    assert e.value.code == -7


@pytest.mark.slow
def test_shared_prefix_full_size_sampled():
    """The 250,000-token shared prefix of 64 requests (+512-token suffixes):
    the tensor-core pass covers 249,984 tokens, the split kernel the rest."""
    w = synth.shared_prefix()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    pool = phs.PagedPool(synth.normal_bf16((w.num_pages, Hkv, 16, D), 51, device="cuda"),
                         synth.normal_bf16((w.num_pages, Hkv, 16, D), 52, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), 53, device="cuda")
    n = (w.n_pre + 1).astype(np.int32)
    shared = (250_000 // 64) * 64
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_shared_prefix(q, pool, dev(w.block_table), dev(n), int(n.max()), shared,
                                        out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = [0, B - 1]
    assert_close(out_np(out)[rows], _oracle_rows(pool, q, w.block_table, n, rows), "config 5")


def test_shared_prefix_checks_every_row_against_row_0():
    """The prefix pass reads row 0's page ids for everyone.  A request whose
    table does not begin with them (one prefix id replaced by another valid
    page of the pool), or that is shorter than the shared prefix, is
    flagged on the device: PHS_ESHAPE in the status word, an all-zero
    output row, and every other row as the oracle gives it."""
    B, Hq, Hkv, shared_len = 8, 32, 8, 1024
    rng = np.random.default_rng(31)
    suffixes = [int(x) for x in rng.integers(1, 700, size=B)]
    pool, q, bt, lens = _shared_case(B, Hq, Hkv, shared_len, suffixes, 31)
    used = set(bt[bt >= 0].ravel().tolist())  # _shared_case leaves two pages unused
    spare = next(i for i in range(pool.k.shape[0]) if i not in used)
    bad_row, short_row = 3, 5
    bt[bad_row, 17] = spare
    lens[short_row] = shared_len - 10
    for out_dtype in (torch.float32, torch.bfloat16):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((B, Hq, 128), float("nan"), dtype=out_dtype, device="cuda")
        phs.attn_decode_shared_prefix(q, pool, dev(bt), dev(lens), int(lens.max()), shared_len,
                                      out=out, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == -2  # PHS_ESHAPE
        got = out_np(out)
        assert np.all(got[bad_row] == 0) and np.all(got[short_row] == 0)
        good = [b for b in range(B) if b not in (bad_row, short_row)]
        assert_close(got[good], _oracle_rows(pool, q, bt, lens, good), "unflagged rows")


def _prefix_steps(B, Hq, Hkv, shared_len, suffix, steps, seed, rows, D=128, fused=False):
    """The decode loop of a batch sharing a prefix: each step appends every
    request's new token (page reference counts checked) and decodes through
    the shared-prefix call (fused: one call that also appends); sampled rows
    are checked against the oracle at every step, on a host copy of their
    pages that the oracle appends to."""
    npref = shared_len // 16
    own = (suffix + steps + 15) // 16
    total = npref + B * own
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    bt = np.empty((B, npref + own), np.int32)
    bt[:, :npref] = perm[:npref]
    for b in range(B):
        bt[b, npref:] = perm[npref + b * own:npref + (b + 1) * own]
    rc = np.ones(total, np.int32)
    rc[perm[:npref]] = B
    kp = synth.normal_bf16((total, Hkv, 16, D), seed + 1, device="cuda")
    vp = synth.normal_bf16((total, Hkv, 16, D), seed + 2, device="cuda")
    pool = phs.PagedPool(kp, vp)
    n_pre = np.full(B, shared_len + suffix, np.int32)
    n_final = n_pre + steps
    hk, bt_s = sub_pool(kp, bt, rows, n_final)
    hv, _ = sub_pool(vp, bt, rows, n_final)
    bt_d, rc_d = dev(bt), dev(rc)
    max_seq = int(n_final.max())
    ws = torch.empty(phs.shared_prefix_workspace_bytes(B, Hq, Hkv, D, max_seq, shared_len),
                     dtype=torch.uint8, device="cuda")
    for k in range(steps):
        n_after = (n_pre + 1 + k).astype(np.int32)
        q = synth.normal_bf16((B, Hq, D), seed + 10 + 3 * k, device="cuda")
        kn = synth.normal_bf16((B, Hkv, D), seed + 11 + 3 * k, device="cuda")
        vn = synth.normal_bf16((B, Hkv, D), seed + 12 + 3 * k, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        sl = dev(n_after)
        if fused:
            kw = dict(k_new=kn, v_new=vn, page_refcount=rc_d)
        else:
            kw = {}
            phs.kv_append_paged(pool, kn, vn, bt_d, sl, page_refcount=rc_d, status=st)
        out = phs.attn_decode_shared_prefix(q, pool, bt_d, sl, max_seq, shared_len,
                                            out_dtype=torch.float32, workspace=ws, status=st,
                                            **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, k
        assert oracle.append_paged(hk, hv, synth.bits(kn)[rows], synth.bits(vn)[rows], bt_s,
                                   n_after[rows]) == 0
        ref, s = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, n_after[rows],
                                          1 / math.sqrt(D))
        assert s == 0
        assert_close(out_np(out)[rows], ref, f"step {k}")


@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_decode_steps_with_append(fused):
    # 64 requests x 8 KV heads (256 query rows per head), suffixes crossing a
    # page boundary during the walk (suffix 505 + 12 steps passes 512)
    _prefix_steps(B=64, Hq=32, Hkv=8, shared_len=4096, suffix=505, steps=12, seed=900,
                  rows=[0, 17, 63], fused=fused)


@pytest.mark.slow
def test_shared_prefix_full_size_steps_with_append():
    """The shared-prefix workload's loop at full size: one 250,000-token
    prefix shared by 64 requests with 512-token suffixes; the bench's one
    call per step (the append fused into the prefix decode) over 4 steps,
    two sampled requests against the oracle each step (the tensor-core pass
    covers the prefix's whole 64-token tiles, 249,984 tokens; the split
    kernel the remaining 16 and the suffix)."""
    w = synth.shared_prefix()
    assert w.extra["prefix_pages"] * 16 == 250_000
    _prefix_steps_full(w, steps=4, rows=[0, w.B - 1])


def _prefix_steps_full(w, steps, rows):
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    kp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 951, device="cuda")
    vp = synth.normal_bf16((w.num_pages, Hkv, 16, D), 952, device="cuda")
    pool = phs.PagedPool(kp, vp)
    n_final = w.n_pre + steps
    hk, bt_s = sub_pool(kp, w.block_table, rows, n_final)
    hv, _ = sub_pool(vp, w.block_table, rows, n_final)
    bt, rcd = dev(w.block_table), dev(w.extra["refcount"])
    shared = (w.extra["prefix_pages"] * 16 // 64) * 64
    max_seq = int(w.n_pre.max()) + w.extra["steps"]
    ws = torch.empty(phs.shared_prefix_workspace_bytes(B, Hq, Hkv, D, max_seq, shared),
                     dtype=torch.uint8, device="cuda")
    for k in range(steps):
        n_after = (w.n_pre + 1 + k).astype(np.int32)
        q = synth.normal_bf16((B, Hq, D), 960 + 3 * k, device="cuda")
        kn = synth.normal_bf16((B, Hkv, D), 961 + 3 * k, device="cuda")
        vn = synth.normal_bf16((B, Hkv, D), 962 + 3 * k, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        sl = dev(n_after)
        out = phs.attn_decode_shared_prefix(q, pool, bt, sl, max_seq, shared,
                                            out_dtype=torch.float32, workspace=ws, status=st,
                                            k_new=kn, v_new=vn, page_refcount=rcd)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, k
        assert oracle.append_paged(hk, hv, synth.bits(kn)[rows], synth.bits(vn)[rows], bt_s,
                                   n_after[rows]) == 0
        ref, s = oracle.decode_full_paged(synth.bits(q)[rows], hk, hv, bt_s, n_after[rows],
                                          w.softmax_scale)
        assert s == 0
        assert_close(out_np(out)[rows], ref, f"config 5 prefix path, step {k}")


def _fused_vs_unfused(B, Hq, Hkv, shared_len, suffixes, seed, rc_override=None, lens_override=None):
    """One step both ways on identical pools: kv_append_paged then the
    shared-prefix call, and the call with the append fused in.  Returns
    (outputs, statuses, pools) of the two, and the case."""
    pool, q, bt, lens = _shared_case(B, Hq, Hkv, shared_len, suffixes, seed)
    if lens_override:
        for b, n in lens_override.items():
            lens[b] = n
    rc = np.ones(pool.k.shape[0], np.int32)
    rc[bt[0, :shared_len // 16]] = B
    for page, count in (rc_override or {}).items():
        rc[page] = count
    kn = synth.normal_bf16((B, Hkv, 128), seed + 20, device="cuda")
    vn = synth.normal_bf16((B, Hkv, 128), seed + 21, device="cuda")
    pools = [phs.PagedPool(pool.k.clone(), pool.v.clone()) for _ in range(2)]
    bt_d, sl, rc_d = dev(bt), dev(lens), dev(rc)
    outs, sts = [], []
    for fused, p in zip((False, True), pools):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if not fused:
            phs.kv_append_paged(p, kn, vn, bt_d, sl, page_refcount=rc_d, status=st)
        kw = dict(k_new=kn, v_new=vn, page_refcount=rc_d) if fused else {}
        out = phs.attn_decode_shared_prefix(q, p, bt_d, sl, int(lens.max()), shared_len,
                                            out_dtype=torch.float32, status=st, **kw)
        torch.cuda.synchronize()
        outs.append(out_np(out))
        sts.append(int(st.item()))
    return outs, sts, pools, (pool, q, bt, lens, kn, vn)


def test_shared_prefix_fused_append_equals_append_then_decode():
    """The append fused into the shared-prefix call (the own-token split
    writes each new token and attends it from the input) gives the
    unfused result bit for bit: outputs and pools.  The suffixes put the
    new token at the first and the last slot of a page and in between."""
    B, Hq, Hkv, shared_len = 16, 32, 8, 1024
    suffixes = [1, 16, 17, 32, 100, 511, 512, 513, 7, 640, 3, 255, 256, 257, 48, 49]
    outs, sts, pools, (pool, q, bt, lens, _, _) = _fused_vs_unfused(B, Hq, Hkv, shared_len,
                                                                    suffixes, 41)
    assert sts == [0, 0]
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(pools[0].k, pools[1].k) and torch.equal(pools[0].v, pools[1].v)
    rows = [0, 6, 9, 15]
    assert_close(outs[1][rows], _oracle_rows(pools[1], q, bt, lens, rows), "fused vs oracle")


def test_shared_prefix_fused_append_refuses_shared_pages():
    """A request whose newest page has a reference count of 2, and one whose
    new token would fall inside the shared prefix (seq_lens == shared_len):
    neither page is written, PHS_ESHARED is recorded, and both ways give the
    same outputs and pools (the refused tokens attended as the pages hold
    them)."""
    B, Hq, Hkv, shared_len = 8, 32, 8, 512
    suffixes = [40, 70, 33, 90, 16, 120, 64, 5]
    pool, _, bt, lens = _shared_case(B, Hq, Hkv, shared_len, suffixes, 43)
    shared_row, at_prefix = 2, 5
    page = int(bt[shared_row, (lens[shared_row] - 1) // 16])
    before = pool.k[page].clone()
    outs, sts, pools, _ = _fused_vs_unfused(B, Hq, Hkv, shared_len, suffixes, 43,
                                            rc_override={page: 2},
                                            lens_override={at_prefix: shared_len})
    assert sts == [-4, -4]  # PHS_ESHARED both ways
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(pools[0].k, pools[1].k) and torch.equal(pools[0].v, pools[1].v)
    assert torch.equal(pools[1].k[page], before)
