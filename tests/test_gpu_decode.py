"""GPU parity: split-KV paged decode, SWA ring decode and the INT8 variant
against the fp64 CPU oracle, at sizes that span several splits, chunks and
ragged tails; plus the layout invariances (page permutation, shared
prefix) that must hold bit for bit on the GPU."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import assert_close, bf16_dev, dev, out_np

pytestmark = pytest.mark.gpu


def paged_case(lens, Hq, Hkv, D, seed, spare=4):
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(np.maximum(lens, 1)), seed)
    npg += spare
    kp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), seed + 1))
    vp = synth.bits(synth.normal_bf16((npg, Hkv, 16, D), seed + 2))
    q = synth.bits(synth.normal_bf16((B, Hq, D), seed + 3))
    return dict(lens=lens, bt=bt, kp=kp, vp=vp, q=q, B=B, Hq=Hq, Hkv=Hkv, D=D)


def run_full(c, out_dtype=torch.float32, tps=0, pool=None):
    pool = pool or phs.PagedPool(bf16_dev(c["kp"]), bf16_dev(c["vp"]))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_full_paged(bf16_dev(c["q"]), pool, dev(c["bt"]), dev(c["lens"]),
                                     int(c["lens"].max()), softmax_scale=1 / math.sqrt(c["D"]),
                                     tokens_per_split=tps, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, int(st.item())
    return out_np(out)


def ref_full(c):
    out, s = oracle.decode_full_paged(c["q"], c["kp"], c["vp"], c["bt"], c["lens"],
                                      1 / math.sqrt(c["D"]))
    assert s == 0
    return out


RAGGED = [1, 15, 16, 17, 100, 1000, 2049, 5000]


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 4, 2), (128, 8, 1), (128, 16, 2),
                                      (64, 32, 2), (128, 8, 8), (64, 2, 2)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_full_decode_ragged(D, Hq, Hkv, out_dtype):
    c = paged_case(RAGGED, Hq, Hkv, D, seed=100 + D + Hq)
    got = run_full(c, out_dtype)
    assert_close(got, ref_full(c), f"D={D} G={Hq // Hkv} {out_dtype}")


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 32, 2), (128, 24, 4), (64, 4, 2)])
def test_full_decode_single_wave_eight_warps(D, Hq, Hkv):
    # a grid of at most one CTA per SM runs 8 warps per CTA: short requests
    # (one 256-token split each), and longer ones in one explicit long split
    c = paged_case([1, 16, 17, 100, 200, 256], Hq, Hkv, D, seed=300 + D + Hq)
    assert_close(run_full(c), ref_full(c), f"short D={D} G={Hq // Hkv}")
    c = paged_case([300, 1000, 2049], Hq, Hkv, D, seed=310 + D + Hq)
    assert_close(run_full(c, tps=4096), ref_full(c), f"long D={D} G={Hq // Hkv}")


@pytest.mark.parametrize("tps", [32, 64, 256, 1024, 4096])
def test_full_decode_any_split(tps):
    c = paged_case([3, 64, 700, 3000, 4096], 32, 8, 128, seed=7)
    got = run_full(c, tps=tps)
    assert_close(got, ref_full(c), f"tokens_per_split={tps}")


def test_full_decode_empty_request_gives_zero():
    c = paged_case([0, 40, 0, 17], 8, 2, 64, seed=9)
    got = run_full(c)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = ref_full(c)
    assert_close(got[[1, 3]], ref[[1, 3]], "non-empty rows")


def test_full_decode_page_permutation_bit_identical():
    c = paged_case([37, 500, 1500], 32, 8, 128, seed=13, spare=11)
    npg = c["kp"].shape[0]
    perm = np.random.default_rng(3).permutation(npg).astype(np.int32)
    inv = np.argsort(perm)
    c2 = dict(c)
    c2["bt"] = np.where(c["bt"] >= 0, perm[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    c2["kp"] = np.ascontiguousarray(c["kp"][inv])
    c2["vp"] = np.ascontiguousarray(c["vp"][inv])
    a = run_full(c, tps=256)
    b = run_full(c2, tps=256)
    assert np.array_equal(a, b)
    assert_close(a, ref_full(c), "permuted pages")


def test_full_decode_shared_prefix_bit_identical():
    # 6 requests: one shared 1024-token prefix + identical 40-token suffixes,
    # once through shared page ids (refcount 6), once through private copies
    Hq, Hkv, D, B = 32, 8, 128, 6
    pre, suf = 1024, 40
    kd = synth.bits(synth.normal_bf16((Hkv, pre + suf, D), 21))
    vd = synth.bits(synth.normal_bf16((Hkv, pre + suf, D), 22))
    q1 = synth.bits(synth.normal_bf16((1, Hq, D), 23))
    q = np.repeat(q1, B, axis=0)
    from paging import dense_to_paged
    npre, nsuf = pre // 16, (suf + 15) // 16
    shared = np.arange(npre, dtype=np.int32)
    bt_sh = np.concatenate([np.tile(shared, (B, 1)),
                            npre + np.arange(B * nsuf, dtype=np.int32).reshape(B, nsuf)], axis=1)
    bt_pr = np.arange(B * (npre + nsuf), dtype=np.int32).reshape(B, -1)
    lens = np.full(B, pre + suf, np.int32)
    c_sh = dict(lens=lens, bt=bt_sh, q=q, D=D, kp=dense_to_paged([kd] * B, bt_sh, bt_sh.max() + 1),
                vp=dense_to_paged([vd] * B, bt_sh, bt_sh.max() + 1))
    c_pr = dict(lens=lens, bt=bt_pr, q=q, D=D, kp=dense_to_paged([kd] * B, bt_pr, bt_pr.max() + 1),
                vp=dense_to_paged([vd] * B, bt_pr, bt_pr.max() + 1))
    a = run_full(c_sh, tps=256)
    b = run_full(c_pr, tps=256)
    assert np.array_equal(a, b)
    for i in range(1, B):
        assert np.array_equal(a[0], a[i])
    assert_close(a, ref_full(c_pr), "shared prefix")


# ------------------------------------------------------------------ ring --
def ring_case(lens, W, Hq, Hkv, D, seed):
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    nr = B + 3
    kr = synth.bits(synth.normal_bf16((nr, Hkv, W, D), seed + 1))
    vr = synth.bits(synth.normal_bf16((nr, Hkv, W, D), seed + 2))
    q = synth.bits(synth.normal_bf16((B, Hq, D), seed + 3))
    ids = np.random.default_rng(seed).permutation(nr)[:B].astype(np.int32)
    pos = synth.ring_positions(B, W, seed + 4)
    return dict(lens=lens, kr=kr, vr=vr, q=q, ids=ids, pos=pos, D=D)


@pytest.mark.parametrize("W", [16, 128, 1024])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 4, 2), (128, 32, 2), (128, 8, 8)])
def test_swa_ring_decode(W, D, Hq, Hkv):
    lens = [1, 5, W - 1, W, W + 1, 3 * W + 7, 40000]
    c = ring_case(lens, W, Hq, Hkv, D, seed=W + D)
    ring = phs.RingPool(bf16_dev(c["kr"]), bf16_dev(c["vr"]))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_swa_ring(bf16_dev(c["q"]), ring, dev(c["pos"]), dev(c["lens"]),
                                   ring_ids=dev(c["ids"]), softmax_scale=1 / math.sqrt(D),
                                   out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, s = oracle.decode_swa_ring(c["q"], c["kr"], c["vr"], c["ids"], c["pos"], c["lens"],
                                    1 / math.sqrt(D))
    assert s == 0
    assert_close(out_np(out), ref, f"W={W} D={D}")


@pytest.mark.parametrize("B", [4, 300, 700, 7200])
def test_swa_ring_decode_launch_shapes(B):
    # the SWA launch picks its shape from the work: one CTA per (request, KV
    # head) unit with its chunks spread over 4 warps when every unit has an
    # SM of its own (4 units), 4 warps x 4 stages when every unit has a warp
    # of its own in one wave (300), and 8 persistent warps x 2 stages for
    # many units (700, 7200)
    W, D, Hq, Hkv = 16, 128, 4, 1
    lens = np.random.default_rng(B).integers(1, 3 * W, B).astype(np.int32)
    c = ring_case(lens, W, Hq, Hkv, D, seed=B)
    ring = phs.RingPool(bf16_dev(c["kr"]), bf16_dev(c["vr"]))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_swa_ring(bf16_dev(c["q"]), ring, dev(c["pos"]), dev(c["lens"]),
                                   ring_ids=dev(c["ids"]), softmax_scale=1 / math.sqrt(D),
                                   out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, s = oracle.decode_swa_ring(c["q"], c["kr"], c["vr"], c["ids"], c["pos"], c["lens"],
                                    1 / math.sqrt(D))
    assert s == 0
    assert_close(out_np(out), ref, f"B={B}")


def test_swa_ring_empty_request_gives_zero():
    W, D, Hq, Hkv = 16, 128, 8, 2
    c = ring_case([0, 1, 17, 0], W, Hq, Hkv, D, seed=55)
    ring = phs.RingPool(bf16_dev(c["kr"]), bf16_dev(c["vr"]))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = phs.attn_decode_swa_ring(bf16_dev(c["q"]), ring, dev(c["pos"]), dev(c["lens"]),
                                   ring_ids=dev(c["ids"]), softmax_scale=1 / math.sqrt(D),
                                   out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out_np(out)
    assert not got[0].any() and not got[3].any()
    ref, s = oracle.decode_swa_ring(c["q"], c["kr"], c["vr"], c["ids"], c["pos"], c["lens"],
                                    1 / math.sqrt(D))
    assert s == 0
    assert_close(got, ref, "empty SWA requests")


# ------------------------------------------------------------------ INT8 --
def int8_case(lens, qlens, Hq, Hkv, D, seed):
    """bf16 pages over the whole sequence; INT8 pages for tokens < qlen,
    produced by the oracle's quantiser (and checked against the GPU's)."""
    c = paged_case(lens, Hq, Hkv, D, seed)
    for name in ("kp", "vp"):
        c[name] = synth.bits(synth.normal_bf16(c[name].shape, seed + (7 if name == "kp" else 8),
                                               outlier_p=0.01))
    qlens = np.asarray(qlens, np.int32)
    nqb = qlens // 32
    qt, nq = synth.block_tables_from_permutation(np.maximum(nqb, 1), seed + 5)
    nq += 2
    kc = np.zeros((nq, Hkv, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nq, Hkv), np.float32)
    vs = np.zeros_like(ks)
    first = np.zeros(len(lens), np.int32)
    assert oracle.quant_int8_block32(c["kp"], c["vp"], c["bt"], kc, vc, ks, vs, qt, first,
                                     nqb) == 0
    c.update(qlens=qlens, nqb=nqb, qt=qt, nq=nq, kc=kc, vc=vc, ks=ks, vs=vs)
    return c


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 8, 2), (128, 32, 2), (128, 8, 8),
                                     (128, 24, 4), (64, 20, 2)])
@pytest.mark.parametrize("tps", [0, 64, 256])
def test_int8_decode(D, Hq, Hkv, tps):
    lens = [33, 1100, 2100, 1056, 5000, 40]
    qlens = [0, 64, 1024, 32, 3968, 32]
    c = int8_case(lens, qlens, Hq, Hkv, D, seed=300 + D + Hq)
    src = phs.PagedPool(bf16_dev(c["kp"]), bf16_dev(c["vp"]))
    i8 = phs.Int8Pool.empty(c["nq"], Hkv, D)
    for t in (i8.k, i8.v):
        t.fill_(128)  # the stored form of code 0
    for t in (i8.k_scale, i8.v_scale):
        t.zero_()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    phs.kv_quant_int8_block32(src, dev(c["bt"]), i8, dev(c["qt"]),
                              dev(np.zeros(len(lens), np.int32)), dev(c["nqb"]),
                              int(c["nqb"].max()), status=st)
    torch.cuda.synchronize()
    gk, gv = i8.codes()
    assert np.array_equal(gk.cpu().numpy(), c["kc"]) and np.array_equal(gv.cpu().numpy(), c["vc"])
    assert np.array_equal(i8.k_scale.cpu().numpy(), c["ks"])
    # the bf16 copy of the INT8 region is not read by decode: scribble on it
    for b, ql in enumerate(c["qlens"]):
        for p in c["bt"][b, :ql // 16]:
            src.k[int(p)].fill_(float("nan"))
            src.v[int(p)].fill_(float("nan"))
    out = phs.attn_decode_full_paged(bf16_dev(c["q"]), src, dev(c["bt"]), dev(c["lens"]),
                                     int(max(lens)), softmax_scale=1 / math.sqrt(D), int8=i8,
                                     qtable=dev(c["qt"]), qlens=dev(c["qlens"]),
                                     tokens_per_split=tps, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, s = oracle.decode_full_paged(
        c["q"], c["kp"], c["vp"], c["bt"], c["lens"], 1 / math.sqrt(D),
        int8=dict(k_codes=c["kc"], v_codes=c["vc"], k_scale=c["ks"], v_scale=c["vs"],
                  qtable=c["qt"], qlens=c["qlens"]))
    assert s == 0
    assert_close(out_np(out), ref, f"int8 D={D} tps={tps}")


# ---------------------------------------------------------- split phases --
def test_split_and_merge_entry_points_match_composed_call():
    c = paged_case([900, 3000, 17, 2500], 32, 8, 128, seed=41)
    pool = phs.PagedPool(bf16_dev(c["kp"]), bf16_dev(c["vp"]))
    q, bt, sl = bf16_dev(c["q"]), dev(c["bt"]), dev(c["lens"])
    ms = int(c["lens"].max())
    ws = torch.empty(phs.decode_workspace_bytes(4, 32, 8, 128, ms, 256), dtype=torch.uint8,
                     device="cuda")
    out1 = torch.empty((4, 32, 128), dtype=torch.float32, device="cuda")
    phs.attn_decode_full_paged_split(q, pool, bt, sl, ms, ws, out1, tokens_per_split=256)
    phs.attn_merge_splits(out1, 8, sl, ms, ws, tokens_per_split=256)
    out2 = phs.attn_decode_full_paged(q, pool, bt, sl, ms, tokens_per_split=256,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    assert_close(out_np(out1), ref_full(c), "split+merge")


# ------------------------------------------------------------ split plan --
def test_split_length_planner():
    # 256 when the longest request has 129..256 tokens and batch x KV heads
    # fits the SMs (one split each); else the longest of 4096, 2048, ..., 128
    # tokens that gives the longest request at least 8 splits and whose grid
    # (batch x KV heads x splits of the longest request) still has 16 CTAs
    # per SM, else 128; an explicit length is kept; the workspace follows
    # the chosen length
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def rule(B, Hkv, n):
        if 128 < n <= 256 and B * Hkv <= sms:
            return 256  # one split per request: no merge after the decode
        t = 4096
        while t > 128 and 8 * t > n:
            t //= 2
        while t > 128 and B * Hkv * -(-n // t) < 16 * sms:
            t //= 2
        return t

    for B, Hkv, n in [(64, 8, 32769), (32, 8, 65537), (256, 8, 131073), (2, 1, 600_000),
                      (1, 1, 100), (8, 8, 8000), (2, 2, 201), (2, 2, 128), (2, 2, 257),
                      (64, 8, 200)]:
        t = phs.decode_tokens_per_split(B, Hkv, n)
        assert t == rule(B, Hkv, n), (B, Hkv, n)
        ws = phs.decode_workspace_bytes(B, 4 * Hkv, Hkv, 128, n)
        assert ws == phs.decode_workspace_bytes(B, 4 * Hkv, Hkv, 128, n, t)
    assert phs.decode_tokens_per_split(64, 8, 32769, 512) == 512
    assert phs.decode_tokens_per_split(64, 8, 32700) == 2048  # the paged batch-64 workload
    assert phs.decode_tokens_per_split(32, 8, 65537) == 4096  # the INT8 workload
