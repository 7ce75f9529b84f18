"""Pins for the CPU oracle, checked against things other than itself:
a library routine on dense inputs, closed forms, invariants stated by the
pages, hand-derived fixtures and brute force on tiny cases.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paging import (bf16_bits_to_f64, dense_to_paged, dense_to_ring, f32_to_bf16_bits,
                    random_bf16, sdpa_reference)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_case(seed, B=3, Hq=8, Hkv=2, D=64, lens=(1, 17, 45), P=16, spare=5):
    rng = np.random.default_rng(seed)
    q = random_bf16(rng, (B, Hq, D))
    k = [random_bf16(rng, (Hkv, n, D)) for n in lens]
    v = [random_bf16(rng, (Hkv, n, D)) for n in lens]
    ppr = [(n + P - 1) // P for n in lens]
    num_pages = sum(ppr) + spare
    perm = rng.permutation(num_pages)
    bt = np.full((B, max(ppr)), -1, np.int32)
    o = 0
    for b, c in enumerate(ppr):
        bt[b, :c] = perm[o:o + c]
        o += c
    return q, k, v, bt, num_pages, np.array(lens, np.int32)


# ---------------------------------------------------------------- decode --
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_full_decode_matches_library_sdpa(seed):
    q, k, v, bt, npg, lens = _random_case(seed)
    kp = dense_to_paged(k, bt, npg)
    vp = dense_to_paged(v, bt, npg)
    scale = 1 / math.sqrt(64)
    out, st = oracle.decode_full_paged(q, kp, vp, bt, lens, scale)
    assert st == 0
    ref = sdpa_reference(q, [bf16_bits_to_f64(x) for x in k], [bf16_bits_to_f64(x) for x in v],
                         scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_full_decode_gqa_grouping_is_contiguous():
    # Hq=4, Hkv=2: q heads 0,1 -> kv head 0; 2,3 -> kv head 1.  Make kv head 1
    # constant V = 5 so heads 2,3 must output exactly 5 and heads 0,1 not.
    rng = np.random.default_rng(3)
    q = random_bf16(rng, (1, 4, 64))
    k = [random_bf16(rng, (2, 20, 64))]
    v = [random_bf16(rng, (2, 20, 64))]
    v[0][1] = f32_to_bf16_bits(np.full((20, 64), 5.0, np.float32))
    bt = np.array([[3, 0]], np.int32)
    kp, vp = dense_to_paged(k, bt, 4), dense_to_paged(v, bt, 4)
    out, st = oracle.decode_full_paged(q, kp, vp, bt, [20], 0.125)
    assert st == 0
    np.testing.assert_allclose(out[0, 2:], 5.0, rtol=0, atol=1e-14)
    assert np.all(np.abs(out[0, :2] - 5.0) > 1.0)


def test_closed_forms():
    rng = np.random.default_rng(7)
    D, n = 64, 40
    bt = np.array([[2, 0, 1]], np.int32)
    v = [random_bf16(rng, (1, n, D))]
    vmean = bf16_bits_to_f64(v[0]).mean(axis=1)
    vp = dense_to_paged(v, bt, 3)
    # all keys equal -> softmax uniform -> output = mean(V)
    k_eq = [np.repeat(random_bf16(rng, (1, 1, D)), n, axis=1)]
    q = random_bf16(rng, (1, 1, D))
    out, _ = oracle.decode_full_paged(q, dense_to_paged(k_eq, bt, 3), vp, bt, [n], 0.3)
    np.testing.assert_allclose(out[0, 0], vmean[0], rtol=0, atol=1e-14)
    # q = 0 -> uniform -> mean(V) for any keys
    k = [random_bf16(rng, (1, n, D))]
    kp = dense_to_paged(k, bt, 3)
    out, _ = oracle.decode_full_paged(np.zeros((1, 1, D), np.uint16), kp, vp, bt, [n], 0.3)
    np.testing.assert_allclose(out[0, 0], vmean[0], rtol=0, atol=1e-14)
    # n = 1 -> output = V[0] exactly
    out, _ = oracle.decode_full_paged(q, kp, vp, bt, [1], 0.3)
    assert np.array_equal(out[0, 0], bf16_bits_to_f64(v[0][0, 0]))
    # one dominant key -> output = that V row
    kd = np.zeros((1, n, D), np.float32)
    kd[0, 23] = 1.0
    qd = f32_to_bf16_bits(np.full((1, 1, D), 8.0, np.float32))
    out, _ = oracle.decode_full_paged(qd, dense_to_paged([f32_to_bf16_bits(kd)], bt, 3), vp, bt,
                                      [n], 1.0)  # score gap 512 -> e^-512 ~ 0
    np.testing.assert_allclose(out[0, 0], bf16_bits_to_f64(v[0][0, 23]), rtol=0, atol=1e-200)


def test_page_permutation_invariance():
    q, k, v, bt, npg, lens = _random_case(11, spare=9)
    out1, _ = oracle.decode_full_paged(q, dense_to_paged(k, bt, npg), dense_to_paged(v, bt, npg),
                                       bt, lens, 0.125)
    perm = np.random.default_rng(5).permutation(npg).astype(np.int32)
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = oracle.decode_full_paged(q, dense_to_paged(k, bt2, npg),
                                       dense_to_paged(v, bt2, npg), bt2, lens, 0.125)
    assert np.array_equal(out1, out2)


def test_shared_prefix_invariance():
    # 4 requests, identical 48-token prefix + identical 9-token suffix:
    # shared prefix pages (refcount 4) vs private copies -> identical output,
    # and equal across requests.
    rng = np.random.default_rng(21)
    B, Hkv, D, P = 4, 2, 64, 16
    n = 57
    kd = random_bf16(rng, (Hkv, n, D))
    vd = random_bf16(rng, (Hkv, n, D))
    q1 = random_bf16(rng, (1, 8, D))
    q = np.repeat(q1, B, axis=0)
    shared = np.array([7, 2, 9], np.int32)
    own = np.array([[0], [1], [3], [4]], np.int32)
    bt_shared = np.concatenate([np.tile(shared, (B, 1)), own], axis=1)
    bt_priv = np.arange(B * 4, dtype=np.int32).reshape(B, 4)
    ks, vs = dense_to_paged([kd] * B, bt_shared, 10), dense_to_paged([vd] * B, bt_shared, 10)
    kp, vp = dense_to_paged([kd] * B, bt_priv, 16), dense_to_paged([vd] * B, bt_priv, 16)
    lens = np.full(B, n, np.int32)
    o_sh, _ = oracle.decode_full_paged(q, ks, vs, bt_shared, lens, 0.125)
    o_pr, _ = oracle.decode_full_paged(q, kp, vp, bt_priv, lens, 0.125)
    assert np.array_equal(o_sh, o_pr)
    for b in range(1, B):
        assert np.array_equal(o_sh[0], o_sh[b])


# ------------------------------------------------------------------ ring --
@pytest.mark.parametrize("n", [1, 5, 37, 128])
def test_swa_equals_full_when_window_covers_sequence(n):
    # n <= W: the sliding window holds the whole sequence.
    rng = np.random.default_rng(n)
    W, D = 128, 64
    q = random_bf16(rng, (1, 4, D))
    k = [random_bf16(rng, (2, n, D))]
    v = [random_bf16(rng, (2, n, D))]
    rp = np.array([int(rng.integers(0, W))], np.int32)
    kr, vr = dense_to_ring(k, rp, W), dense_to_ring(v, rp, W)
    o_swa, st = oracle.decode_swa_ring(q, kr, vr, None, rp, [n], 0.125)
    assert st == 0
    npg = (n + 15) // 16
    bt = np.arange(npg, dtype=np.int32)[None]
    o_full, _ = oracle.decode_full_paged(q, dense_to_paged(k, bt, npg), dense_to_paged(v, bt, npg),
                                         bt, [n], 0.125)
    np.testing.assert_allclose(o_swa, o_full, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("W", [16, 128])
def test_ring_equals_dense_last_window(W):
    rng = np.random.default_rng(W)
    lens = [W + 1, 3 * W + 7, 200]
    B, D = 3, 64
    q = random_bf16(rng, (B, 8, D))
    k = [random_bf16(rng, (2, n, D)) for n in lens]
    v = [random_bf16(rng, (2, n, D)) for n in lens]
    rp = rng.integers(0, W, size=B).astype(np.int32)
    ids = np.array([2, 0, 1], np.int32)
    kr = dense_to_ring(k, rp, W, num_rings=3, ring_ids=ids)
    vr = dense_to_ring(v, rp, W, num_rings=3, ring_ids=ids)
    out, st = oracle.decode_swa_ring(q, kr, vr, ids, rp, lens, 0.125)
    assert st == 0
    kw = [bf16_bits_to_f64(x[:, max(0, x.shape[1] - W):]) for x in k]
    vw = [bf16_bits_to_f64(x[:, max(0, x.shape[1] - W):]) for x in v]
    np.testing.assert_allclose(out, sdpa_reference(q, kw, vw, 0.125), rtol=1e-12, atol=1e-13)


def test_ring_rotation_invariance():
    # rotating the ring's contents together with ring_pos changes nothing
    rng = np.random.default_rng(99)
    W, D, n = 128, 64, 300
    q = random_bf16(rng, (1, 4, D))
    kr = random_bf16(rng, (1, 2, W, D))
    vr = random_bf16(rng, (1, 2, W, D))
    o1, _ = oracle.decode_swa_ring(q, kr, vr, None, [10], [n], 0.2)
    sh = 37
    o2, _ = oracle.decode_swa_ring(q, np.ascontiguousarray(np.roll(kr, sh, axis=2)),
                                   np.ascontiguousarray(np.roll(vr, sh, axis=2)), None,
                                   [(10 + sh) % W], [n], 0.2)
    assert np.array_equal(o1, o2)


# ---------------------------------------------------------------- append --
def test_append_paged_brute_force():
    q, k, v, bt, npg, lens = _random_case(4, lens=(16, 17, 33))
    kp, vp = dense_to_paged(k, bt, npg), dense_to_paged(v, bt, npg)
    rng = np.random.default_rng(8)
    kn = random_bf16(rng, (3, 2, 64))
    vn = random_bf16(rng, (3, 2, 64))
    lens_after = lens + 1
    bt2 = np.concatenate([bt, np.full((3, 1), -1, np.int32)], axis=1)
    # request 0 (16 tokens) needs a new page for token 16
    spare = sorted(set(range(npg)) - set(bt[bt >= 0].tolist()))
    bt2[0, 1] = spare[0]
    kp2, vp2 = kp.copy(), vp.copy()
    st = oracle.append_paged(kp2, vp2, kn, vn, bt2, lens_after)
    assert st == 0
    # expected: the dense sequences with the new token appended
    k_after = [np.concatenate([k[b], kn[b][:, None]], axis=1) for b in range(3)]
    v_after = [np.concatenate([v[b], vn[b][:, None]], axis=1) for b in range(3)]
    for b in range(3):
        for t in range(lens_after[b]):
            assert np.array_equal(kp2[bt2[b, t // 16], :, t % 16], k_after[b][:, t])
            assert np.array_equal(vp2[bt2[b, t // 16], :, t % 16], v_after[b][:, t])
    # exactly B*Hkv*D elements changed in each pool
    assert (kp2 != kp).sum() <= 3 * 2 * 64 and (vp2 != vp).sum() <= 3 * 2 * 64


def test_append_paged_refuses_shared_page():
    rng = np.random.default_rng(2)
    kp = random_bf16(rng, (4, 1, 16, 64))
    vp = random_bf16(rng, (4, 1, 16, 64))
    kn, vn = random_bf16(rng, (2, 1, 64)), random_bf16(rng, (2, 1, 64))
    bt = np.array([[0, 1], [0, 2]], np.int32)   # page 0 shared by both
    rc = np.array([2, 1, 1, 1], np.int32)
    kp2, vp2 = kp.copy(), vp.copy()
    st = oracle.append_paged(kp2, vp2, kn, vn, bt, [5, 20], page_refcount=rc)
    assert st == oracle.ORC_ESHARED
    assert np.array_equal(kp2[0], kp[0])        # shared page untouched
    assert np.array_equal(kp2[2, 0, 3], kn[1, 0])  # private page written


def test_append_ring_writes_one_slot():
    rng = np.random.default_rng(6)
    kr = random_bf16(rng, (3, 2, 128, 64))
    vr = random_bf16(rng, (3, 2, 128, 64))
    kn, vn = random_bf16(rng, (2, 2, 64)), random_bf16(rng, (2, 2, 64))
    kr2, vr2 = kr.copy(), vr.copy()
    st = oracle.append_ring(kr2, vr2, kn, vn, [2, 0], [127, 5])
    assert st == 0
    assert np.array_equal(kr2[2, :, 127], kn[0]) and np.array_equal(vr2[0, :, 5], vn[1])
    assert (kr2 != kr).sum() <= 2 * 2 * 64
    assert np.array_equal(kr2[1], kr[1])


# ------------------------------------------------------------------ INT8 --
def _quant_one_group(x_bits, D):
    """Run the oracle quantiser on one 32 x D group (K side)."""
    kp = x_bits.reshape(2, 1, 16, D).copy()
    vp = np.zeros_like(kp)
    kc = np.zeros((1, 1, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((1, 1), np.float32)
    vs = np.zeros((1, 1), np.float32)
    st = oracle.quant_int8_block32(kp, vp, [[0, 1]], kc, vc, ks, vs, [[0]], [0], [1])
    assert st == 0
    return kc[0, 0], ks[0, 0]


def test_int8_golden_fixture():
    with open(os.path.join(GOLDEN, "int8_block32_hand.json")) as f:
        fx = json.load(f)
    D = fx["head_dim"]
    for g in fx["groups"]:
        x = np.zeros((32, D), np.float32)
        for t, d, val in g["values"]:
            x[t, d] = val
        codes, s = _quant_one_group(f32_to_bf16_bits(x), D)
        assert float(s) == g["scale"], g["name"]
        want = np.zeros((32, D), np.int8)
        for t, d, c in g["codes"]:
            want[t, d] = c
        assert np.array_equal(codes, want), g["name"]


@pytest.mark.parametrize("seed", range(4))
def test_int8_invariants(seed):
    rng = np.random.default_rng(seed)
    D = 128
    x = rng.standard_normal((32, D)).astype(np.float32)
    m = rng.random((32, D)) < 0.01
    x[m] = rng.standard_normal(m.sum()) * 8
    xb = f32_to_bf16_bits(x)
    xf = bf16_bits_to_f64(xb)
    codes, s = _quant_one_group(xb, D)
    a = np.abs(xf).max()
    assert s == np.float32(np.float32(a) / np.float32(127))
    assert codes.min() >= -127 and codes.max() <= 127
    i = np.unravel_index(np.abs(xf).argmax(), xf.shape)
    assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(xf[i])
    deq = codes.astype(np.float64) * float(s)
    # rounding error at most half a step (plus the scale's own rounding)
    assert np.all(np.abs(deq - xf) <= float(s) * (0.5 + 1e-6))


def test_int8_scale_per_block_and_head():
    # two blocks x two heads, each group scaled independently, K and V too
    rng = np.random.default_rng(1)
    D = 64
    kp = random_bf16(rng, (4, 2, 16, D))
    vp = random_bf16(rng, (4, 2, 16, D))
    kp[2, 1] = f32_to_bf16_bits(np.full((16, D), 0.5, np.float32))
    kp[3, 1] = f32_to_bf16_bits(np.full((16, D), -0.25, np.float32))
    kc = np.zeros((3, 2, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((3, 2), np.float32)
    vs = np.zeros((3, 2), np.float32)
    st = oracle.quant_int8_block32(kp, vp, [[0, 1, 2, 3]], kc, vc, ks, vs, [[2, 0]], [0], [2])
    assert st == 0
    # block 1 of the sequence = pages 2,3 -> qpage 0; head 1 is +-constant
    assert ks[0, 1] == np.float32(0.5) / np.float32(127)
    assert np.all(kc[0, 1, :16] == 127) and np.all(kc[0, 1, 16:] == np.int8(np.rint(-0.25 / ks[0, 1])))
    for (qp, pages) in [(2, (0, 1)), (0, (2, 3))]:
        for h in range(2):
            for name, src, sc in [("k", kp, ks), ("v", vp, vs)]:
                xf = bf16_bits_to_f64(np.concatenate([src[pages[0], h], src[pages[1], h]]))
                assert sc[qp, h] == np.float32(np.float32(np.abs(xf).max()) / np.float32(127)), name
    assert np.all(ks[1] == 0) and np.all(kc[1] == 0)   # untouched qpage


def test_int8_decode_matches_library_on_dequantised():
    # tokens [0, 64) from INT8 pages, [64, 75) from bf16 pages
    rng = np.random.default_rng(12)
    Hkv, D, n, qlen = 2, 64, 75, 64
    kd, vd = random_bf16(rng, (Hkv, n, D)), random_bf16(rng, (Hkv, n, D))
    bt = np.arange(5, dtype=np.int32)[None][:, [4, 0, 3, 1, 2]]
    kp, vp = dense_to_paged([kd], bt, 5), dense_to_paged([vd], bt, 5)
    kc = np.zeros((3, Hkv, 32, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((3, Hkv), np.float32)
    vs = np.zeros((3, Hkv), np.float32)
    qt = np.array([[2, 0]], np.int32)
    assert oracle.quant_int8_block32(kp, vp, bt, kc, vc, ks, vs, qt, [0], [2]) == 0
    q = random_bf16(rng, (1, 4, D))
    # make the bf16 copy of the INT8 region garbage: decode must not read it
    kp2, vp2 = kp.copy(), vp.copy()
    for p in bt[0, :4]:
        kp2[p] = 0x3F80
        vp2[p] = 0x3F80
    out, st = oracle.decode_full_paged(
        q, kp2, vp2, bt, [n], 0.125,
        int8=dict(k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs, qtable=qt, qlens=[qlen]))
    assert st == 0
    kdeq = bf16_bits_to_f64(kd).copy()
    vdeq = bf16_bits_to_f64(vd).copy()
    for j in range(2):
        qp = qt[0, j]
        for h in range(Hkv):
            kdeq[h, 32 * j:32 * j + 32] = (kc[qp, h].astype(np.float32) * ks[qp, h]).astype(np.float64)
            vdeq[h, 32 * j:32 * j + 32] = (vc[qp, h].astype(np.float32) * vs[qp, h]).astype(np.float64)
    np.testing.assert_allclose(out, sdpa_reference(q, [kdeq], [vdeq], 0.125), rtol=1e-12,
                               atol=1e-13)


# ----------------------------------------------------------- 1/7 stack --
def test_kv_tokens_stored_closed_form():
    lf = np.array([1 if l % 7 == 6 else 0 for l in range(70)], np.int32)
    assert lf.sum() == 10
    for n in [1, 100, 128, 129, 5000, 131072]:
        got = oracle.kv_tokens_stored(lf, [n], 128)
        assert got == 10 * n + 60 * min(n, 128)
    # ratio to all-Full approaches 1/7 at long lengths (MiMo page, section 1)
    n = 131072
    r = oracle.kv_tokens_stored(lf, [n], 128) / oracle.kv_tokens_stored(np.ones(70, np.int32),
                                                                        [n], 128)
    assert abs(r - (10 * n + 60 * 128) / (70 * n)) < 1e-15
    assert abs(r - 1 / 7) / (1 / 7) < 0.006
    assert round(r, 4) == 0.1437


def test_kv_tokens_stored_on_stack_workload():
    import synth
    w = synth.hybrid_stack()
    lf = w.extra["layer_is_full"]
    full = oracle.kv_tokens_stored(np.ones(70, np.int32), w.n_after, 128)
    hyb = oracle.kv_tokens_stored(lf, w.n_after, 128)
    assert w.n_after.mean() >= 32768
    assert abs(hyb / full - 1 / 7) / (1 / 7) < 0.05


# ------------------------------------------------- SWA segment pages --
def _seg_case(rng, lens, W, Hkv=2, D=64, P=16):
    """Dense sequences, and segment pages holding every page of each
    (page ids from one permutation; pages of different requests disjoint)."""
    k = [random_bf16(rng, (Hkv, n, D)) for n in lens]
    v = [random_bf16(rng, (Hkv, n, D)) for n in lens]
    ppr = [(n + P - 1) // P for n in lens]
    nseg = sum(ppr) + 3
    perm = rng.permutation(nseg)
    bt = np.full((len(lens), max(ppr)), -1, np.int32)
    o = 0
    for b, c in enumerate(ppr):
        bt[b, :c] = perm[o:o + c]
        o += c
    return k, v, bt, nseg


def _window_table(bt, lens, W, P=16):
    """Row b: the segment pages of request b's last window, in token order."""
    rows = []
    for b, n in enumerate(lens):
        lo = n - min(n, W)
        rows.append(bt[b, lo // P:(n + P - 1) // P])
    width = max(len(r) for r in rows)
    out = np.full((len(lens), width), -1, np.int32)
    for b, r in enumerate(rows):
        out[b, :len(r)] = r
    return out


@pytest.mark.parametrize("W", [16, 128])
def test_ring_seeded_from_segment_pages_equals_dense_last_window(W):
    # the ring a request resumes with holds exactly its last W tokens: SWA
    # decode over it equals the library on the dense last-W window (lengths
    # below W, page-aligned and not page-aligned)
    rng = np.random.default_rng(300 + W)
    lens = [5, W, W + 16, 3 * W + 9, 200]
    B, D = len(lens), 64
    k, v, bt, nseg = _seg_case(rng, lens, W)
    ks, vs = dense_to_paged(k, bt, nseg), dense_to_paged(v, bt, nseg)
    ids = rng.permutation(B + 2)[:B].astype(np.int32)
    rp = rng.integers(0, W, size=B).astype(np.int32)
    kr = random_bf16(rng, (B + 2, 2, W, D))
    vr = random_bf16(rng, (B + 2, 2, W, D))
    st = oracle.swa_ring_seed(kr, vr, ks, vs, ids, rp, lens, _window_table(bt, lens, W))
    assert st == 0
    q = random_bf16(rng, (B, 8, D))
    out, st = oracle.decode_swa_ring(q, kr, vr, ids, rp, lens, 0.125)
    assert st == 0
    kw = [bf16_bits_to_f64(x[:, max(0, x.shape[1] - W):]) for x in k]
    vw = [bf16_bits_to_f64(x[:, max(0, x.shape[1] - W):]) for x in v]
    np.testing.assert_allclose(out, sdpa_reference(q, kw, vw, 0.125), rtol=1e-12, atol=1e-13)
    # brute force: every window token sits where the ring formula puts it
    for b, n in enumerate(lens):
        for t in range(n - min(n, W), n):
            assert np.array_equal(kr[ids[b], :, (rp[b] - (n - 1 - t)) % W], k[b][:, t])


def test_ring_save_copies_whole_window_pages():
    rng = np.random.default_rng(310)
    W, D, n = 128, 64, 300          # window [172, 300): pages 11..17 are whole
    k = [random_bf16(rng, (2, n, D))]
    v = [random_bf16(rng, (2, n, D))]
    rp = np.array([77], np.int32)
    kr = dense_to_ring(k, rp, W, num_rings=2, ring_ids=[1])
    vr = dense_to_ring(v, rp, W, num_rings=2, ring_ids=[1])
    ks = np.zeros((9, 2, 16, D), np.uint16)
    vs = np.zeros_like(ks)
    pages = np.arange(11, 18, dtype=np.int32)
    segs = np.arange(7, dtype=np.int32)[::-1].copy() + 2
    one = np.ones(len(pages), np.int32)
    st = oracle.swa_ring_save(kr, vr, ks, vs, one, np.full(len(pages), 77), one * n, pages, segs)
    assert st == 0
    for p, s in zip(pages, segs):
        assert np.array_equal(ks[s], k[0][:, 16 * p:16 * p + 16])
        assert np.array_equal(vs[s], v[0][:, 16 * p:16 * p + 16])
    # page 10 starts before the window (tokens 160..171 were overwritten)
    ks0 = ks.copy()
    st = oracle.swa_ring_save(kr, vr, ks, vs, [1], [77], [n], [10], [0])
    assert st == oracle.ORC_ERANGE and np.array_equal(ks, ks0)


def test_ring_save_then_seed_round_trip():
    # a finished request's whole window pages saved, then seeded into another
    # ring at another newest slot: the SWA decode is unchanged
    rng = np.random.default_rng(320)
    W, D = 64, 64
    lens = [192, 80]                 # page-aligned window starts: 128 and 16
    k = [random_bf16(rng, (2, n, D)) for n in lens]
    v = [random_bf16(rng, (2, n, D)) for n in lens]
    rp = np.array([5, 60], np.int32)
    kr = dense_to_ring(k, rp, W)
    vr = dense_to_ring(v, rp, W)
    q = random_bf16(rng, (2, 4, D))
    ref, _ = oracle.decode_swa_ring(q, kr, vr, None, rp, lens, 0.2)
    ks = np.zeros((10, 2, 16, D), np.uint16)
    vs = np.zeros_like(ks)
    e_ring, e_page, e_seg = [], [], []
    table = np.full((2, W // 16), -1, np.int32)
    s = 0
    for b, n in enumerate(lens):
        for j, p in enumerate(range((n - W) // 16, n // 16)):
            e_ring.append(b)
            e_page.append(p)
            e_seg.append(s)
            table[b, j] = s
            s += 1
    m = len(e_ring)
    assert oracle.swa_ring_save(kr, vr, ks, vs, e_ring, rp[e_ring], np.array(lens)[e_ring],
                                e_page, e_seg) == 0
    rp2 = np.array([31, 2], np.int32)
    kr2 = random_bf16(rng, (2, 2, W, D))
    vr2 = random_bf16(rng, (2, 2, W, D))
    assert oracle.swa_ring_seed(kr2, vr2, ks, vs, None, rp2, lens, table) == 0
    out, _ = oracle.decode_swa_ring(q, kr2, vr2, None, rp2, lens, 0.2)
    assert np.array_equal(out, ref) and m == 8
