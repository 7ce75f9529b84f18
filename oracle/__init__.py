"""CPU oracle for paged hybrid sliding-window decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it: the oracle is plain C in
``phs_oracle.c`` (fp64 reductions), compiled with gcc and reached through
ctypes on numpy arrays.  bf16 tensors are passed as ``uint16`` bit patterns.

Every function here restates, in code of its own, the definition given in
the header of ``phs_oracle.c`` together with the page and section it follows.

Parity status: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, a library routine on dense
inputs, invariants, brute force and hand-derived fixtures); no function is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "phs_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libphs_oracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_EINVAL, ORC_ERANGE, ORC_ESHARED = 0, -1, -3, -4


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp); returns the .so path.
    `src` / `out` build another copy of the source (the pin tests compile
    planted-mistake copies of it this way)."""
    so = out or _SO
    source = src or _SRC
    os.makedirs(os.path.dirname(so), exist_ok=True)
    if (not force and src is None and os.path.exists(so)
            and os.path.getmtime(so) >= os.path.getmtime(_SRC)):
        return so
    tmp = so + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, source, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, so)
    return so


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PHS_ORACLE_MUTANT_LIB: a planted-mistake build, used only by the
            # test that checks the pins catch such mistakes
            path = os.environ.get("PHS_ORACLE_MUTANT_LIB") or build()
            lib = ctypes.CDLL(path)
            P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.phs_oracle_max_threads.restype = I
            lib.phs_oracle_append_paged.argtypes = [P, P, L, I, I, I, P, P, P, I, P, I, P]
            lib.phs_oracle_append_paged.restype = I
            lib.phs_oracle_append_ring.argtypes = [P, P, L, I, I, I, P, P, P, P, I]
            lib.phs_oracle_append_ring.restype = I
            lib.phs_oracle_quant_int8_block32.argtypes = [
                P, P, L, I, I, I, P, I, P, P, P, P, L, P, I, P, P, I]
            lib.phs_oracle_quant_int8_block32.restype = I
            lib.phs_oracle_decode_full_paged.argtypes = [
                P, I, I, I, I, P, P, L, I, P, I, P, P, P, P, P, L, P, I, P, D, P, I, P]
            lib.phs_oracle_decode_full_paged.restype = I
            lib.phs_oracle_decode_swa_ring.argtypes = [
                P, I, I, I, I, P, P, L, I, P, P, P, D, P, I, P]
            lib.phs_oracle_decode_swa_ring.restype = I
            lib.phs_oracle_kv_tokens_stored.argtypes = [P, I, P, I, I]
            lib.phs_oracle_kv_tokens_stored.restype = L
            lib.phs_oracle_swa_ring_save.argtypes = [P, P, L, I, I, I, P, P, L, I, P, P, P, P,
                                                     P, I]
            lib.phs_oracle_swa_ring_save.restype = I
            lib.phs_oracle_swa_ring_seed.argtypes = [P, P, L, I, I, I, P, P, L, I, P, P, P, P,
                                                     I, I]
            lib.phs_oracle_swa_ring_seed.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().phs_oracle_max_threads())


def append_paged(k_pool, v_pool, k_new, v_new, block_table, seq_lens, page_refcount=None):
    """In-place append of token n_b - 1 into the paged pools (uint16 arrays
    of shape [num_pages, Hkv, P, D]).  Returns the oracle status."""
    num_pages, Hkv, P, D = k_pool.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    rc = _c(page_refcount, np.int32)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    return _load().phs_oracle_append_paged(
        _ptr(k_pool), _ptr(v_pool), num_pages, P, Hkv, D, _ptr(kn), _ptr(vn),
        _ptr(bt), bt.shape[1], _ptr(sl), sl.shape[0], _ptr(rc))


def append_ring(k_ring, v_ring, k_new, v_new, ring_ids, ring_pos):
    """In-place write of the new token into ring slot ring_pos[b]."""
    num_rings, Hkv, W, D = k_ring.shape
    rp = _c(ring_pos, np.int32)
    ri = _c(ring_ids, np.int32)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    return _load().phs_oracle_append_ring(
        _ptr(k_ring), _ptr(v_ring), num_rings, W, Hkv, D, _ptr(kn), _ptr(vn),
        _ptr(ri), _ptr(rp), rp.shape[0])


def quant_int8_block32(k_pool, v_pool, src_table, k_codes, v_codes, k_scale, v_scale,
                       dst_qtable, first_qblock, num_qblocks):
    """Quantise 32-token groups into INT8 codes (in place) and fp32 scales."""
    num_pages, Hkv, P, D = k_pool.shape
    st = _c(src_table, np.int32)
    qt = _c(dst_qtable, np.int32)
    fq = _c(first_qblock, np.int32)
    nq = _c(num_qblocks, np.int32)
    return _load().phs_oracle_quant_int8_block32(
        _ptr(k_pool), _ptr(v_pool), num_pages, P, Hkv, D, _ptr(st), st.shape[1],
        _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), k_codes.shape[0],
        _ptr(qt), qt.shape[1], _ptr(fq), _ptr(nq), fq.shape[0])


def decode_full_paged(q, k_pool, v_pool, block_table, seq_lens, scale, rows=None,
                      int8=None):
    """Full-attention decode.  q: uint16 [B, Hq, D].  int8: optional dict with
    k_codes, v_codes [num_qpages, Hkv, 32, D] int8, k_scale, v_scale
    [num_qpages, Hkv] float32, qtable [B, max_qpages] int32, qlens [B].
    Returns (out float64 [B, Hq, D], status); rows not selected stay zero."""
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_pool.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    qq = _c(q, np.uint16)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rws = _c(rows, np.int32)
    if int8 is not None:
        kc, vc = _c(int8["k_codes"], np.int8), _c(int8["v_codes"], np.int8)
        ks, vs = _c(int8["k_scale"], np.float32), _c(int8["v_scale"], np.float32)
        qt, ql = _c(int8["qtable"], np.int32), _c(int8["qlens"], np.int32)
        nq, mq = kc.shape[0], qt.shape[1]
    else:
        kc = vc = ks = vs = qt = ql = None
        nq, mq = 0, 0
    st = _load().phs_oracle_decode_full_paged(
        _ptr(qq), B, Hq, Hkv, D, _ptr(k_pool), _ptr(v_pool), num_pages, P, _ptr(bt),
        bt.shape[1], _ptr(sl), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nq, _ptr(qt), mq,
        _ptr(ql), float(scale), _ptr(rws), 0 if rws is None else rws.shape[0], _ptr(out))
    return out, st


def decode_swa_ring(q, k_ring, v_ring, ring_ids, ring_pos, seq_lens, scale, rows=None):
    """Sliding-window decode over the ring; returns (out float64, status)."""
    B, Hq, D = q.shape
    num_rings, Hkv, W, _ = k_ring.shape
    qq = _c(q, np.uint16)
    ri = _c(ring_ids, np.int32)
    rp = _c(ring_pos, np.int32)
    sl = _c(seq_lens, np.int32)
    rws = _c(rows, np.int32)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = _load().phs_oracle_decode_swa_ring(
        _ptr(qq), B, Hq, Hkv, D, _ptr(k_ring), _ptr(v_ring), num_rings, W, _ptr(ri),
        _ptr(rp), _ptr(sl), float(scale), _ptr(rws), 0 if rws is None else rws.shape[0],
        _ptr(out))
    return out, st


def swa_ring_save(k_ring, v_ring, k_seg, v_seg, ring_ids, ring_pos, seq_lens, page_index,
                  seg_pages):
    """Copy whole pages of requests' SWA windows from the rings (uint16
    [num_rings, Hkv, W, D]) into segment pages (uint16 [num_seg, Hkv, P, D],
    in place).  Returns the oracle status."""
    num_rings, Hkv, W, D = k_ring.shape
    num_seg, _, P, _ = k_seg.shape
    a = [_c(x, np.int32) for x in (ring_ids, ring_pos, seq_lens, page_index, seg_pages)]
    return _load().phs_oracle_swa_ring_save(
        _ptr(k_ring), _ptr(v_ring), num_rings, W, Hkv, D, _ptr(k_seg), _ptr(v_seg), num_seg, P,
        *[_ptr(x) for x in a], a[0].shape[0])


def swa_ring_seed(k_ring, v_ring, k_seg, v_seg, ring_ids, ring_pos, seq_lens, seg_table):
    """Write each request's last min(n, W) tokens from its segment pages
    (seg_table [B, max_seg]) into its ring (in place)."""
    num_rings, Hkv, W, D = k_ring.shape
    num_seg, _, P, _ = k_seg.shape
    ri = _c(ring_ids, np.int32)
    rp, sl, st = _c(ring_pos, np.int32), _c(seq_lens, np.int32), _c(seg_table, np.int32)
    return _load().phs_oracle_swa_ring_seed(
        _ptr(k_ring), _ptr(v_ring), num_rings, W, Hkv, D, _ptr(k_seg), _ptr(v_seg), num_seg, P,
        _ptr(ri), _ptr(rp), _ptr(sl), _ptr(st), st.shape[1], sl.shape[0])


def kv_tokens_stored(layer_is_full, seq_lens, W):
    """Tokens of KV stored per the hybrid stack (sum over layers, requests)."""
    lf = _c(layer_is_full, np.int32)
    sl = _c(seq_lens, np.int32)
    return int(_load().phs_oracle_kv_tokens_stored(_ptr(lf), lf.shape[0], _ptr(sl),
                                                   sl.shape[0], int(W)))
