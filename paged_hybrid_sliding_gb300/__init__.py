"""paged_hybrid_sliding_gb300 -- decode attention over a hybrid paged KV
cache (a paged Full-attention pool plus per-request SWA ring buffers), KV
append and block-32 INT8 quantisation, as hand-written CUDA for sm_103a
behind the C ABI of include/phs.h.

This module only marshals torch tensors into the C ABI: every step runs in
the library's kernels.  Tensors must be CUDA, contiguous and of the dtype
stated; the stream defaults to torch's current stream.  Errors returned by
the library raise PhsError.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _lib

__all__ = [
    "PhsError", "PagedPool", "RingPool", "Int8Pool", "Layer",
    "kv_append_paged", "kv_append_ring", "kv_quant_int8_block32",
    "decode_workspace_bytes", "decode_tokens_per_split",
    "attn_decode_full_paged", "attn_decode_full_paged_split", "attn_merge_splits",
    "attn_decode_full_paged_noalloc", "NOALLOC_SCRATCH_BYTES",
    "attn_decode_shared_prefix", "shared_prefix_workspace_bytes",
    "attn_decode_swa_ring", "attn_decode_hybrid_stack", "hybrid_stack_workspace_bytes",
    "attn_decode_hybrid_stack_fused", "hybrid_stack_fused_workspace_bytes",
    "hybrid_kv_tokens", "copy_d2d", "read_checksum", "copy_pages", "PageAllocator", "RadixTree",
    "window_safe_len", "swa_ring_save", "swa_ring_seed", "lib", "PAGE", "QBLOCK",
]

PAGE = 16
QBLOCK = 32
OUT_BF16, OUT_F32 = 0, 1
NOALLOC_SCRATCH_BYTES = 32 << 20


class PhsError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = lib().phs_status_str(code).decode()
        super().__init__(f"{what}: {msg} ({code})")


def lib():
    return _lib.load()


def _check(code: int, what: str):
    if code != 0:
        raise PhsError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")
    return t


def _opt(t, dtype, name, dims=None):
    return None if t is None else _need(t, dtype, name, dims)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _out_code(dtype):
    if dtype == torch.bfloat16:
        return OUT_BF16
    if dtype == torch.float32:
        return OUT_F32
    raise ValueError("out dtype must be bfloat16 or float32")


@dataclass
class PagedPool:
    """Full-attention pool: k, v bf16 [num_pages, Hkv, 16, D]."""
    k: torch.Tensor
    v: torch.Tensor

    def c(self):
        _need(self.k, torch.bfloat16, "pool.k", 4)
        _need(self.v, torch.bfloat16, "pool.v", 4)
        if self.k.shape != self.v.shape:
            raise ValueError("pool.k and pool.v shapes differ")
        n, h, p, d = self.k.shape
        return _lib.PagedPoolC(self.k.data_ptr(), self.v.data_ptr(), n, p, h, d)

    @staticmethod
    def empty(num_pages, num_kv_heads, head_dim, device="cuda"):
        shape = (num_pages, num_kv_heads, PAGE, head_dim)
        return PagedPool(torch.empty(shape, dtype=torch.bfloat16, device=device),
                         torch.empty(shape, dtype=torch.bfloat16, device=device))


@dataclass
class RingPool:
    """SWA ring pool: k, v bf16 [num_rings, Hkv, W, D]."""
    k: torch.Tensor
    v: torch.Tensor

    def c(self):
        _need(self.k, torch.bfloat16, "ring.k", 4)
        _need(self.v, torch.bfloat16, "ring.v", 4)
        if self.k.shape != self.v.shape:
            raise ValueError("ring.k and ring.v shapes differ")
        n, h, w, d = self.k.shape
        return _lib.RingPoolC(self.k.data_ptr(), self.v.data_ptr(), n, w, h, d)

    @staticmethod
    def empty(num_rings, num_kv_heads, window, head_dim, device="cuda"):
        shape = (num_rings, num_kv_heads, window, head_dim)
        return RingPool(torch.empty(shape, dtype=torch.bfloat16, device=device),
                        torch.empty(shape, dtype=torch.bfloat16, device=device))


# Token held by byte p of a 16-token half of a stored V^T row (see Int8Pool).
VT_TOKEN = tuple(2 * (p >> 2) + (p & 1) + 8 * ((p >> 1) & 1) for p in range(16))


@dataclass
class Int8Pool:
    """INT8 pool in its stored form (each code x as the byte x + 128):
    k uint8 [num_qpages, Hkv, 32 tokens, D]; v uint8 [num_qpages, Hkv, 2,
    D, 16] (transposed per 16-token half; byte p of a row holds token
    VT_TOKEN[p] of its half); scales fp32 [num_qpages, Hkv]."""
    k: torch.Tensor
    v: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor

    def c(self):
        _need(self.k, torch.uint8, "int8.k", 4)
        _need(self.v, torch.uint8, "int8.v", 5)
        _need(self.k_scale, torch.float32, "int8.k_scale", 2)
        _need(self.v_scale, torch.float32, "int8.v_scale", 2)
        n, h, q, d = self.k.shape
        if q != QBLOCK or tuple(self.v.shape) != (n, h, 2, d, QBLOCK // 2) \
                or tuple(self.k_scale.shape) != (n, h) or tuple(self.v_scale.shape) != (n, h):
            raise ValueError("inconsistent INT8 pool shapes")
        return _lib.Int8PoolC(self.k.data_ptr(), self.v.data_ptr(), self.k_scale.data_ptr(),
                              self.v_scale.data_ptr(), n, h, d)

    def codes(self, pages=None):
        """The signed codes (int8) of all pages, or of the page ids in
        `pages`, both token-major [pages, Hkv, 32, D]: a view of the stored
        form for inspection, not used by the decode path."""
        k, v = self.k, self.v
        if pages is not None:
            k, v = k.index_select(0, pages), v.index_select(0, pages)
        # stored row 16 hf + p (half hf, byte p) holds token 16 hf + VT_TOKEN[p]
        order = torch.tensor([16 * hf + t for hf in range(2) for t in VT_TOKEN], device=v.device)
        inv = torch.empty_like(order)
        inv[order] = torch.arange(QBLOCK, device=v.device)
        rows = v.transpose(-1, -2).reshape(*v.shape[:2], QBLOCK, v.shape[3])  # [.., 16 hf + p, D]
        vt = rows.index_select(-2, inv)  # [.., token, D]
        return ((k.to(torch.int16) - 128).to(torch.int8),
                (vt.to(torch.int16) - 128).to(torch.int8).contiguous())

    @staticmethod
    def empty(num_qpages, num_kv_heads, head_dim, device="cuda"):
        return Int8Pool(
            torch.empty((num_qpages, num_kv_heads, QBLOCK, head_dim), dtype=torch.uint8,
                        device=device),
            torch.empty((num_qpages, num_kv_heads, 2, head_dim, QBLOCK // 2), dtype=torch.uint8,
                        device=device),
            torch.empty((num_qpages, num_kv_heads), dtype=torch.float32, device=device),
            torch.empty((num_qpages, num_kv_heads), dtype=torch.float32, device=device))


# ------------------------------------------------------------------ append --
def kv_append_paged(pool: PagedPool, k_new, v_new, block_table, seq_lens, page_refcount=None,
                    status=None, stream=None):
    """Write token seq_lens[b]-1 of every request into its page slot."""
    pc = pool.c()
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _opt(page_refcount, torch.int32, "page_refcount", 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_kv_append_paged(ctypes.byref(pc), _ptr(k_new), _ptr(v_new), _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), seq_lens.shape[0],
                                     _ptr(page_refcount), _ptr(status), _stream(stream)),
           "kv_append_paged")


def kv_append_ring(ring: RingPool, k_new, v_new, ring_pos, ring_ids=None, status=None,
                   stream=None):
    """Write the new token of every request into ring slot ring_pos[b]."""
    rc = ring.c()
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(ring_pos, torch.int32, "ring_pos", 1)
    _opt(ring_ids, torch.int32, "ring_ids", 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_kv_append_ring(ctypes.byref(rc), _ptr(k_new), _ptr(v_new), _ptr(ring_ids),
                                    _ptr(ring_pos), ring_pos.shape[0], _ptr(status),
                                    _stream(stream)), "kv_append_ring")


def kv_quant_int8_block32(src: PagedPool, src_block_table, dst: Int8Pool, dst_qtable,
                          first_qblock, num_qblocks, max_qblocks: int, status=None, stream=None):
    """Quantise 32-token blocks of the bf16 pages into INT8 codes + fp32 scales."""
    sc, dc = src.c(), dst.c()
    _need(src_block_table, torch.int32, "src_block_table", 2)
    _need(dst_qtable, torch.int32, "dst_qtable", 2)
    _need(first_qblock, torch.int32, "first_qblock", 1)
    _need(num_qblocks, torch.int32, "num_qblocks", 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_kv_quant_int8_block32(
        ctypes.byref(sc), _ptr(src_block_table), src_block_table.shape[1], ctypes.byref(dc),
        _ptr(dst_qtable), dst_qtable.shape[1], _ptr(first_qblock), _ptr(num_qblocks),
        int(max_qblocks), first_qblock.shape[0], _ptr(status), _stream(stream)),
        "kv_quant_int8_block32")


# ------------------------------------------------------------------ decode --
def decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                           tokens_per_split=0, has_int8=False) -> int:
    """Workspace bytes for a decode call; 0 if the shape is not supported."""
    return int(lib().phs_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                max_seq_len, tokens_per_split,
                                                int(bool(has_int8))))


def decode_tokens_per_split(batch, num_kv_heads, max_seq_len, tokens_per_split=0) -> int:
    t = lib().phs_decode_tokens_per_split(batch, num_kv_heads, max_seq_len, tokens_per_split)
    _check(min(int(t), 0), "decode_tokens_per_split")
    return int(t)


def _decode_args(q, pool, block_table, seq_lens, int8, qtable, qlens, out, out_dtype, status):
    _need(q, torch.bfloat16, "q", 3)
    pc = pool.c()
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    ic = None
    if int8 is not None:
        ic = int8.c()
        _need(qtable, torch.int32, "qtable", 2)
        _need(qlens, torch.int32, "qlens", 1)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out, out.dtype, "out", 3)
    _opt(status, torch.int32, "status")
    return pc, ic, out


def _append_args(k_new, v_new, page_refcount, B, Hkv, D):
    """Checks of a fused append's new tokens ([B, Hkv, D] bf16, both or
    neither) and page reference counts."""
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        for t, name in ((k_new, "k_new"), (v_new, "v_new")):
            _need(t, torch.bfloat16, name, 3)
            if tuple(t.shape) != (B, Hkv, D):
                raise ValueError(f"{name} must be [batch, Hkv, D]")
    _opt(page_refcount, torch.int32, "page_refcount", 1)


def _workspace(workspace, nbytes, device):
    if workspace is None:
        # a zero size means the library rejects the shape: let the call
        # report the precise status
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    _need(workspace, torch.uint8, "workspace", 1)
    return workspace


def attn_decode_full_paged(q, pool: PagedPool, block_table, seq_lens, max_seq_len: int,
                           softmax_scale=None, int8: Int8Pool | None = None, qtable=None,
                           qlens=None, tokens_per_split=0, out=None, out_dtype=torch.bfloat16,
                           workspace=None, k_new=None, v_new=None, page_refcount=None,
                           status=None, stream=None):
    """Split-KV decode over the paged pool (optionally INT8 below qlens[b]);
    returns out [B, Hq, D].  k_new / v_new ([B, Hkv, D] bf16): append token
    seq_lens[b] - 1 in the same call (as kv_append_paged with page_refcount,
    then this call)."""
    pc, ic, out = _decode_args(q, pool, block_table, seq_lens, int8, qtable, qlens, out,
                               out_dtype, status)
    B, Hq, D = q.shape
    _append_args(k_new, v_new, page_refcount, B, pool.k.shape[1], D)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    need = decode_workspace_bytes(B, Hq, pool.k.shape[1], D, max_seq_len, tokens_per_split,
                                  int8 is not None)
    ws = _workspace(workspace, need, q.device)
    _check(lib().phs_attn_decode_full_paged(
        _ptr(q), Hq, ctypes.byref(pc), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        int(max_seq_len), None if ic is None else ctypes.byref(ic), _ptr(qtable),
        0 if qtable is None else qtable.shape[1], _ptr(qlens), B, scale, int(tokens_per_split),
        _ptr(out), _out_code(out.dtype), _ptr(ws), ws.numel(), _ptr(k_new), _ptr(v_new),
        _ptr(page_refcount), _ptr(status), _stream(stream)), "attn_decode_full_paged")
    return out


def attn_decode_full_paged_noalloc(q, pool: PagedPool, block_table, seq_lens,
                                   max_seq_len: int, out, softmax_scale=None,
                                   int8: Int8Pool | None = None, qtable=None, qlens=None,
                                   tokens_per_split=0, status=None, stream=None):
    """Same as attn_decode_full_paged, for callers that cannot provide a
    workspace (a host framework that owns all device memory, an engine that
    has reserved nearly all of HBM, a loop that must not call cudaMalloc).
    The partials go to the library's built-in 32 MiB scratch per GPU; `out`
    must be given.  Calls that overlap on the GPU share that scratch and
    race, so serialise them.  Raises PhsError (PHS_ESCRATCH) when the
    request needs more scratch than that."""
    pc, ic, out = _decode_args(q, pool, block_table, seq_lens, int8, qtable, qlens, out,
                               out.dtype, status)
    B, Hq, D = q.shape
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    _check(lib().phs_attn_decode_full_paged_noalloc(
        _ptr(q), Hq, ctypes.byref(pc), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        int(max_seq_len), None if ic is None else ctypes.byref(ic), _ptr(qtable),
        0 if qtable is None else qtable.shape[1], _ptr(qlens), B, scale, int(tokens_per_split),
        _ptr(out), _out_code(out.dtype), _ptr(status), _stream(stream)),
        "attn_decode_full_paged_noalloc")
    return out


def shared_prefix_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                  shared_len) -> int:
    """Workspace bytes for attn_decode_shared_prefix; 0 if unsupported."""
    return int(lib().phs_shared_prefix_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                       head_dim, max_seq_len, shared_len))


def attn_decode_shared_prefix(q, pool: PagedPool, block_table, seq_lens, max_seq_len: int,
                              shared_len: int, softmax_scale=None, out=None,
                              out_dtype=torch.bfloat16, workspace=None, k_new=None, v_new=None,
                              page_refcount=None, status=None, stream=None):
    """Decode for a batch whose block tables all start with the same
    shared_len / 16 prefix pages: the prefix is attended once per KV head
    for all requests on the tensor cores, each request's own tokens by the
    split-KV kernel, then merged.  Same result as attn_decode_full_paged.
    k_new / v_new ([B, Hkv, D] bf16): append token seq_lens[b] - 1 in the
    same call (as kv_append_paged with page_refcount, then this call)."""
    pc, _, out = _decode_args(q, pool, block_table, seq_lens, None, None, None, out, out_dtype,
                              status)
    B, Hq, D = q.shape
    _append_args(k_new, v_new, page_refcount, B, pool.k.shape[1], D)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    need = shared_prefix_workspace_bytes(B, Hq, pool.k.shape[1], D, max_seq_len, shared_len)
    ws = _workspace(workspace, need, q.device)
    _check(lib().phs_attn_decode_shared_prefix(
        _ptr(q), Hq, ctypes.byref(pc), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        int(max_seq_len), B, int(shared_len), scale, _ptr(out), _out_code(out.dtype), _ptr(ws),
        ws.numel(), _ptr(k_new), _ptr(v_new), _ptr(page_refcount), _ptr(status), _stream(stream)),
        "attn_decode_shared_prefix")
    return out


def attn_decode_full_paged_split(q, pool: PagedPool, block_table, seq_lens, max_seq_len: int,
                                 workspace, out, softmax_scale=None, int8=None, qtable=None,
                                 qlens=None, tokens_per_split=0, k_new=None, v_new=None,
                                 page_refcount=None, status=None, stream=None):
    """Split phase only (see attn_merge_splits); k_new / v_new as for
    attn_decode_full_paged."""
    pc, ic, out = _decode_args(q, pool, block_table, seq_lens, int8, qtable, qlens, out,
                               out.dtype, status)
    B, Hq, D = q.shape
    _append_args(k_new, v_new, page_refcount, B, pool.k.shape[1], D)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().phs_attn_decode_full_paged_split(
        _ptr(q), Hq, ctypes.byref(pc), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        int(max_seq_len), None if ic is None else ctypes.byref(ic), _ptr(qtable),
        0 if qtable is None else qtable.shape[1], _ptr(qlens), B, scale, int(tokens_per_split),
        _ptr(out), _out_code(out.dtype), _ptr(workspace), workspace.numel(), _ptr(k_new),
        _ptr(v_new), _ptr(page_refcount), _ptr(status), _stream(stream)),
        "attn_decode_full_paged_split")
    return out


def attn_merge_splits(out, num_kv_heads, seq_lens, max_seq_len: int, workspace, qlens=None,
                      has_int8=False, tokens_per_split=0, stream=None):
    """Merge phase only: finishes requests that the split phase cut in pieces."""
    B, Hq, D = out.shape
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _opt(qlens, torch.int32, "qlens", 1)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().phs_attn_merge_splits(B, Hq, num_kv_heads, D, _ptr(seq_lens), int(max_seq_len),
                                       _ptr(qlens), int(bool(has_int8)), int(tokens_per_split),
                                       _ptr(out), _out_code(out.dtype), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "attn_merge_splits")
    return out


def attn_decode_swa_ring(q, ring: RingPool, ring_pos, seq_lens, ring_ids=None,
                         softmax_scale=None, out=None, out_dtype=torch.bfloat16, status=None,
                         stream=None):
    """Sliding-window decode over each request's ring; returns out [B, Hq, D]."""
    _need(q, torch.bfloat16, "q", 3)
    rc = ring.c()
    _need(ring_pos, torch.int32, "ring_pos", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _opt(ring_ids, torch.int32, "ring_ids", 1)
    _opt(status, torch.int32, "status")
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out, out.dtype, "out", 3)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    _check(lib().phs_attn_decode_swa_ring(_ptr(q), Hq, ctypes.byref(rc), _ptr(ring_ids),
                                          _ptr(ring_pos), _ptr(seq_lens), B, scale, _ptr(out),
                                          _out_code(out.dtype), _ptr(status), _stream(stream)),
           "attn_decode_swa_ring")
    return out


@dataclass
class Layer:
    """One layer of a hybrid stack: Full (paged pool) or SWA (ring pool)."""
    q: torch.Tensor
    out: torch.Tensor
    paged: PagedPool | None = None
    ring: RingPool | None = None
    k_new: torch.Tensor | None = None
    v_new: torch.Tensor | None = None

    def c(self):
        L = _lib.LayerC()
        L.is_full = 1 if self.paged is not None else 0
        L.q = self.q.data_ptr()
        L.out = self.out.data_ptr()
        L.k_new = 0 if self.k_new is None else self.k_new.data_ptr()
        L.v_new = 0 if self.v_new is None else self.v_new.data_ptr()
        if self.paged is not None:
            L.paged = self.paged.c()
        else:
            L.ring = self.ring.c()
        return L


def hybrid_stack_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len):
    return int(lib().phs_hybrid_stack_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                      max_seq_len))


def attn_decode_hybrid_stack(layers, num_q_heads, seq_lens, max_seq_len, block_table=None,
                             ring_pos=None, ring_ids=None, softmax_scale=None, do_append=True,
                             workspace=None, status=None, stream=None, page_refcount=None):
    """One decode step (append + attend) over every layer of a hybrid stack.
    page_refcount: optional device int32 [num_pages]; a Full layer's new token
    is not written into a page whose count is not 1."""
    arr = (_lib.LayerC * len(layers))(*[L.c() for L in layers])
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _opt(block_table, torch.int32, "block_table", 2)
    _opt(page_refcount, torch.int32, "page_refcount", 1)
    _opt(ring_pos, torch.int32, "ring_pos", 1)
    _opt(ring_ids, torch.int32, "ring_ids", 1)
    _opt(status, torch.int32, "status")
    B = seq_lens.shape[0]
    q0 = layers[0].q
    D = q0.shape[2]
    out_code = _out_code(layers[0].out.dtype)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    nfull = sum(1 for L in layers if L.paged is not None)
    if workspace is None and nfull:
        hkv = next(L.paged.k.shape[1] for L in layers if L.paged is not None)
        workspace = torch.empty(hybrid_stack_workspace_bytes(B, num_q_heads, hkv, D, max_seq_len),
                                dtype=torch.uint8, device=q0.device)
    _check(lib().phs_attn_decode_hybrid_stack(
        arr, len(layers), num_q_heads, B, _ptr(block_table),
        0 if block_table is None else block_table.shape[1], _ptr(page_refcount),
        _ptr(seq_lens), int(max_seq_len),
        _ptr(ring_ids), _ptr(ring_pos), scale, int(bool(do_append)), out_code, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream)),
        "attn_decode_hybrid_stack")


def hybrid_stack_fused_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                       num_full_layers):
    return int(lib().phs_hybrid_stack_fused_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                            head_dim, max_seq_len,
                                                            num_full_layers))


def attn_decode_hybrid_stack_fused(layers, num_q_heads, seq_lens, max_seq_len, block_table=None,
                                   ring_pos=None, ring_ids=None, softmax_scale=None,
                                   workspace=None, status=None, stream=None, page_refcount=None):
    """One decode step over every layer of a hybrid stack with the appends
    fused into the attention launches (every layer needs k_new / v_new).
    page_refcount as for attn_decode_hybrid_stack."""
    arr = (_lib.LayerC * len(layers))(*[L.c() for L in layers])
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _opt(block_table, torch.int32, "block_table", 2)
    _opt(page_refcount, torch.int32, "page_refcount", 1)
    _opt(ring_pos, torch.int32, "ring_pos", 1)
    _opt(ring_ids, torch.int32, "ring_ids", 1)
    _opt(status, torch.int32, "status")
    B = seq_lens.shape[0]
    q0 = layers[0].q
    D = q0.shape[2]
    out_code = _out_code(layers[0].out.dtype)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    nfull = sum(1 for L in layers if L.paged is not None)
    if workspace is None and nfull:
        hkv = next(L.paged.k.shape[1] for L in layers if L.paged is not None)
        workspace = torch.empty(hybrid_stack_fused_workspace_bytes(B, num_q_heads, hkv, D,
                                                                   max_seq_len, nfull),
                                dtype=torch.uint8, device=q0.device)
    _check(lib().phs_attn_decode_hybrid_stack_fused(
        arr, len(layers), num_q_heads, B, _ptr(block_table),
        0 if block_table is None else block_table.shape[1], _ptr(page_refcount),
        _ptr(seq_lens), int(max_seq_len),
        _ptr(ring_ids), _ptr(ring_pos), scale, out_code, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream)),
        "attn_decode_hybrid_stack_fused")


def hybrid_kv_tokens(layer_is_full, seq_lens_host, window):
    """(Full-layer tokens, SWA-layer tokens) held by a stack; host lists in."""
    import numpy as np
    lf = np.ascontiguousarray(layer_is_full, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    f, w = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().phs_hybrid_kv_tokens(lf.ctypes.data, lf.shape[0], sl.ctypes.data, sl.shape[0],
                                      int(window), ctypes.byref(f), ctypes.byref(w)),
           "hybrid_kv_tokens")
    return f.value, w.value


def copy_d2d(dst, src, stream=None):
    """HBM copy kernel: dst <- src (same byte size, 16-byte multiples)."""
    if dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("copy_d2d size mismatch")
    _check(lib().phs_copy_d2d(_ptr(dst), _ptr(src), src.numel() * src.element_size(),
                              _stream(stream)), "copy_d2d")


def read_checksum(src, sink, stream=None):
    """HBM read kernel: XOR every 32-bit word of `src` (contiguous, a
    multiple of 16 bytes) into sink[0] (CUDA int32 tensor, not cleared)."""
    _need(sink, torch.int32, "sink")
    if not src.is_contiguous():
        raise ValueError("src must be contiguous")
    _check(lib().phs_read_checksum(_ptr(src), src.numel() * src.element_size(), _ptr(sink),
                                   _stream(stream)), "read_checksum")


# ------------------------------------------------------- cache bookkeeping --
def copy_pages(pool: PagedPool, src_pages, dst_pages, status=None, stream=None):
    """Device copy of whole pages (K and V): dst_pages[i] <- src_pages[i]."""
    pc = pool.c()
    _need(src_pages, torch.int32, "src_pages", 1)
    _need(dst_pages, torch.int32, "dst_pages", 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_copy_pages(ctypes.byref(pc), _ptr(src_pages), _ptr(dst_pages),
                                src_pages.shape[0], _ptr(status), _stream(stream)), "copy_pages")


def _i32(a):
    import numpy as np
    return np.ascontiguousarray(a, dtype=np.int32)


class PageAllocator:
    """Refcounted page allocator (host object of the library)."""

    def __init__(self, num_pages: int):
        self.num_pages = int(num_pages)
        self._h = lib().phs_page_allocator_create(self.num_pages)
        if not self._h:
            raise ValueError("bad number of pages")

    def close(self):
        if self._h:
            lib().phs_page_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int):
        import numpy as np
        out = np.empty(max(int(n), 0), dtype=np.int32)
        _check(lib().phs_page_alloc(self._h, int(n), out.ctypes.data), "page_alloc")
        return out

    def incref(self, pages):
        p = _i32(pages)
        _check(lib().phs_page_incref(self._h, p.ctypes.data, p.shape[0]), "page_incref")

    def decref(self, pages):
        p = _i32(pages)
        _check(lib().phs_page_decref(self._h, p.ctypes.data, p.shape[0]), "page_decref")

    def free_count(self) -> int:
        return int(lib().phs_page_free_count(self._h))

    def refcounts(self):
        import numpy as np
        out = np.empty(self.num_pages, dtype=np.int32)
        _check(lib().phs_page_refcounts(self._h, out.ctypes.data), "page_refcounts")
        return out

    def cow(self, page: int) -> int:
        out = ctypes.c_int32()
        _check(lib().phs_page_cow(self._h, int(page), ctypes.byref(out)), "page_cow")
        return out.value


class RadixTree:
    """Radix prefix tree over whole pages, holding references in `alloc`
    (Full pages) and `swa_alloc` (SWA segment pages, optional)."""

    def __init__(self, alloc: PageAllocator, page_size: int = PAGE,
                 swa_alloc: PageAllocator | None = None):
        self.alloc = alloc
        self.swa_alloc = swa_alloc
        self.page_size = int(page_size)
        self._h = lib().phs_radix_create(alloc._h, None if swa_alloc is None else swa_alloc._h,
                                         self.page_size)
        if not self._h:
            raise ValueError("bad radix tree arguments")

    def close(self):
        if self._h:
            lib().phs_radix_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens):
        """Matched page ids (each gets a reference for the caller)."""
        import numpy as np
        t = _i32(tokens)
        cap = t.shape[0] // self.page_size + 1
        out = np.empty(cap, dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().phs_radix_match(self._h, t.ctypes.data, t.shape[0], out.ctypes.data, cap,
                                     ctypes.byref(n)), "radix_match")
        return out[:n.value].copy()

    def match_window_safe(self, tokens, window: int):
        """(Full pages, SWA segment pages of the last window) of the longest
        window-safe match; each id gets a reference for the caller."""
        import numpy as np
        t = _i32(tokens)
        cap = t.shape[0] // self.page_size + 1
        out = np.empty(cap, dtype=np.int32)
        seg = np.empty(cap, dtype=np.int32)
        n, ns = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().phs_radix_match_window_safe(self._h, t.ctypes.data, t.shape[0], int(window),
                                                 out.ctypes.data, cap, ctypes.byref(n),
                                                 seg.ctypes.data, cap, ctypes.byref(ns)),
               "radix_match_window_safe")
        return out[:n.value].copy(), seg[:ns.value].copy()

    def insert(self, tokens, pages, swa_pages=None):
        """Cache the whole pages of `tokens`; swa_pages: per page, the SWA
        segment page holding its SWA-layer KV, or -1 (None: none)."""
        t, p = _i32(tokens), _i32(pages)
        s = None if swa_pages is None else _i32(swa_pages)
        if s is not None and s.shape[0] < t.shape[0] // self.page_size:
            raise ValueError("swa_pages needs one entry per whole page")
        _check(lib().phs_radix_insert(self._h, t.ctypes.data, t.shape[0], p.ctypes.data,
                                      None if s is None else s.ctypes.data), "radix_insert")

    def evict(self, pages: int) -> int:
        freed = ctypes.c_int64()
        _check(lib().phs_radix_evict(self._h, int(pages), ctypes.byref(freed)), "radix_evict")
        return freed.value

    def cached_pages(self) -> int:
        return int(lib().phs_radix_cached_pages(self._h))


def _pool_array(ctype, pools):
    return (ctype * len(pools))(*[p.c() for p in pools])


def swa_ring_save(rings, segs, ring_ids, ring_pos, seq_lens, page_index, seg_pages, status=None,
                  stream=None):
    """Snapshot whole pages of requests' SWA windows into segment pages, in
    every SWA layer: entry i copies logical page page_index[i] of the
    request with ring ring_ids[i] (newest slot ring_pos[i], length
    seq_lens[i]) into segment page seg_pages[i].  rings: list of RingPool,
    segs: list of PagedPool (one per SWA layer)."""
    if len(rings) != len(segs) or not rings:
        raise ValueError("one segment pool per ring pool")
    for name, t in (("ring_ids", ring_ids), ("ring_pos", ring_pos), ("seq_lens", seq_lens),
                    ("page_index", page_index), ("seg_pages", seg_pages)):
        _need(t, torch.int32, name, 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_swa_ring_save(_pool_array(_lib.RingPoolC, rings),
                                   _pool_array(_lib.PagedPoolC, segs), len(rings),
                                   _ptr(ring_ids), _ptr(ring_pos), _ptr(seq_lens),
                                   _ptr(page_index), _ptr(seg_pages), page_index.shape[0],
                                   _ptr(status), _stream(stream)), "swa_ring_save")


def swa_ring_seed(rings, segs, ring_pos, seq_lens, seg_table, ring_ids=None, status=None,
                  stream=None):
    """Fill each request's ring, in every SWA layer, with the last
    min(n, W) tokens from the segment pages of its row of seg_table
    ([B, max_seg] int32), newest token at slot ring_pos[b]."""
    if len(rings) != len(segs) or not rings:
        raise ValueError("one segment pool per ring pool")
    _need(ring_pos, torch.int32, "ring_pos", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(seg_table, torch.int32, "seg_table", 2)
    _opt(ring_ids, torch.int32, "ring_ids", 1)
    _opt(status, torch.int32, "status")
    _check(lib().phs_swa_ring_seed(_pool_array(_lib.RingPoolC, rings),
                                   _pool_array(_lib.PagedPoolC, segs), len(rings),
                                   _ptr(ring_ids), _ptr(ring_pos), _ptr(seq_lens),
                                   _ptr(seg_table), seg_table.shape[1], seq_lens.shape[0],
                                   _ptr(status), _stream(stream)), "swa_ring_seed")


def window_safe_len(swa_valid, match_len: int, window: int, align: int = 1) -> int:
    import numpy as np
    v = np.ascontiguousarray(swa_valid, dtype=np.uint8)
    r = int(lib().phs_window_safe_len(v.ctypes.data, int(match_len), int(window), int(align)))
    _check(min(r, 0), "window_safe_len")
    return r
