// phs_append.cu -- KV append into the paged Full pool or the SWA rings (one
// or many layers per launch), and the plain HBM copy kernel used as the
// in-run bandwidth yardstick.
//
// Sources: "Kimi K3 context caching" page, section 1 (a request extending a
// shared prefix writes only into blocks of its own; shared blocks are held
// by reference count) and "Xiaomi MiMo-V2.5 inference system" page,
// section 2 (Full pool grows on demand; SWA ring evicts by window).
#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

// grid (B, layers); one thread per 16-byte piece of one head's K and V row.
template <int MAXL>
__global__ void phs_append_kernel(const __grid_constant__ AppendParams<MAXL> p) {
  const int b = blockIdx.x, li = blockIdx.y;
  const int per_head = p.D / 8;  // 16-byte pieces per row
  const int t = threadIdx.x;
  if (t >= p.Hkv * per_head) return;
  const int h = t / per_head, piece = t % per_head;
  const AppendLayer& L = p.layer[li];
  int64_t row;  // destination row (token slot) in units of D elements
  if (p.is_ring) {
    const int r = p.table ? p.table[b] : b;
    const int slot = p.ring_pos[b];
    if (r < 0 || r >= L.num || slot < 0 || slot >= p.W) {
      if (t == 0) set_status(p.status, PHS_ERANGE);
      return;
    }
    row = (static_cast<int64_t>(r) * p.Hkv + h) * p.W + slot;
  } else {
    const int n = p.seq_lens[b];
    if (n < 1) return;
    const int tok = n - 1;
    const int lp = tok / kPage;
    if (lp >= p.max_pages) {
      if (t == 0) set_status(p.status, PHS_ERANGE);
      return;
    }
    const int page = p.table[static_cast<size_t>(b) * p.max_pages + lp];
    if (page < 0 || page >= L.num) {
      if (t == 0) set_status(p.status, PHS_ERANGE);
      return;
    }
    if (p.refcount && p.refcount[page] != 1) {
      if (t == 0) set_status(p.status, PHS_ESHARED);
      return;
    }
    row = (static_cast<int64_t>(page) * p.Hkv + h) * kPage + tok % kPage;
  }
  const size_t src = (static_cast<size_t>(b) * p.Hkv + h) * p.D / 8 + piece;
  const size_t dst = static_cast<size_t>(row) * p.D / 8 + piece;
  reinterpret_cast<uint4*>(L.k)[dst] = reinterpret_cast<const uint4*>(L.k_new)[src];
  reinterpret_cast<uint4*>(L.v)[dst] = reinterpret_cast<const uint4*>(L.v_new)[src];
}

template <int MAXL>
int launch_append(const AppendParams<MAXL>& p, cudaStream_t stream) {
  if (p.B <= 0 || p.num_layers <= 0) return PHS_OK;
  const int threads = ((p.Hkv * p.D / 8) + 31) / 32 * 32;
  dim3 grid(p.B, p.num_layers);
  phs_append_kernel<MAXL><<<grid, threads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

template int launch_append<1>(const AppendParams<1>&, cudaStream_t);
template int launch_append<kAppendMaxLayers>(const AppendParams<kAppendMaxLayers>&, cudaStream_t);

// ------------------------------------------------- SWA segment pages --
// Save: CTA (i, layer) copies the 16 tokens of logical page page_index[i]
// of a request from its ring into segment page seg_pages[i].  Seed: CTA
// (b, layer) copies the last min(n, W) tokens of request b from the
// segment pages listed in its row of seg_table into its ring.  Token t of
// a request of length n sits at ring slot (ring_pos - (n - 1 - t)) mod W.
// One thread per 16-byte piece of a token's row (all KV heads), K and V.
template <int MAXL>
__global__ void __launch_bounds__(256) phs_swa_segment_kernel(
    const __grid_constant__ SegCopyParams<MAXL> p) {
  const int i = blockIdx.x;
  const SegCopyLayer& L = p.layer[blockIdx.y];
  const int W = p.W, pieces = p.Hkv * p.D / 8;  // 16-byte pieces per token row
  const int r = p.ring_ids ? p.ring_ids[i] : i;
  const int pos = p.ring_pos[i];
  const int n = p.seq_lens[i];
  if (r < 0 || r >= L.num_rings || pos < 0 || pos >= W || n < 0) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(p.status, PHS_ERANGE);
    return;
  }
  const int t_lo = n - min(n, W);  // the window [t_lo, n)
  int t0, t1, fp = 0;
  int seg = -1;
  if (p.save) {
    t0 = p.page_index[i] * kPage;
    t1 = t0 + kPage;
    seg = p.seg_pages[i];
    if (p.page_index[i] < 0 || t0 < t_lo || t1 > n || seg < 0 || seg >= L.num_seg) {
      if (threadIdx.x == 0 && blockIdx.y == 0) set_status(p.status, PHS_ERANGE);
      return;
    }
  } else {
    t0 = t_lo;
    t1 = n;
    fp = t_lo / kPage;
  }
  const int D8 = p.D / 8;
  for (int e = threadIdx.x; e < (t1 - t0) * pieces; e += blockDim.x) {
    const int t = t0 + e / pieces, rem = e % pieces;
    const int h = rem / D8, c = rem % D8;
    int sp = seg;
    if (!p.save) {
      const int j = t / kPage - fp;
      sp = j < p.max_seg ? p.seg_table[static_cast<size_t>(i) * p.max_seg + j] : -1;
      if (sp < 0 || sp >= L.num_seg) {
        set_status(p.status, PHS_ERANGE);
        continue;
      }
    }
    int slot = (pos - (n - 1 - t)) % W;
    if (slot < 0) slot += W;
    const size_t ring_row = (static_cast<size_t>(r) * p.Hkv + h) * W + slot;
    const size_t seg_row = (static_cast<size_t>(sp) * p.Hkv + h) * kPage + t % kPage;
    const size_t ro = ring_row * D8 + c, so = seg_row * D8 + c;
    if (p.save) {
      reinterpret_cast<uint4*>(L.seg_k)[so] = reinterpret_cast<const uint4*>(L.ring_k)[ro];
      reinterpret_cast<uint4*>(L.seg_v)[so] = reinterpret_cast<const uint4*>(L.ring_v)[ro];
    } else {
      reinterpret_cast<uint4*>(L.ring_k)[ro] = reinterpret_cast<const uint4*>(L.seg_k)[so];
      reinterpret_cast<uint4*>(L.ring_v)[ro] = reinterpret_cast<const uint4*>(L.seg_v)[so];
    }
  }
}

template <int MAXL>
int launch_swa_segment(const SegCopyParams<MAXL>& p, int count, cudaStream_t stream) {
  if (count <= 0 || p.num_layers <= 0) return PHS_OK;
  dim3 grid(count, p.num_layers);
  phs_swa_segment_kernel<MAXL><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

template int launch_swa_segment<kSegMaxLayers>(const SegCopyParams<kSegMaxLayers>&, int,
                                               cudaStream_t);

// ------------------------------------------------------------ page copy --
// grid (n, 2): CTA (i, kv) copies page src[i] -> dst[i] of K (kv 0) or V.
__global__ void __launch_bounds__(256) phs_copy_pages_kernel(uint4* k, uint4* v,
                                                             const int32_t* src,
                                                             const int32_t* dst, int64_t num_pages,
                                                             int page_vecs, int32_t* status) {
  const int i = blockIdx.x;
  const int s = src[i], d = dst[i];
  if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(status, PHS_ERANGE);
    return;
  }
  uint4* base = blockIdx.y ? v : k;
  const uint4* from = base + static_cast<size_t>(s) * page_vecs;
  uint4* to = base + static_cast<size_t>(d) * page_vecs;
  for (int e = threadIdx.x; e < page_vecs; e += blockDim.x) to[e] = from[e];
}

int launch_copy_pages(void* k, void* v, const int32_t* src, const int32_t* dst, int32_t n,
                      int64_t num_pages, int page_bytes, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return PHS_OK;
  dim3 grid(n, 2);
  phs_copy_pages_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<uint4*>(k),
                                                  reinterpret_cast<uint4*>(v), src, dst,
                                                  num_pages, page_bytes / 16, status);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

// ------------------------------------------------------------------ copy --
__global__ void __launch_bounds__(512) phs_copy_kernel(uint4* __restrict__ dst,
                                                       const uint4* __restrict__ src, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = __ldcs(src + i);
    const uint4 b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride);
    const uint4 d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// ------------------------------------------------------------------ read --
// Streaming read of the whole buffer: every 32-bit word XOR-folded, one
// warp-reduced word per warp XORed into *sink (the result is the XOR of all
// words, independent of the launch shape).  Four 16-byte loads in flight per
// thread, like the copy kernel, but no stores: the read-side yardstick.
__global__ void __launch_bounds__(512) phs_read_kernel(const uint4* __restrict__ src, size_t n,
                                                       uint32_t* sink) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = __ldcs(src + i);
    const uint4 b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride);
    const uint4 d = __ldcs(src + i + 3 * stride);
    acc ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^
           (d.x ^ d.y ^ d.z ^ d.w);
  }
  for (; i < n; i += stride) {
    const uint4 a = __ldcs(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0u) atomicXor(sink, acc);
}

// 16 blocks of 512 threads per SM (four waves of resident blocks): measured
// on GB300 over 4 GiB, 7.41 TB/s against 7.13-7.22 TB/s with 2 or 4 blocks
// per SM (and 8 loads in flight per thread did not help).
int launch_read(const void* src, size_t bytes, int num_sms, uint32_t* sink, cudaStream_t stream) {
  const size_t n = bytes / 16;
  if (n == 0) return PHS_OK;
  size_t blocks = static_cast<size_t>(num_sms) * 16;
  const size_t need = (n + 511) / 512;
  if (blocks > need) blocks = need;
  phs_read_kernel<<<static_cast<unsigned>(blocks), 512, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), n, sink);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int launch_copy(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t stream) {
  const size_t n = bytes / 16;
  if (n == 0) return PHS_OK;
  size_t blocks = static_cast<size_t>(num_sms) * 4;
  const size_t need = (n + 511) / 512;
  if (blocks > need) blocks = need;
  phs_copy_kernel<<<static_cast<unsigned>(blocks), 512, 0, stream>>>(
      reinterpret_cast<uint4*>(dst), reinterpret_cast<const uint4*>(src), n);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

}  // namespace phs
