// phs_merge.cuh -- cross-split log-sum-exp merge of split-KV partials,
// shared by the merge kernels and by the persistent SWA kernel (which takes
// the Full layers' merges of a hybrid-stack step as extra work).
//
// Source: the log-sum-exp identity of split softmax attention: with split
// partials (m_s, l_s, o_s) in the log2 domain, M = max m_s, L = sum l_s
// 2^(m_s - M), out = sum 2^(m_s - M) o_s / L.
#pragma once

#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int f32) {
  if (f32)
    reinterpret_cast<float*>(out)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// Number of splits of a request and validation of its INT8 length.
// Returns -1 if the request's lengths are invalid.
// The bf16 region starts at max(qlen, skip): tokens below `skip` (a shared
// prefix) are attended by another kernel.
__device__ __forceinline__ int request_splits(int n, int qlen, int T, int skip = 0) {
  if (n < 0 || qlen < 0 || qlen > n || (qlen % kQBlock) != 0 || n < skip) return -1;
  const int bf0 = max(qlen, skip);
  return (qlen + T - 1) / T + (n - bf0 + T - 1) / T;
}

// Merge of one (request b, KV head h): query rows row0, row0 + step, ...
// each by one whole warp.  The lanes first reduce (max m, sum l) over the
// splits in parallel, then each lane accumulates D/32 output columns over
// the splits with independent vector loads.
template <int D>
__device__ __forceinline__ void merge_request(const MergeArgs& a, const float* ws_o,
                                              const float* ws_ml, void* out, int b, int h,
                                              int row0, int step) {
  constexpr int V = D / 32;  // columns per lane (4 or 2)
  const int lane = threadIdx.x & 31;
  const int G = a.G;
  const int n = min(a.seq_lens[b], a.n_clamp);
  const int qlen = a.qlens ? a.qlens[b] : 0;
  const int ns = min(request_splits(n, qlen, a.T), a.max_splits);
  if (ns <= 1) return;
  const size_t part0 = (static_cast<size_t>(b) * a.Hkv + h) * a.max_splits;
  const size_t out_row0 = (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * G) * D;
  for (int row = row0; row < G; row += step) {
    const float2* ml = reinterpret_cast<const float2*>(ws_ml) + part0 * G + row;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, ml[static_cast<size_t>(s) * G].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Lsum = 0.f;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    const float* ob = ws_o + (part0 * G + row) * D + lane * V;
    for (int s0 = 0; s0 < ns; s0 += 32) {
      // weight of split s0 + lane, then broadcast one split at a time
      float wl = 0.f;
      if (s0 + lane < ns) {
        const float2 v = ml[static_cast<size_t>(s0 + lane) * G];
        wl = v.x == -INFINITY ? 0.f : exp2f(v.x - M);
        Lsum += v.y * wl;
      }
      const int cnt = min(32, ns - s0);
#pragma unroll 16
      for (int k = 0; k < cnt; ++k) {  // up to 16 split loads in flight per lane
        const float w = __shfl_sync(0xffffffffu, wl, k);
        const float* src = ob + static_cast<size_t>(s0 + k) * G * D;
        if constexpr (V == 4) {
          const float4 o = *reinterpret_cast<const float4*>(src);
          acc[0] += w * o.x;
          acc[1] += w * o.y;
          acc[2] += w * o.z;
          acc[3] += w * o.w;
        } else {
          const float2 o = *reinterpret_cast<const float2*>(src);
          acc[0] += w * o.x;
          acc[1] += w * o.y;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      store_out(out, out_row0 + static_cast<size_t>(row) * D + lane * V + i, acc[i] * inv,
                a.out_f32);
  }
}

// The same merge with one warp taking all G rows of (b, h), four rows at a
// time with their loads interleaved, so each group of rows costs the
// latency of one row (the persistent SWA kernel takes the Full layers'
// merges this way, one warp per (layer, request, KV head)).
template <int D>
__device__ __forceinline__ void merge_request_rows4(const MergeArgs& a, const float* ws_o,
                                                    const float* ws_ml, void* out, int b, int h) {
  constexpr int V = D / 32;  // columns per lane (4 or 2)
  constexpr int RB = 4;      // rows merged together
  const int lane = threadIdx.x & 31;
  const int G = a.G;
  const int n = min(a.seq_lens[b], a.n_clamp);
  const int qlen = a.qlens ? a.qlens[b] : 0;
  const int ns = min(request_splits(n, qlen, a.T), a.max_splits);
  if (ns <= 1) return;
  const size_t part0 = (static_cast<size_t>(b) * a.Hkv + h) * a.max_splits;
  const size_t out_row0 = (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * G) * D;
  const float2* ml = reinterpret_cast<const float2*>(ws_ml) + part0 * G;
  for (int r0 = 0; r0 < G; r0 += RB) {
    float M[RB], Lsum[RB], acc[RB][V];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      M[r] = -INFINITY;
      Lsum[r] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[r][i] = 0.f;
    }
    for (int s = lane; s < ns; s += 32)
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (r0 + r < G) M[r] = fmaxf(M[r], ml[static_cast<size_t>(s) * G + r0 + r].x);
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M[r] = fmaxf(M[r], __shfl_xor_sync(0xffffffffu, M[r], o));
    for (int s0 = 0; s0 < ns; s0 += 32) {
      float wl[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        wl[r] = 0.f;
        if (s0 + lane < ns && r0 + r < G) {
          const float2 v = ml[static_cast<size_t>(s0 + lane) * G + r0 + r];
          wl[r] = v.x == -INFINITY ? 0.f : exp2f(v.x - M[r]);
          Lsum[r] += v.y * wl[r];
        }
      }
      const int cnt = min(32, ns - s0);
#pragma unroll 4
      for (int k = 0; k < cnt; ++k) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float w = __shfl_sync(0xffffffffu, wl[r], k);
          if (r0 + r < G) {
            const float* src =
                ws_o + ((part0 + s0 + k) * G + r0 + r) * D + lane * V;
            if constexpr (V == 4) {
              const float4 o = *reinterpret_cast<const float4*>(src);
              acc[r][0] += w * o.x;
              acc[r][1] += w * o.y;
              acc[r][2] += w * o.z;
              acc[r][3] += w * o.w;
            } else {
              const float2 o = *reinterpret_cast<const float2*>(src);
              acc[r][0] += w * o.x;
              acc[r][1] += w * o.y;
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (r0 + r >= G) break;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Lsum[r] += __shfl_xor_sync(0xffffffffu, Lsum[r], o);
      const float inv = Lsum[r] > 0.f ? 1.f / Lsum[r] : 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i)
        store_out(out, out_row0 + static_cast<size_t>(r0 + r) * D + lane * V + i,
                  acc[r][i] * inv, a.out_f32);
    }
  }
}

}  // namespace phs
