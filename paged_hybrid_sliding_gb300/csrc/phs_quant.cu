// phs_quant.cu -- block-32 INT8 KV quantiser.
//
// Source: "Kimi K2.5 architecture deep dive" page, sections 2.2-2.3: the
// warm zone of the KV cache is held as INT8 with block-wise quantisation,
// one scale calibrated per group of 32 tokens.  A group here is 32
// consecutive tokens x D dims of one KV head, K and V separately:
//     a = max |x|,  s = a / 127,  code = clamp(rint(x / s), -127, 127)
// in IEEE single precision (division rounded to nearest even, rint rounding
// half to even; a == 0 gives s = 0 and codes 0).
//
// One CTA of two warps per (request, block, KV head): warp 0 quantises K,
// warp 1 V.  Each warp load covers two (D = 128) or four (D = 64) whole
// token rows with 16-byte loads, keeps the group in registers, reduces the
// absmax with shuffles and writes the codes with 8-byte stores.
#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

template <int D>
__global__ void __launch_bounds__(64) phs_quant_kernel(const QuantArgs a) {
  constexpr int kPieces = D / 8;          // 16-byte pieces per token row
  constexpr int kRowsPerIt = 32 / kPieces;
  constexpr int kIters = kQBlock / kRowsPerIt;
  const int jr = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (jr >= a.num_qblocks[b]) return;
  const int j = a.first_qblock[b] + jr;
  if (j < 0 || j >= a.dst_max_qpages) {
    if (threadIdx.x == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  const int qp = a.dst_qtable[static_cast<size_t>(b) * a.dst_max_qpages + j];
  if (qp < 0 || qp >= a.num_qpages) {
    if (threadIdx.x == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  const __nv_bfloat16* src = warp ? a.v_src : a.k_src;
  int8_t* codes = warp ? a.v_codes : a.k_codes;
  float* scales = warp ? a.v_scale : a.k_scale;
  const int piece = lane % kPieces;

  uint4 x[kIters];
  bool bad = false;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int tt = it * kRowsPerIt + lane / kPieces;  // token within the group
    const int t = j * kQBlock + tt;
    const int lp = t / kPage;
    int page = lp < a.src_max_pages ? a.src_table[static_cast<size_t>(b) * a.src_max_pages + lp] : -1;
    if (page < 0 || page >= a.num_pages) {
      bad = true;
      page = 0;
    }
    const size_t off = ((static_cast<size_t>(page) * a.Hkv + h) * kPage + t % kPage) * D + piece * 8;
    x[it] = *reinterpret_cast<const uint4*>(src + off);
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&x[it]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(v[k]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  auto code = [s](float v) -> uint32_t {
    if (s == 0.f) return 0u;
    int c = __float2int_rn(__fdiv_rn(v, s));
    c = max(-127, min(127, c));
    return static_cast<uint32_t>(c) & 0xFFu;
  };
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int tt = it * kRowsPerIt + lane / kPieces;
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&x[it]);
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 f0 = __bfloat1622float2(v[2 * k]);
      const float2 f1 = __bfloat1622float2(v[2 * k + 1]);
      w[k] = code(f0.x) | (code(f0.y) << 8) | (code(f1.x) << 16) | (code(f1.y) << 24);
    }
    const size_t off = ((static_cast<size_t>(qp) * a.Hkv + h) * kQBlock + tt) * D + piece * 8;
    *reinterpret_cast<uint2*>(codes + off) = make_uint2(w[0], w[1]);
  }
  if (lane == 0) scales[static_cast<size_t>(qp) * a.Hkv + h] = s;
}

int launch_quant(const QuantArgs& a, int max_qblocks, int B, cudaStream_t stream) {
  if (max_qblocks <= 0 || B <= 0) return PHS_OK;
  dim3 grid(max_qblocks, B, a.Hkv);
  if (a.D == 128)
    phs_quant_kernel<128><<<grid, 64, 0, stream>>>(a);
  else if (a.D == 64)
    phs_quant_kernel<64><<<grid, 64, 0, stream>>>(a);
  else
    return PHS_EUNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

}  // namespace phs
