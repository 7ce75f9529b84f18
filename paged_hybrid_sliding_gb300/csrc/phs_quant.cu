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
// token rows with 16-byte streaming loads, keeps the group in registers,
// reduces the absmax in packed bf16 and with shuffles, and writes the codes
// with 8-byte stores.
#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

// Magic-number rounding: for |y| < 2^22, fl(y + 1.5 * 2^23) rounds y to the
// nearest integer (ties to even, the default rounding) and keeps it in the
// low mantissa bits, so the code byte is the low byte of the sum's bits.
constexpr float kRoundMagic = 12582912.0f;

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
  // the group's 32 tokens live in source pages 2j and 2j+1
  int page = -1;
  if (lane < 2) {
    const int lp = 2 * j + lane;
    page = lp < a.src_max_pages ? a.src_table[static_cast<size_t>(b) * a.src_max_pages + lp] : -1;
  }
  const int page0 = __shfl_sync(0xffffffffu, page, 0);
  const int page1 = __shfl_sync(0xffffffffu, page, 1);
  if (page0 < 0 || page0 >= a.num_pages || page1 < 0 || page1 >= a.num_pages) {
    if (lane == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  const __nv_bfloat16* src = warp ? a.v_src : a.k_src;
  int8_t* codes = warp ? a.v_codes : a.k_codes;
  float* scales = warp ? a.v_scale : a.k_scale;
  const int piece = lane % kPieces;

  uint4 x[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int tt = it * kRowsPerIt + lane / kPieces;  // token within the group
    const int pg = tt < kPage ? page0 : page1;
    const size_t off = ((static_cast<size_t>(pg) * a.Hkv + h) * kPage + (tt % kPage)) * D +
                       piece * 8;
    x[it] = __ldcs(reinterpret_cast<const uint4*>(src + off));
  }
  // absmax in packed bf16 (exact: the max of |x| is one of the inputs)
  __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&x[it]);
#pragma unroll
    for (int k = 0; k < 4; ++k) m2 = __hmax2(m2, __habs2(v[k]));
  }
  float amax = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  const float rs = s != 0.f ? __fdiv_rn(1.0f, s) : 0.f;
  // code = rint(x / s) with x / s the IEEE quotient.  y = x * fl(1/s) is
  // within |x/s| * (2^-23 + 2^-48) + ulp/2 <= 1.9e-5 of that quotient (|x/s|
  // <= 127.5), so rint(y) equals rint(x / s) unless y lies within 1.9e-5 of
  // a half-integer; those rare elements take the IEEE division itself.  A
  // scale so small that 1/s overflows (subnormal groups) always divides.
  // |rint(x / s)| <= 127 by construction, so no clamp is needed.  s == 0
  // gives rs == 0 and every code 0.
  const bool always_divide = !(rs < INFINITY);
  auto code = [s, rs, always_divide](float v) -> uint32_t {
    const float y = __fmul_rn(v, rs);
    float t = __fadd_rn(y, kRoundMagic);
    const float r = __fsub_rn(t, kRoundMagic);
    if (always_divide || fabsf(__fsub_rn(y, r)) > 0.4999f)
      t = __fadd_rn(rintf(__fdiv_rn(v, s)), kRoundMagic);
    return __float_as_uint(t);  // code in the low byte
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
      const uint32_t lo = __byte_perm(code(f0.x), code(f0.y), 0x0040);
      const uint32_t hi = __byte_perm(code(f1.x), code(f1.y), 0x0040);
      w[k] = __byte_perm(lo, hi, 0x5410);
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
