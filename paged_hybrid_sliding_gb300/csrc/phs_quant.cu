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
// One CTA of four warps per (request, block, KV head): warps 0-1 quantise
// K, warps 2-3 V, each warp one 16-token source page (a contiguous tile read
// with 16-byte streaming loads and kept in registers).  The two halves of a
// group combine their absmax through shared memory; codes go out with
// 8-byte stores in the same piece order.
#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

// Magic-number rounding: for |y| < 2^22, fl(y + 1.5 * 2^23) rounds y to the
// nearest integer (ties to even, the default rounding) and keeps it in the
// low mantissa bits, so the code byte is the low byte of the sum's bits.
constexpr float kRoundMagic = 12582912.0f;

template <int D>
__global__ void __launch_bounds__(128) phs_quant_kernel(const QuantArgs a) {
  constexpr int kPieces = D / 8;              // 16-byte pieces per token row
  constexpr int kIters = kPage * kPieces / 32;  // pieces of one page tile per lane
  const int jr = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int which = warp >> 1;  // 0 = K, 1 = V
  const int half = warp & 1;    // tokens 16*half .. 16*half+15 = source page 2j+half
  __shared__ float s_amax[4];
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
  const int lp = 2 * j + half;
  const int page =
      lp < a.src_max_pages ? a.src_table[static_cast<size_t>(b) * a.src_max_pages + lp] : -1;
  const bool bad = page < 0 || page >= a.num_pages;  // uniform per warp
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  const __nv_bfloat16* src = which ? a.v_src : a.k_src;
  int8_t* codes = which ? a.v_codes : a.k_codes;
  float* scales = which ? a.v_scale : a.k_scale;
  // one contiguous 16 x D tile: lane takes 16-byte pieces lane, lane + 32, ...
  const uint4* tile =
      reinterpret_cast<const uint4*>(src + (static_cast<size_t>(page) * a.Hkv + h) * kPage * D);
  uint4 x[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) x[it] = __ldcs(tile + it * 32 + lane);
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
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  amax = fmaxf(s_amax[2 * which], s_amax[2 * which + 1]);  // whole 32-token group
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
  // codes of this page tile: rows 16*half .. of INT8 page qp, same piece order
  uint2* out = reinterpret_cast<uint2*>(codes + ((static_cast<size_t>(qp) * a.Hkv + h) * kQBlock +
                                                 kPage * half) * D);
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
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
    out[it * 32 + lane] = make_uint2(w[0], w[1]);
  }
  if (threadIdx.x == 64 * which && half == 0) scales[static_cast<size_t>(qp) * a.Hkv + h] = s;
}

int launch_quant(const QuantArgs& a, int max_qblocks, int B, cudaStream_t stream) {
  if (max_qblocks <= 0 || B <= 0) return PHS_OK;
  dim3 grid(max_qblocks, B, a.Hkv);
  if (a.D == 128)
    phs_quant_kernel<128><<<grid, 128, 0, stream>>>(a);
  else if (a.D == 64)
    phs_quant_kernel<64><<<grid, 128, 0, stream>>>(a);
  else
    return PHS_EUNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

}  // namespace phs
