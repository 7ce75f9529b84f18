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
// K, warps 2-3 V, each warp one 16-token source page, brought into shared
// memory by one 1-D bulk copy.  The two halves of a group combine their
// absmax through shared memory.

// Stored form (the layout the decode kernels' fragments want): each code
// is kept as the byte x + 128.  K codes are token-major, 32 rows of D bytes
// per block and head, written with 8-byte stores in piece order.  V codes
// are transposed per 16-token half: D rows of 16 bytes (one per head dim)
// for tokens 0-15, then D rows for tokens 16-31; byte p of a row holds
// token kI8VtToken(p) of its half.  Each V warp stages its 16 tokens' codes
// in shared memory and writes its half (2 KB, contiguous).
#include "phs_common.cuh"
#include "phs_internal.h"

namespace phs {

// Magic-number rounding: for |y| < 2^22, fl(y + 1.5 * 2^23) rounds y to the
// nearest integer (ties to even, the default rounding) and keeps it in the
// low mantissa bits.  With 128 added to the constant (128 is even, so the
// ties still go to even) the low byte of the sum's bits is the stored byte
// x + 128.
constexpr float kRoundMagicOffset = 12582912.0f + 128.0f;

// Packed fp32 pairs (two lanes of work per instruction on the FMA pipe,
// each rounded to nearest as the scalar instruction would) and the
// three-input min / max.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int D>
// CTAs per SM: each holds its four source pages in shared memory (20.6 KB
// with the V staging), which allows 10 per SM.  Bulk copies instead of
// register-held 16-byte loads free the registers a tile occupied in
// flight, so more CTAs, and 160 KB of copies, fit on an SM (set-up of the
// INT8 workload at batch 32, 12.7 GB: 2.09 -> 1.96 ms, 0.91 -> 0.97 of the
// measured copy rate).
#ifndef PHS_QUANT_MIN_CTAS
#define PHS_QUANT_MIN_CTAS 10
#endif
__global__ void __launch_bounds__(128, PHS_QUANT_MIN_CTAS) phs_quant_kernel(const QuantArgs a) {
  constexpr int kPieces = D / 8;              // 16-byte pieces per token row
  constexpr int kIters = kPage * kPieces / 32;  // pieces of one page tile per lane
  const int jr = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int which = warp >> 1;  // 0 = K, 1 = V
  const int half = warp & 1;    // tokens 16*half .. 16*half+15 = source page 2j+half
  __shared__ float s_amax[4];
  __shared__ __align__(16) uint8_t s_v[kQBlock * D];  // V codes, token-major
  __shared__ __align__(128) uint8_t s_src[4][kPage * D * 2];  // each warp's source page
  __shared__ __align__(8) uint64_t s_bar[4];
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
  uint8_t* codes = which ? a.v_codes : a.k_codes;
  float* scales = which ? a.v_scale : a.k_scale;
  // one contiguous 16 x D tile: lane takes 16-byte pieces lane, lane + 32, ...
  const uint4* tile =
      reinterpret_cast<const uint4*>(src + (static_cast<size_t>(page) * a.Hkv + h) * kPage * D);
  // the page tile by one bulk copy into this warp's shared-memory slot (no
  // registers held while it is in flight)
  const uint32_t bar = smem_u32(&s_bar[warp]);
  const uint4* stile = reinterpret_cast<const uint4*>(s_src[warp]);
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kPage * D * 2);
    bulk_load(smem_u32(s_src[warp]), tile, kPage * D * 2, bar);
  }
  __syncwarp();
  const bool got = __all_sync(0xffffffffu, mbar_wait(bar, 0));
  if (!__syncthreads_and(got)) {
    if (lane == 0) {
      set_status(a.status, PHS_ETIMEOUT);
      (void)mbar_wait(bar, 0);  // drain (bounded) before the CTA exits
    }
    return;
  }
  // absmax in packed bf16 (exact: the max of |x| is one of the inputs).
  // max.xorsign.abs keeps max(|a|, |b|) as the magnitude (its sign is
  // dropped below): one instruction per pair
  uint32_t m2 = 0u;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const uint4 xv = stile[it * 32 + lane];
    const uint32_t* v = reinterpret_cast<const uint32_t*>(&xv);
#pragma unroll
    for (int k = 0; k < 4; ++k) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(v[k]));
  }
  m2 &= 0x7FFF7FFFu;
  float amax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
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
  // a half-integer: a group of 8 codes holding such an element takes the
  // IEEE division for all 8 (rare).  A scale so small that 1/s overflows
  // (subnormal groups) always divides.  |rint(x / s)| <= 127 by
  // construction, so no clamp is needed.  s == 0 gives rs == 0 and every
  // code 0.  The rounding steps run on packed pairs (two elements per
  // instruction, each rounded as the scalar operation would be).
  const bool always_divide = !(rs < INFINITY);
  const uint64_t rs2 = f2_pack(rs, rs), magic2 = f2_pack(kRoundMagicOffset, kRoundMagicOffset);
  const size_t block = static_cast<size_t>(qp) * a.Hkv + h;  // (block, head) of 32 x D codes
  // K: straight to the pool; V: into the shared token-major tile
  uint2* out = which ? reinterpret_cast<uint2*>(s_v + kPage * half * D)
                     : reinterpret_cast<uint2*>(codes + (block * kQBlock + kPage * half) * D);
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const uint4 xv = stile[it * 32 + lane];
    const uint32_t* v = reinterpret_cast<const uint32_t*>(&xv);
    uint32_t t[8];  // fl(rint(code) + 1.5 * 2^23): the code in the low byte
    float dmax = 0.f, dmin = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // bf16 pair -> fp32 pair: the bf16 bits are the high half of the fp32
      const uint64_t f = f2_pack(__uint_as_float(v[k] << 16), __uint_as_float(v[k] & 0xFFFF0000u));
      const uint64_t y = f2_mul(f, rs2);
      const uint64_t tt = f2_add(y, magic2);
      const uint64_t d = f2_sub(y, f2_sub(tt, magic2));  // y - rint(y), in [-1/2, 1/2]
      const float2 dd = f2_unpack(d), tf = f2_unpack(tt);
      dmax = fmax3(dmax, dd.x, dd.y);
      dmin = fmin3(dmin, dd.x, dd.y);
      t[2 * k] = __float_as_uint(tf.x);
      t[2 * k + 1] = __float_as_uint(tf.y);
    }
    if (always_divide || dmax > 0.4999f || dmin < -0.4999f) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xv = __uint_as_float(e & 1 ? v[e >> 1] & 0xFFFF0000u : v[e >> 1] << 16);
        t[e] = __float_as_uint(__fadd_rn(rintf(__fdiv_rn(xv, s)), kRoundMagicOffset));
      }
    }
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t lo = __byte_perm(t[4 * k], t[4 * k + 1], 0x0040);
      const uint32_t hi = __byte_perm(t[4 * k + 2], t[4 * k + 3], 0x0040);
      w[k] = __byte_perm(lo, hi, 0x5410);
    }
    out[it * 32 + lane] = make_uint2(w[0], w[1]);
  }
  if (threadIdx.x == 64 * which && half == 0) scales[block] = s;
  if (which) {
    // V^T: each V warp transposes its own 16-token half (the rows it just
    // staged), lane w taking dims 4w..4w+3.  Output word q of a dim's
    // 16-byte row holds tokens 2q, 2q+1, 2q+8, 2q+9 of the half
    // (kI8VtToken): the 4 x 4 byte transpose of those 4 token rows' words w
    // (two levels of byte permutes).
    __syncwarp();
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(s_v);
    uint4* vt = reinterpret_cast<uint4*>(codes + block * kQBlock * D);
    constexpr int W = D / 4;  // words per token row
    for (int w = lane; w < W; w += 32) {
      uint32_t o[4][4];  // [dim k][word q]
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t0 = 16 * half + kI8VtToken(4 * q);  // tokens t0, t0+1, t0+8, t0+9
        const uint32_t r0 = sw[t0 * W + w], r1 = sw[(t0 + 1) * W + w];
        const uint32_t r2 = sw[(t0 + 8) * W + w], r3 = sw[(t0 + 9) * W + w];
        const uint32_t a = __byte_perm(r0, r1, 0x5140), b = __byte_perm(r0, r1, 0x7362);
        const uint32_t c = __byte_perm(r2, r3, 0x5140), d = __byte_perm(r2, r3, 0x7362);
        o[0][q] = __byte_perm(a, c, 0x5410);
        o[1][q] = __byte_perm(a, c, 0x7632);
        o[2][q] = __byte_perm(b, d, 0x5410);
        o[3][q] = __byte_perm(b, d, 0x7632);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        vt[half * D + 4 * w + k] = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
    }
  }
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
