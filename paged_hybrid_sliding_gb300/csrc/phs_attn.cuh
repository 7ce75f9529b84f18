// phs_attn.cuh -- warp-level building blocks of single-query decode
// attention over 16-token bf16 chunks and 32-token INT8 chunks staged in
// shared memory by TMA with the 128-byte swizzle.
//
// One warp owns one (request, KV head) reduction at a time and packs the
// G = Hq/Hkv query heads of the group into the rows of a 16-row mma tile,
// so every K/V byte read from HBM serves all G heads (GQA packing).  The
// scores S = Q K^T and the update O += P V are m16n8k16 mma.sync
// contractions; the online softmax runs on the accumulator fragments with
// quad shuffles.  The math is the textbook softmax(q K^T * scale) V; the
// running max is kept in the log2 domain (scores pre-multiplied by
// scale * log2(e)) so that each exponential is one exp2f.
#pragma once

#include "phs_common.cuh"

namespace phs {

// swizzled byte offset inside a tile written by TMA with
// CU_TENSOR_MAP_SWIZZLE_128B (tile base 1024-byte aligned)
__device__ __forceinline__ uint32_t swz128(uint32_t off) {
  return off ^ (((off >> 7) & 7u) << 4);
}
// ... and with CU_TENSOR_MAP_SWIZZLE_64B (tile base 512-byte aligned)
__device__ __forceinline__ uint32_t swz64(uint32_t off) { return off ^ (((off >> 7) & 3u) << 4); }

// Bytes of one staged chunk: K + V of 16 bf16 tokens, or of 32 INT8 tokens.
template <int D>
struct ChunkGeom {
  static constexpr int kTileBytes = 16 * D * 2;   // one bf16 16 x D tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSubTiles = D / 64;        // 64-column (128-byte) boxes
  static constexpr int kI8RowBytes = D;           // INT8 row = D bytes
};

// Running state of one warp's softmax reduction.  Rows g (and g+8 when the
// group exceeds 8 heads) are this lane's query heads; the lane holds the
// output columns of its accumulator fragments.
template <int D, bool TWO>
struct WarpState {
  float o[D / 8][4];  // bf16-path layout: o[nt][0..1] = (row g, d 8nt+2q..+1)
  float m[2];         // running max (log2 domain), rows g and g+8
  float l[2];         // this lane's partial sum of exp2 (quad-reduced at the end)
  float u;            // INT8 path: output is stored divided by this V scale

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    u = 1.f;
  }
};

// Q fragments of the group for the bf16 path (standard k order) and for the
// INT8 path (f16, k order matching the ldmatrix layout of 8-bit rows, see
// consume_i8).  Rows >= G are zero.
template <int D, bool TWO>
struct QFrags {
  uint32_t a[D / 16][4];
};

template <int D, bool TWO>
__device__ __forceinline__ void load_q_bf16(QFrags<D, TWO>& f, const __nv_bfloat16* q, int G,
                                            int lane) {
  const int g = lane >> 2, qd = lane & 3;
  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(q);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c0 = 16 * ks + 2 * qd, c1 = c0 + 8;
    f.a[ks][0] = g < G ? __ldg(q32 + (g * D + c0) / 2) : 0u;
    f.a[ks][2] = g < G ? __ldg(q32 + (g * D + c1) / 2) : 0u;
    if (TWO) {
      f.a[ks][1] = g + 8 < G ? __ldg(q32 + ((g + 8) * D + c0) / 2) : 0u;
      f.a[ks][3] = g + 8 < G ? __ldg(q32 + ((g + 8) * D + c1) / 2) : 0u;
    } else {
      f.a[ks][1] = f.a[ks][3] = 0u;
    }
  }
}

// Same, from a row-major [G][D] bf16 copy of the group's queries in shared
// memory.
template <int D, bool TWO>
__device__ __forceinline__ void load_q_bf16_smem(QFrags<D, TWO>& f, uint32_t sq, int G, int lane) {
  const int g = lane >> 2, qd = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c0 = 16 * ks + 2 * qd, c1 = c0 + 8;
    f.a[ks][0] = g < G ? lds32(sq + (g * D + c0) * 2) : 0u;
    f.a[ks][2] = g < G ? lds32(sq + (g * D + c1) * 2) : 0u;
    if (TWO) {
      f.a[ks][1] = g + 8 < G ? lds32(sq + ((g + 8) * D + c0) * 2) : 0u;
      f.a[ks][3] = g + 8 < G ? lds32(sq + ((g + 8) * D + c1) * 2) : 0u;
    } else {
      f.a[ks][1] = f.a[ks][3] = 0u;
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w);
  float2 f = __bfloat1622float2(b);
  return pack_f16(f.x, f.y);
}

// INT8 path: A fragment for k-step ks holds physical columns
// 16ks + 4q .. 16ks + 4q + 3 of each row (see consume_i8).
template <int D, bool TWO>
__device__ __forceinline__ void load_q_f16_i8order(QFrags<D, TWO>& f, const __nv_bfloat16* q,
                                                   int G, int lane) {
  const int g = lane >> 2, qd = lane & 3;
  const uint2* q64 = reinterpret_cast<const uint2*>(q);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c = 16 * ks + 4 * qd;  // 4 consecutive columns, 8 bytes
    uint2 w0 = g < G ? __ldg(q64 + (g * D + c) / 4) : make_uint2(0, 0);
    f.a[ks][0] = bf16x2_to_f16x2(w0.x);
    f.a[ks][2] = bf16x2_to_f16x2(w0.y);
    if (TWO) {
      uint2 w1 = g + 8 < G ? __ldg(q64 + ((g + 8) * D + c) / 4) : make_uint2(0, 0);
      f.a[ks][1] = bf16x2_to_f16x2(w1.x);
      f.a[ks][3] = bf16x2_to_f16x2(w1.y);
    } else {
      f.a[ks][1] = f.a[ks][3] = 0u;
    }
  }
}

// Zero the V rows of tokens whose bit in `valid` is clear, so that
// never-written slots (possibly NaN bit patterns) cannot reach the PV
// product through 0 * NaN.  Generic-proxy writes: the caller issues a
// proxy fence before this stage is refilled by TMA.
template <int D>
__device__ __forceinline__ void zero_invalid_v_rows(uint8_t* sV, uint32_t valid, int lane) {
  constexpr int kChunks = 16 * D * 2 / 16;  // 16-byte units in the tile
#pragma unroll
  for (int i = lane; i < kChunks; i += 32) {
    // a 16-byte unit of the (sub-)tile; row = token within the chunk
    const int sub = i / (16 * 8);
    const int row = (i / 8) % 16;
    if (!((valid >> row) & 1u)) {
      *reinterpret_cast<uint4*>(sV + sub * 2048 + (i % (16 * 8)) * 16) = make_uint4(0, 0, 0, 0);
    }
  }
}

// Online-softmax update of one row given this lane's scores x[] (already in
// the log2 domain, -inf where masked).  Returns the rescale factor for the
// running output and writes p[] in place.
template <int N>
__device__ __forceinline__ float softmax_row_update(float (&x)[N], float& m, float& l) {
  float mx = x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) mx = fmaxf(mx, x[i]);
  mx = warp_max_quad(mx);
  const float m_new = fmaxf(m, mx);
  // all scores seen so far masked: keep the state, contribute nothing
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = exp2f(m - m_use);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    x[i] = exp2f(x[i] - m_use);
    s += x[i];
  }
  l = l * alpha + s;
  m = m_new;
  return alpha;
}

// ----------------------------------------------------------------------
// One 16-token bf16 chunk: K tile at sK, V tile at sV (each D/64 swizzled
// 16 x 64 boxes of 2 KB).  valid: bit t set if token t of the chunk is part
// of the sequence.
// ----------------------------------------------------------------------
template <int D, bool TWO>
__device__ __forceinline__ void consume_bf16(WarpState<D, TWO>& st, const QFrags<D, TWO>& qf,
                                             uint32_t sK, uint32_t sV, uint32_t valid,
                                             float scale_log2, int lane) {
  const int qd = lane & 3;
  const int mi = lane >> 3, r = lane & 7;
  // ---- S = Q K^T : two n-tiles of 8 tokens, two accumulation chains
  float s0[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float s1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int tok = r + ((mi >> 1) << 3);  // matrices 2,3 -> tokens 8..15
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c16 = 2 * ks + (mi & 1);   // 16-byte column unit
      const uint32_t addr = sK + (c16 >> 3) * 2048 + swz128(tok * 128 + (c16 & 7) * 16);
      uint32_t b00, b01, b10, b11;
      ldsm_x4(addr, b00, b01, b10, b11);
      float(&acc)[2][4] = (ks & 1) ? s1 : s0;
      mma_bf16(acc[0], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b00, b01);
      mma_bf16(acc[1], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b10, b11);
    }
  }
  // ---- online softmax, rows g (and g+8)
  uint32_t pa[2][2];  // P as bf16 A fragments: [row half][k half]
#pragma unroll
  for (int rh = 0; rh < (TWO ? 2 : 1); ++rh) {
    float x[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * nt + 2 * qd + e;
        const float v = (s0[nt][2 * rh + e] + s1[nt][2 * rh + e]) * scale_log2;
        x[2 * nt + e] = ((valid >> t) & 1u) ? v : -INFINITY;
      }
    const float alpha = softmax_row_update(x, st.m[rh], st.l[rh]);
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      st.o[nt][2 * rh] *= alpha;
      st.o[nt][2 * rh + 1] *= alpha;
    }
    pa[rh][0] = pack_bf16(x[0], x[1]);
    pa[rh][1] = pack_bf16(x[2], x[3]);
  }
  if (!TWO) pa[1][0] = pa[1][1] = 0u;
  // ---- O += P V : V^T fragments through ldmatrix.trans
  {
    const int tok = r + ((mi & 1) << 3);
#pragma unroll
    for (int np = 0; np < D / 16; ++np) {
      const int c16 = 2 * np + (mi >> 1);
      const uint32_t addr = sV + (c16 >> 3) * 2048 + swz128(tok * 128 + (c16 & 7) * 16);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(addr, v0, v1, v2, v3);
      mma_bf16(st.o[2 * np], pa[0][0], pa[1][0], pa[0][1], pa[1][1], v0, v1);
      mma_bf16(st.o[2 * np + 1], pa[0][0], pa[1][0], pa[0][1], pa[1][1], v2, v3);
    }
  }
}

// ----------------------------------------------------------------------
// One 32-token INT8 chunk: K codes at sK, V codes at sV, each a 32 x D int8
// tile (128-byte swizzle for D = 128, 64-byte swizzle for D = 64).  Scores
// use f16 mma on the exact integer codes; the K scale is folded into the
// score multiplier and the V scale into the output's storage scale st.u,
// so the only rounding beyond the bf16 path is P in f16.
// The output accumulator uses the INT8 column order: o[4J + e][0..1] hold
// columns 32J + 8q + e and 32J + 8q + 4 + e of rows g (g+8).
// ----------------------------------------------------------------------
template <int D>
__device__ __forceinline__ uint32_t i8_off(int row, int c16) {
  if constexpr (D == 128) {
    return swz128(row * 128 + c16 * 16);
  } else {
    return swz64(row * 64 + c16 * 16);
  }
}

template <int D, bool TWO>
__device__ __forceinline__ void consume_i8(WarpState<D, TWO>& st, const QFrags<D, TWO>& qf,
                                           uint32_t sK, uint32_t sV, float k_scale,
                                           float v_scale, float scale_log2, int lane) {
  const int g = lane >> 2, qd = lane & 3;
  const int mi = lane >> 3, r = lane & 7;
  constexpr int KS = D / 16;  // k-steps over the head dim
  // ---- S = Q K^T over 4 n-tiles of 8 tokens
  float s[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hq = 0; hq < KS / 4; ++hq) {
      // matrix mi = 16-byte column unit 4hq + mi of rows 8nt .. 8nt+7
      const uint32_t addr = sK + i8_off<D>(8 * nt + r, 4 * hq + mi);
      uint32_t w[4];
      ldsm_x4(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ks = 4 * hq + i;
        uint32_t b0, b1;
        i8x4_to_f16x2x2(w[i], b0, b1);
        float(&acc)[4] = (i & 1) ? s2 : s[nt];
        mma_f16(acc, qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b0, b1);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] += s2[e];
  }
  // ---- online softmax; the V scale change is folded into the rescale
  const float u_new = v_scale != 0.f ? v_scale : st.u;
  const float ratio = st.u / u_new;
  const float sl = scale_log2 * k_scale;
  uint32_t pa[2][4];  // [row half][a0/a2 for k-step 0, a0/a2 for k-step 1]
#pragma unroll
  for (int rh = 0; rh < (TWO ? 2 : 1); ++rh) {
    float x[8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      x[2 * nt] = s[nt][2 * rh] * sl;
      x[2 * nt + 1] = s[nt][2 * rh + 1] * sl;
    }
    const float alpha = softmax_row_update(x, st.m[rh], st.l[rh]) * ratio;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      st.o[nt][2 * rh] *= alpha;
      st.o[nt][2 * rh + 1] *= alpha;
    }
    // k-step kk covers tokens 16kk .. 16kk+15 = score n-tiles 2kk, 2kk+1
    pa[rh][0] = pack_f16(x[0], x[1]);
    pa[rh][1] = pack_f16(x[2], x[3]);
    pa[rh][2] = pack_f16(x[4], x[5]);
    pa[rh][3] = pack_f16(x[6], x[7]);
  }
  if (!TWO) pa[1][0] = pa[1][1] = pa[1][2] = pa[1][3] = 0u;
  st.u = u_new;
  // ---- O += P V over 2 k-steps of 16 tokens; V^T fragments built from
  // 32-bit shared loads of 4 codes and byte interleaving
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const int r0 = 16 * kk + 2 * qd;
#pragma unroll
    for (int J = 0; J < D / 32; ++J) {
      const int c16 = 2 * J + (g >> 2);
      const uint32_t inner = (g & 3) * 4;
      const uint32_t w0 = lds32(sV + i8_off<D>(r0, c16) + inner);
      const uint32_t w1 = lds32(sV + i8_off<D>(r0 + 1, c16) + inner);
      const uint32_t w2 = lds32(sV + i8_off<D>(r0 + 8, c16) + inner);
      const uint32_t w3 = lds32(sV + i8_off<D>(r0 + 9, c16) + inner);
      uint32_t lo01, hi01, lo23, hi23;
      interleave_bytes(w0, w1, lo01, hi01);
      interleave_bytes(w2, w3, lo23, hi23);
      uint32_t b0[4], b1[4];
      i8x4_to_f16x2x2(lo01, b0[0], b0[1]);
      i8x4_to_f16x2x2(hi01, b0[2], b0[3]);
      i8x4_to_f16x2x2(lo23, b1[0], b1[1]);
      i8x4_to_f16x2x2(hi23, b1[2], b1[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        mma_f16(st.o[4 * J + e], pa[0][2 * kk], pa[1][2 * kk], pa[0][2 * kk + 1],
                pa[1][2 * kk + 1], b0[e], b1[e]);
    }
  }
}

// Column (head-dim index) held by accumulator element (nt, e in {0,1}) of
// lane quad position qd, for the two accumulator orders.
template <bool I8ORDER>
__device__ __forceinline__ int acc_col(int nt, int e, int qd) {
  if (I8ORDER) return 32 * (nt >> 2) + 4 * (2 * qd + e) + (nt & 3);
  return 8 * nt + 2 * qd + e;
}

}  // namespace phs
