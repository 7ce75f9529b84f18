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

// Bytes of one staged chunk: K + V of 16 bf16 tokens, or of 32 INT8 tokens.
template <int D>
struct ChunkGeom {
  static constexpr int kTileBytes = 16 * D * 2;   // one bf16 16 x D tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSubTiles = D / 64;        // 64-column (128-byte) boxes
  static constexpr int kI8RowBytes = D;           // INT8 row = D bytes
};

// Per-lane shared-memory offsets of the mma fragments inside a staged chunk,
// computed once per warp.  TMA's 128-byte swizzle stores byte offset o of a
// tile at o ^ (((o >> 7) & 7) << 4) (the 64-byte swizzle: & 3 instead of
// & 7).  Stage bases are 1024-byte aligned and the
// swizzle only permutes 16-byte units inside 1024-byte blocks, so the
// address of fragment step i is (stage + lane offset) ^ (constant of i) + an
// immediate: one logic op per fragment load instead of the full swizzle.
struct FragOffsets {
  uint32_t bk, bv;  // bf16 chunk: K (ldmatrix) and V (ldmatrix.trans)
  uint32_t ik, iv;  // INT8 chunk: K rows (token order of kI8TokenPerm), V^T rows

  template <int D>
  __device__ __forceinline__ void init(int lane) {
    const int mi = lane >> 3, r = lane & 7, g = lane >> 2, qd = lane & 3;
    // bf16 K: matrix mi = (tokens 8*(mi>>1).., 16-byte unit 2ks + (mi&1))
    bk = (r + ((mi >> 1) << 3)) * 128 + ((((mi & 1) ^ r) & 7) << 4);
    // bf16 V (transposed): (tokens 8*(mi&1).., unit 2np + (mi>>1))
    bv = (r + ((mi & 1) << 3)) * 128 + ((((mi >> 1) ^ r) & 7) << 4);
    (void)g;
    (void)qd;
    // INT8 K (A operand of S^T = K Q^T): matrix mi = (tokens 8(mi&1) + r,
    // 16-byte unit mi>>1 of a k-step pair)
    const int t = r + 8 * (mi & 1);
    if constexpr (D == 128)
      ik = t * 128 + ((((mi >> 1) ^ t) & 7) << 4);  // 128-byte rows and swizzle
    else
      ik = t * 64 + ((((mi >> 1) ^ (t >> 1)) & 3) << 4);  // 64-byte rows and swizzle
    // INT8 V^T (A operand of O^T = V^T P^T): token half th is D rows of 16
    // bytes, i.e. 128-byte row th D/8 + d/8 holds dims d..d+7 of that half,
    // staged with the 128-byte swizzle (unit ^= row & 7).  Matrix mi = (dims
    // 8(mi&1) + r of a 16-dim tile, token half mi>>1): its 8 rows are the 8
    // units of one 128-byte row, so no bank conflicts.
    const int vrow = (mi >> 1) * (D / 8) + (mi & 1);
    iv = vrow * 128 + (((r ^ vrow) & 7) << 4);
  }
};

// Running state of one warp's softmax reduction.  Rows g (and g+8 when the
// group exceeds 8 heads) are this lane's query heads; the lane holds the
// output columns of its accumulator fragments.
template <int D, bool TWO>
struct WarpState {
  static constexpr int R = TWO ? 4 : 2;  // accumulators kept per mma tile
  // bf16 path: o[nt][0..1] = (row g, d 8nt+2q..+1) (+ row g+8: [2..3]).
  // INT8 path (transposed): element (dt, nq, k) of flat index
  // 4 (dt NQ + nq) + k holds (dim 16dt + g + 8(k>>1), query 8nq + 2q + (k&1))
  float o[D / 8][R];
  float m[4];  // running max (log2 domain): bf16 rows g, g+8; INT8 queries 8nq+2q+e at 2nq+e
  float l[4];  // this lane's partial sum of exp2 (reduced across lanes at the end)
  float u;            // INT8 path: output is stored divided by this V scale
  float lu;           // log2(u)

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int r = 0; r < R; ++r) o[i][r] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
    }
    u = 1.f;
    lu = 0.f;
  }
};

// Q fragments of the group for the bf16 path (standard k order) and for the
// INT8 path (f16, k order matching the ldmatrix layout of 8-bit rows, see
// qk_i8).  Rows >= G are zero.
template <int D, bool TWO>
struct QFrags {
  uint32_t a[D / 16][4];
  float qsum[2];  // INT8 path: sum over d of the f16 queries, rows g, g+8
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
// 16ks + 4q .. 16ks + 4q + 3 of each row (see qk_i8).  Also forms the
// row sums of the f16 queries, which remove the code bias from the scores.
__device__ __forceinline__ float f16x2_sum(uint32_t w) {
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&w));
  return f.x + f.y;
}

template <int D, bool TWO>
__device__ __forceinline__ void load_q_f16_i8order(QFrags<D, TWO>& f, const __nv_bfloat16* q,
                                                   int G, int lane) {
  const int g = lane >> 2, qd = lane & 3;
  const uint2* q64 = reinterpret_cast<const uint2*>(q);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c = 16 * ks + 4 * qd;  // 4 consecutive columns, 8 bytes
    uint2 w0 = g < G ? __ldg(q64 + (g * D + c) / 4) : make_uint2(0, 0);
    f.a[ks][0] = bf16x2_to_f16x2(w0.x);
    f.a[ks][2] = bf16x2_to_f16x2(w0.y);
    s0 += f16x2_sum(f.a[ks][0]) + f16x2_sum(f.a[ks][2]);
    if (TWO) {
      uint2 w1 = g + 8 < G ? __ldg(q64 + ((g + 8) * D + c) / 4) : make_uint2(0, 0);
      f.a[ks][1] = bf16x2_to_f16x2(w1.x);
      f.a[ks][3] = bf16x2_to_f16x2(w1.y);
      s1 += f16x2_sum(f.a[ks][1]) + f16x2_sum(f.a[ks][3]);
    } else {
      f.a[ks][1] = f.a[ks][3] = 0u;
    }
  }
  f.qsum[0] = warp_sum_quad(s0);
  f.qsum[1] = warp_sum_quad(s1);
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

// Online-softmax update of one row from this lane's raw scores s[] (-inf
// where masked).  Log2-domain score: x = s * sl - off (sl > 0).  Writes
// p = 2^(x - m_new + lr) into s[] (lr = log2 of a factor folded into P),
// adds sum(p) * inv_ratio to the lane's running sum l and returns the
// rescale factor 2^(m_old - m_new) of the running output.
template <int N>
__device__ __forceinline__ float softmax_row_update(float (&s)[N], float sl, float off, float lr,
                                                    float inv_ratio, float& m, float& l) {
  float mx = s[0];
#pragma unroll
  for (int i = 1; i < N; ++i) mx = fmaxf(mx, s[i]);
  mx = mx == -INFINITY ? -INFINITY : mx * sl - off;
  mx = warp_max_quad(mx);
  const float m_new = fmaxf(m, mx);
  // all scores seen so far masked: keep the state, contribute nothing
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = ex2(m - m_use);
  const float c = off + m_use - lr;
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    s[i] = ex2(fmaf(s[i], sl, -c));
    sum += s[i];
  }
  l = l * alpha + sum * inv_ratio;
  m = m_new;
  return alpha;
}

// Rescale the running output of row half rh by alpha, skipped when no row
// of the warp changed its maximum (the common case once the row max has
// settled).
template <int D, int R>
__device__ __forceinline__ void rescale_rows(float (&o)[D / 8][R], int rh, float alpha) {
  if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      o[nt][2 * rh] *= alpha;
      o[nt][2 * rh + 1] *= alpha;
    }
  }
}

// ----------------------------------------------------------------------
// One 16-token bf16 chunk: K tile at sK, V tile at sV (each D/64 swizzled
// 16 x 64 boxes of 2 KB).  valid: bit t set if token t of the chunk is part
// of the sequence.  Three phases so that a caller can overlap the score
// contraction of the next chunk with the output update of the current one:
//   qk_bf16 (S = Q K^T), softmax_bf16 (online softmax, returns P), pv_bf16.
// ----------------------------------------------------------------------
template <int D, bool TWO>
struct ScoresBf16 {
  float s[2][WarpState<D, TWO>::R];  // n-tiles of 8 tokens
};

template <int D, bool TWO>
__device__ __forceinline__ void qk_bf16(ScoresBf16<D, TWO>& sc, const QFrags<D, TWO>& qf,
                                        const FragOffsets& fo, uint32_t sK) {
  constexpr int R = WarpState<D, TWO>::R;
  float s1[2][R];  // second accumulation chain (odd k-steps)
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r) sc.s[i][r] = s1[i][r] = 0.f;
  const uint32_t kbase = sK + fo.bk;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    // 16-byte unit 2ks + (mi&1) of the (ks/4)-th 64-column box
    const uint32_t addr = (kbase ^ (((2 * ks) & 7) << 4)) + (ks >> 2) * 2048;
    uint32_t b00, b01, b10, b11;
    ldsm_x4(addr, b00, b01, b10, b11);
    if (ks & 1) {
      mma_bf16(s1[0], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b00, b01);
      mma_bf16(s1[1], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b10, b11);
    } else {
      mma_bf16(sc.s[0], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b00, b01);
      mma_bf16(sc.s[1], qf.a[ks][0], qf.a[ks][1], qf.a[ks][2], qf.a[ks][3], b10, b11);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r) sc.s[i][r] += s1[i][r];
}

// P as bf16 A fragments: pa[row half][k half]
template <int D, bool TWO>
__device__ __forceinline__ void softmax_bf16(WarpState<D, TWO>& st, ScoresBf16<D, TWO>& sc,
                                             uint32_t (&pa)[2][2], uint32_t valid,
                                             float scale_log2, int lane) {
  constexpr int R = WarpState<D, TWO>::R;
  const int qd = lane & 3;
#pragma unroll
  for (int rh = 0; rh < (TWO ? 2 : 1); ++rh) {
    float x[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * nt + 2 * qd + e;
        x[2 * nt + e] = ((valid >> t) & 1u) ? sc.s[nt][2 * rh + e] : -INFINITY;
      }
    const float alpha = softmax_row_update(x, scale_log2, 0.f, 0.f, 1.f, st.m[rh], st.l[rh]);
    rescale_rows<D, R>(st.o, rh, alpha);
    pa[rh][0] = pack_bf16(x[0], x[1]);
    pa[rh][1] = pack_bf16(x[2], x[3]);
  }
  if (!TWO) pa[1][0] = pa[1][1] = 0u;
}

// O += P V : V^T fragments through ldmatrix.trans
template <int D, bool TWO>
__device__ __forceinline__ void pv_bf16(WarpState<D, TWO>& st, const uint32_t (&pa)[2][2],
                                        const FragOffsets& fo, uint32_t sV) {
  const uint32_t vbase = sV + fo.bv;
#pragma unroll
  for (int np = 0; np < D / 16; ++np) {
    const uint32_t addr = (vbase ^ (((2 * np) & 7) << 4)) + (np >> 2) * 2048;
    uint32_t v0, v1, v2, v3;
    ldsm_x4_t(addr, v0, v1, v2, v3);
    mma_bf16(st.o[2 * np], pa[0][0], pa[1][0], pa[0][1], pa[1][1], v0, v1);
    mma_bf16(st.o[2 * np + 1], pa[0][0], pa[1][0], pa[0][1], pa[1][1], v2, v3);
  }
}

template <int D, bool TWO>
__device__ __forceinline__ void consume_bf16(WarpState<D, TWO>& st, const QFrags<D, TWO>& qf,
                                             const FragOffsets& fo, uint32_t sK, uint32_t sV,
                                             uint32_t valid, float scale_log2, int lane) {
  ScoresBf16<D, TWO> sc;
  uint32_t pa[2][2];
  qk_bf16(sc, qf, fo, sK);
  softmax_bf16(st, sc, pa, valid, scale_log2, lane);
  pv_bf16(st, pa, fo, sV);
}

// ----------------------------------------------------------------------
// One 32-token INT8 chunk: K codes at sK, a 32 x D tile (128-byte swizzle
// for D = 128, 64-byte for D = 64), and V codes at sV, stored transposed:
// two 16-token halves of D rows of 16 bytes (staged as D/4 rows of 128
// bytes, 128-byte swizzle).  Codes are stored offset by 128 (byte
// u = x + 128), so the low mantissa byte of the f16 1024.0 takes the byte
// as it is: f16 1024 + u = x + 1152, exact.
//
// Both contractions run transposed, S^T = K Q^T and O^T = V^T P^T, so the
// query group (at most 8 heads per n-tile) fills the n = 8 side of the
// m16n8k16 tile instead of 16 rows of which at most 8 are live: half the
// mma instructions of the untransposed form.  K and V^T fragments come
// from ldmatrix on the code tiles (4 codes per lane and row, a permuted k
// order matched by the other operand), and P^T from transposing the packed
// scores in registers (movmatrix).  The K scale is folded into the score
// multiplier and the V scale into P (see softmax_i8), so the only rounding
// beyond the bf16 path is P in f16.  Phases as for bf16 chunks.
// ----------------------------------------------------------------------
template <int D, bool TWO>
struct ScoresI8 {
  static constexpr int NQ = TWO ? 2 : 1;  // query n-tiles of 8
  float s[2][NQ][4];                      // [token tile][query tile][C fragment]
};

// 1024 (the f16 exponent) + 128 (the code offset); removed once per score
// as 1152 * sum(q), not per element
constexpr float kI8Bias = 1152.f;

// four offset codes (bytes of w) -> f16x2 (byte0, byte1) and (byte2, byte3),
// each x + 1152: the byte becomes the low mantissa byte of the f16 1024.0
// (exponent byte 0x64)
__device__ __forceinline__ void u8x4_to_f16x2x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0x64646464u));
}

// the same, exact: x itself (bias subtracted per pair)
__device__ __forceinline__ void u8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  u8x4_to_f16x2x2_biased(w, a, b);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// O^T accumulator element (dt, nq, k) inside the warp state (layout above)
template <int D, bool TWO>
__device__ __forceinline__ float& oT(WarpState<D, TWO>& st, int dt, int nq, int k) {
  constexpr int R = WarpState<D, TWO>::R, NQ = TWO ? 2 : 1;
  const int f = (dt * NQ + nq) * 4 + k;
  return st.o[f / R][f % R];
}

// Sum of the f16 queries of this lane's score columns: query 8nq + 2q + e
// at [nq][e] (the query fragments hold the sums of rows g, g+8).
template <int D, bool TWO>
__device__ __forceinline__ void query_sums_t(const QFrags<D, TWO>& qf, float (&qs)[2][2],
                                             int lane) {
  const int qd = lane & 3;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    qs[0][e] = __shfl_sync(0xffffffffu, qf.qsum[0], 4 * (2 * qd + e));
    qs[1][e] = TWO ? __shfl_sync(0xffffffffu, qf.qsum[1], 4 * (2 * qd + e)) : 0.f;
  }
}

template <int D, bool TWO>
__device__ __forceinline__ void qk_i8(ScoresI8<D, TWO>& sc, const QFrags<D, TWO>& qf,
                                      const FragOffsets& fo, uint32_t sK) {
  constexpr int KS = D / 16;  // k-steps over the head dim
  constexpr int NQ = TWO ? 2 : 1;
  // S^T = (K + 1152) Q^T (the bias is removed in softmax_i8): per 16-token
  // tile mt, k-steps in pairs from one ldmatrix.x4, even and odd k-steps in
  // separate accumulation chains
  const uint32_t kbase = sK + fo.ik;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    float s2[NQ][4];
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
      for (int k = 0; k < 4; ++k) sc.s[mt][nq][k] = s2[nq][k] = 0.f;
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
      uint32_t w[4];
      ldsm_x4((kbase ^ (kp << 5)) + mt * 16 * D, w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int ks = 2 * kp + i;
        uint32_t a0, a1, a2, a3;
        u8x4_to_f16x2x2_biased(w[2 * i], a0, a2);
        u8x4_to_f16x2x2_biased(w[2 * i + 1], a1, a3);
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) {
          const uint32_t b0 = qf.a[ks][nq ? 1 : 0], b1 = qf.a[ks][nq ? 3 : 2];
          if (i)
            mma_f16(s2[nq], a0, a1, a2, a3, b0, b1);
          else
            mma_f16(sc.s[mt][nq], a0, a1, a2, a3, b0, b1);
        }
      }
    }
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
      for (int k = 0; k < 4; ++k) sc.s[mt][nq][k] += s2[nq][k];
  }
}

// Online-softmax update of one score column (a query) from this lane's 4
// raw scores (the reduction runs over the 8 lanes of the same q).  As
// softmax_row_update otherwise.
__device__ __forceinline__ float softmax_col_update(float (&s)[4], float sl, float off, float lr,
                                                    float inv_ratio, float& m, float& l) {
  float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
  mx = mx * sl - off;
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  const float m_new = fmaxf(m, mx);
  const float alpha = ex2(m - m_new);
  const float c = off + m_new - lr;
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s[i] = ex2(fmaf(s[i], sl, -c));
    sum += s[i];
  }
  l = l * alpha + sum * inv_ratio;
  m = m_new;
  return alpha;
}

// Online softmax of an INT8 chunk (every token valid).  The V scale enters
// through P: with the output stored in units of st.u, a chunk scaled by
// v_scale contributes P * (v_scale / st.u) * codes, so log2(v_scale / st.u)
// is added inside the exponent; st.u moves (one rescale) only if that ratio
// leaves 2^+-8.  pb[token tile kk][2 nq + {0, 1}]: the P^T operand (f16) of
// tokens 16kk + 4q, 4q+1 and 4q+2, 4q+3 for query 8nq + g.
template <int D, bool TWO>
__device__ __forceinline__ void softmax_i8(WarpState<D, TWO>& st, const float (&qs)[2][2],
                                           ScoresI8<D, TWO>& sc, uint32_t (&pb)[2][4],
                                           float k_scale, float v_scale, float scale_log2) {
  constexpr int NQ = TWO ? 2 : 1;
  float lr = 0.f, inv_ratio = 1.f;
  if (v_scale > 0.f) {
    const float lv = lg2(v_scale);
    lr = lv - st.lu;
    if (fabsf(lr) > 8.f) {
      const float f = ex2(-lr);  // re-base the stored output on v_scale
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < WarpState<D, TWO>::R; ++e) st.o[nt][e] *= f;
      st.u = v_scale;
      st.lu = lv;
      lr = 0.f;
    }
    inv_ratio = ex2(-lr);
  }
  const float sl = scale_log2 * k_scale;
  float alpha[2][2];
#pragma unroll
  for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      // this lane's tokens of query 8nq + 2q + e: rows g, g+8 of both tiles
      float x[4] = {sc.s[0][nq][e], sc.s[0][nq][2 + e], sc.s[1][nq][e], sc.s[1][nq][2 + e]};
      // scores carry the code bias: subtract 1152 * sum(q) (times sl)
      alpha[nq][e] = softmax_col_update(x, sl, kI8Bias * qs[nq][e] * sl, lr, inv_ratio,
                                        st.m[2 * nq + e], st.l[2 * nq + e]);
      sc.s[0][nq][e] = x[0];
      sc.s[0][nq][2 + e] = x[1];
      sc.s[1][nq][e] = x[2];
      sc.s[1][nq][2 + e] = x[3];
    }
  // rescale the running output, skipped when no column of the warp moved
  bool moved = false;
#pragma unroll
  for (int nq = 0; nq < NQ; ++nq) moved |= alpha[nq][0] != 1.f || alpha[nq][1] != 1.f;
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
        for (int k = 0; k < 4; ++k) oT(st, dt, nq, k) *= alpha[nq][k & 1];
  }
  // P^T operand: the 8 x 8 blocks (tile rows 0-7, 8-15) transposed
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
      pb[kk][2 * nq] = movmatrix_t(pack_f16(sc.s[kk][nq][0], sc.s[kk][nq][1]));
      pb[kk][2 * nq + 1] = movmatrix_t(pack_f16(sc.s[kk][nq][2], sc.s[kk][nq][3]));
    }
  if (!TWO) pb[0][2] = pb[0][3] = pb[1][2] = pb[1][3] = 0u;
}

// O^T += V^T P^T over 2 k-steps of 16 tokens (exact codes: a bias here
// would cost output precision).  One ldmatrix.x4 per 16-dim tile fetches
// both k-steps' A fragments.
template <int D, bool TWO>
__device__ __forceinline__ void pv_i8(WarpState<D, TWO>& st, const uint32_t (&pb)[2][4],
                                      const FragOffsets& fo, uint32_t sV) {
  constexpr int NQ = TWO ? 2 : 1;
  const uint32_t vbase = sV + fo.iv;
#pragma unroll
  for (int dt = 0; dt < D / 16; ++dt) {
    uint32_t w[4];
    // dims 16dt.. of a half are its 128-byte rows 2dt, 2dt+1: (row & 7)
    // gains 2dt mod 8
    ldsm_x4((vbase ^ (((2 * dt) & 7) << 4)) + dt * 2 * 128, w[0], w[1], w[2], w[3]);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t a0, a1, a2, a3;
      u8x4_to_f16x2x2(w[2 * kk], a0, a2);
      u8x4_to_f16x2x2(w[2 * kk + 1], a1, a3);
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq) {
        float c[4] = {oT(st, dt, nq, 0), oT(st, dt, nq, 1), oT(st, dt, nq, 2), oT(st, dt, nq, 3)};
        mma_f16(c, a0, a1, a2, a3, pb[kk][2 * nq], pb[kk][2 * nq + 1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) oT(st, dt, nq, k) = c[k];
      }
    }
  }
}

}  // namespace phs
