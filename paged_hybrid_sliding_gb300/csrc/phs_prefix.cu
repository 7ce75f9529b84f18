// phs_prefix.cu -- decode attention over a prefix shared by a batch of
// requests, on the 5th-generation tensor cores.
//
// Source: "Kimi K3 context caching" page, section 1 (requests hitting the
// same prefix share its physical KV blocks by reference count) and section 4
// (a 250,000-token shared prefix).  When B requests share the prefix, the
// queries of one KV head's group across all B requests (B x G rows) attend
// to the same prefix K/V: one dense contraction per KV head instead of B
// separate decodes that each stream the whole prefix.
//
// One CTA (persistent, one per SM) handles one (KV head, span of the
// prefix) for all rows at once (up to 256 = 2 tiles of 128 rows):
//   warp 8    : TMA producer of 64-token K tiles (four 16-token pages,
//               128-byte swizzle), its copies issued by eight lanes at once
//   warp 10   : the same for V (one 4 KB box per page); K and V stages are
//               released separately (K after Q K^T, V after the P V product)
//   warp 9    : MMA issuer (one lane) of S = Q K^T for row tile 0; owns the
//               tensor-memory allocation
//   warp 11   : MMA issuer (one lane) of S = Q K^T for row tile 1
//   warp 12   : MMA issuer (one lane) of every P V product, so that its long
//               instructions never hold back a Q K^T (decode call 0.2524 ->
//               0.2499 ms against issuing them from warp 9)
//   warps 0-7 : online softmax, one query row per thread
// The tensor pipe holds about one instruction ahead, so an issuing thread
// that waits for its scheduler leaves it idle; the softmax warps keep every
// sub-partition busy, and two issuers on different sub-partitions cover for
// each other (measured: a tile's 20 instructions take 1,600 cycles from one
// issuer next to the softmax load, 1,210 from two).
// Tensor memory (512 columns): S [128 lanes = rows][2 x 64 tokens], Q
// [128 lanes = rows][2 x 64 columns of bf16 pairs], O^T [128 lanes = d][256
// rows].  Per 64-token tile j:
//   S_j = Q K_j^T      tcgen05.mma, A = Q from tensor memory, B = K tile
//                      (K-major), M = 128 per row tile, N = 64, K = 128;
//   softmax            each thread reads its row of S_j (then S is free for
//                      Q K_{j+1}^T), forms P_j = 2^(s * scale log2(e) - m)
//                      in bf16 into shared memory ([row][token], K-major);
//   O^T += V_j^T P_j^T A = V tile (MN-major), B = P_j, M = 128 (d),
//                      N = 256 (rows), K = 64 tokens.
// Putting the rows on N makes the P V product four N = 256 instructions per
// tile instead of eight N = 128 ones, and Q in tensor memory takes the Q
// operand off the shared-memory path; both keep the tensor pipe under the
// HBM time of a tile.  The running max m of a row only moves when it grows
// by more than 2^8 (so P <= 256); only then are the O^T columns of its row
// tile rescaled: every row publishes its factor in shared memory and a
// barrier reduction over the tile's four softmax warps tells them whether
// any row moved.  The CTA writes
// (m, l, O) partials; a merge kernel combines them with the requests' own
// suffix tokens (attended by the split-KV kernel).
#include "phs_attn.cuh"
#include "phs_internal.h"
#include "phs_tc.cuh"

namespace phs {

// Stage counts measured on the 250,000-token prefix (decode call, ms, with
// the separate P V issuer): 3 K / 3 V 0.2467, 4/2 0.2477, 4/4 0.2493,
// 4/3 0.2497, 3/4 0.2499, 3/2 0.2505, 5/3 0.2506, 2/2 0.2528 -- past 3 + 3
// a deeper ring only adds requests in flight, not rate.
#ifndef PHS_PFX_KSTAGES
#define PHS_PFX_KSTAGES 3
#endif
#ifndef PHS_PFX_VSTAGES
#define PHS_PFX_VSTAGES 3
#endif
// P buffers (the softmax of tile j + NP - 1 may run while the value product
// of tile j still reads its P): with 3 K / 3 V stages, 2 buffers 0.2466 ms,
// 3 buffers 0.2372 (192 KB in all); 4 buffers (which leave room for 2 V
// stages only) 0.2461.
#ifndef PHS_PFX_PBUFS
#define PHS_PFX_PBUFS 3
#endif
constexpr int kPfxKStages = PHS_PFX_KSTAGES;  // K tiles in shared memory
constexpr int kPfxVStages = PHS_PFX_VSTAGES;  // V tiles in shared memory
constexpr int kPfxPBufs = PHS_PFX_PBUFS;    // P tiles in shared memory
constexpr int kPfxTile = 64;     // tokens per tile (four pages)
constexpr int kPfxRows = 256;    // query rows per KV head (two tiles of 128)
#ifndef PHS_PFX_PV_WARP
#define PHS_PFX_PV_WARP 1
#endif
// 8 softmax warps, K producer, MMA (row tile 0), V producer, MMA (row tile
// 1), and a thirteenth warp issuing the P V products (PHS_PFX_PV_WARP=0:
// warp 9 issues them after row tile 0's Q K^T)
constexpr int kPfxPvWarp = PHS_PFX_PV_WARP;
constexpr int kPfxThreads = 384 + 32 * kPfxPvWarp;

// tensor-memory columns
constexpr uint32_t kTmS = 0;     // S: row tile mt at kTmS + 64 mt
constexpr uint32_t kTmQ = 128;   // Q: row tile mt at kTmQ + 64 mt
constexpr uint32_t kTmO = 256;   // O^T: row r at column kTmO + r

struct PfxLayout {
  static constexpr int kP = 0;                           // [buf][256 rows][128 B]
  static constexpr int kPBuf = 32 * 1024;
  static constexpr int kTileKV = 16 * 1024;              // one 64-token K or V tile
  static constexpr int kK = kPfxPBufs * kPBuf;           // K ring [KS][16 KB]
  static constexpr int kV = kK + kPfxKStages * kTileKV;  // V ring [VS][16 KB]
  static constexpr int kAlpha = kV + kPfxVStages * kTileKV;  // float [2][256]
  static constexpr int kBar = kAlpha + 2 * kPfxRows * 4;
  // full[KS + VS], empty[KS + VS], sfull[2], sfree[2], pfull[NP], odone[NP], drain
  static constexpr int kNumBars = 2 * (kPfxKStages + kPfxVStages) + 5 + 2 * kPfxPBufs;
  // tmem base, abort flag, softmax failure flags [row tile][tile parity]
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "prefix kernel shared memory above the per-CTA limit");
};

__device__ __forceinline__ uint8_t* pfx_align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Bounded mbarrier wait that also gives up when another role raised abort.
__device__ __forceinline__ bool pfx_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Packed fp32 pairs (two lanes of work per instruction on the FMA pipe) and
// the three-input maximum: they halve the instruction count of the softmax
// rows' scale, sum and max steps, which share their issue slots with the
// exponentials and the P stores.
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// OR of `pred` over the `count` threads of named barrier `id` (all of them
// execute it; it also orders their shared-memory accesses).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kPfxThreads, 1)
    phs_prefix_decode_kernel(const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv, const PrefixArgs a) {
  using L = PfxLayout;
  constexpr int D = 128;
  constexpr int KS = kPfxKStages, VS = kPfxVStages;
  constexpr int NP = kPfxPBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = pfx_align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, split = blockIdx.y;
  // the own-token split launch after this one does not depend on it: it may
  // start in this grid's tail (programmatic dependent launch)
  pdl_launch_dependents();

  // tiles of this CTA
  const int ntiles_all = a.shared_len / kPfxTile;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(ntiles_all, t_begin + a.tiles_per_split);
  const int ntiles = max(0, t_end - t_begin);

  const uint32_t bar_full = sb + L::kBar;                 // [KS + VS] stage loaded (K, then V)
  const uint32_t bar_empty = bar_full + 8 * (KS + VS);    // [KS + VS] stage consumed
  const uint32_t bar_sfull = bar_empty + 8 * (KS + VS);   // [2 row tiles] S_j in tensor memory
  const uint32_t bar_sfree = bar_sfull + 16;              // [2 row tiles] S_j read by its rows
  const uint32_t bar_pfull = bar_sfree + 16;              // [NP]: P buffer written
  const uint32_t bar_odone = bar_pfull + 8 * NP;          // [NP]: P V of that buffer done
  const uint32_t bar_drain = bar_odone + 8 * NP;          // every issued MMA done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* sm_fail = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);

  if (warp == 9) {
    tmem_alloc(sb + L::kMisc, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < KS + VS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, i < KS ? 2 : 1);  // a K stage is read by both Q K^T issuers
    }
    for (int mt = 0; mt < 2; ++mt) {
      mbar_init(bar_sfull + 8 * mt, 1);
      mbar_init(bar_sfree + 8 * mt, 128);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(bar_pfull + 8 * i, 256);
      mbar_init(bar_odone + 8 * i, 1);
    }
    mbar_init(bar_drain, 2 + kPfxPvWarp);
    *abort = 0;
    for (int i = 0; i < 4; ++i) sm_fail[i] = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- queries: thread r puts row r (request r / G, head h*G + r % G) into
  // tensor-memory lane r % 128 of row tile r / 128, as 64 columns of bf16
  // pairs (element 2c in the low half of column c); rows past B*G are zero
  if (warp < 8) {
    const int r = tid;
    const int mt = r >> 7;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool live = r < a.rows;
    const uint4* src = live ? reinterpret_cast<const uint4*>(
                                  a.q + (static_cast<size_t>(r / a.G) * a.Hq + h * a.G + r % a.G) * D)
                            : nullptr;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t qv[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = live ? __ldg(src + half * 8 + c) : make_uint4(0, 0, 0, 0);
        qv[4 * c] = v.x;
        qv[4 * c + 1] = v.y;
        qv[4 * c + 2] = v.z;
        qv[4 * c + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + kTmQ + mt * 64 + half * 32, qv);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 8 || warp == 10) {
    // ------------------------------------------- TMA producers (K, V)
    // The copy engine's cost is per box, so a tile's boxes are issued by
    // several lanes at once: K as eight 2 KB boxes (page i, column half) into
    // [half][64 rows], V as four 4 KB 3-D boxes (one per page) into
    // [page][half][16 rows].  Lane 0 owns the stage barriers.
    if (ntiles > 0) {
      const int kv = warp == 10;  // 0: K, 1: V
      const CUtensorMap* map = kv ? &tv : &tk;
      const int S = kv ? VS : KS;
      const uint32_t full = bar_full + 8 * KS * kv, empty = bar_empty + 8 * KS * kv;
      const uint32_t ring = sb + (kv ? L::kV : L::kK);
      const int nl = kv ? kPfxTile / kPage : 2 * kPfxTile / kPage;  // issuing lanes
      const int pg = kv ? lane : (lane >> 1), half = kv ? 0 : (lane & 1);
      const bool issuer = lane < nl;
      const uint64_t pol = policy_evict_first();
      if (lane == 0) prefetch_tmap(map);
      int issued = 0;
      bool ok = true;
      // page ids are read two tiles ahead, so their latency overlaps the
      // wait for a free stage instead of delaying the copies
      auto page_id = [&](int jt) {
        return issuer ? a.block_table[(t_begin + min(jt, ntiles - 1)) * (kPfxTile / kPage) + pg] : 0;
      };
      int id0 = page_id(0), id1 = page_id(1);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % S;
        int page = id0;
        id0 = id1;
        id1 = page_id(j + 2);
        if (lane == 0 && j >= S) ok = pfx_wait(empty + 8 * st, ((j / S) - 1) & 1, abort);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) {
            set_status(a.status, PHS_ETIMEOUT);
            *abort = 1;
          }
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(full + 8 * st, L::kTileKV);
        __syncwarp();
        if (issuer) {
          if (page < 0 || page >= a.num_pages) {
            set_status(a.status, PHS_ERANGE);
            page = 0;  // keep the byte count: read a valid page, result flagged
          }
          const int row = (page * a.Hkv + h) * kPage;
          const uint32_t stage = ring + st * L::kTileKV;
          if (kv)
            tma_load_3d(stage + pg * 4096, map, 0, row, 0, full + 8 * st, pol);
          else
            tma_load_2d(stage + half * 8192 + pg * 2048, map, half * 64, row, full + 8 * st, pol);
        }
        issued = j + 1;
      }
      // copies still in flight land before the CTA exits (all have landed
      // already unless another role gave up)
      if (lane == 0)
        for (int t = max(0, issued - S); t < issued; ++t) mbar_wait(full + 8 * (t % S), (t / S) & 1);
    }
  } else if (warp == 9 || warp == 11 || warp == 12) {
    // ------------------------------------------------------ MMA issuers
    if (lane == 0 && ntiles > 0) {
      const int mt = warp == 11;  // row tile whose S = Q K^T this thread issues
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kPfxTile, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kPfxRows, true, false);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % KS;
        if (!pfx_wait(bar_full + 8 * st, (j / KS) & 1, abort)) return false;  // K_j
        if (j >= 1 && !pfx_wait(bar_sfree + 8 * mt, (j - 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t kst = sb + L::kK + st * L::kTileKV;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_bf16_ts(tmem + kTmS + mt * kPfxTile, tmem + kTmQ + mt * 64 + ks * 8,
                       sdesc_sw128(kst + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), kIdescQK,
                       ks > 0);
        umma_commit(bar_sfull + 8 * mt);
        umma_commit(bar_empty + 8 * st);  // K stage free once both row tiles' products complete
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int st = j % VS, pb = j % NP;
        if (!pfx_wait(bar_full + 8 * (KS + st), (j / VS) & 1, abort)) return false;  // V_j
        if (!pfx_wait(bar_pfull + 8 * pb, (j / NP) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t vst = sb + L::kV + st * L::kTileKV;
        const uint32_t pst = sb + L::kP + pb * L::kPBuf;
#pragma unroll
        for (int kk = 0; kk < kPfxTile / 16; ++kk)
          umma_bf16(tmem + kTmO, sdesc_sw128(vst + kk * 4096, 2048, 1024),
                    sdesc_sw128(pst + kk * 32, 16, 1024), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar_odone + 8 * pb);
        umma_commit(bar_empty + 8 * (KS + st));  // V stage free once the product completes
        return true;
      };
      bool ok = true;
      if (warp == 12) {  // the P V issuer
        for (int j = 0; ok && j < ntiles; ++j) ok = issue_pv(j);
      } else {
        ok = issue_qk(0);
        for (int j = 0; ok && j < ntiles; ++j) {
          if (j + 1 < ntiles) ok = issue_qk(j + 1);
          if (ok && !kPfxPvWarp && mt == 0) ok = issue_pv(j);
        }
      }
      if (!ok) {
        set_status(a.status, PHS_ETIMEOUT);
        *abort = 1;
      }
      // every MMA issued above completes before tensor memory is released
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------ softmax rows
    const int mt = warp >> 2;
    const int rr = 32 * (warp & 3) + lane;
    const int r = mt * 128 + rr;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const bool got = pfx_wait(bar_sfull + 8 * mt, j & 1, abort);
      uint32_t sv0[32], sv1[32];  // scores of tokens 0..31 and 32..63 of the tile
      if (got) {
        tc_fence_after();
        tmem_ld32(tmem + lane_base + kTmS + mt * kPfxTile, sv0);
        tmem_ld32(tmem + lane_base + kTmS + mt * kPfxTile + 32, sv1);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) sv0[i] = sv1[i] = 0u;
      }
      tc_fence_before();
      mbar_arrive(bar_sfree + 8 * mt);
      auto sv = [&](int i) { return __uint_as_float(i < 32 ? sv0[i] : sv1[i - 32]); };
      float m4[4];  // four independent chains, two scores per step
#pragma unroll
      for (int k = 0; k < 4; ++k) m4[k] = fmaxf(sv(k), sv(4 + k));
#pragma unroll
      for (int i = 8; i < kPfxTile; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], sv(i + k), sv(i + 4 + k));
      float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      mx *= a.scale_log2;
      float alpha = 1.f;
      if (j == 0) {
        m_used = mx;
      } else if (mx > m_used + 8.f) {
        alpha = ex2(m_used - mx);
        m_used = mx;
      }
      float* al = alpha_s + (j & 1) * kPfxRows;
      al[r] = alpha;
      // The 128 threads of this row tile take part in one barrier reduction
      // per tile: whether any row's max moved or any wait failed.  A failed
      // wait is recorded in a flag of this tile's parity before the barrier
      // (a thread cannot write the same flag again before every thread has
      // read it: that would take it past the next tile's barrier), so all of
      // them leave the loop together.
      if (!got) sm_fail[2 * mt + (j & 1)] = 1;
      const bool resc = bar_red_or(1 + mt, 128, !got || alpha != 1.f);
      if (resc && sm_fail[2 * mt + (j & 1)]) {
        ok = false;
        break;
      }
      // P buffer j % NP was last read by P V_{j-NP}; a rescale of O needs P V_{j-1}
      if (j >= NP || (resc && j >= 1)) {
        const int jj = resc ? j - 1 : j - NP;
        if (!pfx_wait(bar_odone + 8 * (jj % NP), (jj / NP) & 1, abort)) {
          ok = false;  // the next tile's reduction ends the loop
          *abort = 1;
        }
        tc_fence_after();
      }
      l *= alpha;
      // P row: 64 bf16 = eight 16-byte units, K-major 128-byte swizzle
      const float c0 = m_used;
      uint8_t* prow = smem + L::kP + (j % NP) * L::kPBuf + r * 128;
      // x = s * scale log2(e) - m for two scores per instruction; the row
      // sum runs as four packed pairs
      const uint64_t scale2 = f2_make(a.scale_log2, a.scale_log2), negm2 = f2_make(-c0, -c0);
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = f2_split(ffma2(f2_make(sv(8 * u + 2 * k), sv(8 * u + 2 * k + 1)),
                                          scale2, negm2));
          const float p0 = ex2(x.x), p1 = ex2(x.y);
          sum2[k] = fadd2(sum2[k], f2_make(p0, p1));
          w[k] = pack_bf16(p0, p1);
        }
        *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      {
        const float2 s0 = f2_split(fadd2(sum2[0], sum2[1])), s1 = f2_split(fadd2(sum2[2], sum2[3]));
        l += (s0.x + s0.y) + (s1.x + s1.y);
      }
      fence_proxy_async_smem();
      if (resc) {
        // this warp rescales O^T lanes d = 32 (warp & 3) .. +31, row columns
        // 128 mt .. +127, by the factors every row published above
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int col0 = 128 * mt + 32 * c;
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kTmO + col0, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * al[col0 + i]);
          tmem_st32(tmem + lane_base + kTmO + col0, ov);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar_pfull + 8 * (j % NP));
    }
    // ---- partial result: O^T columns of this warp's rows, lanes = d
    if (ok && ntiles > 0) {
      const int jl = ntiles - 1;  // the last P V completes after all earlier ones
      ok = pfx_wait(bar_odone + 8 * (jl % NP), (jl / NP) & 1, abort);
    }
    ok = __all_sync(0xffffffffu, ok);
    const size_t part0 = (static_cast<size_t>(h) * a.num_splits + split) * kPfxRows;
    if (ok) {
      tc_fence_after();
      const int d = 32 * (warp & 3) + lane;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int col0 = 128 * mt + 32 * c;
        uint32_t ov[32];
        if (ntiles > 0) {
          tmem_ld32(tmem + lane_base + kTmO + col0, ov);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < a.rows) a.ws_o[(part0 + col0 + i) * D + d] = __uint_as_float(ov[i]);
      }
      if (r < a.rows)
        reinterpret_cast<float2*>(a.ws_ml)[part0 + r] =
            make_float2(ntiles > 0 ? m_used : -INFINITY, ntiles > 0 ? l : 0.f);
    } else if (lane == 0) {
      set_status(a.status, PHS_ETIMEOUT);
      *abort = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the shared-prefix partials with each request's suffix partials.
// One CTA per (request, KV head); warp w merges query rows w, w+4, ...
// Every load a row needs -- the sources' (m, l), this lane's four columns of
// each source's O, and the request's prefix flags -- is issued before any
// of them is used, so the merge costs one memory round trip per chunk of
// sources (the partials were just written and sit in L2); chunks combine
// with a running maximum.
constexpr int kMergeChunk = 24;  // sources per round trip (24 float4 per lane)

__global__ void __launch_bounds__(128) phs_merge_prefix_kernel(const PrefixMergeArgs a) {
  constexpr int D = 128;
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // launched as a dependent of the own-token split, which does not complete
  // before the prefix pass has: both grids' partials are in place after this
  pdl_wait_prior_grid();
  const int G = a.G;
  const int n = min(a.seq_lens[b], a.n_clamp);
  const int ns = n > a.shared_len ? min((n - a.shared_len + a.T - 1) / a.T, a.max_splits) : 0;
  const int total = a.num_psplits + ns;  // sources: prefix splits, then suffix splits
  const size_t out_row0 = (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * G) * D;
  // a request whose table does not begin with the shared pages (or that is
  // shorter than the shared prefix) was flagged by the own-token split: the
  // prefix partials are not its own, so its output row is zeroed
  int bad = 0;
  for (int i = lane; i < a.bad_slots; i += 32)
    bad |= a.prefix_bad[static_cast<size_t>(b) * a.bad_slots + i];
  for (int g = warp; g < G; g += 4) {
    const int r = b * G + g;
    const float2* pml = reinterpret_cast<const float2*>(a.ws_pml) +
                        static_cast<size_t>(h) * a.num_psplits * kPfxRows + r;
    const float2* sml = reinterpret_cast<const float2*>(a.ws_ml) +
                        (static_cast<size_t>(b) * a.Hkv + h) * a.max_splits * G + g;
    // source s's output row: prefix splits kPfxRows rows apart, then the
    // suffix splits G rows apart
    const float* po = a.ws_po + ((static_cast<size_t>(h) * a.num_psplits) * kPfxRows + r) * D;
    const float* so = a.ws_o + (((static_cast<size_t>(b) * a.Hkv + h) * a.max_splits) * G + g) * D;
    auto o_of = [&](int s) -> const float4* {
      return reinterpret_cast<const float4*>(
                 s < a.num_psplits ? po + static_cast<size_t>(s) * kPfxRows * D
                                   : so + static_cast<size_t>(s - a.num_psplits) * G * D) +
             lane;
    };
    float M = -INFINITY, lsum = 0.f;  // lsum: this lane's share of the weighted row sums
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < total; s0 += kMergeChunk) {
      const int cnt = min(kMergeChunk, total - s0);
      const int sl = s0 + lane;
      const float2 ml = lane < cnt ? (sl < a.num_psplits ? pml[static_cast<size_t>(sl) * kPfxRows]
                                                         : sml[static_cast<size_t>(sl - a.num_psplits) * G])
                                   : make_float2(-INFINITY, 0.f);
      float4 o[kMergeChunk];
#pragma unroll
      for (int k = 0; k < kMergeChunk; ++k)
        o[k] = k < cnt ? *o_of(s0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
      float mc = ml.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
      const float mn = fmaxf(M, mc);
      if (mn == -INFINITY) continue;  // no tokens in any source so far
      const float keep = M == -INFINITY ? 0.f : exp2f(M - mn);
      const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mn);
      lsum = lsum * keep + ml.y * w;
      acc.x *= keep;
      acc.y *= keep;
      acc.z *= keep;
      acc.w *= keep;
#pragma unroll
      for (int k = 0; k < kMergeChunk; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        acc.x += wk * o[k].x;
        acc.y += wk * o[k].y;
        acc.z += wk * o[k].z;
        acc.w += wk * o[k].w;
      }
      M = mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const bool zero = __any_sync(0xffffffffu, bad) != 0;
    const float res[4] = {zero ? 0.f : acc.x * inv, zero ? 0.f : acc.y * inv,
                          zero ? 0.f : acc.z * inv, zero ? 0.f : acc.w * inv};
    const size_t idx = out_row0 + static_cast<size_t>(g) * D + lane * 4;
    if (a.out_f32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx) =
          make_float4(res[0], res[1], res[2], res[3]);
    } else {
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(a.out) + idx;
      *reinterpret_cast<uint2*>(ob) = make_uint2(pack_bf16(res[0], res[1]), pack_bf16(res[2], res[3]));
    }
  }
}

int launch_prefix_decode(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixArgs& a,
                         cudaStream_t stream) {
  auto kern = phs_prefix_decode_kernel;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), PfxLayout::kAlloc) != PHS_OK)
    return PHS_ECUDA;
  dim3 grid(a.Hkv, a.num_splits);
  kern<<<grid, kPfxThreads, PfxLayout::kAlloc, stream>>>(tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int launch_merge_prefix(const PrefixMergeArgs& a, int B, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, a.Hkv);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, phs_merge_prefix_kernel, a) == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int prefix_smem_bytes() { return PfxLayout::kAlloc; }

}  // namespace phs
