// phs_decode.cu -- split-KV ("flash-decoding") Full-attention decode over
// the paged pool, with an optional INT8 region, and the cross-split merge.
//
// Grid: one CTA per (split, KV head, request).  A split is a run of
// tokens_per_split tokens of one request; the INT8 region [0, qlen) and the
// bf16 region [qlen, n) are split separately so that every CTA handles one
// chunk kind.  The CTA's 4 warps take the split's chunks round-robin; each
// warp streams its chunks through its own ring of S shared-memory stages
// filled by TMA (per 16-token bf16 page: K and V, each one 4 KB box of
// {64 columns, 16 rows, 2 column halves} for D = 128 or one 16 x 64 box for
// D = 64, 128-byte swizzle; or one 32 x D box each for a 32-token INT8
// page), and reduces them with the GQA-packed mma kernels of phs_attn.cuh.
// The 4 warp states are merged through shared memory; a request with a
// single split writes its output directly, others write (m, l, o) partials
// that phs_merge_kernel (phs_merge.cuh) combines.  The same body serves
// phs_stack_full_kernel (every Full layer of a hybrid-stack step in one
// launch, the append fused in).  Each split CTA signals dependent launches
// at its start (programmatic dependent launch; the merge waits for it).
//
// Sources: "Xiaomi MiMo-V2.5 inference system" page, sections 1-2 (Full
// layers attend over the whole sequence through the authoritative Full
// index; decode cost follows the KV bytes read); "Kimi K3 context caching"
// page, section 1 (KV in non-contiguous physical blocks through a page
// table); "Kimi K2.5 architecture deep dive" page, sections 2.2-2.3 (INT8
// block-wise warm zone, one scale per 32 tokens).
#include <type_traits>

#include "phs_attn.cuh"
#include "phs_internal.h"
#include "phs_merge.cuh"
#include "phs_swa_chunk.cuh"

namespace phs {

constexpr int kSplitWarps = 4;
constexpr int kMaxChunksPerWarp = 64;  // tokens_per_split <= 4096

// Compile-time tunables: TMA stages per warp and the CTAs per SM the
// register allocation must allow (bytes in flight per SM = CTAs x 4 warps x
// stages x 8 KB).  Measured (split kernel, GB/s; bf16 batch 64 / INT8
// batch 32): 2 stages x 3 CTAs 7,192 / 6,165; 3 x 2 7,145 / 5,536; 2 x 2
// 6,960 / 5,577.  More warps per SM with fewer stages each wins: the INT8
// chunks are bound by each warp's dependency chain, and fewer bytes in
// flight per warp cost nothing (168 registers, a few bytes of spill).
#ifndef PHS_SPLIT_STAGES_128
#define PHS_SPLIT_STAGES_128 2
#endif
#ifndef PHS_SPLIT_MIN_CTAS
#define PHS_SPLIT_MIN_CTAS 3
#endif

// NW: warps per CTA (4; 8 for the single-wave bf16 launches)
template <int D, int NW = kSplitWarps>
struct SplitLayout {
  static constexpr int kStage = ChunkGeom<D>::kStageBytes;
  static constexpr int kStages = (D == 128) ? PHS_SPLIT_STAGES_128 : 4;
  static constexpr int kStagesBytes = NW * kStages * kStage;
  static constexpr int kIdsOff = kStagesBytes;
  static constexpr int kIdsBytes = NW * kMaxChunksPerWarp * 12;
  static constexpr int kBarOff = kIdsOff + kIdsBytes;
  static constexpr int kBytes = kBarOff + NW * kStages * 8;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One warp's walk over its chunks of a split.  Stage j is handed back to
// TMA (chunk j + S) right after chunk j is folded into the warp state.
// Returns the index of a chunk whose bounded wait gave up, or -1.
template <bool I8, int D, bool TWO, int S, int NW, typename Issue, typename Patch>
__device__ __forceinline__ int walk_chunks(WarpState<D, TWO>& st, const QFrags<D, TWO>& qf,
                                           const FragOffsets& fo, int my_n, const int32_t* ids,
                                           const float* kss, const float* vss, uint32_t bar0,
                                           uint32_t sbase, uint8_t* smem, int t0, int t1,
                                           int warp, float scale_log2, int lane, Issue&& issue,
                                           Patch&& patch) {
  constexpr int kStage = ChunkGeom<D>::kStageBytes;
  using Scores = typename std::conditional<I8, ScoresI8<D, TWO>, ScoresBf16<D, TWO>>::type;
  Scores sc;
  uint32_t pa[2][I8 ? 4 : 2];
  float qs[2][2];  // INT8: query sums of this lane's score columns
  if constexpr (I8) query_sums_t(qf, qs, lane);
  auto sK = [&](int j) { return sbase + (j % S) * kStage; };
  auto wait = [&](int j) {
    const bool done = mbar_wait(bar0 + 8 * (j % S), (j / S) & 1);
    return __all_sync(0xffffffffu, done);
  };
  // valid-token mask of a bf16 chunk; zero the V rows of the others
  auto prepare = [&](int j) -> uint32_t {
    if constexpr (I8) {
      return 0xFFFFFFFFu;
    } else {
      const int nv = t1 - (t0 + kPage * (warp + j * NW));
      const uint32_t valid = nv >= kPage ? 0xFFFFu : ((1u << nv) - 1u);
      if (valid != 0xFFFFu) {
        zero_invalid_v_rows<D>(smem + (sK(j) + kStage / 2 - smem_u32(smem)), valid, lane);
        __syncwarp();
      }
      return valid;
    }
  };
  auto qk = [&](int j) {
    if constexpr (I8)
      qk_i8(sc, qf, fo, sK(j));
    else
      qk_bf16(sc, qf, fo, sK(j));
  };
  auto softmax = [&](int j, uint32_t valid) {
    if constexpr (I8)
      softmax_i8(st, qs, sc, pa, kss[j], vss[j], scale_log2);
    else
      softmax_bf16(st, sc, pa, valid, scale_log2, lane);
  };
  auto pv = [&](int j) {
    if constexpr (I8)
      pv_i8(st, pa, fo, sK(j) + kStage / 2);
    else
      pv_bf16(st, pa, fo, sK(j) + kStage / 2);
  };
  // In-order walk: each chunk is folded in completely before its stage is
  // refilled.  (Issuing chunk j+1's scores ahead of chunk j's output update
  // was measured slower: it delays the refill, so fewer bytes are in flight.)
  for (int j = 0; j < my_n; ++j) {
    if (!wait(j)) return j;
    const uint32_t valid = prepare(j);
    if (ids[j] >= 0) {
      patch(j, sK(j));  // the stack kernel's fused append: the new row from the input
      qk(j);
      softmax(j, valid);
      pv(j);
    }
    __syncwarp();
    if (lane == 0 && j + S < my_n) {
      fence_proxy_async_smem();
      issue(j + S);
    }
  }
  return -1;
}

// Shared-prefix call: CTA (b, h, s) checks its slice of request b's first
// skip_len / 16 page ids against row 0's (the ids the prefix pass reads)
// and records the result for the merge.  Kept out of line: it runs only in
// that call and must not add to the decode loop's register pressure.
__device__ __noinline__ void check_prefix_ids(const SplitArgs& a, int b, int h, int s) {
  const int slots = a.Hkv * a.max_splits, slot = h * a.max_splits + s;
  const int np = a.skip_len / kPage;
  const int i0 = static_cast<int>(static_cast<long long>(np) * slot / slots);
  const int i1 = static_cast<int>(static_cast<long long>(np) * (slot + 1) / slots);
  const int32_t* row = a.block_table + static_cast<size_t>(b) * a.max_pages;
  int bad = 0;
  if (b > 0)
    for (int i = i0 + static_cast<int>(threadIdx.x); i < i1; i += blockDim.x)
      bad |= __ldg(row + i) != __ldg(a.block_table + i);
  bad = __syncthreads_or(bad || a.seq_lens[b] < a.skip_len);
  if (threadIdx.x == 0) {
    a.prefix_bad[(static_cast<size_t>(b) * a.Hkv + h) * a.max_splits + s] = bad;
    if (bad) set_status(a.status, PHS_ESHAPE);
  }
}

// The work of one CTA: request b, KV head h, split s.  q/out/ws_o/ws_ml are
// the layer's; `app` (k_new null: none) is an append fused into this
// launch, done one of two ways:
//   WRITE_FIRST (single-layer launches): the CTA holding token n-1 writes it
//     into its page before it issues its copies, which then read it back --
//     nothing in the chunk loop, so no register cost there;
//   otherwise (the stack kernel, whose layers may share one pool): it writes
//     the page and patches its staged copy from the input in the loop, so
//     each layer attends its own token even when another layer of the same
//     launch writes the same slot.
// MIXED: the launch may hold INT8 splits (a.qlens set); without them the
// INT8 walk is compiled out, which leaves the bf16 walk its registers.
template <int D, bool TWO, bool MIXED, bool WRITE_FIRST, int NW = kSplitWarps>
__device__ __forceinline__ void split_body(const CUtensorMap* tk, const CUtensorMap* tv,
                                           const CUtensorMap* tk8, const CUtensorMap* tv8,
                                           const SplitArgs& a, const __nv_bfloat16* q,
                                           void* out, float* ws_o, float* ws_ml,
                                           const FusedAppend& app, int b, int h, int s) {
  using L = SplitLayout<D, NW>;
  constexpr int S = L::kStages;
  constexpr int GR = TWO ? 16 : 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // a dependent launch (merge, or the next layers' SWA work) may start as
  // soon as every CTA of this grid is running; it waits for our results
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;

  if (a.prefix_bad != nullptr) check_prefix_ids(a, b, h, s);

  int n = a.seq_lens[b];
  // a fused append has a slot for the new token only inside the table
  const bool appends = app.k_new != nullptr && n >= 1 && n <= a.n_clamp;
  if (n > a.n_clamp) {  // longer than its block table or the stated bound
    if (s == 0 && h == 0 && threadIdx.x == 0) set_status(a.status, PHS_ERANGE);
    n = a.n_clamp;
  }
  const int qlen = MIXED && a.qlens ? a.qlens[b] : 0;
  const int T = a.T;
  const int ns = min(request_splits(n, qlen, T, a.skip_len), a.max_splits);
  if (ns < 0) {
    if (s == 0 && h == 0 && threadIdx.x == 0) set_status(a.status, PHS_ERANGE);
    return;
  }
  // a fused append writes bf16 pages only: a new token inside the request's
  // INT8 region is not written and is an error
  if (MIXED && app.k_new != nullptr && n >= 1 && n - 1 < qlen && s == 0 && h == 0 &&
      threadIdx.x == 0)
    set_status(a.status, PHS_ERANGE);
  const size_t out_row0 = (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * G) * D;
  if (ns == 0) {  // empty request: zero output (unless another kernel owns it)
    // a fused append whose new token falls inside the shared prefix (n ==
    // skip_len): its page is one of the shared ones, so it is not written
    if (app.k_new != nullptr && n >= 1 && n - 1 < a.skip_len && s == 0 && threadIdx.x == 0)
      set_status(a.status, PHS_ESHARED);
    if (s == 0 && !a.force_partial)
      for (int e = threadIdx.x; e < G * D; e += blockDim.x) store_out(out, out_row0 + e, 0.f, a.out_f32);
    return;
  }
  if (s >= ns) return;

  const int nsq = (qlen + T - 1) / T;
  const bool is_i8 = MIXED && s < nsq;
  int t0, t1, nch;
  if (is_i8) {
    t0 = s * T;
    t1 = min(t0 + T, qlen);
    nch = (t1 - t0) / kQBlock;
  } else {
    t0 = max(qlen, a.skip_len) + (s - nsq) * T;
    t1 = min(t0 + T, n);
    nch = (t1 - t0 + kPage - 1) / kPage;
  }
  const int my_n = warp < nch ? (nch - warp + NW - 1) / NW : 0;

  // ---- chunk ids (physical page / INT8 page) of this warp; the INT8
  // scales, which need the ids, are loaded after the first copies are issued
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L::kIdsOff) + warp * kMaxChunksPerWarp * 3;
  float* kss = reinterpret_cast<float*>(ids + kMaxChunksPerWarp);
  float* vss = kss + kMaxChunksPerWarp;
  for (int j = lane; j < my_n; j += 32) {
    const int ci = warp + j * NW;
    int id;
    if (is_i8) {
      const int lq = t0 / kQBlock + ci;
      id = lq < a.max_qpages ? a.qtable[static_cast<size_t>(b) * a.max_qpages + lq] : -1;
      if (id < 0 || id >= a.num_qpages) {
        set_status(a.status, PHS_ERANGE);
        id = -1;
      }
    } else {
      const int lp = t0 / kPage + ci;  // < max_pages: n was clamped above
      id = a.block_table[static_cast<size_t>(b) * a.max_pages + lp];
      if (id < 0 || id >= a.num_pages) {
        set_status(a.status, PHS_ERANGE);
        id = -1;
      }
    }
    ids[j] = id;
  }
  const uint32_t bar0 = smem_u32(smem + L::kBarOff) + warp * S * 8;
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint32_t sbase = smem_u32(smem) + warp * S * L::kStage;
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int j) {  // lane 0 only
    const uint32_t bar = bar0 + 8 * (j % S);
    const uint32_t dst = sbase + (j % S) * L::kStage;
    const int id = ids[j];
    if (id < 0) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      return;
    }
    mbar_arrive_expect_tx(bar, L::kStage);
    if (is_i8) {  // K: 32 rows of D codes; V^T: D/4 rows of 128 bytes
      const int kv = id * a.Hkv + h;
      tma_load_2d(dst, tk8, 0, kv * kQBlock, bar, pol);
      tma_load_2d(dst + L::kStage / 2, tv8, 0, kv * (D / 4), bar, pol);
    } else {
      const int row = (id * a.Hkv + h) * kPage;
      if constexpr (D == 128) {  // one 4 KB box per page: [half][16 rows]
        tma_load_3d(dst, tk, 0, row, 0, bar, pol);
        tma_load_3d(dst + L::kStage / 2, tv, 0, row, 0, bar, pol);
      } else {
        tma_load_2d(dst, tk, 0, row, bar, pol);
        tma_load_2d(dst + L::kStage / 2, tv, 0, row, bar, pol);
      }
    }
  };
  // fused append, before any copy is issued: the warp whose chunk holds
  // token n - 1 (the request's last token, so in this split only if it is the
  // last bf16 split) writes the new row into its page -- unless the page is
  // shared -- and the chunk's copy reads it back like any other row.  The
  // proxy fences order those generic stores before the copies.
  if (WRITE_FIRST && appends && !is_i8 && n - 1 >= t0 && n - 1 < t1) {
    const int ci = (n - 1 - t0) / kPage;  // chunk within the split
    if (ci % NW == warp) {
      const int id = ids[ci / NW], r = (n - 1) % kPage;
      if (id >= 0) {
        if (a.page_refcount != nullptr && __ldg(a.page_refcount + id) != 1) {
          if (lane == 0) set_status(a.status, PHS_ESHARED);  // a shared page: left as it is
        } else {
          const int op = lane >> 4, c = lane & 15;  // lanes 0-15 K, 16-31 V
          if (c < D / 8) {
            const size_t src = (static_cast<size_t>(b) * a.Hkv + h) * D + c * 8;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>((op ? app.v_new : app.k_new) + src));
            __nv_bfloat16* pool = op ? app.v_pool : app.k_pool;
            *reinterpret_cast<uint4*>(
                pool + ((static_cast<size_t>(id) * a.Hkv + h) * kPage + r) * D + c * 8) = v;
            fence_proxy_async_global();
          }
        }
      }
      __syncwarp();
      if (lane == 0) fence_proxy_async_global();
    }
  }
  if (lane == 0) {
    if (is_i8) {
      prefetch_tmap(tk8);
      prefetch_tmap(tv8);
    } else {
      prefetch_tmap(tk);
      prefetch_tmap(tv);
    }
    for (int j = 0; j < S && j < my_n; ++j) issue(j);
  }
  if (is_i8) {
    for (int j = lane; j < my_n; j += 32) {
      const int id = ids[j];
      kss[j] = id >= 0 ? __ldg(a.k_scale + static_cast<size_t>(id) * a.Hkv + h) : 0.f;
      vss[j] = id >= 0 ? __ldg(a.v_scale + static_cast<size_t>(id) * a.Hkv + h) : 0.f;
    }
  }

  // ---- queries of the group (overlaps the first loads)
  QFrags<D, TWO> qf;
  const __nv_bfloat16* qg = q + out_row0;
  if (is_i8)
    load_q_f16_i8order(qf, qg, G, lane);
  else
    load_q_bf16(qf, qg, G, lane);
  __syncwarp();  // every lane's scales are in shared memory

  WarpState<D, TWO> st;
  st.reset();
  FragOffsets fo;
  fo.init<D>(lane);
  auto no_patch = [](int, uint32_t) {};
  // in-loop append (stack kernel): row (n-1) % 16 of the chunk holding token
  // n-1; lanes 0-15 carry K, 16-31 V, 16 bytes each (the staged tile is
  // [half][16 rows][128 B] with the 128-byte swizzle)
  auto patch = [&](int j, uint32_t stage) {
    if (app.k_new == nullptr) return;
    const int r = n - 1 - (t0 + kPage * (warp + j * NW));
    if (r < 0 || r >= kPage) return;
    // (a length past the table was clamped: no slot for its new token; read
    // again here so that nothing extra stays live across the loop)
    if (__ldg(a.seq_lens + b) > a.n_clamp) return;
    if (a.page_refcount != nullptr && __ldg(a.page_refcount + ids[j]) != 1) {
      // a shared page: leave it (and the staged copy of it) as it is
      if (lane == 0) set_status(a.status, PHS_ESHARED);
      return;
    }
    const int op = lane >> 4, c = lane & 15;
    if (c < D / 8) {
      const size_t src = (static_cast<size_t>(b) * a.Hkv + h) * D + c * 8;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>((op ? app.v_new : app.k_new) + src));
      const uint32_t dst = stage + op * (L::kStage / 2) + (c >> 3) * 2048 + r * 128 +
                           (((c & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(smem + (dst - smem_u32(smem))) = v;
      __nv_bfloat16* pool = op ? app.v_pool : app.k_pool;
      *reinterpret_cast<uint4*>(
          pool + ((static_cast<size_t>(ids[j]) * a.Hkv + h) * kPage + r) * D + c * 8) = v;
    }
    __syncwarp();
  };
  int failed;
  if (is_i8)
    failed = walk_chunks<true, D, TWO, S, NW>(st, qf, fo, my_n, ids, kss, vss, bar0, sbase, smem, t0,
                                          t1, warp, a.scale_log2, lane, issue, no_patch);
  else if constexpr (WRITE_FIRST)
    failed = walk_chunks<false, D, TWO, S, NW>(st, qf, fo, my_n, ids, kss, vss, bar0, sbase, smem,
                                           t0, t1, warp, a.scale_log2, lane, issue, no_patch);
  else
    failed = walk_chunks<false, D, TWO, S, NW>(st, qf, fo, my_n, ids, kss, vss, bar0, sbase, smem,
                                           t0, t1, warp, a.scale_log2, lane, issue, patch);
  if (failed >= 0 && lane == 0) {
    // gave up: record it and drain (bounded) the loads still in flight
    set_status(a.status, PHS_ETIMEOUT);
    for (int k = failed; k < my_n && k < failed + S; ++k)
      (void)mbar_wait(bar0 + 8 * (k % S), (k / S) & 1);
  }

  // ---- warp result -> shared memory -> CTA merge
  const int g = lane >> 2, qd = lane & 3;
  float lsum[4];
  if (is_i8) {  // query columns: reduce over the 8 lanes of the same q
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v = st.l[i];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      lsum[i] = v;
    }
  } else {  // query rows: reduce over the quad
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) lsum[rh] = warp_sum_quad(st.l[rh]);
  }
  __syncthreads();  // every warp is done with its stages
  float* sO = reinterpret_cast<float*>(smem);
  float* sM = sO + NW * GR * D;
  float* sL = sM + NW * GR;
  if (is_i8) {
    // O^T element (dt, nq, k): dim 16dt + g + 8(k>>1), query 8nq + 2q + (k&1);
    // the output is held in units of the V scale st.u
#pragma unroll
    for (int nq = 0; nq < (TWO ? 2 : 1); ++nq)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * nq + 2 * qd + e;
        if (row < G) {
#pragma unroll
          for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              sO[(warp * GR + row) * D + 16 * dt + 8 * hh + g] = oT(st, dt, nq, 2 * hh + e) * st.u;
          if (g == 0) {
            sM[warp * GR + row] = st.m[2 * nq + e];
            sL[warp * GR + row] = lsum[2 * nq + e];
          }
        }
      }
  } else {
#pragma unroll
    for (int rh = 0; rh < (TWO ? 2 : 1); ++rh) {
      const int row = g + 8 * rh;
      if (row < G) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) sO[(warp * GR + row) * D + 8 * nt + 2 * qd + e] = st.o[nt][2 * rh + e];
        if (qd == 0) {
          sM[warp * GR + row] = st.m[rh];
          sL[warp * GR + row] = lsum[rh];
        }
      }
    }
  }
  __syncthreads();
  const size_t part = (static_cast<size_t>(b) * a.Hkv + h) * a.max_splits + s;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int row = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sM[w * GR + row]);
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = sM[w * GR + row];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      Lsum += sL[w * GR + row] * f;
      O += sO[(w * GR + row) * D + d] * f;
    }
    if (ns == 1 && !a.force_partial) {
      store_out(out, out_row0 + e, Lsum > 0.f ? O / Lsum : 0.f, a.out_f32);
    } else {
      ws_o[(part * G + row) * D + d] = O;
      if (d == 0) {
        ws_ml[(part * G + row) * 2] = M;
        ws_ml[(part * G + row) * 2 + 1] = Lsum;
      }
    }
  }
}

// request index fastest: CTAs that read the same shared-prefix pages for
// different requests run close together in time and share them through L2
template <int D, bool TWO, bool MIXED, int NW = kSplitWarps>
__global__ void __launch_bounds__(NW * 32, NW == kSplitWarps ? PHS_SPLIT_MIN_CTAS : 1)
    phs_split_decode_kernel(const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv,
                            const __grid_constant__ CUtensorMap tk8,
                            const __grid_constant__ CUtensorMap tv8, const SplitArgs a) {
  split_body<D, TWO, MIXED, true, NW>(&tk, &tv, &tk8, &tv8, a, a.q, a.out, a.ws_o, a.ws_ml, a.app,
                                  blockIdx.x, blockIdx.y, blockIdx.z);
  // started early beside an independent grid: one CTA holds this grid open
  // until that grid has finished, so a launch that waits for this grid also
  // sees the other's results
  if (a.wait_prior_at_exit && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    pdl_wait_prior_grid();
}

// Every Full layer of a hybrid stack in one launch: blockIdx.z = layer *
// max_splits + split; each layer brings its own pool maps, queries, output,
// partials and new token.  Source: "Xiaomi MiMo-V2.5 inference system" page,
// section 2 (layer-wise overlap of the step; whole-step replay).  The Full
// layers of a stack hold bf16 pages only.
template <int D, bool TWO, int NW = kSplitWarps>
__global__ void __launch_bounds__(NW * 32, NW == kSplitWarps ? PHS_SPLIT_MIN_CTAS : 1)
    phs_stack_full_kernel(const __grid_constant__ StackFullParams p) {
  const int l = blockIdx.z / p.a.max_splits, s = blockIdx.z - l * p.a.max_splits;
  const StackFullLayer& L = p.layer[l];
  split_body<D, TWO, false, false, NW>(&L.tk, &L.tv, &L.tk, &L.tv, p.a, L.q, L.out, L.ws_o, L.ws_ml,
                                   L.app, blockIdx.x, blockIdx.y, s);
}

// A whole small hybrid step in one launch (every request in one split, so
// nothing to merge, and all CTAs in one wave): CTAs [0, full_ctas) run the
// Full layers' splits, the rest one SWA unit each.  Both bodies are the
// ones the two separate launches run, so the results are the same; the step
// pays one launch instead of two (2-layer hybrid step at batch 2, replayed as
// a CUDA graph: 8.2 -> 6.2 us; two launches cost the same whether dependent or
// parallel).  Source: "Xiaomi MiMo-V2.5 inference system" page, section 2
// (the step's layers in few launches; whole-step replay).
template <int D, bool TWO>
__global__ void __launch_bounds__(2 * kSplitWarps * 32, 1)
    phs_stack_small_kernel(const __grid_constant__ StackSmallParams p) {
  const int i = blockIdx.x;
  if (i < p.full_ctas) {
    const int B = p.B, Hkv = p.full.a.Hkv;
    const int b = i % B, h = (i / B) % Hkv, l = i / (B * Hkv);
    const StackFullLayer& L = p.full.layer[l];
    split_body<D, TWO, false, false, 2 * kSplitWarps>(&L.tk, &L.tv, &L.tk, &L.tv, p.full.a, L.q,
                                                      L.out, L.ws_o, L.ws_ml, L.app, b, h, 0);
  } else {
    swa_chunked_unit<D, TWO, kSwaMaxLayers>(p.swa, i - p.full_ctas);
  }
}

int stack_small_smem_bytes(int D, int G, int smem_optin) {
  const int split = D == 128 ? SplitLayout<128, 2 * kSplitWarps>::kAlloc
                             : SplitLayout<64, 2 * kSplitWarps>::kAlloc;
  const int swa = SwaChunkLayout(D, G).total;
  const int need = split > swa ? split : swa;
  return need <= smem_optin ? need : 0;
}

// Cross-split merge of one (request, KV head): warp w of the CTA merges
// query rows w, w+4, ...
template <int D>
__device__ __forceinline__ void merge_body(const MergeArgs& a, const float* ws_o,
                                           const float* ws_ml, void* out, int b, int h) {
  pdl_wait_prior_grid();  // launched as a dependent of the split launch
  merge_request<D>(a, ws_o, ws_ml, out, b, h, threadIdx.x >> 5, blockDim.x >> 5);
}

template <int D>
__global__ void __launch_bounds__(128) phs_merge_kernel(const MergeArgs a) {
  merge_body<D>(a, a.ws_o, a.ws_ml, a.out, blockIdx.x, blockIdx.y);
}

// The merges of every Full layer of a hybrid stack in one launch (z = layer).
template <int D>
__global__ void __launch_bounds__(128) phs_stack_merge_kernel(const __grid_constant__ StackMergeParams p) {
  const StackMergeLayer& L = p.layer[blockIdx.z];
  merge_body<D>(p.a, L.ws_o, L.ws_ml, L.out, blockIdx.x, blockIdx.y);
}

// ------------------------------------------------------------ launchers --
// A bf16 launch whose grid has at most one CTA per SM (a latency-bound small
// step) runs 8 warps per CTA, halving each warp's chain of chunks.
static bool single_wave(const SplitArgs& a, long long ctas) {
  return a.qlens == nullptr && a.num_sms > 0 && ctas <= a.num_sms;
}

template <int D, bool TWO>
static int launch_split_t(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tk8,
                          const CUtensorMap& tv8, const SplitArgs& a, int B, cudaStream_t stream,
                          bool dependent) {
  const bool wide = single_wave(a, 1LL * B * a.Hkv * a.max_splits);
  auto kern = wide ? phs_split_decode_kernel<D, TWO, false, 2 * kSplitWarps>
              : a.qlens ? phs_split_decode_kernel<D, TWO, true>
                        : phs_split_decode_kernel<D, TWO, false>;
  const int nw = wide ? 2 * kSplitWarps : kSplitWarps;
  const int smem = wide ? SplitLayout<D, 2 * kSplitWarps>::kAlloc : SplitLayout<D>::kAlloc;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != PHS_OK) return PHS_ECUDA;
  dim3 grid(B, a.Hkv, a.max_splits);
  if (!dependent) {
    kern<<<grid, nw * 32, smem, stream>>>(tk, tv, tk8, tv8, a);
    return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(nw * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, tk8, tv8, a) == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int launch_split_decode(int D, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tk8, const CUtensorMap& tv8, const SplitArgs& a,
                        int B, cudaStream_t stream, bool dependent) {
  const bool two = a.G > 8;
  if (D == 128) {
    return two ? launch_split_t<128, true>(tk, tv, tk8, tv8, a, B, stream, dependent)
               : launch_split_t<128, false>(tk, tv, tk8, tv8, a, B, stream, dependent);
  }
  if (D == 64) {
    return two ? launch_split_t<64, true>(tk, tv, tk8, tv8, a, B, stream, dependent)
               : launch_split_t<64, false>(tk, tv, tk8, tv8, a, B, stream, dependent);
  }
  return PHS_EUNSUPPORTED;
}

template <int D, bool TWO>
static int launch_stack_full_t(const StackFullParams& p, int B, cudaStream_t stream) {
  const bool wide = single_wave(p.a, 1LL * B * p.a.Hkv * p.a.max_splits * p.num_layers);
  auto kern = wide ? phs_stack_full_kernel<D, TWO, 2 * kSplitWarps> : phs_stack_full_kernel<D, TWO>;
  const int nw = wide ? 2 * kSplitWarps : kSplitWarps;
  const int smem = wide ? SplitLayout<D, 2 * kSplitWarps>::kAlloc : SplitLayout<D>::kAlloc;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != PHS_OK) return PHS_ECUDA;
  dim3 grid(B, p.a.Hkv, p.a.max_splits * p.num_layers);
  kern<<<grid, nw * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

template <int D, bool TWO>
static int launch_stack_small_t(const StackSmallParams& p, int swa_units, int smem,
                                cudaStream_t stream) {
  auto kern = phs_stack_small_kernel<D, TWO>;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != PHS_OK) return PHS_ECUDA;
  kern<<<static_cast<unsigned>(p.full_ctas + swa_units), 2 * kSplitWarps * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int launch_stack_small(int D, const StackSmallParams& p, int swa_units, cudaStream_t stream) {
  if (p.full.a.max_splits != 1 || p.full.num_layers <= 0 || p.swa.num_layers <= 0) return PHS_EINVAL;
  const int smem = stack_small_smem_bytes(D, p.full.a.G, 1 << 30);
  const bool two = p.full.a.G > 8;
  if (D == 128)
    return two ? launch_stack_small_t<128, true>(p, swa_units, smem, stream)
               : launch_stack_small_t<128, false>(p, swa_units, smem, stream);
  if (D == 64)
    return two ? launch_stack_small_t<64, true>(p, swa_units, smem, stream)
               : launch_stack_small_t<64, false>(p, swa_units, smem, stream);
  return PHS_EUNSUPPORTED;
}

int launch_stack_full(int D, const StackFullParams& p, int B, cudaStream_t stream) {
  if (p.num_layers <= 0 || p.num_layers > kStackMaxFull || p.a.qlens) return PHS_EINVAL;
  if (static_cast<long long>(p.a.max_splits) * p.num_layers > 65535) return PHS_EUNSUPPORTED;
  const bool two = p.a.G > 8;
  if (D == 128)
    return two ? launch_stack_full_t<128, true>(p, B, stream)
               : launch_stack_full_t<128, false>(p, B, stream);
  if (D == 64)
    return two ? launch_stack_full_t<64, true>(p, B, stream)
               : launch_stack_full_t<64, false>(p, B, stream);
  return PHS_EUNSUPPORTED;
}

// Launch as a programmatic dependent of the previous launch on the stream
// (the kernel waits for that grid before reading its results).
template <typename Kern, typename Arg>
static int launch_dependent(Kern kern, dim3 grid, dim3 block, int smem, cudaStream_t stream,
                            const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, arg) == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

int launch_stack_merge(int D, const StackMergeParams& p, int B, int num_layers,
                       cudaStream_t stream) {
  if (num_layers <= 0 || num_layers > kStackMaxFull) return PHS_EINVAL;
  dim3 grid(B, p.a.Hkv, num_layers);
  if (D == 128) return launch_dependent(phs_stack_merge_kernel<128>, grid, 128, 0, stream, p);
  if (D == 64) return launch_dependent(phs_stack_merge_kernel<64>, grid, 128, 0, stream, p);
  return PHS_EUNSUPPORTED;
}

int launch_merge(int D, const MergeArgs& a, int B, cudaStream_t stream) {
  dim3 grid(B, a.Hkv);
  if (D == 128) return launch_dependent(phs_merge_kernel<128>, grid, 128, 0, stream, a);
  if (D == 64) return launch_dependent(phs_merge_kernel<64>, grid, 128, 0, stream, a);
  return PHS_EUNSUPPORTED;
}

}  // namespace phs
