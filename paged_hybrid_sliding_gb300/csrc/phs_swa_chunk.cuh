// phs_swa_chunk.cuh -- the chunked shape of the sliding-window decode: one
// CTA per (layer, request, KV head) unit, the unit's chunks spread over its
// warps.  Shared by the SWA launch (phs_swa.cu) and by the one-launch small
// hybrid step (phs_decode.cu).
//
// Source: "Xiaomi MiMo-V2.5 inference system" page, section 1 (SWA layers
// attend to the most recent 128 tokens) and section 2 (a ring buffer of W
// slots per request).
#pragma once

#include "phs_attn.cuh"
#include "phs_internal.h"
#include "phs_merge.cuh"

namespace phs {

__device__ __forceinline__ uint8_t* swa_align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct SwaUnit {
  int l, b, h, ring, pos, n;
  bool ok;
};

// Latency shape for small steps: one CTA per (layer, request, KV head)
// unit, its warps taking the unit's chunks round-robin (warp w: chunks w,
// w + 4, ...).  A 128-slot ring is then two chunks per warp instead of eight
// in one warp's dependent chain (2-layer hybrid step at batch 2: the SWA
// launch spent ~15,000 SM cycles on one warp's serial chunk chain, issue
// mostly stalled on fixed-latency dependencies).  The warps' states meet in
// shared memory, over the finished stages.  Used when every unit has an SM
// of its own.
constexpr int kSwaChunkWarps = 4;
constexpr int kSwaChunkStages = 2;

struct SwaChunkLayout {
  int kv, qslot, q_off, bar_off, total;
  __host__ __device__ SwaChunkLayout(int D, int G) {
    kv = 64 * D;                                            // K + V tile of 16 tokens
    qslot = (G * D * 2 + 127) / 128 * 128;                  // the group's queries
    q_off = kSwaChunkWarps * kSwaChunkStages * kv;
    bar_off = q_off + qslot;
    total = bar_off + (kSwaChunkWarps * kSwaChunkStages + 1) * 8 + 1024;  // + alignment slack
  }
};

// One unit of the chunked shape, by the calling CTA (of kSwaChunkWarps warps
// or more: the warps past them take no chunks and only help write the
// output, so the result does not depend on the CTA's size).
template <int D, bool TWO, int MAXL>
__device__ __forceinline__ void swa_chunked_unit(const SwaParams<MAXL>& p, int unit) {
  constexpr int NW = kSwaChunkWarps, S = kSwaChunkStages;
  constexpr int GR = TWO ? 16 : 8;  // query rows a warp state holds
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = swa_align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, G = p.G, W = p.W;
  const SwaChunkLayout L(D, G);
  const int CPU = W / kPage;
  const int BH = p.B * Hkv;
  SwaUnit u;
  u.l = unit / BH;
  const int rem = unit - u.l * BH;
  u.b = rem / Hkv;
  u.h = rem - u.b * Hkv;
  u.ring = p.ring_ids ? __ldg(p.ring_ids + u.b) : u.b;
  u.pos = __ldg(p.ring_pos + u.b);
  u.n = __ldg(p.seq_lens + u.b);
  u.ok = u.ring >= 0 && u.ring < p.num_rings[u.l] && u.pos >= 0 && u.pos < W && u.n >= 0;
  // this warp's stage barriers and stages (used by warps < NW only)
  const uint32_t bar0 = sb + L.bar_off + warp * S * 8;
  const uint32_t qbar = sb + L.bar_off + NW * S * 8;
  const uint32_t sbase = sb + warp * S * L.kv;
  const uint32_t qs = sb + L.q_off;
  __shared__ int fail;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * S + 1; ++i) mbar_init(sb + L.bar_off + 8 * i, 1);
    fence_mbar_init();
    fail = 0;
  }
  __syncthreads();
  const int my = warp < NW && warp < CPU ? (CPU - warp + NW - 1) / NW : 0;  // this warp's chunks
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int jj) {  // lane 0: chunk warp + NW jj into stage jj % S
    const uint32_t bar = bar0 + 8 * (jj % S), dst = sbase + (jj % S) * L.kv;
    mbar_arrive_expect_tx(bar, L.kv);
    const int row = (u.ring * Hkv + u.h) * W + kPage * (warp + NW * jj);
    if constexpr (D == 128) {  // one 4 KB box per 16-row block: [half][16 rows]
      tma_load_3d(dst, &p.tk[u.l], 0, row, 0, bar, pol);
      tma_load_3d(dst + L.kv / 2, &p.tv[u.l], 0, row, 0, bar, pol);
    } else {
      tma_load_2d(dst, &p.tk[u.l], 0, row, bar, pol);
      tma_load_2d(dst + L.kv / 2, &p.tv[u.l], 0, row, bar, pol);
    }
  };
  if (u.ok) {
    if (threadIdx.x == 0) {
      const uint32_t qbytes = static_cast<uint32_t>(G * D * 2);
      mbar_arrive_expect_tx(qbar, qbytes);
      bulk_load(qs, p.q[u.l] + (static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G) * D,
                qbytes, qbar);
    }
    if (lane == 0)
      for (int jj = 0; jj < S && jj < my; ++jj) issue(jj);
  } else if (threadIdx.x == 0) {
    set_status(p.status, PHS_ERANGE);
  }

  WarpState<D, TWO> st;
  st.reset();
  if (u.ok && warp < NW) {
    QFrags<D, TWO> qf;
    FragOffsets fo;
    fo.init<D>(lane);
    bool ok = __all_sync(0xffffffffu, mbar_wait(qbar, 0));
    if (ok) load_q_bf16_smem<D, TWO>(qf, qs, G, lane);
    const int nv = min(u.n, W);  // valid slots: the last nv tokens
    const FusedAppend& app = p.app[u.l];
    const bool appends = app.k_new != nullptr && u.n > 0;
    int jj = 0;
    for (; ok && jj < my; ++jj) {
      const int ci = warp + NW * jj, stg = jj % S;
      if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * stg, (jj / S) & 1))) {
        ok = false;
        break;
      }
      const uint32_t sK = sbase + stg * L.kv, sV = sK + L.kv / 2;
      if (appends) {
        // fused append: the new token sits in slot u.pos; write it into the
        // ring and patch the staged row from the input (lanes 0-15 K, 16-31 V)
        const int r = u.pos - kPage * ci;
        if (r >= 0 && r < kPage) {
          const int op = lane >> 4, cc = lane & 15;
          if (cc < D / 8) {
            const size_t src = (static_cast<size_t>(u.b) * Hkv + u.h) * D + cc * 8;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>((op ? app.v_new : app.k_new) + src));
            const uint32_t dst =
                (op ? sV : sK) + (cc >> 3) * 2048 + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + (dst - sb)) = v;
            __nv_bfloat16* ring = op ? app.v_pool : app.k_pool;
            *reinterpret_cast<uint4*>(
                ring + ((static_cast<size_t>(u.ring) * Hkv + u.h) * W + u.pos) * D + cc * 8) = v;
          }
          __syncwarp();
        }
      }
      uint32_t valid = 0xFFFFu;
      if (nv < W) {
        int dist = u.pos - (kPage * ci + (lane & 15));  // age of the token in this slot
        if (dist < 0) dist += W;
        valid = __ballot_sync(0xffffffffu, dist < nv) & 0xFFFFu;
      }
      if (valid != 0u) {
        if (valid != 0xFFFFu) {
          zero_invalid_v_rows<D>(smem + (sV - sb), valid, lane);
          __syncwarp();
        }
        consume_bf16<D, TWO>(st, qf, fo, sK, sV, valid, p.scale_log2, lane);
      }
      __syncwarp();
      if (lane == 0 && jj + S < my) {
        fence_proxy_async_smem();
        issue(jj + S);
      }
    }
    if (!ok && lane == 0) {
      // gave up: drain (bounded) this warp's copies still in flight
      set_status(p.status, PHS_ETIMEOUT);
      fail = 1;
      for (int t = jj; t < my && t < jj + S; ++t) (void)mbar_wait(bar0 + 8 * (t % S), (t / S) & 1);
      if (warp == 0) (void)mbar_wait(qbar, 0);
    }
  }
  // ---- the warps' states, combined through shared memory (over the
  // stages, which every warp has finished with)
  const int g = lane >> 2, qd = lane & 3;
  float lsum[2];
#pragma unroll
  for (int rh = 0; rh < 2; ++rh) lsum[rh] = warp_sum_quad(st.l[rh]);
  __syncthreads();
  const bool write = u.ok && !fail;
  float* sO = reinterpret_cast<float*>(smem);
  float* sM = sO + NW * GR * D;
  float* sL = sM + NW * GR;
  if (write && warp < NW) {
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
  if (write) {
    const size_t out_row0 = (static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G) * D;
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
      store_out(p.out[u.l], out_row0 + e, Lsum > 0.f ? O / Lsum : 0.f, p.out_f32);
    }
  }
}

}  // namespace phs
