// phs_swa.cu -- sliding-window decode over SWA ring buffers, one or many
// layers per launch.
//
// Work unit: (layer, request, KV head) = the W ring slots of one head, read
// as W/16 chunks of 16 slots.  The kernel is persistent: each warp walks a
// strided list of units and streams their chunks back to back through its
// own ring of S shared-memory stages, so loads of the next unit overlap the
// tail of the current one.  A stage holds a 16-slot K tile and V tile (TMA,
// 128-byte swizzle); the stage that carries a unit's first chunk also gets
// the group's queries in a slot of its own (1-D bulk copy).  A unit's output
// is written straight from the accumulators: no split, no workspace.  In a
// hybrid-stack step (phs_attn_decode_hybrid_stack_fused) the warp holding a
// request's newest slot also appends the new token (ring write + patch of
// the staged row from the input), and the warps take the Full layers'
// cross-split merges after their SWA units, once the split launch before
// them has finished (programmatic dependent launch).  Small steps (at most
// one unit per SM) take the chunked shape instead: one CTA per unit, its
// chunks spread over the CTA's warps (phs_swa_chunk.cuh).
//
// Sources: "Xiaomi MiMo-V2.5 inference system" page, section 1 (SWA layers
// keep and attend to the most recent 128 tokens) and section 2 (ring
// buffer of capacity W per request, storage O(W); SWA reads overlap layer
// by layer).
#include "phs_attn.cuh"
#include "phs_internal.h"
#include "phs_merge.cuh"
#include "phs_swa_chunk.cuh"

namespace phs {

// Shared-memory stages per warp.  Measured on 60 layers x batch 256: 2
// stages 6,845 GB/s, 3 stages 6,471, 4 (4 warps per CTA) 5,990 -- fewer
// copies in flight per SM run faster here.
#ifndef PHS_SWA_STAGES
#define PHS_SWA_STAGES 2
#endif
constexpr int kSwaStages = PHS_SWA_STAGES;
// Warps per CTA when their stages fit (one CTA per SM).  Measured with 2
// stages, same workload: 6 warps 6,679 GB/s, 7 6,850, 8 6,949, 10 6,715,
// 12 6,721.
#ifndef PHS_SWA_WARPS
#define PHS_SWA_WARPS 8
#endif
constexpr int kSwaWarps = PHS_SWA_WARPS;

// Shared-memory layout for NW warps of S stages: [stages][bars][query
// slots].  It does not depend on the batch: each warp reads its units'
// ring id, newest slot and length from global memory, one unit ahead.
struct SwaLayout {
  int kv, qslot, stages_bytes, bar_off, q_off, total;
  __host__ __device__ SwaLayout(int D, int G, int NW, int S) {
    kv = 64 * D;                                   // K + V tile of 16 tokens
    qslot = (G * D * 2 + 127) / 128 * 128;         // one group's queries
    stages_bytes = NW * S * kv;
    bar_off = stages_bytes;
    q_off = bar_off + NW * S * 8;
    total = q_off + NW * S * qslot + 1024;         // + base alignment slack
  }
};

template <int D, bool TWO, int MAXL, int NW, int S>
__global__ void __launch_bounds__(NW * 32, 1)
    phs_swa_decode_kernel(const __grid_constant__ SwaParams<MAXL> p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = swa_align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G, W = p.W;
  const SwaLayout L(D, G, NW, S);

  const int CPU = W / kPage;  // chunks per unit
  const int BH = B * Hkv;
  const int units = p.num_layers * BH;
  const int gw = blockIdx.x * NW + warp;
  const int tw = gridDim.x * NW;
  const int my_units = gw < units ? (units - gw + tw - 1) / tw : 0;
  const int total = my_units * CPU;

  const uint32_t bar0 = smem_u32(smem + L.bar_off) + warp * S * 8;
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t sbase = smem_u32(smem) + warp * S * L.kv;
  const uint32_t qbase = smem_u32(smem + L.q_off) + warp * S * L.qslot;
  const uint64_t pol = policy_evict_first();

  // unit k of this warp: its layer, request and KV head, and the request's
  // ring id, newest slot and length (read from global memory; validated
  // where used)
  auto unit_at = [&](int k) {
    SwaUnit u;
    const int id = gw + k * tw;
    u.l = id / BH;
    const int rem = id - u.l * BH;
    u.b = rem / Hkv;
    u.h = rem - u.b * Hkv;
    u.ring = p.ring_ids ? __ldg(p.ring_ids + u.b) : u.b;
    u.pos = __ldg(p.ring_pos + u.b);
    u.n = __ldg(p.seq_lens + u.b);
    return u;
  };
  auto checked = [&](SwaUnit u) {
    u.ok = u.ring >= 0 && u.ring < p.num_rings[u.l] && u.pos >= 0 && u.pos < W && u.n >= 0;
    return u;
  };

  // issuer state (lane 0): unit index, chunk within it, stage
  int ik = 0, ic = 0, ist = 0;
  SwaUnit iu;
  if (total > 0) iu = checked(unit_at(0));
  auto issue_next = [&]() {  // lane 0 only
    const uint32_t bar = bar0 + 8 * ist;
    const uint32_t dst = sbase + ist * L.kv;
    if (!iu.ok) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    } else {
      const uint32_t qbytes = ic == 0 ? static_cast<uint32_t>(G * D * 2) : 0u;
      mbar_arrive_expect_tx(bar, L.kv + qbytes);
      const int row = (iu.ring * Hkv + iu.h) * W + kPage * ic;
      if constexpr (D == 128) {  // one 4 KB box per 16-row block: [half][16 rows]
        tma_load_3d(dst, &p.tk[iu.l], 0, row, 0, bar, pol);
        tma_load_3d(dst + L.kv / 2, &p.tv[iu.l], 0, row, 0, bar, pol);
      } else {
        tma_load_2d(dst, &p.tk[iu.l], 0, row, bar, pol);
        tma_load_2d(dst + L.kv / 2, &p.tv[iu.l], 0, row, bar, pol);
      }
      if (ic == 0) {
        const __nv_bfloat16* q =
            p.q[iu.l] + (static_cast<size_t>(iu.b) * p.Hq + static_cast<size_t>(iu.h) * G) * D;
        bulk_load(qbase + ist * L.qslot, q, qbytes, bar);
      }
    }
    if (++ist == S) ist = 0;
    if (++ic == CPU) {
      ic = 0;
      if (++ik < my_units) iu = checked(unit_at(ik));
    }
  };

  if (lane == 0)
    for (int j = 0; j < S && j < total; ++j) issue_next();

  WarpState<D, TWO> st;
  QFrags<D, TWO> qf;
  FragOffsets fo;
  fo.init<D>(lane);
  const int g = lane >> 2, qd = lane & 3;
  int k = 0, c = 0, cst = 0;
  uint32_t phase = 0;
  SwaUnit u;
  // the consumer's next unit, loaded while the current one streams
  SwaUnit next;
  if (total > 0) next = unit_at(0);
  int j = 0;
  for (; j < total; ++j) {
    const uint32_t bar = bar0 + 8 * cst;
    const bool done = mbar_wait(bar, phase);
    if (!__all_sync(0xffffffffu, done)) {
      if (lane == 0) set_status(p.status, PHS_ETIMEOUT);
      break;
    }
    const uint32_t sK = sbase + cst * L.kv;
    const uint32_t sV = sK + L.kv / 2;
    if (c == 0) {
      u = checked(next);
      if (k + 1 < my_units) next = unit_at(k + 1);
      st.reset();
      if (u.ok)
        load_q_bf16_smem<D, TWO>(qf, qbase + cst * L.qslot, G, lane);
      else if (lane == 0)
        set_status(p.status, PHS_ERANGE);
    }
    if (u.ok && p.app[u.l].k_new != nullptr && u.n > 0) {
      // fused append: the new token sits in slot u.pos; write it into the
      // ring and patch the staged row from the input (lanes 0-15 K, 16-31 V)
      const int r = u.pos - kPage * c;
      if (r >= 0 && r < kPage) {
        const FusedAppend& app = p.app[u.l];
        const int op = lane >> 4, cc = lane & 15;
        if (cc < D / 8) {
          const size_t src = (static_cast<size_t>(u.b) * Hkv + u.h) * D + cc * 8;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>((op ? app.v_new : app.k_new) + src));
          const uint32_t dst = (op ? sV : sK) + (cc >> 3) * 2048 + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(smem + (dst - smem_u32(smem))) = v;
          __nv_bfloat16* ring = op ? app.v_pool : app.k_pool;
          *reinterpret_cast<uint4*>(
              ring + ((static_cast<size_t>(u.ring) * Hkv + u.h) * W + u.pos) * D + cc * 8) = v;
        }
        __syncwarp();
      }
    }
    if (u.ok) {
      const int nv = min(u.n, W);  // valid slots: the last nv tokens
      uint32_t valid = 0xFFFFu;
      if (nv < W) {
        const int slot = kPage * c + (lane & 15);
        int dist = u.pos - slot;  // age of the token in this slot
        if (dist < 0) dist += W;
        valid = __ballot_sync(0xffffffffu, dist < nv) & 0xFFFFu;
      }
      if (valid != 0u) {
        if (valid != 0xFFFFu) {
          zero_invalid_v_rows<D>(smem + (sV - smem_u32(smem)), valid, lane);
          __syncwarp();
        }
        consume_bf16<D, TWO>(st, qf, fo, sK, sV, valid, p.scale_log2, lane);
      }
      if (c == CPU - 1) {
        // finalize the unit: out = o / l for the group's query heads
        void* outp = p.out[u.l];
        const size_t row0 = (static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G) * D;
#pragma unroll
        for (int rh = 0; rh < (TWO ? 2 : 1); ++rh) {
          const float lsum = warp_sum_quad(st.l[rh]);
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          const int row = g + 8 * rh;
          if (row < G) {
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
              const size_t idx = row0 + static_cast<size_t>(row) * D + 8 * nt + 2 * qd;
              const float v0 = st.o[nt][2 * rh] * inv, v1 = st.o[nt][2 * rh + 1] * inv;
              if (p.out_f32) {
                *reinterpret_cast<float2*>(reinterpret_cast<float*>(outp) + idx) =
                    make_float2(v0, v1);
              } else {
                *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(outp) + idx) =
                    __floats2bfloat162_rn(v0, v1);
              }
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + S < total) {
      fence_proxy_async_smem();
      issue_next();
    }
    if (++cst == S) {
      cst = 0;
      phase ^= 1u;
    }
    if (++c == CPU) {
      c = 0;
      ++k;
    }
  }
  if (j < total && lane == 0) {
    // gave up: drain (bounded) the loads still in flight for this warp
    for (int i = 0; i < S && j + i < total; ++i) {
      (void)mbar_wait(bar0 + 8 * cst, phase);
      if (++cst == S) {
        cst = 0;
        phase ^= 1u;
      }
    }
  }
  // ---- a hybrid-stack step's Full-layer merges: one warp per (layer,
  // request, KV head), after this warp's SWA units.  Without merges, one
  // thread still waits for the split grid this launch started beside, so
  // that this grid's completion (which later launches are ordered after)
  // implies that one's.
  if (p.num_merge_layers == 0 && p.wait_prior_at_exit && blockIdx.x == 0 && threadIdx.x == 0)
    pdl_wait_prior_grid();
  if (p.num_merge_layers > 0) {
    // the split launch before this one (this grid may start while it runs)
    pdl_wait_prior_grid();
    const int mu = p.num_merge_layers * BH;
    for (int id = gw; id < mu; id += tw) {
      const int l = id / BH, rem = id - l * BH;
      const int b = rem / Hkv, h = rem - (rem / Hkv) * Hkv;
      const StackMergeLayer& M = p.merge_layer[l];
      merge_request_rows4<D>(p.merge, M.ws_o, M.ws_ml, M.out, b, h);
    }
  }
}

template <int D, bool TWO, int MAXL, int NW, int S>
static int launch_swa_t(const SwaParams<MAXL>& p, int num_sms, cudaStream_t stream,
                        bool dependent) {
  auto kern = phs_swa_decode_kernel<D, TWO, MAXL, NW, S>;
  const int smem = SwaLayout(D, p.G, NW, S).total;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != PHS_OK) return PHS_ECUDA;
  const long long units = std::max(static_cast<long long>(p.num_layers),
                                   static_cast<long long>(p.num_merge_layers)) *
                          p.B * p.Hkv;  // SWA units, or merge units if more
  long long blocks = (units + NW - 1) / NW;
  if (blocks > num_sms) blocks = num_sms;
  if (blocks < 1) blocks = 1;
  if (!dependent) {
    kern<<<static_cast<int>(blocks), NW * 32, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
  }
  // programmatic dependent of the previous launch (a hybrid-stack step's
  // Full split): the SWA units need nothing from it and overlap its last
  // wave; the folded merges wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

// The chunked shape as a launch of its own (the layout, the unit body and
// their rationale are in phs_swa_chunk.cuh).  The Full layers' merges of a
// hybrid-stack step, when they ride on the launch, follow the unit (one warp
// per merge unit, as in the persistent kernel).
template <int D, bool TWO, int MAXL>
__global__ void __launch_bounds__(kSwaChunkWarps * 32, 1)
    phs_swa_chunked_kernel(const __grid_constant__ SwaParams<MAXL> p) {
  constexpr int NW = kSwaChunkWarps;
  const int warp = threadIdx.x >> 5;
  const int Hkv = p.Hkv;
  const int BH = p.B * Hkv;
  swa_chunked_unit<D, TWO, MAXL>(p, blockIdx.x);
  if (p.num_merge_layers > 0) {
    // the split launch before this one (this grid may start while it runs)
    pdl_wait_prior_grid();
    const int mu = p.num_merge_layers * BH;
    for (int id = blockIdx.x * NW + warp; id < mu; id += gridDim.x * NW) {
      const int l = id / BH, r = id - l * BH;
      const int b = r / Hkv, h = r - b * Hkv;
      const StackMergeLayer& M = p.merge_layer[l];
      merge_request_rows4<D>(p.merge, M.ws_o, M.ws_ml, M.out, b, h);
    }
  } else if (p.wait_prior_at_exit && blockIdx.x == 0 && threadIdx.x == 0) {
    // launched beside the split launch before it: this grid's completion
    // (which later launches are ordered after) implies that one's
    pdl_wait_prior_grid();
  }
}

template <int D, bool TWO, int MAXL>
static int launch_swa_chunked(const SwaParams<MAXL>& p, cudaStream_t stream, bool dependent) {
  auto kern = phs_swa_chunked_kernel<D, TWO, MAXL>;
  const int smem = SwaChunkLayout(D, p.G).total;
  if (ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != PHS_OK) return PHS_ECUDA;
  const unsigned blocks = static_cast<unsigned>(p.num_layers * p.B * p.Hkv);
  if (!dependent) {
    kern<<<blocks, kSwaChunkWarps * 32, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kSwaChunkWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

// Launch shapes (warps per CTA x stages per warp):
//   latency  4 x 4: when every unit gets a warp of its own in one wave, a
//            unit's W/16 chunks are the whole chain, and 4 stages take it in
//            half the round trips of 2 (one SWA layer of a batch-2 hybrid
//            step: 13.5 -> 12.3 us per step; 8 stages for D = 64 gave the
//            same);
//   stream   kSwaWarps x kSwaStages: many units per warp, the copies of the
//            next unit overlap the current one;
//   small    4 x kSwaStages: when the stream shape's shared memory does not fit;
//   chunked  one CTA per unit, its chunks spread over 4 warps (above): when
//            every unit has an SM of its own.
enum SwaMode { kSwaNone = 0, kSwaLatency, kSwaStream, kSwaSmall, kSwaChunked };

SwaMode swa_mode(int D, int G, long long units, int num_sms, int smem_optin) {
  if (units <= num_sms && SwaChunkLayout(D, G).total <= smem_optin) return kSwaChunked;
  if (units <= 4LL * num_sms && SwaLayout(D, G, 4, 4).total <= smem_optin) return kSwaLatency;
  if (SwaLayout(D, G, kSwaWarps, kSwaStages).total <= smem_optin) return kSwaStream;
  if (SwaLayout(D, G, 4, kSwaStages).total <= smem_optin) return kSwaSmall;
  return kSwaNone;
}

int swa_smem_bytes(int D, int G) { return SwaLayout(D, G, 4, kSwaStages).total; }

template <int MAXL>
int launch_swa_decode(int D, const SwaParams<MAXL>& p, int num_sms, int smem_optin,
                      cudaStream_t stream, bool dependent) {
  if (static_cast<long long>(p.num_layers) * p.B * p.Hkv > INT32_MAX / 2) return PHS_EUNSUPPORTED;
  const SwaMode mode = swa_mode(D, p.G, static_cast<long long>(p.num_layers) * p.B * p.Hkv,
                                num_sms, smem_optin);
  if (mode == kSwaNone) return PHS_EUNSUPPORTED;
  const bool two = p.G > 8;
#define PHS_SWA_LAUNCH(DD, TT)                                                               \
  switch (mode) {                                                                            \
    case kSwaChunked: return launch_swa_chunked<DD, TT, MAXL>(p, stream, dependent);          \
    case kSwaLatency: return launch_swa_t<DD, TT, MAXL, 4, 4>(p, num_sms, stream, dependent); \
    case kSwaStream:                                                                         \
      return launch_swa_t<DD, TT, MAXL, kSwaWarps, kSwaStages>(p, num_sms, stream, dependent); \
    default: return launch_swa_t<DD, TT, MAXL, 4, kSwaStages>(p, num_sms, stream, dependent);  \
  }
  if (D == 128) {
    if (two) PHS_SWA_LAUNCH(128, true);
    PHS_SWA_LAUNCH(128, false);
  }
  if (D == 64) {
    if (two) PHS_SWA_LAUNCH(64, true);
    PHS_SWA_LAUNCH(64, false);
  }
#undef PHS_SWA_LAUNCH
  return PHS_EUNSUPPORTED;
}

template int launch_swa_decode<1>(int, const SwaParams<1>&, int, int, cudaStream_t, bool);
template int launch_swa_decode<kSwaMaxLayers>(int, const SwaParams<kSwaMaxLayers>&, int, int,
                                              cudaStream_t, bool);

}  // namespace phs
