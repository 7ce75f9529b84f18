// phs_swa.cu -- sliding-window decode over SWA ring buffers, one or many
// layers per launch.
//
// Work unit: (layer, request, KV head) = the W ring slots of one head, read
// as W/16 chunks of 16 slots.  The kernel is persistent: each warp walks a
// strided list of units and streams their chunks back to back through its
// own ring of shared-memory stages, so loads of the next unit overlap the
// tail of the current one.  Each stage holds a 16-slot K tile and V tile
// (TMA, 128-byte swizzle) and, for the first chunk of a unit, the group's
// queries (1-D bulk copy).  The output of a unit is written straight from
// the accumulators: no split, no workspace.
//
// Sources: "Xiaomi MiMo-V2.5 inference system" page, section 1 (SWA layers
// keep and attend to the most recent 128 tokens) and section 2 (ring
// buffer of capacity W per request, storage O(W); SWA reads overlap layer
// by layer).
#include "phs_attn.cuh"
#include "phs_internal.h"

namespace phs {

constexpr int kSwaWarps = 4;
constexpr int kSwaStages = 4;

template <int D, bool TWO>
struct SwaLayout {
  static constexpr int kKV = ChunkGeom<D>::kStageBytes;
  static constexpr int kQSlot = ((TWO ? 16 : 8) * D * 2 + 1023) / 1024 * 1024;
  static constexpr int kStage = kKV + kQSlot;
  static constexpr int kStagesBytes = kSwaWarps * kSwaStages * kStage;
  static constexpr int kBarOff = kStagesBytes;
  static constexpr int kInfoOff = kBarOff + kSwaWarps * kSwaStages * 8;
  static constexpr int kFixed = kInfoOff + 1024;  // + 12 bytes per request
};

__device__ __forceinline__ uint8_t* swa_align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool TWO, int MAXL>
__global__ void __launch_bounds__(kSwaWarps * 32, 1)
    phs_swa_decode_kernel(const __grid_constant__ SwaParams<MAXL> p) {
  using L = SwaLayout<D, TWO>;
  constexpr int S = kSwaStages;
  constexpr int NW = kSwaWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = swa_align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G, W = p.W;

  // ---- per-request ring id, newest slot and length, cached in smem
  int32_t* s_ring = reinterpret_cast<int32_t*>(smem + L::kInfoOff);
  int32_t* s_pos = s_ring + B;
  int32_t* s_n = s_pos + B;
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    s_ring[i] = p.ring_ids ? p.ring_ids[i] : i;
    s_pos[i] = p.ring_pos[i];
    s_n[i] = p.seq_lens[i];
  }
  __syncthreads();

  const int CPU = W / kPage;  // chunks per unit
  const long long units = static_cast<long long>(p.num_layers) * B * Hkv;
  const long long gw = static_cast<long long>(blockIdx.x) * NW + warp;
  const long long tw = static_cast<long long>(gridDim.x) * NW;
  const long long my_units = gw < units ? (units - gw + tw - 1) / tw : 0;
  const long long total = my_units * CPU;

  const uint32_t bar0 = smem_u32(smem + L::kBarOff) + warp * S * 8;
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t sbase = smem_u32(smem) + warp * S * L::kStage;
  const uint64_t pol = policy_evict_first();

  struct Unit {
    int l, b, h, ring, pos, n;
    bool ok;
  };
  auto unit_of = [&](long long k) {
    Unit u;
    const long long id = gw + k * tw;
    u.l = static_cast<int>(id / (static_cast<long long>(B) * Hkv));
    const int rem = static_cast<int>(id % (static_cast<long long>(B) * Hkv));
    u.b = rem / Hkv;
    u.h = rem % Hkv;
    u.ring = s_ring[u.b];
    u.pos = s_pos[u.b];
    u.n = s_n[u.b];
    u.ok = u.ring >= 0 && u.ring < p.num_rings[u.l] && u.pos >= 0 && u.pos < W && u.n >= 0;
    return u;
  };

  auto issue = [&](long long j) {  // lane 0 only
    const uint32_t bar = bar0 + 8 * (j % S);
    const uint32_t dst = sbase + (j % S) * L::kStage;
    const Unit u = unit_of(j / CPU);
    const int c = static_cast<int>(j % CPU);
    if (!u.ok) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      return;
    }
    const uint32_t qbytes = c == 0 ? static_cast<uint32_t>(G * D * 2) : 0u;
    mbar_arrive_expect_tx(bar, L::kKV + qbytes);
    const int row = (u.ring * Hkv + u.h) * W + kPage * c;
#pragma unroll
    for (int sub = 0; sub < D / 64; ++sub) {
      tma_load_2d(dst + sub * 2048, &p.tk[u.l], sub * 64, row, bar, pol);
      tma_load_2d(dst + L::kKV / 2 + sub * 2048, &p.tv[u.l], sub * 64, row, bar, pol);
    }
    if (c == 0) {
      const __nv_bfloat16* q =
          p.q[u.l] + (static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G) * D;
      bulk_load(dst + L::kKV, q, qbytes, bar);
    }
  };

  if (lane == 0)
    for (long long j = 0; j < S && j < total; ++j) issue(j);

  WarpState<D, TWO> st;
  QFrags<D, TWO> qf;
  const int g = lane >> 2, qd = lane & 3;
  long long j = 0;
  for (; j < total; ++j) {
    const uint32_t bar = bar0 + 8 * (j % S);
    const bool done = mbar_wait(bar, static_cast<uint32_t>((j / S) & 1));
    if (!__all_sync(0xffffffffu, done)) {
      if (lane == 0) set_status(p.status, PHS_ETIMEOUT);
      break;
    }
    const Unit u = unit_of(j / CPU);
    const int c = static_cast<int>(j % CPU);
    const uint32_t sK = sbase + (j % S) * L::kStage;
    const uint32_t sV = sK + L::kKV / 2;
    if (c == 0) {
      st.reset();
      if (u.ok) load_q_bf16_smem<D, TWO>(qf, sK + L::kKV, G, lane);
    }
    if (u.ok) {
      const int nv = min(u.n, W);  // valid slots: the last nv tokens
      uint32_t valid = 0xFFFFu;
      if (nv < W) {
        const int slot = kPage * c + (lane & 15);
        const int dist = ((u.pos - slot) % W + W) % W;  // age of the token in this slot
        valid = __ballot_sync(0xffffffffu, dist < nv) & 0xFFFFu;
      }
      if (valid != 0u) {
        if (valid != 0xFFFFu) {
          zero_invalid_v_rows<D>(smem + (sV - smem_u32(smem)), valid, lane);
          __syncwarp();
        }
        consume_bf16<D, TWO>(st, qf, sK, sV, valid, p.scale_log2, lane);
      }
    } else if (c == 0 && lane == 0) {
      set_status(p.status, PHS_ERANGE);
    }
    if (c == CPU - 1 && u.ok) {
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
              *reinterpret_cast<float2*>(reinterpret_cast<float*>(outp) + idx) = make_float2(v0, v1);
            } else {
              *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(outp) + idx) =
                  __floats2bfloat162_rn(v0, v1);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + S < total) {
      fence_proxy_async_smem();
      issue(j + S);
    }
  }
  if (j < total && lane == 0) {
    for (long long k = j; k < total && k < j + S; ++k)
      (void)mbar_wait(bar0 + 8 * (k % S), static_cast<uint32_t>((k / S) & 1));
  }
}

template <int D, bool TWO, int MAXL>
static int launch_swa_t(const SwaParams<MAXL>& p, int num_sms, cudaStream_t stream) {
  using L = SwaLayout<D, TWO>;
  auto kern = phs_swa_decode_kernel<D, TWO, MAXL>;
  const int smem = L::kFixed + 12 * p.B + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return PHS_ECUDA;
  const long long units = static_cast<long long>(p.num_layers) * p.B * p.Hkv;
  long long blocks = (units + kSwaWarps - 1) / kSwaWarps;
  if (blocks > num_sms) blocks = num_sms;
  if (blocks < 1) blocks = 1;
  kern<<<static_cast<int>(blocks), kSwaWarps * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PHS_OK : PHS_ECUDA;
}

template <int MAXL>
int launch_swa_decode(int D, const SwaParams<MAXL>& p, int num_sms, cudaStream_t stream) {
  const bool two = p.G > 8;
  if (D == 128)
    return two ? launch_swa_t<128, true, MAXL>(p, num_sms, stream)
               : launch_swa_t<128, false, MAXL>(p, num_sms, stream);
  if (D == 64)
    return two ? launch_swa_t<64, true, MAXL>(p, num_sms, stream)
               : launch_swa_t<64, false, MAXL>(p, num_sms, stream);
  return PHS_EUNSUPPORTED;
}

template int launch_swa_decode<1>(int, const SwaParams<1>&, int, cudaStream_t);
template int launch_swa_decode<kSwaMaxLayers>(int, const SwaParams<kSwaMaxLayers>&, int,
                                              cudaStream_t);

// Shared-memory bytes the ring kernel needs for `batch` requests.
int swa_smem_bytes(int D, int G, int batch) {
  const bool two = G > 8;
  int fixed;
  if (D == 128)
    fixed = two ? SwaLayout<128, true>::kFixed : SwaLayout<128, false>::kFixed;
  else
    fixed = two ? SwaLayout<64, true>::kFixed : SwaLayout<64, false>::kFixed;
  return fixed + 12 * batch + 1024;
}

}  // namespace phs
