// phs_api.cu -- the extern "C" entry points declared in include/phs.h:
// argument validation, TMA tensor-map encoding, split planning, and the
// hybrid layer-stack driver.  All compute happens in the kernels of
// phs_decode.cu, phs_swa.cu, phs_append.cu and phs_quant.cu.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <map>
#include <mutex>
#include <utility>

#include "phs_internal.h"

namespace phs {

int swa_smem_bytes(int D, int G);

int ensure_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHS_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({kernel, dev});
  if (it != done.end() && it->second >= bytes) return PHS_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return PHS_ECUDA;
  done[{kernel, dev}] = bytes;
  return PHS_OK;
}

namespace {

constexpr int kMaxSplitTokens = 4096;
constexpr int kMaxWindow = 4096;
// The append kernel gives one thread to each 16-byte piece of a token's K
// (and V) row over all KV heads, in one CTA.
constexpr int kMaxAppendThreads = 1024;

// ---------------------------------------------------------- device info --
struct DevInfo {
  int device = -1;
  int sms = 0;
  int smem_optin = 0;
};

int dev_info(DevInfo& out) {
  thread_local DevInfo cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHS_ECUDA;
  if (cache.device != dev) {
    DevInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PHS_ECUDA;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return PHS_ECUDA;
    cache = d;
  }
  out = cache;
  return PHS_OK;
}

// ---------------------------------------------------------- tensor maps --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 pool viewed as a 2-D tensor of `rows` rows of D elements; boxes of
// 16 rows x 64 columns (128 bytes) with the 128-byte swizzle.
int map_bf16_rows(CUtensorMap* m, const void* base, int64_t rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PHS_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHS_OK : PHS_ECUDA;
}

// bf16 pool (D = 128) viewed as a 3-D tensor {64 columns, rows, 2 column
// halves} (strides 256 B, 128 B): one box of {64, 16, 2} fetches a whole
// 16-row page block as [half][16 rows][128 B] with the 128-byte swizzle --
// one 4 KB copy instead of two 2 KB ones (the copy engine's cost is per box).
int map_bf16_pages3d(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PHS_ECUDA;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), 2};
  cuuint64_t strides[2] = {256, 128};
  cuuint32_t box[3] = {64, 16, 2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHS_OK : PHS_ECUDA;
}

// Map for the per-page K/V copies of the decode kernels: one 3-D box per
// 16-row block when D = 128, two 2-D boxes of 64 columns otherwise (D = 64:
// one box).  Both land as [column half][16 rows][128 B] in shared memory.
int map_bf16_kv(CUtensorMap* m, const void* base, int64_t rows, int D) {
  return D == 128 ? map_bf16_pages3d(m, base, rows) : map_bf16_rows(m, base, rows, D);
}

// int8 codes, rows of D bytes; boxes of 32 rows x D with the 128-byte
// (D = 128) or 64-byte (D = 64) swizzle.
int map_i8_rows(CUtensorMap* m, const void* base, int64_t rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PHS_ECUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(D), 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHS_OK : PHS_ECUDA;
}

// int8 V^T codes (D x 32 bytes per block and head) viewed as rows of 128
// bytes (4 head dims each); boxes of D/4 rows (a whole block) with the
// 128-byte swizzle: the same copy shape as a K block.
int map_i8_vt(CUtensorMap* m, const void* base, int64_t rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PHS_ECUDA;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(D / 4)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHS_OK : PHS_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(int Hq, int Hkv, int D) {
  if (Hq <= 0 || Hkv <= 0) return PHS_EINVAL;
  if (Hq % Hkv != 0) return PHS_ESHAPE;
  if (Hq / Hkv > 16) return PHS_EUNSUPPORTED;
  if (D != 64 && D != 128) return PHS_EUNSUPPORTED;
  return PHS_OK;
}

int check_paged(const phs_paged_pool* pool) {
  if (!pool || !pool->k || !pool->v) return PHS_EINVAL;
  if (pool->num_pages <= 0 || pool->num_kv_heads <= 0) return PHS_EINVAL;
  if (pool->page_size != kPage) return PHS_EUNSUPPORTED;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PHS_EUNSUPPORTED;
  if (pool->num_pages * pool->num_kv_heads * kPage > INT32_MAX) return PHS_EUNSUPPORTED;
  if (int64_t{pool->num_kv_heads} * pool->head_dim / 8 > kMaxAppendThreads) return PHS_EUNSUPPORTED;
  if (!aligned16(pool->k) || !aligned16(pool->v)) return PHS_EALIGN;
  return PHS_OK;
}

int check_ring(const phs_ring_pool* ring) {
  if (!ring || !ring->k || !ring->v) return PHS_EINVAL;
  if (ring->num_rings <= 0 || ring->num_kv_heads <= 0 || ring->window <= 0) return PHS_EINVAL;
  if (ring->window % kPage != 0 || ring->window > kMaxWindow) return PHS_EUNSUPPORTED;
  if (ring->head_dim != 64 && ring->head_dim != 128) return PHS_EUNSUPPORTED;
  if (ring->num_rings * ring->num_kv_heads * ring->window > INT32_MAX) return PHS_EUNSUPPORTED;
  if (int64_t{ring->num_kv_heads} * ring->head_dim / 8 > kMaxAppendThreads) return PHS_EUNSUPPORTED;
  if (!aligned16(ring->k) || !aligned16(ring->v)) return PHS_EALIGN;
  return PHS_OK;
}

int check_int8(const phs_int8_pool* p) {
  if (!p || !p->k || !p->v || !p->k_scale || !p->v_scale) return PHS_EINVAL;
  if (p->num_qpages <= 0 || p->num_kv_heads <= 0) return PHS_EINVAL;
  if (p->head_dim != 64 && p->head_dim != 128) return PHS_EUNSUPPORTED;
  // TMA row coordinates are int32: 32 K rows and D/4 V^T rows per block and head
  if (p->num_qpages * p->num_kv_heads * kQBlock > INT32_MAX) return PHS_EUNSUPPORTED;
  if (!aligned16(p->k) || !aligned16(p->v)) return PHS_EALIGN;
  return PHS_OK;
}

// Default split length: the longest of 4096, 2048, ... 128 tokens that
// gives the longest request at least 8 splits and whose grid (B x Hkv x
// splits of the longest request) still has 16 CTAs per SM.  Long splits
// amortise each CTA's set-up (queries, page ids, the first copies) and keep
// the partial results small; 8 splits of the longest request keep the last
// wave fine-grained.  Measured (GB/s, whole step, each set on one box; 1024
// / 2048 / 4096 tokens): paged batch 64, lengths to 32K, 7,114 / 7,170 /
// 7,134; INT8 batch 32 at 65K 6,033 / 6,557 / 6,753; 70-layer stack batch
// 256, lengths to 128K, 7,042 / 7,206 / 7,306.
// Short requests in a grid that one wave holds anyway (B x Hkv <= SMs, the
// longest request 129..256 tokens) take one split of 256: no merge then
// follows the decode.  Measured on the 2-layer hybrid step at batch 2
// (lengths 37 and 201, replayed as a CUDA graph): 12.3 -> 10.3 us per step.
#ifndef PHS_SPLIT_T_MAX
#define PHS_SPLIT_T_MAX 4096
#endif
#ifndef PHS_SPLIT_CTAS_PER_SM
#define PHS_SPLIT_CTAS_PER_SM 16
#endif

int32_t plan_tokens_per_split(int B, int Hkv, int max_seq, int requested, int sms) {
  if (requested > 0) return requested;
  if (max_seq > 128 && max_seq <= 256 && static_cast<long long>(B) * Hkv <= sms) return 256;
  int t = PHS_SPLIT_T_MAX;
  while (t > 128 && 8LL * t > max_seq) t /= 2;
  const long long target = static_cast<long long>(PHS_SPLIT_CTAS_PER_SM) * std::max(sms, 1);
  while (t > 128) {
    const long long ctas = static_cast<long long>(B) * Hkv * ((max_seq + t - 1) / t);
    if (ctas >= target) break;
    t /= 2;
  }
  return t;
}

int max_splits_for(int max_seq, int T, bool has_int8) {
  return std::max(1, (max_seq + T - 1) / T + (has_int8 ? 1 : 0));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t ws_o_bytes(int B, int Hkv, int ms, int G, int D) {
  return align256(static_cast<size_t>(B) * Hkv * ms * G * D * sizeof(float));
}

size_t ws_bytes(int B, int Hkv, int ms, int G, int D) {
  return ws_o_bytes(B, Hkv, ms, G, D) +
         align256(static_cast<size_t>(B) * Hkv * ms * G * 2 * sizeof(float));
}

struct DecodePlan {
  int T = 0, max_splits = 0, G = 0, D = 0, Hkv = 0;
  bool has_int8 = false;
  size_t need = 0;
};

int make_plan(DecodePlan& pl, int B, int Hq, int Hkv, int D, int max_seq, int tps,
              bool has_int8) {
  int st = check_dims(Hq, Hkv, D);
  if (st) return st;
  if (B <= 0 || max_seq < 0) return PHS_EINVAL;
  if (tps < 0 || (tps > 0 && (tps % kQBlock != 0 || tps > kMaxSplitTokens)))
    return PHS_EUNSUPPORTED;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  pl.T = plan_tokens_per_split(B, Hkv, max_seq, tps, di.sms);
  pl.max_splits = max_splits_for(max_seq, pl.T, has_int8);
  pl.G = Hq / Hkv;
  pl.D = D;
  pl.Hkv = Hkv;
  pl.has_int8 = has_int8;
  if (pl.max_splits > 65535) return PHS_EUNSUPPORTED;  // grid z limit
  pl.need = ws_bytes(B, Hkv, pl.max_splits, pl.G, D);
  return PHS_OK;
}

// Shared preamble of the decode entry points.
struct DecodeCall {
  DecodePlan pl;
  SplitArgs a;
  MergeArgs m;
  CUtensorMap tk, tv, tk8, tv8;
};

int prepare_decode(DecodeCall& c, const void* q, int Hq, const phs_paged_pool* pool,
                   const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                   int max_seq, const phs_int8_pool* int8, const int32_t* qtable, int max_qpages,
                   const int32_t* qlens, int B, float softmax_scale, int tps, void* out,
                   int out_dtype, void* workspace, size_t ws_size, const void* k_new,
                   const void* v_new, const int32_t* page_refcount, int32_t* dev_status) {
  int st = check_paged(pool);
  if (st) return st;
  if (!q || !block_table || !seq_lens || !out) return PHS_EINVAL;
  if ((k_new == nullptr) != (v_new == nullptr)) return PHS_EINVAL;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PHS_EALIGN;
  if (max_pages <= 0 || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  const int D = pool->head_dim, Hkv = pool->num_kv_heads;
  if (int8) {
    if ((st = check_int8(int8))) return st;
    if (!qtable || !qlens || max_qpages <= 0) return PHS_EINVAL;
    if (int8->head_dim != D || int8->num_kv_heads != Hkv) return PHS_ESHAPE;
  }
  if ((st = make_plan(c.pl, B, Hq, Hkv, D, max_seq, tps, int8 != nullptr))) return st;
  if (!workspace || ws_size < c.pl.need) return PHS_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PHS_EALIGN;
  if (!aligned16(q)) return PHS_EALIGN;

  std::memset(&c.a, 0, sizeof(c.a));
  c.a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  c.a.block_table = block_table;
  c.a.seq_lens = seq_lens;
  c.a.qtable = int8 ? qtable : nullptr;
  c.a.qlens = int8 ? qlens : nullptr;
  c.a.k_scale = int8 ? int8->k_scale : nullptr;
  c.a.v_scale = int8 ? int8->v_scale : nullptr;
  c.a.out = out;
  c.a.ws_o = reinterpret_cast<float*>(workspace);
  c.a.ws_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) +
                                       ws_o_bytes(B, Hkv, c.pl.max_splits, c.pl.G, D));
  c.a.status = dev_status;
  c.a.num_pages = pool->num_pages;
  c.a.num_qpages = int8 ? int8->num_qpages : 0;
  c.a.Hq = Hq;
  c.a.Hkv = Hkv;
  c.a.G = c.pl.G;
  c.a.max_pages = max_pages;
  c.a.max_qpages = int8 ? max_qpages : 0;
  c.a.n_clamp = static_cast<int>(std::min<long long>(max_seq, 1LL * max_pages * kPage));
  c.a.T = c.pl.T;
  c.a.max_splits = c.pl.max_splits;
  c.a.out_f32 = out_dtype == PHS_OUT_F32;
  c.a.scale_log2 = softmax_scale * 1.4426950408889634f;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  c.a.num_sms = di.sms;
  if (k_new) {  // the step's append, fused into the split launch
    c.a.app = FusedAppend{reinterpret_cast<const __nv_bfloat16*>(k_new),
                          reinterpret_cast<const __nv_bfloat16*>(v_new),
                          reinterpret_cast<__nv_bfloat16*>(pool->k),
                          reinterpret_cast<__nv_bfloat16*>(pool->v)};
    c.a.page_refcount = page_refcount;
  }

  std::memset(&c.m, 0, sizeof(c.m));
  c.m.seq_lens = seq_lens;
  c.m.qlens = c.a.qlens;
  c.m.ws_o = c.a.ws_o;
  c.m.ws_ml = c.a.ws_ml;
  c.m.out = out;
  c.m.Hq = Hq;
  c.m.Hkv = Hkv;
  c.m.G = c.pl.G;
  c.m.n_clamp = c.a.n_clamp;
  c.m.T = c.pl.T;
  c.m.max_splits = c.pl.max_splits;
  c.m.out_f32 = c.a.out_f32;

  const int64_t rows = pool->num_pages * Hkv * kPage;
  if ((st = map_bf16_kv(&c.tk, pool->k, rows, D))) return st;
  if ((st = map_bf16_kv(&c.tv, pool->v, rows, D))) return st;
  if (int8) {
    const int64_t blocks = int8->num_qpages * Hkv;
    if ((st = map_i8_rows(&c.tk8, int8->k, blocks * kQBlock, D))) return st;
    if ((st = map_i8_vt(&c.tv8, int8->v, blocks * (D / 4), D))) return st;
  } else {
    c.tk8 = c.tk;  // unused by bf16-only launches
    c.tv8 = c.tv;
  }
  return PHS_OK;
}

}  // namespace
}  // namespace phs

using namespace phs;

extern "C" {

int32_t phs_version(void) { return 1; }

const char* phs_status_str(int s) {
  switch (s) {
    case PHS_OK: return "ok";
    case PHS_EINVAL: return "invalid argument";
    case PHS_ESHAPE: return "inconsistent shapes";
    case PHS_ERANGE: return "index out of range";
    case PHS_ESHARED: return "append into a shared page";
    case PHS_EWORKSPACE: return "workspace missing or too small";
    case PHS_ECUDA: return "CUDA call failed";
    case PHS_EUNSUPPORTED: return "unsupported shape";
    case PHS_ETIMEOUT: return "device wait timed out";
    case PHS_EALIGN: return "pointer not aligned";
    case PHS_ESCRATCH: return "request exceeds the no-allocation entry point's built-in scratch";
    case PHS_ENOSPACE: return "not enough free pages";
    default: return "unknown status";
  }
}

int phs_kv_append_paged(const phs_paged_pool* pool, const void* k_new, const void* v_new,
                        const int32_t* block_table, int32_t max_pages_per_seq,
                        const int32_t* seq_lens, int32_t batch, const int32_t* page_refcount,
                        int32_t* dev_status, void* stream) {
  int st = check_paged(pool);
  if (st) return st;
  if (!k_new || !v_new || !block_table || !seq_lens || batch < 0 || max_pages_per_seq <= 0)
    return PHS_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PHS_EALIGN;
  if (batch == 0) return PHS_OK;
  AppendParams<1> p;
  std::memset(&p, 0, sizeof(p));
  p.layer[0] = AppendLayer{pool->k, pool->v, k_new, v_new, pool->num_pages};
  p.table = block_table;
  p.seq_lens = seq_lens;
  p.refcount = page_refcount;
  p.status = dev_status;
  p.num_layers = 1;
  p.B = batch;
  p.Hkv = pool->num_kv_heads;
  p.D = pool->head_dim;
  p.max_pages = max_pages_per_seq;
  p.is_ring = 0;
  return launch_append<1>(p, reinterpret_cast<cudaStream_t>(stream));
}

int phs_kv_append_ring(const phs_ring_pool* ring, const void* k_new, const void* v_new,
                       const int32_t* ring_ids, const int32_t* ring_pos, int32_t batch,
                       int32_t* dev_status, void* stream) {
  int st = check_ring(ring);
  if (st) return st;
  if (!k_new || !v_new || !ring_pos || batch < 0) return PHS_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PHS_EALIGN;
  if (batch == 0) return PHS_OK;
  AppendParams<1> p;
  std::memset(&p, 0, sizeof(p));
  p.layer[0] = AppendLayer{ring->k, ring->v, k_new, v_new, ring->num_rings};
  p.table = ring_ids;
  p.ring_pos = ring_pos;
  p.status = dev_status;
  p.num_layers = 1;
  p.B = batch;
  p.Hkv = ring->num_kv_heads;
  p.D = ring->head_dim;
  p.W = ring->window;
  p.is_ring = 1;
  return launch_append<1>(p, reinterpret_cast<cudaStream_t>(stream));
}

int phs_kv_quant_int8_block32(const phs_paged_pool* src, const int32_t* src_block_table,
                              int32_t src_max_pages, const phs_int8_pool* dst,
                              const int32_t* dst_qtable, int32_t dst_max_qpages,
                              const int32_t* first_qblock, const int32_t* num_qblocks,
                              int32_t max_qblocks, int32_t batch, int32_t* dev_status,
                              void* stream) {
  int st = check_paged(src);
  if (st) return st;
  if ((st = check_int8(dst))) return st;
  if (!src_block_table || !dst_qtable || !first_qblock || !num_qblocks) return PHS_EINVAL;
  if (src_max_pages <= 0 || dst_max_qpages <= 0 || batch < 0 || max_qblocks < 0)
    return PHS_EINVAL;
  if (dst->head_dim != src->head_dim || dst->num_kv_heads != src->num_kv_heads) return PHS_ESHAPE;
  if (batch == 0 || max_qblocks == 0) return PHS_OK;
  QuantArgs a;
  std::memset(&a, 0, sizeof(a));
  a.k_src = reinterpret_cast<const __nv_bfloat16*>(src->k);
  a.v_src = reinterpret_cast<const __nv_bfloat16*>(src->v);
  a.src_table = src_block_table;
  a.k_codes = dst->k;
  a.v_codes = dst->v;
  a.k_scale = dst->k_scale;
  a.v_scale = dst->v_scale;
  a.dst_qtable = dst_qtable;
  a.first_qblock = first_qblock;
  a.num_qblocks = num_qblocks;
  a.status = dev_status;
  a.num_pages = src->num_pages;
  a.num_qpages = dst->num_qpages;
  a.src_max_pages = src_max_pages;
  a.dst_max_qpages = dst_max_qpages;
  a.Hkv = src->num_kv_heads;
  a.D = src->head_dim;
  return launch_quant(a, max_qblocks, batch, reinterpret_cast<cudaStream_t>(stream));
}

int32_t phs_decode_tokens_per_split(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len,
                                    int32_t tokens_per_split) {
  DevInfo di;
  if (dev_info(di)) return PHS_ECUDA;
  if (tokens_per_split < 0 || (tokens_per_split > 0 && (tokens_per_split % kQBlock != 0 ||
                                                        tokens_per_split > kMaxSplitTokens)))
    return PHS_EUNSUPPORTED;
  return plan_tokens_per_split(batch, num_kv_heads, max_seq_len, tokens_per_split, di.sms);
}

size_t phs_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len,
                                  int32_t tokens_per_split, int32_t has_int8) {
  DecodePlan pl;
  if (make_plan(pl, batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, tokens_per_split,
                has_int8 != 0))
    return 0;
  return pl.need;
}

int phs_attn_decode_full_paged_split(const void* q, int32_t num_q_heads,
                                     const phs_paged_pool* pool, const int32_t* block_table,
                                     int32_t max_pages_per_seq, const int32_t* seq_lens,
                                     int32_t max_seq_len, const phs_int8_pool* int8,
                                     const int32_t* qtable, int32_t max_qpages_per_seq,
                                     const int32_t* qlens, int32_t batch, float softmax_scale,
                                     int32_t tokens_per_split, void* out, int32_t out_dtype,
                                     void* workspace, size_t workspace_bytes, const void* k_new,
                                     const void* v_new, const int32_t* page_refcount,
                                     int32_t* dev_status, void* stream) {
  DecodeCall c;
  int st = prepare_decode(c, q, num_q_heads, pool, block_table, max_pages_per_seq, seq_lens,
                          max_seq_len, int8, qtable, max_qpages_per_seq, qlens, batch,
                          softmax_scale, tokens_per_split, out, out_dtype, workspace,
                          workspace_bytes, k_new, v_new, page_refcount, dev_status);
  if (st) return st;
  return launch_split_decode(c.pl.D, c.tk, c.tv, c.tk8, c.tv8, c.a, batch,
                             reinterpret_cast<cudaStream_t>(stream));
}

int phs_attn_merge_splits(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, const int32_t* seq_lens, int32_t max_seq_len,
                          const int32_t* qlens, int32_t has_int8, int32_t tokens_per_split,
                          void* out, int32_t out_dtype, const void* workspace,
                          size_t workspace_bytes, void* stream) {
  DecodePlan pl;
  int st = make_plan(pl, batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                     tokens_per_split, has_int8 != 0);
  if (st) return st;
  if (!seq_lens || !out) return PHS_EINVAL;
  if (has_int8 && !qlens) return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  if (!workspace || workspace_bytes < pl.need) return PHS_EWORKSPACE;
  MergeArgs m;
  std::memset(&m, 0, sizeof(m));
  m.seq_lens = seq_lens;
  m.qlens = has_int8 ? qlens : nullptr;
  m.ws_o = reinterpret_cast<const float*>(workspace);
  m.ws_ml = reinterpret_cast<const float*>(reinterpret_cast<const char*>(workspace) +
                                           ws_o_bytes(batch, num_kv_heads, pl.max_splits, pl.G,
                                                      head_dim));
  m.out = out;
  m.Hq = num_q_heads;
  m.Hkv = num_kv_heads;
  m.G = pl.G;
  m.n_clamp = max_seq_len;
  m.T = pl.T;
  m.max_splits = pl.max_splits;
  m.out_f32 = out_dtype == PHS_OUT_F32;
  return launch_merge(head_dim, m, batch, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The decode call; allow_wide = false keeps 4 warps per CTA whatever the
// grid (the unfused stack decides for the whole step, as the fused one does).
int decode_full_paged(const void* q, int32_t num_q_heads, const phs_paged_pool* pool,
                      const int32_t* block_table, int32_t max_pages_per_seq,
                      const int32_t* seq_lens, int32_t max_seq_len, const phs_int8_pool* int8,
                      const int32_t* qtable, int32_t max_qpages_per_seq, const int32_t* qlens,
                      int32_t batch, float softmax_scale, int32_t tokens_per_split, void* out,
                      int32_t out_dtype, void* workspace, size_t workspace_bytes,
                      const void* k_new, const void* v_new, const int32_t* page_refcount,
                      int32_t* dev_status, void* stream, bool allow_wide) {
  DecodeCall c;
  int st = prepare_decode(c, q, num_q_heads, pool, block_table, max_pages_per_seq, seq_lens,
                          max_seq_len, int8, qtable, max_qpages_per_seq, qlens, batch,
                          softmax_scale, tokens_per_split, out, out_dtype, workspace,
                          workspace_bytes, k_new, v_new, page_refcount, dev_status);
  if (st) return st;
  if (!allow_wide) c.a.num_sms = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_split_decode(c.pl.D, c.tk, c.tv, c.tk8, c.tv8, c.a, batch, s))) return st;
  if (c.pl.max_splits == 1) return PHS_OK;  // every request finished in its only split
  return launch_merge(c.pl.D, c.m, batch, s);
}

}  // namespace

int phs_attn_decode_full_paged(const void* q, int32_t num_q_heads, const phs_paged_pool* pool,
                               const int32_t* block_table, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, int32_t max_seq_len,
                               const phs_int8_pool* int8, const int32_t* qtable,
                               int32_t max_qpages_per_seq, const int32_t* qlens, int32_t batch,
                               float softmax_scale, int32_t tokens_per_split, void* out,
                               int32_t out_dtype, void* workspace, size_t workspace_bytes,
                               const void* k_new, const void* v_new,
                               const int32_t* page_refcount, int32_t* dev_status, void* stream) {
  return decode_full_paged(q, num_q_heads, pool, block_table, max_pages_per_seq, seq_lens,
                           max_seq_len, int8, qtable, max_qpages_per_seq, qlens, batch,
                           softmax_scale, tokens_per_split, out, out_dtype, workspace,
                           workspace_bytes, k_new, v_new, page_refcount, dev_status, stream, true);
}

int phs_attn_decode_swa_ring(const void* q, int32_t num_q_heads, const phs_ring_pool* ring,
                             const int32_t* ring_ids, const int32_t* ring_pos,
                             const int32_t* seq_lens, int32_t batch, float softmax_scale,
                             void* out, int32_t out_dtype, int32_t* dev_status, void* stream) {
  int st = check_ring(ring);
  if (st) return st;
  if (!q || !ring_pos || !seq_lens || !out || batch < 0) return PHS_EINVAL;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  const int D = ring->head_dim, Hkv = ring->num_kv_heads;
  if ((st = check_dims(num_q_heads, Hkv, D))) return st;
  if (!aligned16(q)) return PHS_EALIGN;
  if (batch == 0) return PHS_OK;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  if (swa_smem_bytes(D, num_q_heads / Hkv) > di.smem_optin) return PHS_EUNSUPPORTED;
  SwaParams<1> p;
  std::memset(&p, 0, sizeof(p));
  if ((st = map_bf16_kv(&p.tk[0], ring->k, ring->num_rings * Hkv * ring->window, D))) return st;
  if ((st = map_bf16_kv(&p.tv[0], ring->v, ring->num_rings * Hkv * ring->window, D))) return st;
  p.q[0] = reinterpret_cast<const __nv_bfloat16*>(q);
  p.out[0] = out;
  p.num_rings[0] = ring->num_rings;
  p.ring_ids = ring_ids;
  p.ring_pos = ring_pos;
  p.seq_lens = seq_lens;
  p.status = dev_status;
  p.num_layers = 1;
  p.B = batch;
  p.Hq = num_q_heads;
  p.Hkv = Hkv;
  p.G = num_q_heads / Hkv;
  p.W = ring->window;
  p.out_f32 = out_dtype == PHS_OUT_F32;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_swa_decode<1>(D, p, di.sms, di.smem_optin, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------- shared-prefix decode --
namespace {

struct PrefixPlan {
  int G = 0, rows = 0, T = 0, ms = 0, ntiles = 0, tps = 0, nsp = 0;
  size_t off_ml = 0, off_po = 0, off_pml = 0, off_bad = 0, need = 0;
};

int make_prefix_plan(PrefixPlan& pl, int B, int Hq, int Hkv, int D, int max_seq, int shared_len) {
  int st = check_dims(Hq, Hkv, D);
  if (st) return st;
  if (D != 128) return PHS_EUNSUPPORTED;
  if (B <= 0 || shared_len <= 0 || max_seq < shared_len) return PHS_EINVAL;
  if (shared_len % 64 != 0) return PHS_EUNSUPPORTED;
  pl.G = Hq / Hkv;
  pl.rows = B * pl.G;
  if (pl.rows > 256) return PHS_EUNSUPPORTED;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  if (prefix_smem_bytes() > di.smem_optin) return PHS_EUNSUPPORTED;
  const int suffix = std::max(1, max_seq - shared_len);
  // own-token splits of at least 256 tokens: they run beside the prefix pass
  // on the spare SMs, where fewer and longer CTAs spend less on set-up per
  // byte (250,000-token prefix, 64 requests with 512-640 own tokens: 128 ->
  // 256 tokens per split took the call from 0.2300 to 0.2270-0.2275 ms)
  pl.T = std::max(256, plan_tokens_per_split(B, Hkv, suffix, 0, di.sms));
  pl.ms = std::max(1, (suffix + pl.T - 1) / pl.T);
  pl.ntiles = shared_len / 64;
  // One CTA per SM: each KV head's prefix is spread over (SMs - spare) / Hkv
  // CTAs.  The spare SMs run the own-token split while the prefix pass runs
  // (its CTAs cannot share an SM with a prefix CTA; without spare SMs they
  // all run in the pass's tail).  spare balances the two: own tokens at the
  // split kernel's rate against prefix tokens at the prefix pass's (about
  // 48 and 32 GB/s per SM), over the longest own suffix.  Measured on the
  // 250,000-token prefix, 64 requests (decode call): 0 spare SMs 0.2405 ms,
  // 8 0.2381, 16 0.2349, 24 0.2375; this rule gives 16 there.
  const double own = static_cast<double>(B) * std::max(0, max_seq - shared_len);
  const double share = own / (own + 1.5 * static_cast<double>(shared_len));
  const int spare = std::min(di.sms / 2, static_cast<int>(share * di.sms + 0.5));
  const int target = std::max(1, (di.sms - spare) / Hkv);
  pl.tps = (pl.ntiles + target - 1) / target;
  pl.nsp = (pl.ntiles + pl.tps - 1) / pl.tps;
  if (pl.nsp > 65535) return PHS_EUNSUPPORTED;
  pl.off_ml = ws_o_bytes(B, Hkv, pl.ms, pl.G, D);
  pl.off_po = pl.off_ml + align256(static_cast<size_t>(B) * Hkv * pl.ms * pl.G * 2 * sizeof(float));
  pl.off_pml = pl.off_po + align256(static_cast<size_t>(Hkv) * pl.nsp * 256 * D * sizeof(float));
  pl.off_bad = pl.off_pml + align256(static_cast<size_t>(Hkv) * pl.nsp * 256 * 2 * sizeof(float));
  pl.need = pl.off_bad + align256(static_cast<size_t>(B) * Hkv * pl.ms * sizeof(int32_t));
  return PHS_OK;
}

}  // namespace

size_t phs_shared_prefix_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t max_seq_len,
                                         int32_t shared_len) {
  PrefixPlan pl;
  if (make_prefix_plan(pl, batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, shared_len))
    return 0;
  return pl.need;
}

int phs_attn_decode_shared_prefix(const void* q, int32_t num_q_heads, const phs_paged_pool* pool,
                                  const int32_t* block_table, int32_t max_pages_per_seq,
                                  const int32_t* seq_lens, int32_t max_seq_len, int32_t batch,
                                  int32_t shared_len, float softmax_scale, void* out,
                                  int32_t out_dtype, void* workspace, size_t workspace_bytes,
                                  const void* k_new, const void* v_new,
                                  const int32_t* page_refcount, int32_t* dev_status,
                                  void* stream) {
  int st = check_paged(pool);
  if (st) return st;
  if (!q || !block_table || !seq_lens || !out) return PHS_EINVAL;
  if ((k_new == nullptr) != (v_new == nullptr)) return PHS_EINVAL;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PHS_EALIGN;
  if (max_pages_per_seq <= 0 || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  const int D = pool->head_dim, Hkv = pool->num_kv_heads;
  PrefixPlan pl;
  if ((st = make_prefix_plan(pl, batch, num_q_heads, Hkv, D, max_seq_len, shared_len))) return st;
  if (shared_len / kPage > max_pages_per_seq) return PHS_ESHAPE;
  if (!workspace || workspace_bytes < pl.need) return PHS_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || !aligned16(q)) return PHS_EALIGN;
  char* ws = reinterpret_cast<char*>(workspace);
  CUtensorMap tk;  // 64-column boxes: the prefix kernel's K tile is [half][64 rows]
  const int64_t rows = pool->num_pages * Hkv * kPage;
  if ((st = map_bf16_rows(&tk, pool->k, rows, D))) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  // 1. the shared prefix, all requests at once (tensor cores)
  PrefixArgs pa;
  std::memset(&pa, 0, sizeof(pa));
  pa.q = reinterpret_cast<const __nv_bfloat16*>(q);
  pa.block_table = block_table;  // row 0 holds the shared prefix pages
  pa.status = dev_status;
  pa.ws_o = reinterpret_cast<float*>(ws + pl.off_po);
  pa.ws_ml = reinterpret_cast<float*>(ws + pl.off_pml);
  pa.num_pages = pool->num_pages;
  pa.Hq = num_q_heads;
  pa.Hkv = Hkv;
  pa.G = pl.G;
  pa.rows = pl.rows;
  pa.shared_len = shared_len;
  pa.tiles_per_split = pl.tps;
  pa.num_splits = pl.nsp;
  pa.scale_log2 = scale_log2;
  CUtensorMap tk3, tv3;  // per-page boxes (split kernel K/V, prefix kernel V)
  if ((st = map_bf16_pages3d(&tk3, pool->k, rows))) return st;
  if ((st = map_bf16_pages3d(&tv3, pool->v, rows))) return st;
  if ((st = launch_prefix_decode(tk, tv3, pa, s))) return st;
  // 2. each request's own tokens [shared_len, n) (split-KV, partials only)
  SplitArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = pa.q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.ws_o = reinterpret_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float*>(ws + pl.off_ml);
  a.status = dev_status;
  a.num_pages = pool->num_pages;
  a.Hq = num_q_heads;
  a.Hkv = Hkv;
  a.G = pl.G;
  a.max_pages = max_pages_per_seq;
  a.n_clamp = static_cast<int>(std::min<long long>(max_seq_len, 1LL * max_pages_per_seq * kPage));
  a.T = pl.T;
  a.max_splits = pl.ms;
  a.out_f32 = out_dtype == PHS_OUT_F32;
  a.scale_log2 = scale_log2;
  a.skip_len = shared_len;
  a.force_partial = 1;
  a.prefix_bad = reinterpret_cast<int32_t*>(ws + pl.off_bad);
  a.wait_prior_at_exit = 1;  // started beside the prefix pass (independent tokens)
  if (k_new) {  // the new tokens are own tokens: the own-token split appends them
    a.app = FusedAppend{reinterpret_cast<const __nv_bfloat16*>(k_new),
                        reinterpret_cast<const __nv_bfloat16*>(v_new),
                        reinterpret_cast<__nv_bfloat16*>(pool->k),
                        reinterpret_cast<__nv_bfloat16*>(pool->v)};
    a.page_refcount = page_refcount;
  }
  if ((st = launch_split_decode(D, tk3, tv3, tk3, tv3, a, batch, s, true))) return st;
  // 3. merge prefix and suffix partials
  PrefixMergeArgs m;
  std::memset(&m, 0, sizeof(m));
  m.seq_lens = seq_lens;
  m.prefix_bad = a.prefix_bad;
  m.bad_slots = Hkv * pl.ms;
  m.ws_o = a.ws_o;
  m.ws_ml = a.ws_ml;
  m.ws_po = pa.ws_o;
  m.ws_pml = pa.ws_ml;
  m.out = out;
  m.Hq = num_q_heads;
  m.Hkv = Hkv;
  m.G = pl.G;
  m.n_clamp = a.n_clamp;
  m.T = pl.T;
  m.max_splits = pl.ms;
  m.num_psplits = pl.nsp;
  m.shared_len = shared_len;
  m.out_f32 = a.out_f32;
  return launch_merge_prefix(m, batch, s);
}

size_t phs_hybrid_stack_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_seq_len) {
  return phs_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, 0, 0);
}

int phs_attn_decode_hybrid_stack(const phs_layer* layers, int32_t num_layers,
                                 int32_t num_q_heads, int32_t batch, const int32_t* block_table,
                                 int32_t max_pages_per_seq, const int32_t* page_refcount,
                                 const int32_t* seq_lens, int32_t max_seq_len,
                                 const int32_t* ring_ids, const int32_t* ring_pos,
                                 float softmax_scale, int32_t do_append, int32_t out_dtype,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 void* stream) {
  if (!layers || num_layers <= 0 || batch < 0 || !seq_lens) return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return PHS_EINVAL;
  if (batch == 0) return PHS_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int st;
  // ---- validate every layer before launching anything
  int D = -1, Hkv = -1, W = -1;
  int nfull = 0, nswa = 0;
  for (int i = 0; i < num_layers; ++i) {
    const phs_layer& L = layers[i];
    if (!L.q || !L.out) return PHS_EINVAL;
    if (do_append && (!L.k_new || !L.v_new)) return PHS_EINVAL;
    int d, h;
    if (L.is_full) {
      if ((st = check_paged(&L.paged))) return st;
      d = L.paged.head_dim;
      h = L.paged.num_kv_heads;
      ++nfull;
    } else {
      if ((st = check_ring(&L.ring))) return st;
      d = L.ring.head_dim;
      h = L.ring.num_kv_heads;
      if (W < 0) W = L.ring.window;
      if (L.ring.window != W) return PHS_ESHAPE;
      ++nswa;
    }
    if (D < 0) {
      D = d;
      Hkv = h;
    }
    if (d != D || h != Hkv) return PHS_ESHAPE;
    if (!aligned16(L.q) || (do_append && (!aligned16(L.k_new) || !aligned16(L.v_new))))
      return PHS_EALIGN;
  }
  if ((st = check_dims(num_q_heads, Hkv, D))) return st;
  if (nfull && (!block_table || max_pages_per_seq <= 0)) return PHS_EINVAL;
  if (nswa && !ring_pos) return PHS_EINVAL;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  if (nswa && swa_smem_bytes(D, num_q_heads / Hkv) > di.smem_optin) return PHS_EUNSUPPORTED;
  // 8 warps per split CTA only if all Full layers' grids together fit one
  // wave (the fused call's launch shape, so both give the same results)
  bool wide = false;
  if (nfull) {
    DecodePlan pl;
    if ((st = make_plan(pl, batch, num_q_heads, Hkv, D, max_seq_len, 0, false))) return st;
    if (!workspace || workspace_bytes < pl.need) return PHS_EWORKSPACE;
    wide = 1LL * batch * Hkv * pl.max_splits * nfull <= di.sms;
  }

  // ---- appends: all Full layers in one launch, all SWA layers in one
  if (do_append) {
    for (int pass = 0; pass < 2; ++pass) {
      const bool full = pass == 0;
      AppendParams<kAppendMaxLayers> p;
      std::memset(&p, 0, sizeof(p));
      p.table = full ? block_table : ring_ids;
      p.seq_lens = seq_lens;
      p.ring_pos = ring_pos;
      p.refcount = full ? page_refcount : nullptr;
      p.status = dev_status;
      p.B = batch;
      p.Hkv = Hkv;
      p.D = D;
      p.max_pages = max_pages_per_seq;
      p.W = W;
      p.is_ring = full ? 0 : 1;
      for (int i = 0; i < num_layers; ++i) {
        const phs_layer& L = layers[i];
        if ((L.is_full != 0) != full) continue;
        p.layer[p.num_layers++] =
            full ? AppendLayer{L.paged.k, L.paged.v, L.k_new, L.v_new, L.paged.num_pages}
                 : AppendLayer{L.ring.k, L.ring.v, L.k_new, L.v_new, L.ring.num_rings};
        if (p.num_layers == kAppendMaxLayers) {
          if ((st = launch_append<kAppendMaxLayers>(p, s))) return st;
          p.num_layers = 0;
        }
      }
      if (p.num_layers && (st = launch_append<kAppendMaxLayers>(p, s))) return st;
    }
  }

  // ---- SWA layers: one launch (per 64 layers)
  if (nswa) {
    SwaParams<kSwaMaxLayers>* p = new SwaParams<kSwaMaxLayers>();
    std::memset(p, 0, sizeof(*p));
    p->ring_ids = ring_ids;
    p->ring_pos = ring_pos;
    p->seq_lens = seq_lens;
    p->status = dev_status;
    p->B = batch;
    p->Hq = num_q_heads;
    p->Hkv = Hkv;
    p->G = num_q_heads / Hkv;
    p->W = W;
    p->out_f32 = out_dtype == PHS_OUT_F32;
    p->scale_log2 = softmax_scale * 1.4426950408889634f;
    st = PHS_OK;
    for (int i = 0; i < num_layers && st == PHS_OK; ++i) {
      const phs_layer& L = layers[i];
      if (L.is_full) continue;
      const int k = p->num_layers;
      const int64_t rows = L.ring.num_rings * Hkv * W;
      if ((st = map_bf16_kv(&p->tk[k], L.ring.k, rows, D))) break;
      if ((st = map_bf16_kv(&p->tv[k], L.ring.v, rows, D))) break;
      p->q[k] = reinterpret_cast<const __nv_bfloat16*>(L.q);
      p->out[k] = L.out;
      p->num_rings[k] = L.ring.num_rings;
      if (++p->num_layers == kSwaMaxLayers) {
        st = launch_swa_decode<kSwaMaxLayers>(D, *p, di.sms, di.smem_optin, s);
        p->num_layers = 0;
      }
    }
    if (st == PHS_OK && p->num_layers) st = launch_swa_decode<kSwaMaxLayers>(D, *p, di.sms, di.smem_optin, s);
    delete p;
    if (st) return st;
  }

  // ---- Full layers: split + merge per layer, reusing the workspace
  for (int i = 0; i < num_layers; ++i) {
    const phs_layer& L = layers[i];
    if (!L.is_full) continue;
    st = decode_full_paged(L.q, num_q_heads, &L.paged, block_table, max_pages_per_seq, seq_lens,
                           max_seq_len, nullptr, nullptr, 0, nullptr, batch, softmax_scale, 0,
                           L.out, out_dtype, workspace, workspace_bytes, nullptr, nullptr, nullptr,
                           dev_status, stream, wide);
    if (st) return st;
  }
  return PHS_OK;
}

size_t phs_hybrid_stack_fused_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t max_seq_len, int32_t num_full_layers) {
  if (num_full_layers <= 0) return 0;
  const size_t one =
      phs_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, 0, 0);
  return one * static_cast<size_t>(num_full_layers);
}

int phs_attn_decode_hybrid_stack_fused(const phs_layer* layers, int32_t num_layers,
                                       int32_t num_q_heads, int32_t batch,
                                       const int32_t* block_table, int32_t max_pages_per_seq,
                                       const int32_t* page_refcount,
                                       const int32_t* seq_lens, int32_t max_seq_len,
                                       const int32_t* ring_ids, const int32_t* ring_pos,
                                       float softmax_scale, int32_t out_dtype, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status,
                                       void* stream) {
  if (!layers || num_layers <= 0 || batch < 0 || !seq_lens) return PHS_EINVAL;
  if (out_dtype != PHS_OUT_BF16 && out_dtype != PHS_OUT_F32) return PHS_EINVAL;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return PHS_EINVAL;
  if (batch == 0) return PHS_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int st;
  // ---- validate every layer before launching anything
  int D = -1, Hkv = -1, W = -1, nfull = 0, nswa = 0;
  int64_t min_pages = 0;  // the Full pools share the block table: ids must fit all of them
  for (int i = 0; i < num_layers; ++i) {
    const phs_layer& L = layers[i];
    if (!L.q || !L.out || !L.k_new || !L.v_new) return PHS_EINVAL;
    int d, h;
    if (L.is_full) {
      if ((st = check_paged(&L.paged))) return st;
      d = L.paged.head_dim;
      h = L.paged.num_kv_heads;
      min_pages = nfull == 0 ? L.paged.num_pages : std::min(min_pages, L.paged.num_pages);
      ++nfull;
    } else {
      if ((st = check_ring(&L.ring))) return st;
      d = L.ring.head_dim;
      h = L.ring.num_kv_heads;
      if (W < 0) W = L.ring.window;
      if (L.ring.window != W) return PHS_ESHAPE;
      ++nswa;
    }
    if (D < 0) {
      D = d;
      Hkv = h;
    }
    if (d != D || h != Hkv) return PHS_ESHAPE;
    if (!aligned16(L.q) || !aligned16(L.k_new) || !aligned16(L.v_new)) return PHS_EALIGN;
  }
  if ((st = check_dims(num_q_heads, Hkv, D))) return st;
  if (nfull && (!block_table || max_pages_per_seq <= 0)) return PHS_EINVAL;
  if (nswa && !ring_pos) return PHS_EINVAL;
  DevInfo di;
  if ((st = dev_info(di))) return st;
  if (nswa && swa_smem_bytes(D, num_q_heads / Hkv) > di.smem_optin) return PHS_EUNSUPPORTED;
  DecodePlan pl;
  if (nfull) {
    if ((st = make_plan(pl, batch, num_q_heads, Hkv, D, max_seq_len, 0, false))) return st;
    if (!workspace || workspace_bytes < pl.need * static_cast<size_t>(nfull))
      return PHS_EWORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PHS_EALIGN;
  }
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  StackMergeParams fold_merges;  // Full-layer merges handed to the SWA launch
  std::memset(&fold_merges, 0, sizeof(fold_merges));
  int fold_layers = 0;

  // A small step (every request in one split, so nothing to merge, and the
  // Full CTAs and SWA units together in one wave) goes in one launch that
  // runs both kinds of layer (phs_stack_small_kernel); the parameter blocks
  // below are built as for the two launches and handed to it.
  std::unique_ptr<StackSmallParams> small;
  if (nfull && nswa && nfull < kStackMaxFull && nswa < kSwaMaxLayers && pl.max_splits == 1 &&
      1LL * batch * Hkv * (nfull + nswa) <= di.sms &&
      stack_small_smem_bytes(D, num_q_heads / Hkv, di.smem_optin) > 0) {
    small.reset(new StackSmallParams());
    std::memset(small.get(), 0, sizeof(StackSmallParams));
  }

  // ---- launch 1 (per 16 Full layers): split-KV decode of every Full layer,
  // each CTA holding a request's newest token also appends it
  if (nfull) {
    StackFullParams* p = new StackFullParams();
    std::memset(p, 0, sizeof(*p));
    StackMergeParams* m = new StackMergeParams();
    std::memset(m, 0, sizeof(*m));
    SplitArgs& a = p->a;
    a.block_table = block_table;
    a.page_refcount = page_refcount;
    a.seq_lens = seq_lens;
    a.status = dev_status;
    a.num_pages = min_pages;
    a.Hq = num_q_heads;
    a.Hkv = Hkv;
    a.G = pl.G;
    a.max_pages = max_pages_per_seq;
    a.n_clamp = static_cast<int>(std::min<long long>(max_seq_len, 1LL * max_pages_per_seq * kPage));
    a.T = pl.T;
    a.max_splits = pl.max_splits;
    a.out_f32 = out_dtype == PHS_OUT_F32;
    a.scale_log2 = scale_log2;
    // 8 warps per CTA only if all Full layers' grids together fit one wave
    a.num_sms = 1LL * batch * Hkv * pl.max_splits * nfull <= di.sms ? di.sms : 0;
    MergeArgs& ma = m->a;
    ma.seq_lens = seq_lens;
    ma.Hq = num_q_heads;
    ma.Hkv = Hkv;
    ma.G = pl.G;
    ma.n_clamp = a.n_clamp;
    ma.T = pl.T;
    ma.max_splits = pl.max_splits;
    ma.out_f32 = a.out_f32;
    const size_t off_ml = ws_o_bytes(batch, Hkv, pl.max_splits, pl.G, D);
    char* ws = reinterpret_cast<char*>(workspace);
    int k = 0, done = 0;
    st = PHS_OK;
    for (int i = 0; i < num_layers && st == PHS_OK; ++i) {
      const phs_layer& L = layers[i];
      if (!L.is_full) continue;
      StackFullLayer& F = p->layer[k];
      const int64_t rows = L.paged.num_pages * Hkv * kPage;
      if ((st = map_bf16_kv(&F.tk, L.paged.k, rows, D))) break;
      if ((st = map_bf16_kv(&F.tv, L.paged.v, rows, D))) break;
      char* lw = ws + pl.need * static_cast<size_t>(done + k);
      F.q = reinterpret_cast<const __nv_bfloat16*>(L.q);
      F.out = L.out;
      F.ws_o = reinterpret_cast<float*>(lw);
      F.ws_ml = reinterpret_cast<float*>(lw + off_ml);
      F.app = FusedAppend{reinterpret_cast<const __nv_bfloat16*>(L.k_new),
                          reinterpret_cast<const __nv_bfloat16*>(L.v_new),
                          reinterpret_cast<__nv_bfloat16*>(L.paged.k),
                          reinterpret_cast<__nv_bfloat16*>(L.paged.v)};
      m->layer[k] = StackMergeLayer{F.ws_o, F.ws_ml, L.out};
      if (++k == kStackMaxFull) {
        p->num_layers = k;
        if ((st = launch_stack_full(D, *p, batch, s))) break;
        if (pl.max_splits > 1 && (st = launch_stack_merge(D, *m, batch, k, s))) break;
        done += k;
        k = 0;
      }
    }
    if (st == PHS_OK && k) {
      p->num_layers = k;
      if (small)
        small->full = *p;  // launched with the SWA layers below
      else
        st = launch_stack_full(D, *p, batch, s);
      // the last batch of Full layers is merged by the SWA launch when there
      // is one (two launches per step); otherwise by a merge launch
      if (st == PHS_OK && pl.max_splits > 1) {
        if (nswa) {
          fold_merges = *m;
          fold_layers = k;
        } else {
          st = launch_stack_merge(D, *m, batch, k, s);
        }
      }
    }
    delete p;
    delete m;
    if (st) return st;
  }

  // ---- launch 2: every SWA layer (one persistent launch per 64 layers),
  // each unit holding a request's newest slot also appends it
  if (nswa) {
    SwaParams<kSwaMaxLayers>* p = new SwaParams<kSwaMaxLayers>();
    std::memset(p, 0, sizeof(*p));
    p->ring_ids = ring_ids;
    p->ring_pos = ring_pos;
    p->seq_lens = seq_lens;
    p->status = dev_status;
    p->B = batch;
    p->Hq = num_q_heads;
    p->Hkv = Hkv;
    p->G = num_q_heads / Hkv;
    p->W = W;
    p->out_f32 = out_dtype == PHS_OUT_F32;
    p->scale_log2 = scale_log2;
    p->wait_prior_at_exit = nfull > 0;  // every SWA launch here is a dependent launch
    if (fold_layers) {  // the Full layers' merges ride on the first SWA launch
      for (int i = 0; i < fold_layers; ++i) p->merge_layer[i] = fold_merges.layer[i];
      p->merge = fold_merges.a;
      p->num_merge_layers = fold_layers;
    }
    st = PHS_OK;
    for (int i = 0; i < num_layers && st == PHS_OK; ++i) {
      const phs_layer& L = layers[i];
      if (L.is_full) continue;
      const int k = p->num_layers;
      const int64_t rows = L.ring.num_rings * Hkv * W;
      if ((st = map_bf16_kv(&p->tk[k], L.ring.k, rows, D))) break;
      if ((st = map_bf16_kv(&p->tv[k], L.ring.v, rows, D))) break;
      p->q[k] = reinterpret_cast<const __nv_bfloat16*>(L.q);
      p->out[k] = L.out;
      p->num_rings[k] = L.ring.num_rings;
      p->app[k] = FusedAppend{reinterpret_cast<const __nv_bfloat16*>(L.k_new),
                              reinterpret_cast<const __nv_bfloat16*>(L.v_new),
                              reinterpret_cast<__nv_bfloat16*>(L.ring.k),
                              reinterpret_cast<__nv_bfloat16*>(L.ring.v)};
      if (++p->num_layers == kSwaMaxLayers) {
        st = launch_swa_decode<kSwaMaxLayers>(D, *p, di.sms, di.smem_optin, s, nfull > 0);
        p->num_layers = 0;
        p->num_merge_layers = 0;
      }
    }
    if (st == PHS_OK && p->num_layers) {
      if (small) {
        small->swa = *p;
        small->B = batch;
        small->full_ctas = batch * Hkv * nfull;
        st = launch_stack_small(D, *small, batch * Hkv * p->num_layers, s);
      } else {
        st = launch_swa_decode<kSwaMaxLayers>(D, *p, di.sms, di.smem_optin, s, nfull > 0);
      }
    }
    delete p;
    if (st) return st;
  }
  return PHS_OK;
}

int phs_hybrid_kv_tokens(const int32_t* layer_is_full_host, int32_t num_layers,
                         const int32_t* seq_lens_host, int32_t batch, int32_t window,
                         int64_t* full_tokens, int64_t* swa_tokens) {
  if (!layer_is_full_host || !seq_lens_host || !full_tokens || !swa_tokens) return PHS_EINVAL;
  if (num_layers < 0 || batch < 0 || window <= 0) return PHS_EINVAL;
  int64_t f = 0, w = 0;
  for (int l = 0; l < num_layers; ++l)
    for (int b = 0; b < batch; ++b) {
      const int64_t n = seq_lens_host[b] > 0 ? seq_lens_host[b] : 0;
      if (layer_is_full_host[l])
        f += n;
      else
        w += std::min<int64_t>(n, window);
    }
  *full_tokens = f;
  *swa_tokens = w;
  return PHS_OK;
}

int phs_copy_pages(const phs_paged_pool* pool, const int32_t* src_pages, const int32_t* dst_pages,
                   int32_t n, int32_t* dev_status, void* stream) {
  int st = check_paged(pool);
  if (st) return st;
  if (n < 0 || (n > 0 && (!src_pages || !dst_pages))) return PHS_EINVAL;
  const int page_bytes = pool->num_kv_heads * kPage * pool->head_dim * 2;
  return launch_copy_pages(pool->k, pool->v, src_pages, dst_pages, n, pool->num_pages,
                           page_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace phs {
namespace {

// Shared checks and launch of the SWA segment save / seed calls.
int swa_segment_call(const phs_ring_pool* rings, const phs_paged_pool* segs, int32_t num_layers,
                     SegCopyParams<kSegMaxLayers>& p, int count, cudaStream_t s) {
  if (!rings || !segs || num_layers <= 0) return PHS_EINVAL;
  int st;
  for (int l = 0; l < num_layers; ++l) {
    if ((st = check_ring(&rings[l]))) return st;
    if ((st = check_paged(&segs[l]))) return st;
    if (rings[l].window != rings[0].window || rings[l].num_kv_heads != rings[0].num_kv_heads ||
        rings[l].head_dim != rings[0].head_dim || segs[l].num_kv_heads != rings[0].num_kv_heads ||
        segs[l].head_dim != rings[0].head_dim)
      return PHS_ESHAPE;
  }
  if (count == 0) return PHS_OK;
  p.Hkv = rings[0].num_kv_heads;
  p.D = rings[0].head_dim;
  p.W = rings[0].window;
  for (int l0 = 0; l0 < num_layers; l0 += kSegMaxLayers) {
    p.num_layers = std::min(kSegMaxLayers, num_layers - l0);
    for (int k = 0; k < p.num_layers; ++k) {
      const phs_ring_pool& R = rings[l0 + k];
      const phs_paged_pool& S = segs[l0 + k];
      p.layer[k] = SegCopyLayer{R.k, R.v, S.k, S.v, R.num_rings, S.num_pages};
    }
    if ((st = launch_swa_segment<kSegMaxLayers>(p, count, s))) return st;
  }
  return PHS_OK;
}

}  // namespace
}  // namespace phs

extern "C" {

int phs_swa_ring_save(const phs_ring_pool* rings, const phs_paged_pool* segs, int32_t num_layers,
                      const int32_t* ring_ids, const int32_t* ring_pos, const int32_t* seq_lens,
                      const int32_t* page_index, const int32_t* seg_pages, int32_t count,
                      int32_t* dev_status, void* stream) {
  if (count < 0 || (count > 0 && (!ring_ids || !ring_pos || !seq_lens || !page_index ||
                                   !seg_pages)))
    return PHS_EINVAL;
  SegCopyParams<kSegMaxLayers>* p = new SegCopyParams<kSegMaxLayers>();
  std::memset(p, 0, sizeof(*p));
  p->ring_ids = ring_ids;
  p->ring_pos = ring_pos;
  p->seq_lens = seq_lens;
  p->page_index = page_index;
  p->seg_pages = seg_pages;
  p->status = dev_status;
  p->save = 1;
  const int st = swa_segment_call(rings, segs, num_layers, *p, count,
                                  reinterpret_cast<cudaStream_t>(stream));
  delete p;
  return st;
}

int phs_swa_ring_seed(const phs_ring_pool* rings, const phs_paged_pool* segs, int32_t num_layers,
                      const int32_t* ring_ids, const int32_t* ring_pos, const int32_t* seq_lens,
                      const int32_t* seg_table, int32_t max_seg_pages, int32_t batch,
                      int32_t* dev_status, void* stream) {
  if (batch < 0 || (batch > 0 && (!ring_pos || !seq_lens || !seg_table || max_seg_pages <= 0)))
    return PHS_EINVAL;
  SegCopyParams<kSegMaxLayers>* p = new SegCopyParams<kSegMaxLayers>();
  std::memset(p, 0, sizeof(*p));
  p->ring_ids = ring_ids;
  p->ring_pos = ring_pos;
  p->seq_lens = seq_lens;
  p->seg_table = seg_table;
  p->max_seg = max_seg_pages;
  p->status = dev_status;
  p->save = 0;
  const int st = swa_segment_call(rings, segs, num_layers, *p, batch,
                                  reinterpret_cast<cudaStream_t>(stream));
  delete p;
  return st;
}

int phs_copy_d2d(void* dst, const void* src, size_t bytes, void* stream) {
  if (!dst || !src) return PHS_EINVAL;
  if (!aligned16(dst) || !aligned16(src) || (bytes & 15u)) return PHS_EALIGN;
  DevInfo di;
  int st = dev_info(di);
  if (st) return st;
  return launch_copy(dst, src, bytes, di.sms, reinterpret_cast<cudaStream_t>(stream));
}

int phs_read_checksum(const void* src, size_t bytes, uint32_t* dev_sink, void* stream) {
  if (!src || !dev_sink) return PHS_EINVAL;
  if (!aligned16(src) || (bytes & 15u)) return PHS_EALIGN;
  if ((reinterpret_cast<uintptr_t>(dev_sink) & 3u) != 0) return PHS_EALIGN;
  DevInfo di;
  int st = dev_info(di);
  if (st) return st;
  return launch_read(src, bytes, di.sms, dev_sink, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation decode.  The split partials go to this file-scope array
// instead of a caller workspace.  In host code the array's name is only a
// stand-in: its device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char phs_noalloc_scratch[PHS_NOALLOC_SCRATCH_BYTES];

namespace phs {
namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if none or on
// failure).  A context re-created after a device reset gets a new id, so a
// cached device address is never reused across contexts.
unsigned long long current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch in the current context: looked up with
// cudaGetSymbolAddress on the first call in each context (after a device
// reset the new context looks it up again), or null if the lookup fails.
void* noalloc_scratch_on_current_device() {
  static std::mutex mu;
  static std::map<unsigned long long, void*> addr;  // context id -> address
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0) {
    auto it = addr.find(id);
    if (it != addr.end()) return it->second;
  }
  // first call in this context (or no context yet: the lookup makes the
  // device's primary context current)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, phs_noalloc_scratch) != cudaSuccess) return nullptr;
  const unsigned long long now = current_context_id();
  if (now != 0) addr[now] = p;
  return p;
}

}  // namespace
}  // namespace phs

extern "C" int phs_attn_decode_full_paged_noalloc(
    const void* q, int32_t num_q_heads, const phs_paged_pool* pool, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
    const phs_int8_pool* int8, const int32_t* qtable, int32_t max_qpages_per_seq,
    const int32_t* qlens, int32_t batch, float softmax_scale, int32_t tokens_per_split, void* out,
    int32_t out_dtype, int32_t* dev_status, void* stream) {
  int st = check_paged(pool);
  if (st) return st;
  // choose a split length whose partials fit the scratch
  const bool has_int8 = int8 != nullptr;
  DecodePlan pl;
  if ((st = make_plan(pl, batch, num_q_heads, pool->num_kv_heads, pool->head_dim, max_seq_len,
                      tokens_per_split, has_int8)))
    return st;
  int tps = pl.T;
  while (pl.need > PHS_NOALLOC_SCRATCH_BYTES && tokens_per_split == 0 && tps < kMaxSplitTokens) {
    tps *= 2;
    if ((st = make_plan(pl, batch, num_q_heads, pool->num_kv_heads, pool->head_dim, max_seq_len,
                        tps, has_int8)))
      return st;
  }
  if (pl.need > PHS_NOALLOC_SCRATCH_BYTES) return PHS_ESCRATCH;
  void* scratch = noalloc_scratch_on_current_device();
  if (!scratch) return PHS_ECUDA;
  DecodeCall c;
  st = prepare_decode(c, q, num_q_heads, pool, block_table, max_pages_per_seq, seq_lens,
                      max_seq_len, int8, qtable, max_qpages_per_seq, qlens, batch, softmax_scale,
                      tps, out, out_dtype, scratch, PHS_NOALLOC_SCRATCH_BYTES, nullptr, nullptr,
                      nullptr, dev_status);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_split_decode(c.pl.D, c.tk, c.tv, c.tk8, c.tv8, c.a, batch, s))) return st;
  if (c.pl.max_splits == 1) return PHS_OK;  // every request finished in its only split
  return launch_merge(c.pl.D, c.m, batch, s);
}
