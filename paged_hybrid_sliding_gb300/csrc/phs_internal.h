// phs_internal.h -- argument blocks and launchers shared between the
// kernels' translation units and the C-ABI front end (phs_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "phs.h"

namespace phs {

constexpr int kPage = 16;    // tokens per Full-pool page
constexpr int kQBlock = 32;  // tokens per INT8 page / scale group

// Token held by byte p (0..15) of a 16-token half of an INT8 V^T row:
// bytes 4q, 4q+1 hold tokens 2q, 2q+1 and bytes 4q+2, 4q+3 tokens 8+2q,
// 9+2q.  The decode kernel transposes the two 8 x 8 blocks of a tile's
// packed scores (movmatrix), which gives lane q the P^T operand of exactly
// those tokens, in the order ldmatrix delivers bytes 4q..4q+3 of a V^T row.
constexpr int kI8VtToken(int p) { return 2 * (p >> 2) + (p & 1) + 8 * ((p >> 1) & 1); }

// ----------------------------------------------------- split-KV decode --
// New token of each request for an append fused into a decode kernel: the
// kernel writes it to its page (or ring slot) and attends to it from these
// inputs instead of reading it back.  k_new null: no append.
struct FusedAppend {
  const __nv_bfloat16* k_new;  // [B][Hkv][D]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;       // paged [num_pages][Hkv][16][D] / ring [rings][Hkv][W][D]
  __nv_bfloat16* v_pool;
};

struct SplitArgs {
  const __nv_bfloat16* q;   // [B][Hq][D]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qtable;    // INT8 page table, or null
  const int32_t* qlens;     // INT8 lengths, or null
  const float* k_scale;
  const float* v_scale;
  void* out;
  float* ws_o;              // [B][Hkv][max_splits][G][D]
  float* ws_ml;             // [B][Hkv][max_splits][G][2]
  int32_t* status;
  int64_t num_pages;
  int64_t num_qpages;
  int Hq, Hkv, G;
  int wait_prior_at_exit;   // launched beside an independent grid (programmatic
                            // dependent): do not complete before it has
  int max_pages;            // block table row length
  int max_qpages;           // INT8 table row length
  int n_clamp;              // lengths above this are an error and clamped
  int T;                    // tokens per split (multiple of 32)
  int max_splits;
  int out_f32;
  float scale_log2;         // softmax_scale * log2(e)
  int skip_len;             // tokens [0, skip_len) are attended elsewhere (shared prefix)
  int force_partial;        // write partials even for single-split requests
  // fused append: page reference counts, or null; a new
  // token whose page count is not 1 is neither written nor attended from
  // the input (the page is shared; copy on write is the caller's job)
  const int32_t* page_refcount;
  // shared-prefix call (skip_len > 0): per (request, KV head, split) CTA,
  // 1 if its slice of the request's first skip_len / 16 page ids differs
  // from row 0's, or the request is shorter than skip_len; else 0
  int32_t* prefix_bad;
  // append fused into a split launch (the shared-prefix call's own-token
  // split; k_new null: none).  The stack kernel takes each layer's from its
  // own parameter block instead.
  FusedAppend app;
  // SMs of the device (0: unknown).  A bf16 launch whose grid has at most
  // one CTA per SM runs 8 warps per CTA instead of 4, so that each warp's
  // chain of chunks is half as long (latency-bound small steps).
  int num_sms;
};


// ------------------------------------- hybrid stack: Full layers at once --
constexpr int kStackMaxFull = 16;  // Full layers per launch

struct StackFullLayer {
  CUtensorMap tk, tv;        // per-page K / V boxes of this layer's pool
  const __nv_bfloat16* q;    // [B][Hq][D]
  void* out;
  float* ws_o;               // this layer's partials (split kernel layout)
  float* ws_ml;
  FusedAppend app;
};

struct StackFullParams {
  StackFullLayer layer[kStackMaxFull];
  SplitArgs a;               // fields shared by the layers (q/out/ws_* unused)
  int num_layers;
};

struct StackMergeLayer {
  const float* ws_o;
  const float* ws_ml;
  void* out;
};

// ------------------------------------------------- shared-prefix decode --
struct PrefixArgs {
  const __nv_bfloat16* q;   // [B][Hq][D]
  const int32_t* block_table;  // page ids of the shared prefix (row 0 of the table)
  int32_t* status;
  float* ws_o;              // [Hkv][num_splits][256][D]
  float* ws_ml;             // [Hkv][num_splits][256][2]
  int64_t num_pages;
  int Hq, Hkv, G;
  int rows;                 // B * G <= 256
  int shared_len;           // tokens, multiple of 64
  int tiles_per_split;
  int num_splits;
  float scale_log2;
};

struct PrefixMergeArgs {
  const int32_t* seq_lens;
  const int32_t* prefix_bad;  // [B][Hkv][max_splits] from the own-token split
  int bad_slots;              // Hkv * max_splits
  const float* ws_o;        // suffix partials (split kernel layout)
  const float* ws_ml;
  const float* ws_po;       // prefix partials
  const float* ws_pml;
  void* out;
  int Hq, Hkv, G;
  int n_clamp;
  int T;
  int max_splits;           // suffix split slots
  int num_psplits;
  int shared_len;
  int out_f32;
};

int launch_prefix_decode(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixArgs& a,
                         cudaStream_t stream);
int launch_merge_prefix(const PrefixMergeArgs& a, int B, cudaStream_t stream);
int prefix_smem_bytes();

struct MergeArgs {
  const int32_t* seq_lens;
  const int32_t* qlens;
  const float* ws_o;
  const float* ws_ml;
  void* out;
  int Hq, Hkv, G;
  int n_clamp;
  int T;
  int max_splits;
  int out_f32;
};

int launch_split_decode(int D, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tk8, const CUtensorMap& tv8, const SplitArgs& a,
                        int B, cudaStream_t stream, bool dependent = false);
int launch_merge(int D, const MergeArgs& a, int B, cudaStream_t stream);

// The cross-split merges of every Full layer of a hybrid stack: one launch
// for a stack without SWA layers, else extra work of the SWA launch.
struct StackMergeParams {
  StackMergeLayer layer[kStackMaxFull];
  MergeArgs a;               // fields shared by the layers (ws_*/out unused)
};
int launch_stack_full(int D, const StackFullParams& p, int B, cudaStream_t stream);
int launch_stack_merge(int D, const StackMergeParams& p, int B, int num_layers,
                       cudaStream_t stream);

// ------------------------------------------------------------ SWA ring --
constexpr int kSwaMaxLayers = 64;

template <int MAXL>
struct SwaParams {
  CUtensorMap tk[MAXL];
  CUtensorMap tv[MAXL];
  const __nv_bfloat16* q[MAXL];
  void* out[MAXL];
  int64_t num_rings[MAXL];
  FusedAppend app[MAXL];    // per layer; k_new null: no fused append
  const int32_t* ring_ids;  // null = identity
  const int32_t* ring_pos;
  const int32_t* seq_lens;
  int32_t* status;
  int num_layers, B, Hq, Hkv, G, W;
  int out_f32;
  float scale_log2;
  // The Full layers' cross-split merges of a hybrid-stack step, taken as
  // extra work after the SWA units (the split launch ran before this one on
  // the stream): layer l's partials and output, shared merge fields.
  StackMergeLayer merge_layer[kStackMaxFull];
  MergeArgs merge;
  int num_merge_layers;     // 0: none
  int wait_prior_at_exit;   // launched beside the split launch before it
                            // (programmatic dependent): do not complete
                            // before it has
};

template <int MAXL>
int launch_swa_decode(int D, const SwaParams<MAXL>& p, int num_sms, int smem_optin,
                      cudaStream_t stream, bool dependent = false);

// ---------------------------------------------- one-launch small step --
// A whole small hybrid step in one launch: CTAs [0, full_ctas) run the Full
// layers' splits (one split per request, 8 warps), the rest one SWA unit
// each (the chunked shape).
struct StackSmallParams {
  StackFullParams full;
  SwaParams<kSwaMaxLayers> swa;
  int B;
  int full_ctas;  // B x Hkv x Full layers
};

// Dynamic shared memory of the one-launch step (0: does not fit).
int stack_small_smem_bytes(int D, int G, int smem_optin);
int launch_stack_small(int D, const StackSmallParams& p, int swa_units, cudaStream_t stream);

// -------------------------------------------------------------- append --
constexpr int kAppendMaxLayers = 64;

struct AppendLayer {
  void* k;
  void* v;
  const void* k_new;
  const void* v_new;
  int64_t num;  // pages (paged) or rings (ring)
};

template <int MAXL>
struct AppendParams {
  AppendLayer layer[MAXL];
  const int32_t* table;     // paged: block table; ring: ring ids (may be null)
  const int32_t* seq_lens;  // paged
  const int32_t* ring_pos;  // ring
  const int32_t* refcount;  // paged, may be null
  int32_t* status;
  int num_layers, B, Hkv, D;
  int max_pages;            // paged
  int W;                    // ring
  int is_ring;
};

template <int MAXL>
int launch_append(const AppendParams<MAXL>& p, cudaStream_t stream);

// ---------------------------------------------- SWA segment pages (save /
// seed a ring from page snapshots of its window) --
constexpr int kSegMaxLayers = 64;

struct SegCopyLayer {
  void* ring_k;
  void* ring_v;
  void* seg_k;   // segment pool, paged layout [num_seg][Hkv][16][D]
  void* seg_v;
  int64_t num_rings;
  int64_t num_seg;
};

template <int MAXL>
struct SegCopyParams {
  SegCopyLayer layer[MAXL];
  const int32_t* ring_ids;    // per entry (save) / request (seed); may be null (seed)
  const int32_t* ring_pos;    // newest slot
  const int32_t* seq_lens;    // tokens of the request
  const int32_t* page_index;  // save: logical page to snapshot
  const int32_t* seg_pages;   // save: destination segment page
  const int32_t* seg_table;   // seed: [B][max_seg] segment pages of the window
  int32_t* status;
  int num_layers, Hkv, D, W, max_seg;
  int save;                   // 1 save (ring -> segment), 0 seed (segment -> ring)
};

template <int MAXL>
int launch_swa_segment(const SegCopyParams<MAXL>& p, int count, cudaStream_t stream);

// ----------------------------------------------------------- quantiser --
struct QuantArgs {
  const __nv_bfloat16* k_src;
  const __nv_bfloat16* v_src;
  const int32_t* src_table;
  uint8_t* k_codes;  // stored form of phs_int8_pool
  uint8_t* v_codes;
  float* k_scale;
  float* v_scale;
  const int32_t* dst_qtable;
  const int32_t* first_qblock;
  const int32_t* num_qblocks;
  int32_t* status;
  int64_t num_pages, num_qpages;
  int src_max_pages, dst_max_qpages;
  int Hkv, D;
};

int launch_quant(const QuantArgs& a, int max_qblocks, int B, cudaStream_t stream);

// ---------------------------------------------------------------- copy --
int launch_copy(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t stream);
int launch_read(const void* src, size_t bytes, int num_sms, uint32_t* sink, cudaStream_t stream);
int launch_copy_pages(void* k, void* v, const int32_t* src, const int32_t* dst, int32_t n,
                      int64_t num_pages, int page_bytes, int32_t* status, cudaStream_t stream);

int swa_smem_bytes(int D, int G);

// Raise a kernel's dynamic shared-memory limit once per (kernel, device);
// later calls are a lookup (no CUDA call, so launches stay cheap and safe to
// record into a CUDA graph).
int ensure_dynamic_smem(const void* kernel, int bytes);

}  // namespace phs
