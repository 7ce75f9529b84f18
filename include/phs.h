/*
 * phs.h -- C ABI of the paged hybrid sliding-window decode library
 * (libphs.so, CUDA, sm_103a).
 *
 * The library computes one decode step of attention for a batch of requests
 * whose KV cache is split into two pools, as described on the "Xiaomi
 * MiMo-V2.5 inference system" page (section 2, "KVCache system rebuild",
 * dual pools):
 *   - a Full-attention pool of fixed-size pages reached through per-request
 *     block tables; pages may be shared by several requests through a
 *     reference count ("Kimi K3 context caching" page, section 1: copy on
 *     write and reference counts in the page table);
 *   - a sliding-window (SWA) pool that is a per-request ring buffer of W
 *     tokens (MiMo page, section 2: ring buffer, storage O(W)).
 * plus the KV append that writes each new token into its page or ring slot
 * and a block-wise INT8 quantiser with one fp32 absmax scale per 32 tokens per
 * KV head ("Kimi K2.5 architecture deep dive" page, sections 2.2 and 2.3).
 *
 * Conventions (all entry points):
 *   - Every pointer argument named *dev / pool / table / q / out / workspace
 *     is a DEVICE pointer unless the comment says "host".  The caller owns
 *     all memory.  The library allocates nothing and keeps no state between
 *     calls except a per-thread cache of device properties (and the built-in
 *     scratch of phs_attn_decode_full_paged_noalloc, described there).
 *   - bf16 tensors are IEEE bfloat16 (2 bytes).  Layouts are C order:
 *       Full pool  K, V : [num_pages][Hkv][page_size][D]       bf16
 *       SWA ring   K, V : [num_rings][Hkv][window][D]          bf16
 *       INT8 pool  K, V : [num_qpages][Hkv][32][D]             int8
 *       INT8 scales     : [num_qpages][Hkv]                    fp32
 *       q, out          : [batch][Hq][D]                       bf16 / fp32
 *       k_new, v_new    : [batch][Hkv][D]                      bf16
 *       block_table     : [batch][max_pages_per_seq]           int32
 *   - Query head i attends with KV head i / (Hq / Hkv).
 *   - seq_lens[b] is the request's length AFTER this step's token has been
 *     appended; decode is "append, then attend", so the new token attends to
 *     itself.  Token t of request b lives in page block_table[b][t / 16] at
 *     slot t % 16.  In the ring the newest token is at slot ring_pos[b] and
 *     token t at (ring_pos[b] - (seq_lens[b] - 1 - t)) mod W; an SWA layer
 *     attends to the last min(seq_lens[b], W) tokens.
 *   - All work is queued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).
 *   - Argument errors are detected on the host and returned synchronously as
 *     a negative phs_status, before anything is launched.
 *   - Errors that depend on device data (a page id outside the pool, a
 *     sequence longer than its block table, an append into a shared page, a
 *     wait that timed out) are recorded in *dev_status when dev_status is not
 *     NULL: a device int32 the caller zeroes; the first error code written
 *     wins.  The offending item is skipped; nothing traps.
 *   - Supported shapes: page_size 16, head_dim 64 or 128, Hq a multiple of Hkv
 *     with group size Hq/Hkv <= 16, window a multiple of 16 (<= 4096),
 *     Hkv * head_dim <= 8192 (Hkv <= 64 at head_dim 128).
 *     Anything else returns PHS_EUNSUPPORTED.
 */
#ifndef PHS_H_
#define PHS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PHS_OK = 0,
    PHS_EINVAL = -1,        /* null pointer, non-positive size, bad enum */
    PHS_ESHAPE = -2,        /* inconsistent shapes between arguments */
    PHS_ERANGE = -3,        /* (device) index outside its pool or table */
    PHS_ESHARED = -4,       /* (device) append into a page with refcount != 1 */
    PHS_EWORKSPACE = -5,    /* workspace missing or too small */
    PHS_ECUDA = -6,         /* a CUDA runtime/driver call failed */
    PHS_EUNSUPPORTED = -7,  /* valid but unsupported shape */
    PHS_ETIMEOUT = -8,      /* (device) a bounded wait gave up */
    PHS_EALIGN = -9,        /* a pointer is not 16-byte aligned */
    PHS_ESCRATCH = -10,     /* request needs more than the built-in scratch of
                               phs_attn_decode_full_paged_noalloc */
    PHS_ENOSPACE = -11      /* page allocator has fewer free pages than asked */
} phs_status;

enum { PHS_OUT_BF16 = 0, PHS_OUT_F32 = 1 };

/* Paged Full-attention pool. */
typedef struct {
    void *k;              /* device, bf16 [num_pages][Hkv][page_size][D] */
    void *v;              /* device, same layout as k */
    int64_t num_pages;
    int32_t page_size;    /* tokens per page; must be 16 */
    int32_t num_kv_heads; /* Hkv */
    int32_t head_dim;     /* D: 64 or 128 */
} phs_paged_pool;

/* SWA ring pool: one ring of `window` token slots per ring id. */
typedef struct {
    void *k;              /* device, bf16 [num_rings][Hkv][window][D] */
    void *v;
    int64_t num_rings;
    int32_t window;       /* W, a multiple of 16 */
    int32_t num_kv_heads;
    int32_t head_dim;
} phs_ring_pool;

/* INT8 pool: 32-token pages of codes plus one fp32 scale per page and head.
 * A code x in [-127, 127] is stored as the byte x + 128.  K is token-major.
 * V is transposed per 16-token half of the page: D rows of 16 bytes (one per
 * head dim) for tokens 0-15, then D rows for tokens 16-31; byte p of a row
 * holds token 2(p/4) + (p%2) + 8((p/2)%2) of its half.  These are the orders
 * in which the decode kernel's mma fragments read the codes.  Each is
 * 32 * D bytes per page and head. */
typedef struct {
    uint8_t *k;           /* device, [num_qpages][Hkv][32 tokens][D] */
    uint8_t *v;           /* device, [num_qpages][Hkv][2 halves][D][16 tokens, order above] */
    float *k_scale;       /* device, fp32 [num_qpages][Hkv] */
    float *v_scale;
    int64_t num_qpages;
    int32_t num_kv_heads;
    int32_t head_dim;
} phs_int8_pool;

/* ------------------------------------------------------------------------
 * KV append, Full pool.
 * Source: "Kimi K3 context caching" page, section 1 (a request that extends
 * a shared prefix gets new physical blocks only for its own new tokens) and
 * MiMo page, section 2 (the Full pool grows on demand).
 * For each request b with seq_lens[b] >= 1, copies k_new[b] and v_new[b]
 * ([Hkv][D] bf16) into slot (seq_lens[b]-1) % 16 of page
 * block_table[b][(seq_lens[b]-1) / 16], for every KV head.  A byte copy.
 * page_refcount (device, int32 [num_pages], may be NULL): when given, a
 * target page whose count is not 1 is not written and PHS_ESHARED is
 * recorded in *dev_status (copy on write is the allocator's job).
 * Out-of-range page ids / table positions record PHS_ERANGE.
 * ---------------------------------------------------------------------- */
int phs_kv_append_paged(const phs_paged_pool *pool, const void *k_new, const void *v_new,
                        const int32_t *block_table, int32_t max_pages_per_seq,
                        const int32_t *seq_lens, int32_t batch,
                        const int32_t *page_refcount, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * KV append, SWA ring.
 * Source: MiMo page, section 2 (ring buffer of W slots, window-based
 * eviction: the new token overwrites the one leaving the window).
 * Writes k_new[b], v_new[b] into slot ring_pos[b] of ring ring_ids[b]
 * (ring_ids may be NULL: request b owns ring b).  ring_pos is the slot of
 * the token being appended (device, int32 [batch], in [0, W)).
 * ---------------------------------------------------------------------- */
int phs_kv_append_ring(const phs_ring_pool *ring, const void *k_new, const void *v_new,
                       const int32_t *ring_ids, const int32_t *ring_pos, int32_t batch,
                       int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Block-32 INT8 quantiser.
 * Source: "Kimi K2.5 architecture deep dive" page, sections 2.2-2.3 (warm
 * KV as INT8 with block-wise quantisation, a scale per group of 32 tokens).
 * For each request b and each 32-token block j in
 * [first_qblock[b], first_qblock[b] + num_qblocks[b]) (device int32 arrays),
 * for each KV head, separately for K and V: reads the 32 x D bf16 group
 * (tokens 32j .. 32j+31 through src_block_table), computes in IEEE fp32
 *     a = max |x|,  s = a / 127,  code = clamp(rint(x / s), -127, 127)
 * (rint rounds half to even; a == 0 gives s = 0 and all codes 0), and stores
 * the codes in INT8 page dst_qtable[b][j] (in the stored form and layout of
 * phs_int8_pool) and s in the matching scale slot.
 * max_qblocks bounds num_qblocks[b] (host int; sizes the grid).
 * ---------------------------------------------------------------------- */
int phs_kv_quant_int8_block32(const phs_paged_pool *src, const int32_t *src_block_table,
                              int32_t src_max_pages, const phs_int8_pool *dst,
                              const int32_t *dst_qtable, int32_t dst_max_qpages,
                              const int32_t *first_qblock, const int32_t *num_qblocks,
                              int32_t max_qblocks, int32_t batch, int32_t *dev_status,
                              void *stream);

/* ------------------------------------------------------------------------
 * Workspace for split-KV Full-attention decode, in bytes.
 * tokens_per_split: 0 = the library's choice (the same choice the decode
 * call makes for the same arguments); otherwise a positive multiple of 32.
 * has_int8: 1 if the decode call will pass an INT8 pool.
 * ---------------------------------------------------------------------- */
size_t phs_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len,
                                  int32_t tokens_per_split, int32_t has_int8);

/* The split length (tokens) the decode call uses for these arguments: 256
 * when max_seq_len is 129..256 and batch x num_kv_heads is at most the
 * GPU's SM count (one split per request, no merge); otherwise the longest
 * of 4096, 2048, ..., 128 that gives a max_seq_len request at least 8
 * splits and whose grid (batch x num_kv_heads x the splits of a
 * max_seq_len request) has at least 16 CTAs per SM, else 128;
 * tokens_per_split > 0 is returned as given. */
int32_t phs_decode_tokens_per_split(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len,
                                    int32_t tokens_per_split);

/* ------------------------------------------------------------------------
 * Full-attention decode over the paged pool, one query token per request.
 * Source: MiMo page, section 1 (Full layers attend over the whole sequence;
 * decode latency follows the KV bytes read) and the textbook definition
 *     out[b][i] = softmax_t(softmax_scale * q[b][i] . K_b[t]) V_b[t],
 *     t in [0, seq_lens[b]).
 * Optional INT8 region (int8 != NULL): tokens t < qlens[b] (a multiple of
 * 32) are read from INT8 page qtable[b][t / 32] (device int32
 * [batch][max_qpages_per_seq]) and dequantised as (float)code * scale;
 * tokens t >= qlens[b] are read from bf16 pages block_table[b][t / 16].
 * The sequence is cut into splits of tokens_per_split tokens (INT8 and bf16
 * regions are split separately); one CTA reduces one (request, KV head,
 * split) for all Hq/Hkv query heads of the group; a second kernel merges the
 * splits by log-sum-exp.  max_seq_len (host int) bounds seq_lens[b].
 * out: [batch][Hq][D], bf16 (out_dtype PHS_OUT_BF16) or fp32.
 * workspace: device, at least phs_decode_workspace_bytes(...) bytes, 256-byte
 * aligned; contents need no initialisation and are overwritten.
 * Requests with seq_lens[b] == 0 get an all-zero output row.
 * Fused append (k_new and v_new both given, device bf16 [batch][Hkv][D],
 * 16-byte aligned; both NULL: none): each request's new token, token
 * seq_lens[b] - 1, is written into its bf16 page by the CTA that attends
 * it, which attends it from k_new/v_new.  The result equals
 * phs_kv_append_paged (with the same page_refcount) followed by this call.
 * A page whose count is not 1 is not written (PHS_ESHARED), and its tokens
 * are attended as the page holds them.  A new token inside the request's
 * INT8 region (seq_lens[b] - 1 < qlens[b]) is not written and records
 * PHS_ERANGE.
 * ---------------------------------------------------------------------- */
int phs_attn_decode_full_paged(const void *q, int32_t num_q_heads, const phs_paged_pool *pool,
                               const int32_t *block_table, int32_t max_pages_per_seq,
                               const int32_t *seq_lens, int32_t max_seq_len,
                               const phs_int8_pool *int8, const int32_t *qtable,
                               int32_t max_qpages_per_seq, const int32_t *qlens,
                               int32_t batch, float softmax_scale, int32_t tokens_per_split,
                               void *out, int32_t out_dtype, void *workspace,
                               size_t workspace_bytes, const void *k_new, const void *v_new,
                               const int32_t *page_refcount, int32_t *dev_status,
                               void *stream);

/* The two phases of phs_attn_decode_full_paged, exposed separately so that
 * each kernel can be timed on its own.  The split phase writes every
 * single-split request's final output directly and the partial (m, l, o)
 * of multi-split requests into the workspace; the merge phase finishes the
 * multi-split requests.  Same arguments and meaning as above. */
int phs_attn_decode_full_paged_split(const void *q, int32_t num_q_heads,
                                     const phs_paged_pool *pool, const int32_t *block_table,
                                     int32_t max_pages_per_seq, const int32_t *seq_lens,
                                     int32_t max_seq_len, const phs_int8_pool *int8,
                                     const int32_t *qtable, int32_t max_qpages_per_seq,
                                     const int32_t *qlens, int32_t batch, float softmax_scale,
                                     int32_t tokens_per_split, void *out, int32_t out_dtype,
                                     void *workspace, size_t workspace_bytes,
                                     const void *k_new, const void *v_new,
                                     const int32_t *page_refcount, int32_t *dev_status,
                                     void *stream);

/* Cross-split merge: for each (request, query head) with more than one
 * split, M = max_s m_s, L = sum_s l_s 2^(m_s - M),
 * out = sum_s 2^(m_s - M) o_s / L.  qlens may be NULL (no INT8 region). */
int phs_attn_merge_splits(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, const int32_t *seq_lens, int32_t max_seq_len,
                          const int32_t *qlens, int32_t has_int8, int32_t tokens_per_split,
                          void *out, int32_t out_dtype, const void *workspace,
                          size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Full-attention decode that allocates nothing: the same computation, the
 * same arguments and the same results as phs_attn_decode_full_paged, minus
 * the workspace.  The pages have no counterpart to this call; it exists for
 * callers that cannot hand the library a workspace: plug-ins and callbacks
 * running inside a host framework that owns all device memory and does not
 * expose its allocator, serving engines that reserve nearly all of HBM for
 * the KV pool up front (so a late cudaMalloc would fail), and latency-bound
 * decode loops where cudaMalloc/cudaFree and the device-wide synchronisation
 * they imply are not acceptable.
 *
 * Scratch: the split partials live in a file-scope device array of
 * PHS_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU which loads the library
 * holds until the process exits.  The library's first call of this entry
 * point on a device looks up the array's device address (no allocation);
 * make that first call before any stream capture.  The address is cached
 * per CUDA context: after a device reset the first call in the new context
 * looks it up again (make that call outside a capture too).  All calls share the one
 * array and keep no state in it between calls, so calls that overlap on
 * the GPU (on different streams, or from several threads) race: serialise
 * them.  When tokens_per_split is 0 the library picks the split length as
 * the decode call does and, if the partials would not fit, lengthens the
 * splits (up to 4096 tokens); a request that still does not fit, or an
 * explicit tokens_per_split that does not fit, returns PHS_ESCRATCH before
 * anything is launched.  Nothing here calls cudaMalloc, cudaFree or any
 * allocating routine.
 * ---------------------------------------------------------------------- */
#define PHS_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int phs_attn_decode_full_paged_noalloc(const void *q, int32_t num_q_heads,
                                       const phs_paged_pool *pool, const int32_t *block_table,
                                       int32_t max_pages_per_seq, const int32_t *seq_lens,
                                       int32_t max_seq_len, const phs_int8_pool *int8,
                                       const int32_t *qtable, int32_t max_qpages_per_seq,
                                       const int32_t *qlens, int32_t batch, float softmax_scale,
                                       int32_t tokens_per_split, void *out, int32_t out_dtype,
                                       int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Full-attention decode of a batch that shares a prefix, on the tensor
 * cores.  Source: "Kimi K3 context caching" page, sections 1 and 4 (requests
 * hitting a cached prefix share its physical blocks; a 250,000-token shared
 * prefix).  Computes exactly what phs_attn_decode_full_paged computes, for
 * a batch whose block tables all begin with the same shared_len / 16 page
 * ids (row 0 of the table is read for them):
 *   - tokens [0, shared_len) of every request are attended in one pass over
 *     the prefix per KV head, with the B x G query rows of that head as one
 *     dense tile (tcgen05.mma), so the prefix is read from HBM once;
 *   - tokens [shared_len, n_b) by the split-KV kernel;
 *   - a merge combines both by log-sum-exp.
 * Limits: head_dim 128, batch x (Hq/Hkv) <= 256, shared_len a positive
 * multiple of 64 with max_seq_len >= shared_len (else PHS_EUNSUPPORTED /
 * PHS_EINVAL).  workspace: phs_shared_prefix_workspace_bytes(...) bytes,
 * 256-byte aligned.
 * Checked on the device: a request whose first shared_len / 16 page ids
 * differ from row 0's, or whose seq_lens[b] < shared_len, records
 * PHS_ESHAPE in *dev_status and gets an all-zero output row; the other
 * requests are unaffected.
 * Fused append (k_new and v_new both given, device bf16 [batch][Hkv][D],
 * 16-byte aligned; both NULL: none): the step's new token of each request,
 * token seq_lens[b] - 1, is written into its page by the CTA that attends
 * it, which attends it from k_new/v_new.  The result equals
 * phs_kv_append_paged (with the same page_refcount) followed by this call.
 * A page whose count is not 1 is not written (PHS_ESHARED), and its tokens
 * are attended as the page holds them.  A new token inside the shared
 * prefix (seq_lens[b] == shared_len) is never written and records
 * PHS_ESHARED.
 * ---------------------------------------------------------------------- */
size_t phs_shared_prefix_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t max_seq_len, int32_t shared_len);

int phs_attn_decode_shared_prefix(const void *q, int32_t num_q_heads, const phs_paged_pool *pool,
                                  const int32_t *block_table, int32_t max_pages_per_seq,
                                  const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                                  int32_t shared_len, float softmax_scale, void *out,
                                  int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                  const void *k_new, const void *v_new,
                                  const int32_t *page_refcount, int32_t *dev_status,
                                  void *stream);

/* ------------------------------------------------------------------------
 * Sliding-window decode over the SWA ring.
 * Source: MiMo page, section 1 (SWA layers, window 128, attend to the most
 * recent tokens) and section 2 (ring buffer of capacity W).
 * out[b][i] = softmax attention of q[b][i] over the last min(seq_lens[b], W)
 * tokens of request b, read from ring ring_ids[b] (NULL = identity) whose
 * newest token is at slot ring_pos[b].  No workspace.
 * ---------------------------------------------------------------------- */
int phs_attn_decode_swa_ring(const void *q, int32_t num_q_heads, const phs_ring_pool *ring,
                             const int32_t *ring_ids, const int32_t *ring_pos,
                             const int32_t *seq_lens, int32_t batch, float softmax_scale,
                             void *out, int32_t out_dtype, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * One decode step of a hybrid layer stack.
 * Source: MiMo page, section 1 (70 layers: 10 Full attention, 60 sliding
 * window of 128) and section 2 (dual pools; SWA reads overlap layer by
 * layer).  For every layer in `layers` (host array): if do_append, append
 * k_new/v_new into the layer's pool (paged for Full layers through the
 * shared block_table, ring slot ring_pos for SWA layers), then attend:
 * Full layers through phs_attn_decode_full_paged, SWA layers through the
 * ring.  All SWA layers go into one launch per 64 layers; each Full layer is one split
 * launch plus one merge launch when a request has several splits, all
 * reusing `workspace` (phs_hybrid_stack_workspace_bytes).  Layers are independent: the step
 * runs each layer on its own q (no model weights are involved).
 * page_refcount (device, int32 [num_pages], may be NULL) is checked as by
 * phs_kv_append_paged: a Full layer's new token whose page count is not 1
 * is not written (PHS_ESHARED in *dev_status); the Full pools share the
 * block table, so one count per page id serves every Full layer.
 * Every argument is checked before anything is launched (softmax_scale
 * must be positive and finite).
 * ---------------------------------------------------------------------- */
typedef struct {
    int32_t is_full;      /* 1 = Full-attention layer, 0 = SWA layer */
    const void *q;        /* device, bf16 [batch][Hq][D] */
    const void *k_new;    /* device, bf16 [batch][Hkv][D] (used if do_append) */
    const void *v_new;
    void *out;            /* device, [batch][Hq][D], out_dtype */
    phs_paged_pool paged; /* Full layers */
    phs_ring_pool ring;   /* SWA layers */
} phs_layer;

int phs_attn_decode_hybrid_stack(const phs_layer *layers, int32_t num_layers,
                                 int32_t num_q_heads, int32_t batch,
                                 const int32_t *block_table, int32_t max_pages_per_seq,
                                 const int32_t *page_refcount,
                                 const int32_t *seq_lens, int32_t max_seq_len,
                                 const int32_t *ring_ids, const int32_t *ring_pos,
                                 float softmax_scale, int32_t do_append, int32_t out_dtype,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream);

/* Workspace bytes for phs_attn_decode_hybrid_stack with these shapes (the
 * split partials of one Full layer at a time: the layers reuse it); 0 if the
 * shape is not supported.  Host call, no device work. */
size_t phs_hybrid_stack_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_seq_len);

/* ------------------------------------------------------------------------
 * One decode step of a hybrid layer stack, appends fused into the attention
 * launches.  Source: MiMo page, section 1 (10 Full + 60 SWA layers) and
 * section 2 (layer-wise overlap of a step; the whole step replayed as a
 * graph).  Same contract as phs_attn_decode_hybrid_stack with do_append = 1:
 * every layer's k_new/v_new ([batch][Hkv][D] bf16, 16-byte aligned,
 * required) is written into slot seq_lens[b]-1 of its page (Full, through
 * the shared block_table) or into ring slot ring_pos[b] (SWA), and attended
 * as the newest token -- the kernels take it from k_new/v_new instead of
 * reading it back.  Launches: one split-KV launch for up to 16 Full layers
 * at once and one persistent launch for up to 64 SWA layers, whose warps
 * also run the Full layers' cross-split merges after their SWA work (a
 * stack without SWA layers gets a merge launch instead).  A 70-layer
 * stack of 10 Full + 60 SWA layers: two launches per step instead of
 * twenty-three.  A small
 * step (every request in one split, fewer than 16 Full and 64 SWA layers,
 * and all its CTAs in one wave) goes in a single launch.  The Full layers'
 * partials live side by side, so the workspace is
 * phs_hybrid_stack_fused_workspace_bytes (256-byte aligned).
 * Outputs and pool contents equal those of the unfused call.
 * Errors as phs_attn_decode_hybrid_stack (PHS_EINVAL also for a missing
 * k_new/v_new); block-table ids must be valid for every Full pool.  With
 * page_refcount, a new token whose page is shared is neither written nor
 * attended from k_new/v_new (the layer attends to the page as it stands,
 * as the unfused call does after its refused append) and PHS_ESHARED is
 * recorded.
 * ---------------------------------------------------------------------- */
int phs_attn_decode_hybrid_stack_fused(const phs_layer *layers, int32_t num_layers,
                                       int32_t num_q_heads, int32_t batch,
                                       const int32_t *block_table, int32_t max_pages_per_seq,
                                       const int32_t *page_refcount,
                                       const int32_t *seq_lens, int32_t max_seq_len,
                                       const int32_t *ring_ids, const int32_t *ring_pos,
                                       float softmax_scale, int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       void *stream);

/* Workspace of phs_attn_decode_hybrid_stack_fused: one split-partials area
 * per Full layer (0 when num_full_layers <= 0). */
size_t phs_hybrid_stack_fused_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t max_seq_len, int32_t num_full_layers);

/* KV tokens held by a hybrid stack (host arrays in, host results out):
 * Full layers hold seq_lens[b] tokens per request, SWA layers
 * min(seq_lens[b], window).  Source: MiMo page, section 1 (the 10/60 stack
 * holds about 1/7 of an all-Full stack's KV at long lengths). */
int phs_hybrid_kv_tokens(const int32_t *layer_is_full_host, int32_t num_layers,
                         const int32_t *seq_lens_host, int32_t batch, int32_t window,
                         int64_t *full_tokens, int64_t *swa_tokens);

/* Plain device-to-device copy kernel (16-byte vector loads and stores), the
 * in-run HBM bandwidth yardstick.  dst and src 16-byte aligned, bytes a
 * multiple of 16. */
int phs_copy_d2d(void *dst, const void *src, size_t bytes, void *stream);

/* Streaming read of a device buffer, the in-run read-side HBM yardstick
 * (the decode kernels read almost only, and a read stream runs faster than
 * a copy's combined read + write rate).  XORs every 32-bit word of
 * src[0, bytes) into *dev_sink (device, uint32, 4-byte aligned; not
 * cleared first).  src 16-byte aligned, bytes a multiple of 16. */
int phs_read_checksum(const void *src, size_t bytes, uint32_t *dev_sink, void *stream);

/* ========================================================================
 * Host-side cache bookkeeping that produces the block tables and page
 * reference counts the kernels consume.  Host memory in, host memory out;
 * every object is thread-safe (one mutex per object).
 * ====================================================================== */

/* Refcounted page allocator over the pages of a Full pool.
 * Source: "Kimi K3 context caching" page, section 1: requests that hit a
 * shared prefix increment the reference count of its physical blocks in the
 * page table (copy on write); only a request's own new tokens get new
 * blocks. */
typedef struct phs_page_allocator phs_page_allocator;
phs_page_allocator *phs_page_allocator_create(int64_t num_pages); /* NULL on bad size */
/* Releases the caller's handle; a radix tree created on the allocator keeps
 * it alive (the object is freed when the last tree using it is destroyed). */
void phs_page_allocator_destroy(phs_page_allocator *a);
/* n fresh pages with count 1 into out_pages (host); PHS_ENOSPACE if fewer free. */
int phs_page_alloc(phs_page_allocator *a, int32_t n, int32_t *out_pages);
/* +1 / -1 on each listed page (all must be live, else PHS_ERANGE and no
 * change); pages reaching 0 return to the free list. */
int phs_page_incref(phs_page_allocator *a, const int32_t *pages, int32_t n);
int phs_page_decref(phs_page_allocator *a, const int32_t *pages, int32_t n);
int64_t phs_page_free_count(phs_page_allocator *a);
/* Snapshot of all counts into out (host int32 [num_pages]); copy it to the
 * device for the refcount check of phs_kv_append_paged. */
int phs_page_refcounts(phs_page_allocator *a, int32_t *out);
/* Copy on write before appending into `page`: if its count is 1 the page is
 * returned unchanged; otherwise a fresh page (count 1) is allocated, the
 * shared page loses one reference, and the fresh id is returned -- the
 * caller copies the contents with phs_copy_pages and updates its table. */
int phs_page_cow(phs_page_allocator *a, int32_t page, int32_t *out_page);

/* Device copy of whole pages (K and V, all heads): dst_pages[i] <- src_pages[i]
 * (device int32 arrays).  Out-of-range ids record PHS_ERANGE. */
int phs_copy_pages(const phs_paged_pool *pool, const int32_t *src_pages,
                   const int32_t *dst_pages, int32_t n, int32_t *dev_status, void *stream);

/* Radix prefix tree over whole pages.
 * Source: "Kimi K3 context caching" page, sections 1 and 3 (global radix
 * tree, longest-prefix match, insert of newly computed blocks) and "Xiaomi
 * MiMo-V2.5 inference system" page, section 2 (prefix-tree rebuild: each
 * node carries the Full segment index and the SWA mapping).  Only whole
 * pages are cached and shared.  The tree holds one reference on each Full
 * page it caches (in `alloc`) and on each SWA segment page it maps (in
 * `swa_alloc`, may be NULL when no SWA KV is cached; must differ from
 * `alloc`).  An SWA segment page is a 16-token snapshot of the SWA-layer KV
 * of one cached page (see phs_swa_ring_save); its id means the same page
 * in every SWA layer's segment pool. */
typedef struct phs_radix_tree phs_radix_tree;
phs_radix_tree *phs_radix_create(phs_page_allocator *alloc, phs_page_allocator *swa_alloc,
                                 int32_t page_size);
void phs_radix_destroy(phs_radix_tree *t); /* drops the tree's page references */
/* Longest cached whole-page prefix of tokens[0..n): its page ids go to
 * out_pages (capacity max_pages, else PHS_ESHAPE), their number to
 * *out_num_pages (matched tokens = that * page_size).  Each matched page
 * gets one more reference (the caller's request); release with
 * phs_page_decref when the request ends. */
int phs_radix_match(phs_radix_tree *t, const int32_t *tokens, int64_t n, int32_t *out_pages,
                    int32_t max_pages, int32_t *out_num_pages);
/* Same, cut back to the window-safe length of a hybrid stack.  Source:
 * "Xiaomi MiMo-V2.5 inference system" page, section 2 (prefix tree
 * rebuild): a match is valid only where at least the last W tokens still
 * have valid SWA slots.  Here: the longest page-aligned L <= match whose
 * last min(L, window) tokens all lie in pages that map an SWA segment page
 * (window a multiple of page_size, else PHS_EUNSUPPORTED).  Returns the
 * L / page_size Full pages as phs_radix_match does, and in out_swa_pages
 * (capacity max_swa_pages, else PHS_ESHAPE) the segment pages of that last
 * window, in token order: min(L, window) / page_size of them, the first
 * holding tokens [L - min(L, window), ... + page_size).  Each returned
 * segment page gets one more reference in swa_alloc (the caller's: release
 * it with phs_page_decref once phs_swa_ring_seed has copied it). */
int phs_radix_match_window_safe(phs_radix_tree *t, const int32_t *tokens, int64_t n,
                                int32_t window, int32_t *out_pages, int32_t max_pages,
                                int32_t *out_num_pages, int32_t *out_swa_pages,
                                int32_t max_swa_pages, int32_t *out_num_swa_pages);
/* Cache the whole pages of tokens[0..n) with page ids pages[0..n/page_size).
 * Positions already cached keep the tree's pages (the caller's ids for them
 * are not referenced); new pages get a tree reference.  swa_pages (host,
 * [n/page_size], may be NULL = none) gives, per page, the SWA segment page
 * holding that page's SWA-layer KV, or -1; a cached page that has none
 * takes the caller's (with a tree reference in swa_alloc), one that has one
 * keeps it.  A finished request typically saves the pages of its last
 * window (phs_swa_ring_save) and passes their segment ids here. */
int phs_radix_insert(phs_radix_tree *t, const int32_t *tokens, int64_t n, const int32_t *pages,
                     const int32_t *swa_pages);
/* Evict least-recently-used leaves whose pages (Full and SWA segment) only
 * the tree references until at least `pages` Full pages were freed or none
 * is evictable; their SWA segment pages are released too. */
int phs_radix_evict(phs_radix_tree *t, int64_t pages, int64_t *out_freed);
int64_t phs_radix_cached_pages(phs_radix_tree *t);
/* Window-safe length as a plain function: the largest L <= match_len, L a
 * multiple of align, with swa_valid[t] != 0 (host uint8) for every t in
 * [max(0, L - window), L); 0 if none. */
int64_t phs_window_safe_len(const uint8_t *swa_valid, int64_t match_len, int32_t window,
                            int32_t align);

/* ------------------------------------------------------------------------
 * SWA segment pages: snapshots of ring contents by whole pages, so that a
 * cached prefix can seed a new request's ring.
 * Source: "Xiaomi MiMo-V2.5 inference system" page, section 2 (dual pools:
 * the SWA pool keeps only each request's last W tokens; a prefix-cache hit
 * is usable only at a window-safe length, and the node's SWA mapping says
 * where that window's SWA KV is).
 * rings / segs: host arrays of num_layers descriptors, one per SWA layer
 * (same window, Hkv and head_dim throughout); segs[l] is a segment pool in
 * the Full-pool layout [num_seg_pages][Hkv][16][D] bf16.  A segment page id
 * names the same page in every layer.  Token t of a request of length n
 * sits at ring slot (ring_pos - (n - 1 - t)) mod W, as for decode.
 *
 * phs_swa_ring_save: for each entry i < count (device int32 arrays), copies
 * tokens [16 * page_index[i], 16 * page_index[i] + 16) of the request whose
 * ring is ring_ids[i], newest slot ring_pos[i], length seq_lens[i], into
 * segment page seg_pages[i], in every layer.  The page must lie inside the
 * ring's window [n - min(n, W), n), else PHS_ERANGE (entry skipped).
 *
 * phs_swa_ring_seed: for each request b < batch, writes the last
 * min(n, W) tokens (n = seq_lens[b]) into ring ring_ids[b] (NULL =
 * identity) so that its newest token sits at slot ring_pos[b]; token t is
 * read from segment page seg_table[b][t / 16 - first] (device int32
 * [batch][max_seg_pages]), first = (n - min(n, W)) / 16, at slot t % 16.
 * Out-of-range ids record PHS_ERANGE and skip the token.  After seeding, a
 * decode step appends token n at slot (ring_pos[b] + 1) mod W.
 * ---------------------------------------------------------------------- */
int phs_swa_ring_save(const phs_ring_pool *rings, const phs_paged_pool *segs, int32_t num_layers,
                      const int32_t *ring_ids, const int32_t *ring_pos, const int32_t *seq_lens,
                      const int32_t *page_index, const int32_t *seg_pages, int32_t count,
                      int32_t *dev_status, void *stream);
int phs_swa_ring_seed(const phs_ring_pool *rings, const phs_paged_pool *segs, int32_t num_layers,
                      const int32_t *ring_ids, const int32_t *ring_pos, const int32_t *seq_lens,
                      const int32_t *seg_table, int32_t max_seg_pages, int32_t batch,
                      int32_t *dev_status, void *stream);

const char *phs_status_str(int status);
int32_t phs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PHS_H_ */
