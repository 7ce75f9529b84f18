/*
 * phs_oracle.c -- the CPU oracle for paged hybrid sliding-window decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it.  It shares
 * no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Sources of what is computed (page title, section):
 *  - "Xiaomi MiMo-V2.5 inference system" (IT Home news page), section 1
 *    "why Hybrid SWA": 70 layers, 10 Full-attention, 60 sliding-window of
 *    128 tokens; SWA layers keep only the most recent W tokens.
 *  - same page, section 2, "KVCache system rebuild / dual pools": a Full KV
 *    pool that grows on demand and an SWA KV pool that is a ring buffer of
 *    capacity W per request (storage O(W)); the Full index is authoritative.
 *  - "Kimi K3 context caching" page (xdnf.cn), section 1 "global radix tree":
 *    KV lives in non-contiguous physical blocks reached through a page
 *    table; requests sharing a prefix share blocks by reference count and
 *    new tokens get new blocks of their own.
 *  - "Kimi K2.5 architecture deep dive" page (framerc.cn), sections 2.2
 *    (turn one: warm-zone KV stored as INT8 with block-wise quantisation) and
 *    2.3 (one scale calibrated per group of 32 tokens).
 *  - Attention itself is the textbook single-query softmax(q K^T * scale) V,
 *    one query token per request, evaluated over the logical sequence.
 *
 * Precision: every floating-point reduction is done in double.  bf16 inputs
 * are widened exactly.  The INT8 quantiser is the exception: its steps are
 * written in explicit IEEE single precision, because the codes and scales it
 * produces are compared byte for byte.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *  - seq_lens passed here are the lengths AFTER this step's append, so the
 *    query of the new token attends to itself.
 *  - query head i uses KV head i / (Hq / Hkv) (contiguous groups).
 *  - the ring's newest token sits at slot ring_pos[b]; token t of a request
 *    of length n sits at slot (ring_pos - (n - 1 - t)) mod W; the window is
 *    the last min(n, W) tokens, including the new one.
 *  - INT8: one scale per (32 consecutive tokens, KV head), separately for K
 *    and V; s = absmax / 127 in fp32; code = round-half-even(x / s) clamped
 *    to [-127, 127]; an all-zero group gets s = 0 and codes 0; dequantised
 *    value = (float)code * s in fp32.
 *  - INT8 region: tokens [0, qlen_b) come from INT8 pages through the
 *    32-token table qtable[b][t / 32]; tokens [qlen_b, n_b) come from bf16
 *    pages through block_table[b][t / P] (the block table is indexed by the
 *    absolute token position).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ERANGE -3
#define ORC_ESHARED -4

/* bf16 -> single: a bf16 value is the upper half of a binary32 value. */
static float bf16_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double bf16_to_double(uint16_t h) { return (double)bf16_to_float(h); }

/* Non-negative remainder. */
static int64_t pos_mod(int64_t a, int64_t m) {
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

int phs_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * KV append into the paged Full pool (Kimi K3 page, section 1: the new token
 * goes to a block owned by this request alone; MiMo page, section 2: the
 * Full pool grows on demand).
 * Pool layout [num_pages][Hkv][P][D] bf16; k_new/v_new [B][Hkv][D].
 * The token index written is n_b - 1.  If page_refcount is given, a page
 * whose count is not 1 is shared and is not written (status ORC_ESHARED).
 * ---------------------------------------------------------------------- */
int phs_oracle_append_paged(uint16_t *k_pool, uint16_t *v_pool, int64_t num_pages,
                            int P, int Hkv, int D, const uint16_t *k_new,
                            const uint16_t *v_new, const int32_t *block_table,
                            int max_pages, const int32_t *seq_lens, int B,
                            const int32_t *page_refcount) {
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int64_t n = seq_lens[b];
        if (n < 1) continue; /* nothing appended for an empty request */
        int64_t t = n - 1; /* the new token's position */
        int64_t lp = t / P;
        if (lp >= max_pages) { status = ORC_ERANGE; continue; }
        int64_t page = block_table[(int64_t)b * max_pages + lp];
        if (page < 0 || page >= num_pages) { status = ORC_ERANGE; continue; }
        if (page_refcount && page_refcount[page] != 1) { status = ORC_ESHARED; continue; }
        int64_t slot = t % P;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t dst = ((page * Hkv + h) * P + slot) * D + d;
                int64_t src = ((int64_t)b * Hkv + h) * D + d;
                k_pool[dst] = k_new[src];
                v_pool[dst] = v_new[src];
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * KV append into the SWA ring (MiMo page, section 2: ring buffer of capacity
 * W, window-based eviction).  Writing slot ring_pos[b] overwrites the token
 * that left the window.  Ring layout [num_rings][Hkv][W][D] bf16.
 * ring_ids may be NULL (request b owns ring b).
 * ---------------------------------------------------------------------- */
int phs_oracle_append_ring(uint16_t *k_ring, uint16_t *v_ring, int64_t num_rings, int W,
                           int Hkv, int D, const uint16_t *k_new, const uint16_t *v_new,
                           const int32_t *ring_ids, const int32_t *ring_pos, int B) {
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int64_t r = ring_ids ? ring_ids[b] : b;
        int64_t slot = ring_pos[b];
        if (r < 0 || r >= num_rings || slot < 0 || slot >= W) { status = ORC_ERANGE; continue; }
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t dst = ((r * Hkv + h) * W + slot) * D + d;
                int64_t src = ((int64_t)b * Hkv + h) * D + d;
                k_ring[dst] = k_new[src];
                v_ring[dst] = v_new[src];
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * Block-32 INT8 quantiser (Kimi K2.5 page, sections 2.2 and 2.3: INT8 with
 * block-wise quantisation, one scale calibrated per group of 32 tokens).
 * One group = 32 consecutive tokens x D dims of one KV head, K and V
 * separately.  Steps in IEEE single precision:
 *   a = max |x| ; s = a / 127 ; code = clamp(rint(x / s), -127, 127)
 * with rint rounding half to even (the default rounding mode), and s = 0,
 * codes 0 when a == 0.
 * Source: bf16 pages [num_pages][Hkv][P][D] through src_table[b][t / P].
 * Destination: codes [num_qpages][Hkv][32][D] int8, scales
 * [num_qpages][Hkv] fp32, through dst_qtable[b][j] for 32-token block j.
 * Blocks j in [first_qblock[b], first_qblock[b] + num_qblocks[b]).
 * ---------------------------------------------------------------------- */
static float quant_scale(float absmax) { return absmax / 127.0f; }

static int8_t quant_code(float x, float s) {
    if (s == 0.0f) return 0;
    float r = rintf(x / s);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int8_t)r;
}

int phs_oracle_quant_int8_block32(const uint16_t *k_pool, const uint16_t *v_pool,
                                  int64_t num_pages, int P, int Hkv, int D,
                                  const int32_t *src_table, int src_max_pages,
                                  int8_t *k_codes, int8_t *v_codes, float *k_scale,
                                  float *v_scale, int64_t num_qpages,
                                  const int32_t *dst_qtable, int dst_max_qpages,
                                  const int32_t *first_qblock, const int32_t *num_qblocks,
                                  int B) {
    const int Q = 32;
    int status = ORC_OK;
    if (Q % P != 0 && P % Q != 0) return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        for (int64_t j = first_qblock[b]; j < (int64_t)first_qblock[b] + num_qblocks[b]; ++j) {
            if (j < 0 || j >= dst_max_qpages) { status = ORC_ERANGE; continue; }
            int64_t qp = dst_qtable[(int64_t)b * dst_max_qpages + j];
            if (qp < 0 || qp >= num_qpages) { status = ORC_ERANGE; continue; }
            for (int h = 0; h < Hkv; ++h) {
                for (int which = 0; which < 2; ++which) {
                    const uint16_t *src = which ? v_pool : k_pool;
                    int8_t *codes = which ? v_codes : k_codes;
                    float *scales = which ? v_scale : k_scale;
                    /* gather the 32 x D group through the block table */
                    float x[32 * 256];
                    int ok = 1;
                    if (D > 256) return ORC_EINVAL;
                    for (int tt = 0; tt < Q && ok; ++tt) {
                        int64_t t = j * Q + tt;
                        int64_t lp = t / P;
                        if (lp >= src_max_pages) { ok = 0; break; }
                        int64_t page = src_table[(int64_t)b * src_max_pages + lp];
                        if (page < 0 || page >= num_pages) { ok = 0; break; }
                        for (int d = 0; d < D; ++d)
                            x[tt * D + d] = bf16_to_float(src[((page * Hkv + h) * P + t % P) * D + d]);
                    }
                    if (!ok) { status = ORC_ERANGE; continue; }
                    float a = 0.0f;
                    for (int e = 0; e < Q * D; ++e) {
                        float m = fabsf(x[e]);
                        if (m > a) a = m;
                    }
                    float s = quant_scale(a);
                    scales[qp * Hkv + h] = s;
                    for (int tt = 0; tt < Q; ++tt)
                        for (int d = 0; d < D; ++d)
                            codes[((qp * Hkv + h) * Q + tt) * D + d] = quant_code(x[tt * D + d], s);
                }
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * Attention of one query row over a gathered logical sequence, in double:
 *   s_t = scale * sum_d q[d] K[t][d];  p_t = exp(s_t - max_u s_u);
 *   o = sum_t p_t V[t] / sum_t p_t.
 * K and V are given as callbacks that return row t widened to double.
 * ---------------------------------------------------------------------- */
typedef void (*row_fn)(const void *ctx, int64_t t, int is_v, double *row);

static void attend_one(const double *q, int D, int64_t t0, int64_t t1, double scale,
                       row_fn get_row, const void *ctx, double *out) {
    int64_t n = t1 - t0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n <= 0) return;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double row[256];
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        get_row(ctx, t, 0, row);
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * row[d];
        s[t - t0] = acc * scale;
        if (s[t - t0] > m) m = s[t - t0];
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        double p = exp(s[t - t0] - m);
        l += p;
        get_row(ctx, t, 1, row);
        for (int d = 0; d < D; ++d) out[d] += p * row[d];
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    free(s);
}

/* Logical sequence of request b, KV head h, in the Full pool (bf16 pages and
 * an optional INT8 prefix). */
typedef struct {
    const uint16_t *k_pool, *v_pool;
    int64_t num_pages;
    int P, Hkv, D;
    const int32_t *bt_row; /* block_table + b * max_pages */
    int max_pages;
    const int8_t *k_codes, *v_codes;
    const float *k_scale, *v_scale;
    int64_t num_qpages;
    const int32_t *qt_row; /* qtable + b * max_qpages */
    int max_qpages;
    int64_t qlen;
    int h;
    int *bad; /* set to 1 on an out-of-range index */
} full_ctx;

static void full_row(const void *vctx, int64_t t, int is_v, double *row) {
    const full_ctx *c = (const full_ctx *)vctx;
    if (t < c->qlen) {
        int64_t j = t / 32;
        int64_t qp = j < c->max_qpages ? c->qt_row[j] : -1;
        if (qp < 0 || qp >= c->num_qpages) {
            *c->bad = 1;
            for (int d = 0; d < c->D; ++d) row[d] = 0.0;
            return;
        }
        const int8_t *codes = is_v ? c->v_codes : c->k_codes;
        float s = (is_v ? c->v_scale : c->k_scale)[qp * c->Hkv + c->h];
        const int8_t *r = codes + ((qp * c->Hkv + c->h) * 32 + t % 32) * c->D;
        for (int d = 0; d < c->D; ++d) row[d] = (double)((float)r[d] * s);
        return;
    }
    int64_t lp = t / c->P;
    int64_t page = lp < c->max_pages ? c->bt_row[lp] : -1;
    if (page < 0 || page >= c->num_pages) {
        *c->bad = 1;
        for (int d = 0; d < c->D; ++d) row[d] = 0.0;
        return;
    }
    const uint16_t *pool = is_v ? c->v_pool : c->k_pool;
    const uint16_t *r = pool + ((page * c->Hkv + c->h) * c->P + t % c->P) * c->D;
    for (int d = 0; d < c->D; ++d) row[d] = bf16_to_double(r[d]);
}

/* ------------------------------------------------------------------------
 * Full-attention decode over the paged pool.  q [B][Hq][D] bf16 -> out
 * [B][Hq][D] double.  rows (nullable) selects which requests to compute;
 * the others are left untouched.  qlens == NULL means no INT8 region.
 * ---------------------------------------------------------------------- */
int phs_oracle_decode_full_paged(const uint16_t *q, int B, int Hq, int Hkv, int D,
                                 const uint16_t *k_pool, const uint16_t *v_pool,
                                 int64_t num_pages, int P, const int32_t *block_table,
                                 int max_pages, const int32_t *seq_lens,
                                 const int8_t *k_codes, const int8_t *v_codes,
                                 const float *k_scale, const float *v_scale,
                                 int64_t num_qpages, const int32_t *qtable, int max_qpages,
                                 const int32_t *qlens, double scale, const int32_t *rows,
                                 int nrows, double *out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D > 256) return ORC_EINVAL;
    const int G = Hq / Hkv;
    int nsel = rows ? nrows : B;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t w = 0; w < (int64_t)nsel * Hq; ++w) {
        int b = rows ? rows[w / Hq] : (int)(w / Hq);
        int i = (int)(w % Hq);
        int h = i / G;
        int local_bad = 0;
        full_ctx c = {k_pool, v_pool, num_pages, P, Hkv, D,
                      block_table + (int64_t)b * max_pages, max_pages,
                      k_codes, v_codes, k_scale, v_scale, num_qpages,
                      qtable ? qtable + (int64_t)b * max_qpages : NULL, max_qpages,
                      qlens ? qlens[b] : 0, h, &local_bad};
        double qd[256];
        for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[((int64_t)b * Hq + i) * D + d]);
        attend_one(qd, D, 0, seq_lens[b], scale, full_row, &c, out + ((int64_t)b * Hq + i) * D);
        bad |= local_bad;
    }
    return bad ? ORC_ERANGE : ORC_OK;
}

/* Logical sequence of request b, KV head h, in its SWA ring. */
typedef struct {
    const uint16_t *k_ring, *v_ring;
    int64_t ring;
    int W, Hkv, D, h;
    int64_t newest_slot, n;
} ring_ctx;

static void ring_row(const void *vctx, int64_t t, int is_v, double *row) {
    const ring_ctx *c = (const ring_ctx *)vctx;
    int64_t slot = pos_mod(c->newest_slot - (c->n - 1 - t), c->W);
    const uint16_t *base = is_v ? c->v_ring : c->k_ring;
    const uint16_t *r = base + ((c->ring * c->Hkv + c->h) * c->W + slot) * c->D;
    for (int d = 0; d < c->D; ++d) row[d] = bf16_to_double(r[d]);
}

/* ------------------------------------------------------------------------
 * Sliding-window decode over the ring (MiMo page, section 1: an SWA layer
 * attends to the most recent W tokens; section 2: ring of capacity W).
 * Window = tokens [max(0, n - W), n).
 * ---------------------------------------------------------------------- */
int phs_oracle_decode_swa_ring(const uint16_t *q, int B, int Hq, int Hkv, int D,
                               const uint16_t *k_ring, const uint16_t *v_ring,
                               int64_t num_rings, int W, const int32_t *ring_ids,
                               const int32_t *ring_pos, const int32_t *seq_lens,
                               double scale, const int32_t *rows, int nrows, double *out) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D > 256 || W <= 0) return ORC_EINVAL;
    const int G = Hq / Hkv;
    int nsel = rows ? nrows : B;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t w = 0; w < (int64_t)nsel * Hq; ++w) {
        int b = rows ? rows[w / Hq] : (int)(w / Hq);
        int i = (int)(w % Hq);
        int64_t r = ring_ids ? ring_ids[b] : b;
        int64_t n = seq_lens[b];
        if (r < 0 || r >= num_rings || ring_pos[b] < 0 || ring_pos[b] >= W) {
            bad = 1;
            continue;
        }
        ring_ctx c = {k_ring, v_ring, r, W, Hkv, D, i / G, ring_pos[b], n};
        double qd[256];
        for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[((int64_t)b * Hq + i) * D + d]);
        int64_t t0 = n > W ? n - W : 0;
        attend_one(qd, D, t0, n, scale, ring_row, &c, out + ((int64_t)b * Hq + i) * D);
    }
    return bad ? ORC_ERANGE : ORC_OK;
}

/* ------------------------------------------------------------------------
 * SWA segment pages (MiMo page, section 2: a prefix-cache hit of a hybrid
 * stack is usable only at a window-safe length, and the tree's SWA mapping
 * says where that window's SWA KV lives).  A segment page holds the
 * SWA-layer KV of P consecutive tokens, layout [num_seg][Hkv][P][D] bf16.
 * In a ring of W slots, token t of a request of length n sits at slot
 * (ring_pos - (n - 1 - t)) mod W (as for decode).
 *
 * save: entry i copies tokens [P * page_index[i], P * page_index[i] + P) of
 * the request whose ring is ring_ids[i] (newest slot ring_pos[i], length
 * seq_lens[i]) into segment page seg_pages[i].  Every one of those tokens
 * must be in the ring's window [n - min(n, W), n) (else ORC_ERANGE, entry
 * skipped).
 * ---------------------------------------------------------------------- */
int phs_oracle_swa_ring_save(const uint16_t *k_ring, const uint16_t *v_ring, int64_t num_rings,
                             int W, int Hkv, int D, uint16_t *k_seg, uint16_t *v_seg,
                             int64_t num_seg, int P, const int32_t *ring_ids,
                             const int32_t *ring_pos, const int32_t *seq_lens,
                             const int32_t *page_index, const int32_t *seg_pages, int count) {
    int status = ORC_OK;
    for (int i = 0; i < count; ++i) {
        int64_t r = ring_ids[i], pos = ring_pos[i], n = seq_lens[i], sp = seg_pages[i];
        int64_t first = (int64_t)page_index[i] * P;
        int64_t lo = n - (n < W ? n : W);
        if (r < 0 || r >= num_rings || pos < 0 || pos >= W || sp < 0 || sp >= num_seg ||
            page_index[i] < 0 || first < lo || first + P > n) {
            status = ORC_ERANGE;
            continue;
        }
        for (int64_t t = first; t < first + P; ++t) {
            int64_t slot = pos_mod(pos - (n - 1 - t), W);
            for (int h = 0; h < Hkv; ++h)
                for (int d = 0; d < D; ++d) {
                    int64_t src = ((r * Hkv + h) * W + slot) * D + d;
                    int64_t dst = ((sp * Hkv + h) * P + t % P) * D + d;
                    k_seg[dst] = k_ring[src];
                    v_seg[dst] = v_ring[src];
                }
        }
    }
    return status;
}

/* seed: request b (length n = seq_lens[b], ring ring_ids[b] or b when
 * ring_ids is NULL, newest slot ring_pos[b]) gets the last min(n, W) tokens
 * written into its ring; token t is read from segment page
 * seg_table[b][t / P - first] at slot t % P, first = (n - min(n, W)) / P.
 * A token whose page id is missing or out of range is skipped (ORC_ERANGE). */
int phs_oracle_swa_ring_seed(uint16_t *k_ring, uint16_t *v_ring, int64_t num_rings, int W,
                             int Hkv, int D, const uint16_t *k_seg, const uint16_t *v_seg,
                             int64_t num_seg, int P, const int32_t *ring_ids,
                             const int32_t *ring_pos, const int32_t *seq_lens,
                             const int32_t *seg_table, int max_seg, int B) {
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int64_t r = ring_ids ? ring_ids[b] : b, pos = ring_pos[b], n = seq_lens[b];
        if (r < 0 || r >= num_rings || pos < 0 || pos >= W || n < 0) {
            status = ORC_ERANGE;
            continue;
        }
        int64_t lo = n - (n < W ? n : W);
        int64_t first = lo / P;
        for (int64_t t = lo; t < n; ++t) {
            int64_t j = t / P - first;
            int64_t sp = j < max_seg ? seg_table[(int64_t)b * max_seg + j] : -1;
            if (sp < 0 || sp >= num_seg) {
                status = ORC_ERANGE;
                continue;
            }
            int64_t slot = pos_mod(pos - (n - 1 - t), W); /* seed: ring slot of token t */
            for (int h = 0; h < Hkv; ++h)
                for (int d = 0; d < D; ++d) {
                    int64_t src = ((sp * Hkv + h) * P + t % P) * D + d;
                    int64_t dst = ((r * Hkv + h) * W + slot) * D + d;
                    k_ring[dst] = k_seg[src];
                    v_ring[dst] = v_seg[src];
                }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * KV tokens stored by a layer stack (MiMo page, section 1: SWA layers keep
 * only the last W tokens, so the 10 Full + 60 SWA stack stores about 1/7 of
 * an all-Full stack at long lengths).  Per layer and request: a Full layer
 * stores n_b tokens, an SWA layer min(n_b, W).  Returns the sum over layers
 * and requests; multiply by Hkv * D * 2 (K and V) * element bytes for bytes.
 * ---------------------------------------------------------------------- */
int64_t phs_oracle_kv_tokens_stored(const int32_t *layer_is_full, int L,
                                    const int32_t *seq_lens, int B, int W) {
    int64_t total = 0;
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b) {
            int64_t n = seq_lens[b];
            total += layer_is_full[l] ? n : (n < W ? n : W);
        }
    return total;
}
