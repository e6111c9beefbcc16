/*
 * oracle/attn_ref.c -- plain fp64 CPU oracle for the paged-KV attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file; only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library under paged_kv_cache_token_gb300/csrc/.
 *
 * What it computes is the plain definition of the method's result:
 *
 *   * causal softmax attention of each new query row over ALL keys of its
 *     request up to and including its own position, on contiguous K/V
 *     (no pages, no chunks, no splits) -- hotelren.com/news/6181127 §1.1
 *     (position i depends on 0..i), §2.1 (upper triangle masked to -inf
 *     before a row-wise softmax, then times V), §3.1 (decode: append the new
 *     K,V, then score against all S+t keys) and the §5.1 skeleton
 *     (softmax(q K_all^T) V_all);  niuwancheng.cn "11. chunked prefill and
 *     unified scheduling", section "cutting long input into chunks" (a chunk
 *     reads the earlier chunks' K/V like a decode and the result is the same
 *     as one-shot prefill) -- so one-shot attention over the contiguous
 *     sequence IS the expected output of every chunked / paged step;
 *
 *   * the page contents that appending new K/V through a block table must
 *     produce -- lshu.cn/news/11576 §2.2 (K/V written by page index into a
 *     pre-allocated pool of fixed-size pages), §2.3 (16 tokens per block);
 *
 *   * the per-token KV byte count 2 x L x n_kv_heads x d_head x bytes --
 *     hotelren.com/news/6181127 §2.3;
 *
 *   * the INT8 codes of a per-channel quantised KV cache and attention over
 *     the values they stand for -- wmrh.cn/news/64708 §4.3, §5.4.
 *
 * Arithmetic is IEEE double throughout; inputs arrive as the exact 16-bit
 * patterns (bf16 or IEEE binary16) and are widened here, exactly.
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math: IEEE semantics).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PAGE_TOKENS 16 /* lshu.cn/news/11576 §2.3: 16 tokens per block */

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

/* ---------------------------------------------------------------------- */
/* Exact widening of 16-bit float patterns to double.                      */
/* ---------------------------------------------------------------------- */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double mag;
    if (e == 0xFF)
        mag = f ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexp((double)f, -126 - 7); /* subnormal: 0.f x 2^-126 */
    else
        mag = ldexp((double)(128 + f), e - 127 - 7); /* 1.f x 2^(e-127) */
    return sign ? -mag : mag;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0x1F)
        mag = f ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexp((double)f, -14 - 10);
    else
        mag = ldexp((double)(1024 + f), e - 15 - 10);
    return sign ? -mag : mag;
}

static double widen(int dtype, uint16_t x)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(x) : oracle_fp16_to_double(x);
}

/* Widen a whole array (used by tests to compare against the same decoding). */
int oracle_widen(int dtype, const uint16_t* src, int64_t n, double* dst)
{
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16) return -1;
    for (int64_t i = 0; i < n; ++i) dst[i] = widen(dtype, src[i]);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Per-token KV bytes: 2 (K and V) x layers x kv heads x head dim x bytes. */
/* hotelren.com/news/6181127 §2.3.                                         */
/* ---------------------------------------------------------------------- */
int64_t oracle_kv_bytes_per_token(int64_t layers, int64_t n_kv_heads, int64_t d_head,
                                  int64_t bytes_per_elem)
{
    return 2 * layers * n_kv_heads * d_head * bytes_per_elem;
}

/* ---------------------------------------------------------------------- */
/* Causal softmax attention over contiguous K/V, any set of query rows.    */
/*                                                                         */
/* q     [n_rows, Hq, D]   16-bit patterns                                  */
/* pos   [n_rows]          absolute position of each query row; row i      */
/*                         attends keys 0..pos[i] inclusive                 */
/* k, v  [n_kv, Hkv, D]    16-bit patterns, the request's whole sequence   */
/* out   [n_rows, Hq, D]   double                                           */
/* Query head h reads KV head h / (Hq / Hkv) (consecutive query heads share */
/* one KV head; the pages do not fix the grouping).                         */
/*                                                                         */
/* For each (row, head):  s_j = scale * <q, k_j>  (j = 0..pos)             */
/*                        m = max_j s_j,  w_j = exp(s_j - m),  Z = sum w_j */
/*                        out = sum_j (w_j / Z) v_j                         */
/* Returns 0, -1 on a bad argument (nothing written), -3 when out of memory. */
/* ---------------------------------------------------------------------- */
/* The same, on K/V already widened to double (kd, vd: [n_kv, Hkv, D]). */
static int attention_core(int dtype, const uint16_t* q, const int32_t* pos, int32_t n_rows,
                          const double* kd, const double* vd, int32_t Hq, int32_t Hkv,
                          int32_t D, double scale, double* out)
{
    const int32_t group = Hq / Hkv;
    const int64_t units = (int64_t)n_rows * Hq;
#pragma omp parallel
    {
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int32_t i = (int32_t)(u / Hq);
            const int32_t h = (int32_t)(u % Hq);
            const int32_t g = h / group;
            const int32_t p = pos[i];
            for (int32_t d = 0; d < D; ++d) qd[d] = widen(dtype, q[((int64_t)i * Hq + h) * D + d]);

            /* pass 1: the row maximum of the scores s_j = scale * <q, k_j>, j = 0..p */
            double m = -INFINITY;
            for (int32_t j = 0; j <= p; ++j) {
                const double* kj = kd + ((int64_t)j * Hkv + g) * D;
                double s = 0.0;
                for (int32_t d = 0; d < D; ++d) s += qd[d] * kj[d];
                s *= scale;
                if (s > m) m = s;
            }
            /* pass 2: weights w_j = exp(s_j - m), normaliser Z, weighted sum of V */
            double* o = out + ((int64_t)i * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            double Z = 0.0;
            for (int32_t j = 0; j <= p; ++j) {
                const double* kj = kd + ((int64_t)j * Hkv + g) * D;
                const double* vj = vd + ((int64_t)j * Hkv + g) * D;
                double s = 0.0;
                for (int32_t d = 0; d < D; ++d) s += qd[d] * kj[d];
                s *= scale;
                const double w = exp(s - m);
                Z += w;
                for (int32_t d = 0; d < D; ++d) o[d] += w * vj[d];
            }
            for (int32_t d = 0; d < D; ++d) o[d] /= Z;
        }
        free(qd);
    }
    return 0;
}

static int rows_ok(int dtype, const int32_t* pos, int32_t n_rows, int32_t n_kv, int32_t Hq,
                   int32_t Hkv, int32_t D)
{
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16) return 0;
    if (n_rows < 0 || n_kv < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return 0;
    for (int32_t i = 0; i < n_rows; ++i)
        if (pos[i] < 0 || pos[i] >= n_kv) return 0;
    return 1;
}

int oracle_attention_rows(int dtype, const uint16_t* q, const int32_t* pos, int32_t n_rows,
                          const uint16_t* k, const uint16_t* v, int32_t n_kv, int32_t Hq,
                          int32_t Hkv, int32_t D, double scale, double* out)
{
    if (!rows_ok(dtype, pos, n_rows, n_kv, Hq, Hkv, D)) return -1;
    const int64_t kv_elems = (int64_t)n_kv * Hkv * D;

    /* widen K and V once (exact), then work in double only */
    double* kd = (double*)malloc(sizeof(double) * (size_t)(kv_elems ? kv_elems : 1));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(kv_elems ? kv_elems : 1));
    if (!kd || !vd) {
        free(kd);
        free(vd);
        return -3;
    }
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < kv_elems; ++e) {
        kd[e] = widen(dtype, k[e]);
        vd[e] = widen(dtype, v[e]);
    }
    attention_core(dtype, q, pos, n_rows, kd, vd, Hq, Hkv, D, scale, out);
    free(kd);
    free(vd);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* INT8 KV cache: wmrh.cn/news/64708 §4.3 (the KV cache in INT8 instead of  */
/* FP16 halves its memory and bandwidth) and §5.4 (calibrate the KV cache   */
/* per channel: the channels' value ranges differ widely).  One scale per  */
/* (KV head, dim) channel for K and one for V, fixed by calibration.        */
/*                                                                         */
/* The code of a 16-bit value x in a channel with scale s > 0:             */
/*     code = clamp(rint(x / s), -127, 127)                                 */
/* where x / s is the IEEE single-precision quotient of the exact float    */
/* value of x and s (round to nearest even), rint rounds to nearest with   */
/* ties to even, and the value the code stands for is code * s.            */
/*                                                                         */
/* x [n_tok, H, D] 16-bit patterns, scale [H, D], out [n_tok, H, D].        */
/* Returns 0; -1 on a bad argument (a scale not > 0 included).              */
/* ---------------------------------------------------------------------- */
int oracle_quantize_int8(int dtype, const uint16_t* x, int64_t n_tok, int32_t H, int32_t D,
                         const float* scale, int8_t* out)
{
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16) return -1;
    if (n_tok < 0 || H <= 0 || D <= 0) return -1;
    for (int64_t c = 0; c < (int64_t)H * D; ++c)
        if (!(scale[c] > 0.0f)) return -1;
    for (int64_t t = 0; t < n_tok; ++t)
        for (int64_t c = 0; c < (int64_t)H * D; ++c) {
            const float xf = (float)widen(dtype, x[t * H * D + c]); /* exact */
            const float quot = xf / scale[c];                          /* IEEE single */
            float r = rintf(quot);                                     /* ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            out[t * H * D + c] = (int8_t)r;
        }
    return 0;
}

/* Attention as oracle_attention_rows, over an INT8 cache: key and value j of channel  */
/* (g, d) stand for code * scale (exact in double); q stays 16-bit.                    */
int oracle_attention_rows_int8(int dtype, const uint16_t* q, const int32_t* pos,
                               int32_t n_rows, const int8_t* kc, const int8_t* vc,
                               const float* k_scale, const float* v_scale, int32_t n_kv,
                               int32_t Hq, int32_t Hkv, int32_t D, double scale, double* out)
{
    if (!rows_ok(dtype, pos, n_rows, n_kv, Hq, Hkv, D)) return -1;
    const int64_t ch = (int64_t)Hkv * D;
    const int64_t kv_elems = (int64_t)n_kv * ch;
    double* kd = (double*)malloc(sizeof(double) * (size_t)(kv_elems ? kv_elems : 1));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(kv_elems ? kv_elems : 1));
    if (!kd || !vd) {
        free(kd);
        free(vd);
        return -3;
    }
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < kv_elems; ++e) {
        kd[e] = (double)kc[e] * (double)k_scale[e % ch];
        vd[e] = (double)vc[e] * (double)v_scale[e % ch];
    }
    attention_core(dtype, q, pos, n_rows, kd, vd, Hq, Hkv, D, scale, out);
    free(kd);
    free(vd);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Expected page pool after appending one step's new K/V.                  */
/*                                                                         */
/* Token t of the step belongs to request r when                            */
/*   sum_{r'<r} q_lens[r'] <= t < sum_{r'<=r} q_lens[r'];                   */
/* its logical position is p = context_lens[r] + (t - start of r), its page */
/* is block_table[r * max_pages + p / 16] and its slot in the page p % 16.  */
/* Pool layout: [num_pages][Hkv][16][D] (one contiguous 16 x D block per    */
/* page and KV head).  The global slot index is page * 16 + p % 16.         */
/*                                                                         */
/* k_pool / v_pool are updated in place (untouched entries keep whatever   */
/* the caller put there); slot_mapping[T] receives the global slot indices */
/* (may be NULL).  Returns 0; -1 on a bad argument; -2 when a position runs */
/* past the block-table row or a page id is outside [0, num_pages) (the     */
/* pool is then left partially written up to that token).                  */
/* ---------------------------------------------------------------------- */
int oracle_kv_append(int32_t num_reqs, const int32_t* q_lens, const int32_t* context_lens,
                     const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                     int32_t Hkv, int32_t D, const uint16_t* k_new, const uint16_t* v_new,
                     uint16_t* k_pool, uint16_t* v_pool, int64_t* slot_mapping)
{
    if (num_reqs < 0 || max_pages < 0 || num_pages < 0 || Hkv <= 0 || D <= 0) return -1;
    int64_t t = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        if (q_lens[r] < 0 || context_lens[r] < 0) return -1;
        for (int32_t i = 0; i < q_lens[r]; ++i, ++t) {
            const int64_t p = (int64_t)context_lens[r] + i;
            const int64_t logical_page = p / ORACLE_PAGE_TOKENS;
            if (logical_page >= max_pages) return -2;
            const int64_t page = block_table[(int64_t)r * max_pages + logical_page];
            if (page < 0 || page >= num_pages) return -2;
            const int64_t in_page = p % ORACLE_PAGE_TOKENS;
            if (slot_mapping) slot_mapping[t] = page * ORACLE_PAGE_TOKENS + in_page;
            for (int32_t h = 0; h < Hkv; ++h) {
                const int64_t dst = ((page * Hkv + h) * ORACLE_PAGE_TOKENS + in_page) * D;
                const int64_t src = (t * Hkv + h) * D;
                for (int32_t d = 0; d < D; ++d) {
                    k_pool[dst + d] = k_new[src + d];
                    v_pool[dst + d] = v_new[src + d];
                }
            }
        }
    }
    return 0;
}
