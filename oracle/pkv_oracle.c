/*
 * pkv_oracle.c -- slow, plain CPU reference for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check of the entry module and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library; it is compiled by gcc alone.
 *
 * Everything is computed from plain definitions, in double precision where the
 * data is floating point, in the order the definitions give:
 *
 *   element decoding   IEEE 754 binary16, bfloat16 (upper half of binary32) and
 *                      OCP FP8 E4M3 ("fn": bias 7, no infinities, S.1111.111 is
 *                      NaN, largest finite 448, subnormals m * 2^-9).
 *   element encoding   E4M3 with round-to-nearest-even and saturation to +-448,
 *                      written from the format definition.
 *   kv_append          a decode round computes K and V for the new token only and
 *                      keeps them -- 「KV 缓存与分页注意力」 §02; the token goes to
 *                      the slot the block table hands out -- same page, §07 块表.
 *   copy_blocks        copy-on-write: copy the shared block, write into the copy
 *                      -- same page, §08 共用，写时复制.
 *   decode attention   the new token's query attends over the K/V of every cached
 *                      token, which are fetched block by block through the block
 *                      table -- same page, §02 and §07; grouped heads share one
 *                      K/V head -- same page, §11 后来的做法.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#define _POSIX_C_SOURCE 200809L
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { DT_F16 = 0, DT_BF16 = 1, DT_E4M3 = 2 };

/* ------------------------------------------------------------------------ */
/* element decoding                                                          */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pkvo_dec_f16(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0x1f)
        v = (m == 0) ? INFINITY : NAN;
    else if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return s ? -v : v;
}

/* bfloat16 is the upper 16 bits of an IEEE binary32 value. */
double pkvo_dec_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * No infinities; exponent 1111 with mantissa 111 is NaN. */
double pkvo_dec_e4m3(uint8_t x)
{
    int s = (x >> 7) & 1;
    int e = (x >> 3) & 0xf;
    int m = x & 7;
    double v;
    if (e == 0xf && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

static double dec_elem(int dtype, const void* base, int64_t idx)
{
    switch (dtype) {
    case DT_F16:  return pkvo_dec_f16(((const uint16_t*)base)[idx]);
    case DT_BF16: return pkvo_dec_bf16(((const uint16_t*)base)[idx]);
    case DT_E4M3: return pkvo_dec_e4m3(((const uint8_t*)base)[idx]);
    default:      return NAN;
    }
}

/* Bulk forms of the element conversions, for the tests. */
void pkvo_dec_array(int dtype, const void* src, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dec_elem(dtype, src, i);
}

static int elem_bytes(int dtype)
{
    return dtype == DT_E4M3 ? 1 : 2;
}

/* ------------------------------------------------------------------------ */
/* E4M3 encoding: round to nearest, ties to even, saturate finite to +-448.  */
/* ------------------------------------------------------------------------ */

uint8_t pkvo_enc_e4m3(float y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    if (isnan(y))
        return (uint8_t)(sign | 0x7f);
    double a = fabs((double)y);
    if (a >= 448.0)                                /* largest finite: 1.75 * 2^8 */
        return (uint8_t)(sign | 0x7e);

    /* spacing of representable values around a */
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);                  /* subnormal range */
    } else {
        int ex;
        frexp(a, &ex);                             /* a = f * 2^ex, f in [0.5,1) */
        quantum = ldexp(1.0, (ex - 1) - 3);        /* 3 mantissa bits */
    }
    /* a / quantum is exact (power-of-two divisor); rint rounds half to even
       in the default rounding mode */
    double r = rint(a / quantum) * quantum;
    if (r >= 448.0)
        return (uint8_t)(sign | 0x7e);
    if (r == 0.0)
        return sign;

    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)(int)(r / ldexp(1.0, -9)); /* exponent field 0 */
    } else {
        int ex;
        double f = frexp(r, &ex);                  /* r = (2f) * 2^(ex-1) */
        int e = (ex - 1) + 7;
        int m = (int)((2.0 * f - 1.0) * 8.0);
        code = (uint8_t)((e << 3) | m);
    }
    return (uint8_t)(sign | code);
}

void pkvo_enc_e4m3_array(const float* y, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_enc_e4m3(y[i]);
}

/* ------------------------------------------------------------------------ */
/* sizing                                                                    */
/* ------------------------------------------------------------------------ */

/* Bytes one token occupies in the cache: a key and a value vector for every
 * KV head of every layer -- 「KV 缓存与分页注意力」 §03 一个词元 800 KB. */
int64_t pkvo_kv_bytes_per_token(int64_t num_kv_heads, int64_t head_dim,
                                int64_t num_layers, int64_t elem_size)
{
    return 2 * num_kv_heads * head_dim * num_layers * elem_size;
}

/* Physical blocks a sequence of n tokens holds when a block is only taken once
 * the previous one is full -- same page, §07 块表. */
int64_t pkvo_blocks_for_tokens(int64_t n, int64_t block_size)
{
    int64_t blocks = 0;
    int64_t room = 0;                  /* free slots left in the last block */
    for (int64_t t = 0; t < n; ++t) {
        if (room == 0) {
            ++blocks;
            room = block_size;
        }
        --room;
    }
    return blocks;
}

/* ------------------------------------------------------------------------ */
/* cache addressing: cache[block][kv_head][offset][d], K and V alike         */
/* ------------------------------------------------------------------------ */

static int64_t cache_index(int64_t blk, int64_t head, int64_t off, int64_t d,
                           int32_t num_kv_heads, int32_t block_size, int32_t head_dim)
{
    return ((blk * num_kv_heads + head) * block_size + off) * head_dim + d;
}

/* Logical-order gather of one KV head of one sequence: row t of `out` is the
 * vector of token t, found in physical block table[t / BS] at offset t % BS
 * -- 「Paged Attention in LLMs」 section "Block Table".  Returns -1 if a table
 * entry is outside the pool. */
int pkvo_gather(const void* cache, int cache_dtype, int64_t num_blocks,
                int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                const int32_t* table_row, int32_t context_len, int32_t kv_head,
                double scale_factor, double* out /* [context_len][head_dim] */)
{
    for (int32_t t = 0; t < context_len; ++t) {
        int64_t logical = t / block_size;
        int64_t off = t % block_size;
        int64_t phys = table_row[logical];
        if (phys < 0 || phys >= num_blocks)
            return -1;
        for (int32_t d = 0; d < head_dim; ++d) {
            int64_t i = cache_index(phys, kv_head, off, d, num_kv_heads, block_size, head_dim);
            out[(int64_t)t * head_dim + d] = dec_elem(cache_dtype, cache, i) * scale_factor;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* kv_append                                                                  */
/* ------------------------------------------------------------------------ */

/* Write token t's K and V (all KV heads) at slot_mapping[t]: block slot / BS,
 * offset slot % BS.  A negative slot means "no write".  When the cache holds the
 * input's own type the bytes are copied; an E4M3 cache stores
 * e4m3(fp32(x) * fp32(1 / scale)).  Returns the number of tokens skipped
 * because their slot lies outside the pool, or -1 for an unsupported pairing. */
int64_t pkvo_kv_append(void* k_cache, void* v_cache, int64_t num_blocks,
                       int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                       int cache_dtype, float k_scale, float v_scale,
                       const void* k, const void* v, int in_dtype,
                       const int64_t* slot_mapping, int64_t num_tokens)
{
    if (in_dtype == DT_E4M3)
        return -1;
    if (cache_dtype != in_dtype && cache_dtype != DT_E4M3)
        return -1;
    int cb = elem_bytes(cache_dtype);
    int ib = elem_bytes(in_dtype);
    float k_inv = 1.0f / k_scale;
    float v_inv = 1.0f / v_scale;
    int64_t skipped = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size) {
            ++skipped;
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
                int64_t dst = cache_index(blk, h, off, d, num_kv_heads, block_size, head_dim);
                if (cache_dtype == in_dtype) {
                    memcpy((char*)k_cache + dst * cb, (const char*)k + src * ib, (size_t)cb);
                    memcpy((char*)v_cache + dst * cb, (const char*)v + src * ib, (size_t)cb);
                } else {
                    float xk = (float)dec_elem(in_dtype, k, src);
                    float xv = (float)dec_elem(in_dtype, v, src);
                    float yk = xk * k_inv;
                    float yv = xv * v_inv;
                    ((uint8_t*)k_cache)[dst] = pkvo_enc_e4m3(yk);
                    ((uint8_t*)v_cache)[dst] = pkvo_enc_e4m3(yv);
                }
            }
        }
    }
    return skipped;
}

/* ------------------------------------------------------------------------ */
/* copy_blocks                                                               */
/* ------------------------------------------------------------------------ */

/* For every layer and every (src, dst) pair, the whole dst block (all heads,
 * all slots, K and V) becomes a copy of the src block as it was before the call.
 * Returns -1 if a block id is outside the pool (nothing is written then). */
int pkvo_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                     int64_t num_blocks, int64_t block_bytes,
                     const int64_t* pairs, int64_t num_pairs)
{
    for (int64_t i = 0; i < 2 * num_pairs; ++i)
        if (pairs[i] < 0 || pairs[i] >= num_blocks)
            return -1;
    if (num_pairs == 0)
        return 0;
    /* snapshot of every source block first, then the writes */
    size_t snap_bytes = (size_t)(2 * num_layers * num_pairs * block_bytes);
    char* snap = (char*)malloc(snap_bytes);
    if (!snap)
        return -2;
    for (int32_t l = 0; l < num_layers; ++l)
        for (int64_t p = 0; p < num_pairs; ++p) {
            int64_t src = pairs[2 * p];
            char* sk = snap + ((2 * (int64_t)l) * num_pairs + p) * block_bytes;
            char* sv = snap + ((2 * (int64_t)l + 1) * num_pairs + p) * block_bytes;
            memcpy(sk, (const char*)k_caches[l] + src * block_bytes, (size_t)block_bytes);
            memcpy(sv, (const char*)v_caches[l] + src * block_bytes, (size_t)block_bytes);
        }
    for (int32_t l = 0; l < num_layers; ++l)
        for (int64_t p = 0; p < num_pairs; ++p) {
            int64_t dst = pairs[2 * p + 1];
            const char* sk = snap + ((2 * (int64_t)l) * num_pairs + p) * block_bytes;
            const char* sv = snap + ((2 * (int64_t)l + 1) * num_pairs + p) * block_bytes;
            memcpy((char*)k_caches[l] + dst * block_bytes, sk, (size_t)block_bytes);
            memcpy((char*)v_caches[l] + dst * block_bytes, sv, (size_t)block_bytes);
        }
    free(snap);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* decode attention                                                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    const void* k_cache;
    const void* v_cache;
    int cache_dtype;
    int64_t num_blocks;
    int32_t num_kv_heads, block_size, head_dim;
    double k_scale, v_scale;
    const void* q;
    int q_dtype;
    int32_t num_seqs, num_heads;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    double scale;
    int32_t t_begin, t_end;       /* token range; t_end < 0 means "whole context" */
    double* out;                  /* [S][H][D] */
    double* lse_max;              /* optional [S][H]: max logit of the range */
    double* lse_sum;              /* optional [S][H]: sum of exp(x - max) */
    int unnormalised;             /* 1: out holds sum_t exp(x_t - max) v_t */
    int64_t next;                 /* work counter (s*H + h), guarded by mu */
    pthread_mutex_t mu;
    int status;
} decode_job;

/* One (sequence, query head): plain two-pass softmax attention in double.
 *   kv head      g   = h / (H / Hkv)           (consecutive query heads share)
 *   logit        x_t = scale * sum_d q[d] * k_t[d]
 *   weight       w_t = exp(x_t - max_t x_t)
 *   output       o   = sum_t w_t v_t / sum_t w_t                              */
static int decode_one(decode_job* J, int32_t s, int32_t h, double* xbuf, double* kv)
{
    int32_t D = J->head_dim;
    int32_t group = J->num_heads / J->num_kv_heads;
    int32_t g = h / group;
    int32_t ctx = J->context_lens[s];
    const int32_t* row = J->block_tables + (int64_t)s * J->max_blocks_per_seq;
    double* o = J->out + ((int64_t)s * J->num_heads + h) * D;
    int32_t t0 = J->t_begin;
    int32_t t1 = J->t_end < 0 ? ctx : (J->t_end < ctx ? J->t_end : ctx);

    for (int32_t d = 0; d < D; ++d)
        o[d] = 0.0;
    if (ctx > J->max_blocks_per_seq * J->block_size)
        return -1;
    if (t1 <= t0) {
        if (J->lse_max) J->lse_max[(int64_t)s * J->num_heads + h] = -INFINITY;
        if (J->lse_sum) J->lse_sum[(int64_t)s * J->num_heads + h] = 0.0;
        return 0;
    }

    /* keys in logical order, then the logits */
    if (pkvo_gather(J->k_cache, J->cache_dtype, J->num_blocks, J->num_kv_heads,
                    J->block_size, D, row, t1, g, J->k_scale, kv) != 0)
        return -1;
    const int64_t qbase = ((int64_t)s * J->num_heads + h) * D;
    double m = -INFINITY;
    for (int32_t t = t0; t < t1; ++t) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += dec_elem(J->q_dtype, J->q, qbase + d) * kv[(int64_t)t * D + d];
        xbuf[t] = J->scale * dot;
        if (xbuf[t] > m)
            m = xbuf[t];
    }

    /* values in logical order, then the weighted sum */
    if (pkvo_gather(J->v_cache, J->cache_dtype, J->num_blocks, J->num_kv_heads,
                    J->block_size, D, row, t1, g, J->v_scale, kv) != 0)
        return -1;
    double l = 0.0;
    for (int32_t t = t0; t < t1; ++t) {
        double w = exp(xbuf[t] - m);
        l += w;
        for (int32_t d = 0; d < D; ++d)
            o[d] += w * kv[(int64_t)t * D + d];
    }
    if (!J->unnormalised)
        for (int32_t d = 0; d < D; ++d)
            o[d] /= l;
    if (J->lse_max) J->lse_max[(int64_t)s * J->num_heads + h] = m;
    if (J->lse_sum) J->lse_sum[(int64_t)s * J->num_heads + h] = l;
    return 0;
}

static void* decode_worker(void* arg)
{
    decode_job* J = (decode_job*)arg;
    int64_t total = (int64_t)J->num_seqs * J->num_heads;
    int32_t max_ctx = J->max_blocks_per_seq * J->block_size;
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    double* kv = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1) * (size_t)J->head_dim);
    int bad = (xbuf == NULL || kv == NULL);
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t w = J->next++;
        if (bad) J->status = -2;
        pthread_mutex_unlock(&J->mu);
        if (w >= total || bad)
            break;
        int32_t s = (int32_t)(w / J->num_heads);
        int32_t h = (int32_t)(w % J->num_heads);
        if (decode_one(J, s, h, xbuf, kv) != 0) {
            pthread_mutex_lock(&J->mu);
            J->status = -1;
            pthread_mutex_unlock(&J->mu);
        }
    }
    free(xbuf);
    free(kv);
    return NULL;
}

static int run_decode(decode_job* J, int nthreads)
{
    if (J->num_kv_heads <= 0 || J->num_heads % J->num_kv_heads != 0)
        return -3;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    J->next = 0;
    J->status = 0;
    pthread_mutex_init(&J->mu, NULL);
    if (nthreads == 1) {
        decode_worker(J);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int i = 0; i < nthreads; ++i)
            if (pthread_create(&th[i], NULL, decode_worker, J) == 0)
                ++started;
        if (started == 0)
            decode_worker(J);
        for (int i = 0; i < started; ++i)
            pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J->mu);
    return J->status;
}

/* Decode attention of every (sequence, query head) over its whole context.
 * out[s][h][d] in double.  Returns 0, or -1 if a block id or a context length
 * is outside what the table and the pool hold, -3 for bad head counts. */
int pkvo_paged_attention_decode(const void* k_cache, const void* v_cache, int cache_dtype,
                                int64_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                                int32_t head_dim, float k_scale, float v_scale,
                                const void* q, int q_dtype, int32_t num_seqs, int32_t num_heads,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, float scale,
                                double* out, int nthreads)
{
    decode_job J;
    memset(&J, 0, sizeof J);
    J.k_cache = k_cache; J.v_cache = v_cache; J.cache_dtype = cache_dtype;
    J.num_blocks = num_blocks; J.num_kv_heads = num_kv_heads; J.block_size = block_size;
    J.head_dim = head_dim; J.k_scale = (double)k_scale; J.v_scale = (double)v_scale;
    J.q = q; J.q_dtype = q_dtype; J.num_seqs = num_seqs; J.num_heads = num_heads;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.scale = (double)scale;
    J.t_begin = 0; J.t_end = -1; J.out = out;
    return run_decode(&J, nthreads);
}

/* The same attention restricted to tokens [t_begin, t_end) of every context,
 * returned unnormalised: out = sum_t exp(x_t - m) v_t, with m = max logit of the
 * range (lse_max) and l = sum_t exp(x_t - m) (lse_sum).  A range that holds no
 * token gives m = -inf, l = 0, out = 0. */
int pkvo_attention_range(const void* k_cache, const void* v_cache, int cache_dtype,
                         int64_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                         int32_t head_dim, float k_scale, float v_scale,
                         const void* q, int q_dtype, int32_t num_seqs, int32_t num_heads,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, float scale,
                         int32_t t_begin, int32_t t_end,
                         double* out, double* lse_max, double* lse_sum, int nthreads)
{
    decode_job J;
    memset(&J, 0, sizeof J);
    J.k_cache = k_cache; J.v_cache = v_cache; J.cache_dtype = cache_dtype;
    J.num_blocks = num_blocks; J.num_kv_heads = num_kv_heads; J.block_size = block_size;
    J.head_dim = head_dim; J.k_scale = (double)k_scale; J.v_scale = (double)v_scale;
    J.q = q; J.q_dtype = q_dtype; J.num_seqs = num_seqs; J.num_heads = num_heads;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.scale = (double)scale;
    J.t_begin = t_begin; J.t_end = t_end; J.out = out;
    J.lse_max = lse_max; J.lse_sum = lse_sum; J.unnormalised = 1;
    return run_decode(&J, nthreads);
}
