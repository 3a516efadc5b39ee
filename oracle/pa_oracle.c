/*
 * Oracle for paged KV-cache decode: plain, slow, fp64 C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * under paged_kv_cache_blocks_gb300/) includes, links or calls this file; only
 * the tests, the package's smoke check and the CPU-baseline leg of the bench
 * use it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where that is defined:
 *
 *   - KV layout.  The cache is cut into fixed blocks of `block_size` (16)
 *     tokens; a per-sequence block table maps logical block j to a physical
 *     block id, like a page table maps virtual pages to frames.
 *       "vLLM Nedir? PagedAttention ile Production LLM Serving", section
 *       "PagedAttention"; "vLLM ve Triton ile maliyet optimizasyonu",
 *       section 03 ("Yontem"), steps 1 and 2.
 *     Physical layout (the pages leave it open; our reading): one array per
 *     K and per V of shape [num_blocks][num_kv_heads][block_size][head_dim].
 *
 *   - Cache write: the new token's key/value rows are copied to the slot the
 *     allocator handed out, slot = block_id * block_size + offset.
 *       "vLLM Nedir?", section "Bir istek motorun icinde", step 2
 *       (allocate_slots); "vLLM ve Triton", section 03, step 3.
 *
 *   - Copy-on-write: a shared block is copied to a fresh block before one of
 *     its holders writes into it.  "vLLM ve Triton", section 03.
 *
 *   - Chunked prefill: several query tokens of one sequence (the last piece
 *     of its prompt) attend causally over its paged K/V; see oracle_prefill.
 *
 *   - Attention: the maths of scaled dot-product attention is unchanged by
 *     paging, only where K and V are read from changes:
 *       out = softmax(q K^T / sqrt(d_k)) V  over the sequence's tokens.
 *       "vLLM ve Triton", section 03, the paragraph on scaled dot-product
 *       attention (its formula was lost in extraction; this is the standard
 *       definition it names).
 *     Grouped-query attention: several query heads share one KV head.
 *       "Yerel LLM sistemlerinde backpressure ve olcekleme", section
 *       "KV butcesi" (64 attention heads, 8 KV heads).
 *     Our reading: query head i uses KV head i / G, G = Hq / Hkv (contiguous
 *     groups).
 *
 * Method: gather every sequence's blocks into a contiguous fp64 K and V
 * (exact conversion from fp16/bf16), then textbook softmax attention in fp64:
 * scores, subtract the maximum, exp (libm), normalise, weighted sum of V.
 * No online softmax, no partitions, no blocking.
 *
 * Element types are passed as raw 16-bit patterns: dtype 0 = IEEE binary16,
 * dtype 1 = bfloat16; FP8 caches as E4M3 bytes with per-KV-head scales.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- 16-bit float decoding, written from the IEEE 754 / bfloat16 layouts ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);           /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: the top 16 bits of an IEEE binary32 (1, 8 bits bias 127, 7). */
static double bf16_bits_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -133);          /* subnormal: f * 2^-126 * 2^-7 */
    } else if (e == 255) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -mag : mag;
}

static double to_double(uint16_t bits, int dtype) {
    return dtype == 0 ? half_bits_to_double(bits) : bf16_bits_to_double(bits);
}

/* Exposed so the tests can check the decoding against numpy / torch. */
void oracle_bits_to_double(const uint16_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = to_double(bits[i], dtype);
}

/* ---- FP8 (E4M3) KV cache ----
 *
 * An FP8 cache halves the bytes per token at some accuracy risk ("Yerel LLM
 * sistemlerinde backpressure ve olcekleme", section "1. KV cache tuketimi
 * ve GPU bellek tasmasi", the FP8 KV cache paragraph).  E4M3 ("fn"): 1 sign
 * bit, 4 exponent bits with bias 7, 3 fraction bits, no infinities, the
 * code S.1111.111 is NaN, largest finite 448.  Stored code =
 * E4M3(fp32(x) * fp32(1 / scale)), rounded to nearest-even and saturated to
 * +-448; value = code * scale.  Scales are per KV head, for K and for V.
 * Our layout reading: K blocks [num_blocks][Hkv][16][D] bytes as for 16-bit
 * caches, V blocks stored dimension-major [num_blocks][Hkv][D][16].
 */
static double e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 7;
    double mag;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) mag = ldexp((double)f, -9);              /* f/8 * 2^-6 */
    else mag = ldexp((double)(8 + f), e - 10);           /* (1 + f/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Round a float to the nearest E4M3 code (ties to even), saturating. */
static uint8_t double_to_e4m3(double x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 464.0) return sign | 0x7e;                  /* 464 ties to 448; above saturates */
    if (a < ldexp(1.0, -6)) {                            /* subnormal grid: k * 2^-9 */
        double k = a * 512.0;
        double r = nearbyint(k);                          /* default mode: ties to even */
        return sign | (uint8_t)r;                        /* r == 8 is the code of 2^-6 */
    }
    int e2;
    frexp(a, &e2);                                       /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                                      /* a in [2^e, 2^(e+1)) */
    double k = ldexp(a, 3 - e) - 8.0;                    /* fraction in eighths, [0, 8) */
    double r = nearbyint(k);
    if (r >= 8.0) { r = 0.0; e += 1; }
    if (e > 8) return sign | 0x7e;
    return sign | (uint8_t)(((e + 7) << 3) | (int)r);
}

void oracle_e4m3_to_double(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
}

void oracle_float_to_e4m3(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_e4m3((double)x[i]);
}

/*
 * FP8 cache write: like oracle_cache_write, with every value quantised as
 * E4M3(fp32(value) * fp32(1 / scale[h])), K row-major per token, V written
 * into the dimension-major V block.
 */
int64_t oracle_cache_write_fp8(const uint16_t* k, const uint16_t* v, int dtype,
                               const int64_t* slot_mapping, int64_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               const float* k_scale, const float* v_scale, uint8_t* k_cache,
                               uint8_t* v_cache, int64_t num_blocks);

/* ---- cache write ---- */

/*
 * For every token t with slot s = slot_mapping[t] >= 0: copy the head_dim
 * 16-bit values of k[t][h] to k_cache[s / block_size][h][s % block_size] and
 * likewise for v, for every KV head h.  Negative slots are padding and are
 * skipped.  Returns the number of tokens whose slot lies past the pool
 * (those are skipped too).
 */
int64_t oracle_cache_write(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                           int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, uint16_t* k_cache, uint16_t* v_cache,
                           int64_t num_blocks) {
    int64_t out_of_range = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        if (blk >= num_blocks) { ++out_of_range; continue; }
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
            int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                k_cache[dst + d] = k[src + d];
                v_cache[dst + d] = v[src + d];
            }
        }
    }
    return out_of_range;
}

int64_t oracle_cache_write_fp8(const uint16_t* k, const uint16_t* v, int dtype,
                               const int64_t* slot_mapping, int64_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               const float* k_scale, const float* v_scale, uint8_t* k_cache,
                               uint8_t* v_cache, int64_t num_blocks) {
    int64_t out_of_range = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        if (blk >= num_blocks) { ++out_of_range; continue; }
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            float inv_k = 1.0f / k_scale[h];
            float inv_v = 1.0f / v_scale[h];
            int64_t src = (t * num_kv_heads + h) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                float xk = (float)to_double(k[src + d], dtype) * inv_k;
                float xv = (float)to_double(v[src + d], dtype) * inv_v;
                k_cache[((blk * num_kv_heads + h) * block_size + off) * (int64_t)head_dim + d] =
                    double_to_e4m3((double)xk);
                v_cache[((blk * num_kv_heads + h) * (int64_t)head_dim + d) * block_size + off] =
                    double_to_e4m3((double)xv);
            }
        }
    }
    return out_of_range;
}

/* ---- copy-on-write block copy ---- */

/*
 * For every pair i: every KV head's 16 rows of block src[i] are copied to
 * block dst[i], in K and in V.  A block shared by several sequences is
 * copied when one holder writes into it ("vLLM ve Triton ile maliyet
 * optimizasyonu", section 03, the copy-on-write paragraph).  Pairs with an
 * id outside the pool are skipped (counted in the return value).
 */
int64_t oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, int64_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           const int32_t* src, const int32_t* dst, int64_t n_pairs) {
    int64_t skipped = 0;
    int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t i = 0; i < n_pairs; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
            ++skipped;
            continue;
        }
        for (int64_t e = 0; e < per_block; ++e) {
            k_cache[dst[i] * per_block + e] = k_cache[src[i] * per_block + e];
            v_cache[dst[i] * per_block + e] = v_cache[src[i] * per_block + e];
        }
    }
    return skipped;
}

/* ---- gather ---- */

/*
 * Logical token t of a sequence lives in physical block table_row[t / bs] at
 * row t % bs.  Writes the seq_len x head_dim values of KV head h, converted
 * to fp64, to `dst` in token order.
 */
void oracle_gather(const uint16_t* cache, int dtype, const int32_t* table_row, int32_t seq_len,
                   int32_t num_kv_heads, int32_t h, int32_t head_dim, int32_t block_size,
                   double* dst) {
    for (int32_t t = 0; t < seq_len; ++t) {
        int64_t phys = table_row[t / block_size];
        int64_t row = ((phys * num_kv_heads + h) * block_size + (t % block_size)) * (int64_t)head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            dst[(int64_t)t * head_dim + d] = to_double(cache[row + d], dtype);
    }
}

/* ---- decode attention ---- */

/*
 * q:            [num_seqs][num_q_heads][head_dim] 16-bit patterns
 * k/v_cache:    [num_blocks][num_kv_heads][block_size][head_dim]
 * block_tables: [num_seqs][max_blocks]; only the first ceil(len/bs) entries
 *               of a row are read
 * seq_lens:     [num_seqs], tokens to attend over (the new one included)
 * out:          [num_seqs][num_q_heads][head_dim] fp64
 * A sequence of length 0 has an empty softmax; our reading defines its
 * output as 0.
 * Returns 0, or -1 if scratch memory could not be allocated.
 */
int oracle_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int dtype,
                  const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, double scale, double* out, int num_threads) {
    const int32_t G = num_q_heads / num_kv_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    int64_t n_pairs = (int64_t)num_seqs * num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t pair = 0; pair < n_pairs; ++pair) {
        int32_t b = (int32_t)(pair / num_kv_heads);
        int32_t h = (int32_t)(pair % num_kv_heads);
        int32_t L = seq_lens[b];
        if (L <= 0) {
            for (int32_t g = 0; g < G; ++g) {
                double* o = out + ((int64_t)b * num_q_heads + (int64_t)h * G + g) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            }
            continue;
        }
        double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!K || !V || !s || !qd) {
            free(K); free(V); free(s); free(qd);
            failed |= 1;
            continue;
        }
        const int32_t* row = block_tables + (int64_t)b * max_blocks;
        oracle_gather(k_cache, dtype, row, L, num_kv_heads, h, head_dim, block_size, K);
        oracle_gather(v_cache, dtype, row, L, num_kv_heads, h, head_dim, block_size, V);
        for (int32_t g = 0; g < G; ++g) {
            int32_t i = h * G + g; /* query head i reads KV head i / G */
            const uint16_t* qi = q + ((int64_t)b * num_q_heads + i) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) qd[d] = to_double(qi[d], dtype);
            /* scores */
            double smax = -INFINITY;
            for (int32_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int32_t d = 0; d < head_dim; ++d) acc += qd[d] * K[(int64_t)t * head_dim + d];
                s[t] = scale * acc;
                if (s[t] > smax) smax = s[t];
            }
            /* softmax weights */
            double denom = 0.0;
            for (int32_t t = 0; t < L; ++t) {
                s[t] = exp(s[t] - smax);
                denom += s[t];
            }
            /* weighted sum of values */
            double* o = out + ((int64_t)b * num_q_heads + i) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int32_t t = 0; t < L; ++t) acc += s[t] * V[(int64_t)t * head_dim + d];
                o[d] = acc / denom;
            }
        }
        free(K); free(V); free(s); free(qd);
    }
    return failed ? -1 : 0;
}

/*
 * Decode over an FP8 cache: the same textbook attention as oracle_decode on
 * the dequantised values K = code * k_scale[h], V = code * v_scale[h]
 * (V read from its dimension-major blocks).  q is 16-bit (dtype).
 */
int oracle_decode_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                      const float* k_scale, const float* v_scale, int dtype,
                      const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, double scale, double* out,
                      int num_threads) {
    const int32_t G = num_q_heads / num_kv_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    int64_t n_pairs = (int64_t)num_seqs * num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t pair = 0; pair < n_pairs; ++pair) {
        int32_t b = (int32_t)(pair / num_kv_heads);
        int32_t h = (int32_t)(pair % num_kv_heads);
        int32_t L = seq_lens[b];
        if (L <= 0) {
            for (int32_t g = 0; g < G; ++g) {
                double* o = out + ((int64_t)b * num_q_heads + (int64_t)h * G + g) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            }
            continue;
        }
        double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
        double* sc = (double*)malloc(sizeof(double) * (size_t)L);
        double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!K || !V || !sc || !qd) {
            free(K); free(V); free(sc); free(qd);
            failed |= 1;
            continue;
        }
        const int32_t* row = block_tables + (int64_t)b * max_blocks;
        for (int32_t t = 0; t < L; ++t) {
            int64_t phys = row[t / block_size];
            int64_t off = t % block_size;
            for (int32_t d = 0; d < head_dim; ++d) {
                K[(int64_t)t * head_dim + d] =
                    e4m3_to_double(k_cache[((phys * num_kv_heads + h) * block_size + off) * head_dim + d]) *
                    (double)k_scale[h];
                V[(int64_t)t * head_dim + d] =
                    e4m3_to_double(v_cache[((phys * num_kv_heads + h) * head_dim + d) * block_size + off]) *
                    (double)v_scale[h];
            }
        }
        for (int32_t g = 0; g < G; ++g) {
            int32_t i = h * G + g;
            const uint16_t* qi = q + ((int64_t)b * num_q_heads + i) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) qd[d] = to_double(qi[d], dtype);
            double smax = -INFINITY;
            for (int32_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int32_t d = 0; d < head_dim; ++d) acc += qd[d] * K[(int64_t)t * head_dim + d];
                sc[t] = scale * acc;
                if (sc[t] > smax) smax = sc[t];
            }
            double denom = 0.0;
            for (int32_t t = 0; t < L; ++t) {
                sc[t] = exp(sc[t] - smax);
                denom += sc[t];
            }
            double* o = out + ((int64_t)b * num_q_heads + i) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int32_t t = 0; t < L; ++t) acc += sc[t] * V[(int64_t)t * head_dim + d];
                o[d] = acc / denom;
            }
        }
        free(K); free(V); free(sc); free(qd);
    }
    return failed ? -1 : 0;
}

/* ---- multi-query (chunked prefill) attention ---- */

/*
 * Chunked prefill: a long prompt is not processed in one iteration but cut
 * into pieces that fit the step's token budget; each iteration computes one
 * piece together with the running sequences' single decode tokens, and the
 * piece's K/V fill the sequence's blocks over several steps.
 *   "Yerel LLM sistemlerinde backpressure ve olcekleme", section
 *   "4. Prefill ve decode" (the chunked prefill paragraph and diagram);
 *   "vLLM Nedir? PagedAttention ile Production LLM Serving", section
 *   "Chunked prefill".
 * Our reading of what one iteration's attention computes: sequence b holds
 * seq_lens[b] tokens in its blocks after the piece's K/V were written; its
 * piece is the last Qn = q_offsets[b+1] - q_offsets[b] of them (a decode
 * token is a piece of one), so query j of the piece sits at position
 * p = seq_lens[b] - Qn + j and attends causally to tokens 0 .. p.
 *
 * q:          [num_q_tokens][num_q_heads][head_dim] 16-bit patterns, the
 *             pieces of all sequences back to back (q_offsets[num_seqs] =
 *             num_q_tokens)
 * rows:       the query tokens to compute (indices into q), or NULL for all
 * out:        [n_rows][num_q_heads][head_dim] fp64
 * Returns 0; -1 if scratch memory could not be allocated; -2 if a piece is
 * longer than its sequence or q_offsets is not non-decreasing from 0.
 */
int oracle_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int dtype,
                   const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                   const int32_t* q_offsets, int32_t num_seqs, const int64_t* rows, int64_t n_rows,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   double scale, double* out, int num_threads) {
    const int32_t G = num_q_heads / num_kv_heads;
    const int64_t num_q_tokens = q_offsets[num_seqs];
    if (q_offsets[0] != 0) return -2;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t piece = q_offsets[b + 1] - q_offsets[b];
        if (piece < 0 || piece > seq_lens[b]) return -2;
    }
    if (!rows) n_rows = num_q_tokens;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    int64_t n_tasks = n_rows * num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t task = 0; task < n_tasks; ++task) {
        int64_t r = task / num_kv_heads;
        int32_t h = (int32_t)(task % num_kv_heads);
        int64_t tok = rows ? rows[r] : r;
        if (tok < 0 || tok >= num_q_tokens) {
            failed |= 2;
            continue;
        }
        /* the sequence whose piece holds query token tok */
        int32_t b = 0;
        while (q_offsets[b + 1] <= tok) ++b;
        int32_t piece_len = q_offsets[b + 1] - q_offsets[b];
        int32_t j = (int32_t)(tok - q_offsets[b]);
        int32_t pos = seq_lens[b] - piece_len + j;
        int32_t n_visible = pos + 1; /* causal: tokens 0 .. pos */
        double* K = (double*)malloc(sizeof(double) * (size_t)n_visible * head_dim);
        double* V = (double*)malloc(sizeof(double) * (size_t)n_visible * head_dim);
        double* sc = (double*)malloc(sizeof(double) * (size_t)n_visible);
        double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!K || !V || !sc || !qd) {
            free(K); free(V); free(sc); free(qd);
            failed |= 1;
            continue;
        }
        const int32_t* trow = block_tables + (int64_t)b * max_blocks;
        oracle_gather(k_cache, dtype, trow, n_visible, num_kv_heads, h, head_dim, block_size, K);
        oracle_gather(v_cache, dtype, trow, n_visible, num_kv_heads, h, head_dim, block_size, V);
        for (int32_t g = 0; g < G; ++g) {
            int32_t head = h * G + g; /* query head reads KV head head / G */
            const uint16_t* qrow = q + (tok * num_q_heads + head) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) qd[d] = to_double(qrow[d], dtype);
            double smax = -INFINITY;
            for (int32_t t = 0; t < n_visible; ++t) {
                double acc = 0.0;
                for (int32_t d = 0; d < head_dim; ++d) acc += qd[d] * K[(int64_t)t * head_dim + d];
                sc[t] = scale * acc;
                if (sc[t] > smax) smax = sc[t];
            }
            double denom = 0.0;
            for (int32_t t = 0; t < n_visible; ++t) {
                sc[t] = exp(sc[t] - smax);
                denom += sc[t];
            }
            double* o = out + (r * num_q_heads + head) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int32_t t = 0; t < n_visible; ++t) acc += sc[t] * V[(int64_t)t * head_dim + d];
                o[d] = acc / denom;
            }
        }
        free(K); free(V); free(sc); free(qd);
    }
    if (failed & 2) return -2;
    return failed ? -1 : 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
