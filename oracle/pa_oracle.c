/*
 * pa_oracle.c -- plain float64 CPU oracle for paged KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header or constant
 * with the CUDA library: it has its own float16 / bfloat16 decoding, its own address
 * translation and its own attention, all written for clarity, not speed.
 *
 * What it computes (sources, by page title and section):
 *
 *  - Address translation, "locate_kv": a logical token position t maps to
 *    logical block t / block_size and slot t % block_size, and the block
 *    table turns the logical block into a physical block id.  ("Unveiling the
 *    NVIDIA driver stack: GPU page tables and vLLM PagedAttention",
 *    section 6, "code view"; worked example: position 37 with table
 *    [7, 42, 9, 103] lands in physical block 9, slot 5.)
 *
 *  - The cache write: a new token's K and V go into the next free slot of the
 *    sequence's last block.  The slot is given here as one flat number
 *    slot = physical_block * block_size + offset; negative slots are padding
 *    and are skipped.  ("vLLM PagedAttention source walk-through", section
 *    3.2, append_token and _write_kv_to_block; "Efficient Memory Management
 *    for LLM Serving with PagedAttention -- in-depth reading", sections 3.2
 *    and 3.4, step 1.)
 *
 *  - Decode attention: paged attention is mathematically the same as ordinary
 *    attention over the sequence's keys and values ("in-depth reading",
 *    section 4.4; "walk-through", section 3.4).  So the oracle gathers the
 *    ctx valid keys and values of a sequence through the block table into
 *    contiguous arrays and applies the textbook softmax: scores
 *    x_i = scale * q . k_i, m = max_i x_i, p_i = exp(x_i - m) / sum_j
 *    exp(x_j - m), out = sum_i p_i v_i (the two-pass form the walk-through's
 *    section 3.4 calls "traditional").  Query head h reads KV head
 *    h / (num_heads / num_kv_heads) (grouped-query attention with consecutive
 *    groups; the pages do not fix the mapping).
 *
 *  - Prefill: each query row of a prompt (or of a chunk of it) attends to
 *    every earlier position of its sequence and to its own; with the
 *    queries' own K/V already in the cache, a row at position p is decode
 *    attention over the first p + 1 tokens ("in-depth reading", section
 *    5.1, item 5; "vAttention", paged prefill).
 *
 *  - FP8 caches: the block's contents are compressed and the attention
 *    kernel dequantises them ("PagedAttention: when the KV cache meets OS
 *    paging", section 6, the layer diagram).  The page names FP8 and nothing
 *    more; the oracle reads it as OCP E4M3 ("e4m3fn") codes with one float
 *    scale for the K pool and one for the V pool: the write stores the code
 *    nearest to x / scale, the read uses code value * scale.
 *
 *  The K and V pools have the layout [num_blocks, block_size, num_kv_heads,
 *  head_dim]; values are IEEE binary16 or bfloat16 bit patterns, or E4M3
 *  bytes, each decoded by its own routine below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_BLOCK 2
#define ORACLE_BAD_CONTEXT 3
#define ORACLE_DUPLICATE_SLOT 4
#define ORACLE_BAD_SLOT 5
#define ORACLE_NO_MEMORY 6

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits.  Exponent 0 encodes zero and
 * subnormals (fraction * 2^-24), exponent 31 encodes infinities and NaNs. */
double pa_oracle_half_to_double(uint16_t bits) {
    const int sign = (bits >> 15) & 1;
    const int expo = (bits >> 10) & 0x1f;
    const int frac = bits & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 -> double, from the format's definition: 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits.  Exponent 0 encodes zero and subnormals
 * (fraction * 2^-133), exponent 255 encodes infinities and NaNs. */
double pa_oracle_bf16_to_double(uint16_t bits) {
    const int sign = (bits >> 15) & 1;
    const int expo = (bits >> 7) & 0xff;
    const int frac = bits & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), expo - 134);
    }
    return sign ? -v : v;
}

/* FP8 E4M3 (OCP "e4m3fn") -> double, from the format's definition: 1 sign
 * bit, 4 exponent bits (bias 7), 3 fraction bits; exponent 0 encodes zero
 * and subnormals (fraction * 2^-9); no infinities; exponent 15 with fraction
 * 7 is NaN, so the largest finite value is 1.75 * 2^8 = 448. */
double pa_oracle_e4m3_to_double(uint8_t bits) {
    const int sign = (bits >> 7) & 1;
    const int expo = (bits >> 3) & 0xf;
    const int frac = bits & 0x7;
    double v;
    if (expo == 15 && frac == 7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexp((double)frac, -9);
    } else {
        v = ldexp((double)(8 + frac), expo - 10);
    }
    return sign ? -v : v;
}

/* Round half to even of a non-negative double to an integer-valued double. */
static double round_half_even(double a) {
    const double f = floor(a);
    const double r = a - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* The E4M3 code of x / scale: the quotient is taken in float32 (correctly
 * rounded), then rounded to the nearest E4M3 value, ties to even; finite
 * values beyond 448 saturate to +-448 and so do infinities; NaN gives NaN. */
uint8_t pa_oracle_quantize_e4m3(float x, float scale) {
    const float v = x / scale;
    if (isnan(v)) return 0x7f;
    const int sign = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    int code;
    if (a >= 448.0) {
        code = 0x7e;
    } else if (a < ldexp(1.0, -6)) {             /* subnormal quanta of 2^-9 */
        code = (int)round_half_even(a / ldexp(1.0, -9)); /* 8 becomes the smallest normal */
    } else {
        int e = (int)floor(log2(a));
        if (ldexp(1.0, e) > a) --e;                /* guard log2 rounding */
        if (ldexp(1.0, e + 1) <= a) ++e;
        double m = round_half_even(a / ldexp(1.0, e - 3)); /* 8 .. 16 */
        if (m == 16.0) {
            m = 8.0;
            ++e;
        }
        code = ((e + 7) << 3) | ((int)m - 8);
        if (code > 0x7e) code = 0x7e;
    }
    return (uint8_t)((sign << 7) | code);
}

#define ORACLE_FP16 0
#define ORACLE_BF16 1

static double decode_elem(uint16_t bits, int dtype) {
    return dtype == ORACLE_BF16 ? pa_oracle_bf16_to_double(bits) : pa_oracle_half_to_double(bits);
}

/* Logical token position -> (physical block, slot in block). */
int pa_oracle_locate_kv(int64_t logical_token_idx, const int32_t* block_table, int block_size,
                        int32_t* physical_block, int32_t* offset_in_block) {
    if (logical_token_idx < 0 || block_size <= 0 || !block_table) return ORACLE_BAD_ARG;
    const int64_t logical_block = logical_token_idx / block_size;
    *offset_in_block = (int32_t)(logical_token_idx % block_size);
    *physical_block = block_table[logical_block];
    return ORACLE_OK;
}

static int cmp_i64(const void* a, const void* b) {
    const int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/* Write each new token's K and V rows (all KV heads) into its slot.  The
 * pools are updated in place; slots < 0 are skipped; slots must be distinct. */
int pa_oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint16_t* k_cache,
                                uint16_t* v_cache, const int64_t* slot_mapping, int64_t num_tokens,
                                int64_t num_blocks, int block_size, int num_kv_heads, int head_dim) {
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;
    if (num_tokens == 0) return ORACLE_OK;
    /* precondition: distinct non-negative slots */
    int64_t* sorted = (int64_t*)malloc(sizeof(int64_t) * (size_t)num_tokens);
    if (!sorted) return ORACLE_NO_MEMORY;
    memcpy(sorted, slot_mapping, sizeof(int64_t) * (size_t)num_tokens);
    qsort(sorted, (size_t)num_tokens, sizeof(int64_t), cmp_i64);
    for (int64_t i = 1; i < num_tokens; ++i) {
        if (sorted[i] >= 0 && sorted[i] == sorted[i - 1]) {
            free(sorted);
            return ORACLE_DUPLICATE_SLOT;
        }
    }
    free(sorted);
    const int64_t row = (int64_t)num_kv_heads * head_dim; /* elements of one token, all heads */
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) return ORACLE_BAD_SLOT;
        const int64_t block = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int j = 0; j < head_dim; ++j) {
                const int64_t src = t * row + (int64_t)h * head_dim + j;
                const int64_t dst = ((block * block_size + off) * num_kv_heads + h) * head_dim + j;
                k_cache[dst] = key[src];
                v_cache[dst] = value[src];
            }
        }
    }
    return ORACLE_OK;
}

/* The cache write into an FP8 E4M3 cache ("when the KV cache meets OS
 * paging", section 6: compress inside the block): each element of the new token's K
 * (V) row, decoded from key (value) of dtype 0 (binary16) or 1 (bfloat16), is
 * stored as pa_oracle_quantize_e4m3(x, k_scale) (v_scale).  Slots as in
 * pa_oracle_reshape_and_cache. */
int pa_oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, uint8_t* k_cache,
                                    uint8_t* v_cache, const int64_t* slot_mapping, int64_t num_tokens,
                                    int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                                    int dtype, float k_scale, float v_scale) {
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) return ORACLE_BAD_SLOT;
        for (int64_t e = 0; e < row; ++e) {
            const float kx = (float)decode_elem(key[t * row + e], dtype);
            const float vx = (float)decode_elem(value[t * row + e], dtype);
            k_cache[slot * row + e] = pa_oracle_quantize_e4m3(kx, k_scale);
            v_cache[slot * row + e] = pa_oracle_quantize_e4m3(vx, v_scale);
        }
    }
    return ORACLE_OK;
}

/* Copy whole blocks, the copy step of copy-on-write ("Unveiling the NVIDIA
 * driver stack", section 4; "in-depth reading", section 2.4): for each pair
 * (src, dst) the dst block of both pools becomes a copy of the src block.
 * Pairs with an id outside the pool or src == dst are skipped; destinations
 * must be distinct and must not be the source of another pair. */
int pa_oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int64_t* block_mapping,
                          int64_t num_pairs, int64_t num_blocks, int block_size, int num_kv_heads,
                          int head_dim) {
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;
#define COPIES(k) (block_mapping[2 * (k)] >= 0 && block_mapping[2 * (k) + 1] >= 0 && \
                   block_mapping[2 * (k)] < num_blocks && block_mapping[2 * (k) + 1] < num_blocks && \
                   block_mapping[2 * (k)] != block_mapping[2 * (k) + 1])
    /* precondition, over the pairs that copy (the others write nothing) */
    for (int64_t i = 0; i < num_pairs; ++i) {
        if (!COPIES(i)) continue;
        for (int64_t j = 0; j < num_pairs; ++j) {
            if (i == j || !COPIES(j)) continue;
            const int64_t dst_i = block_mapping[2 * i + 1];
            if (dst_i == block_mapping[2 * j + 1] || dst_i == block_mapping[2 * j]) return ORACLE_BAD_ARG;
        }
    }
    const int64_t elems = (int64_t)block_size * num_kv_heads * head_dim;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = block_mapping[2 * i];
        const int64_t dst = block_mapping[2 * i + 1];
        if (!COPIES(i)) continue;
        for (int64_t e = 0; e < elems; ++e) {
            k_cache[dst * elems + e] = k_cache[src * elems + e];
            v_cache[dst * elems + e] = v_cache[src * elems + e];
        }
    }
#undef COPIES
    return ORACLE_OK;
}

/* Element `idx` of a cache of cache_dtype 0/1 (16-bit) or 2 (E4M3 bytes,
 * multiplied by its scale). */
static double cache_elem(const void* cache, int64_t idx, int cache_dtype, double cache_scale) {
    if (cache_dtype == 2) return pa_oracle_e4m3_to_double(((const uint8_t*)cache)[idx]) * cache_scale;
    return decode_elem(((const uint16_t*)cache)[idx], cache_dtype);
}

/* One (sequence, query head): gather, score, softmax, weighted sum. */
static int decode_one(double* out, const uint16_t* q_row, const void* k_cache,
                      const void* v_cache, const int32_t* table, int max_blocks_per_seq,
                      int ctx, int num_kv_heads, int kv_head, int head_dim, int block_size,
                      int64_t num_blocks, double scale, int dtype, int cache_dtype, double k_scale,
                      double v_scale) {
    if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_CONTEXT;
    for (int j = 0; j < head_dim; ++j) out[j] = 0.0;
    if (ctx == 0) return ORACLE_OK; /* an empty sequence yields zeros */

    double* K = (double*)malloc(sizeof(double) * (size_t)ctx * head_dim);
    double* V = (double*)malloc(sizeof(double) * (size_t)ctx * head_dim);
    double* x = (double*)malloc(sizeof(double) * (size_t)ctx);
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!K || !V || !x || !qd) {
        free(K); free(V); free(x); free(qd);
        return ORACLE_NO_MEMORY;
    }
    int rc = ORACLE_OK;
    /* gather the valid keys and values into contiguous [ctx, head_dim] arrays */
    for (int i = 0; i < ctx && rc == ORACLE_OK; ++i) {
        int32_t phys, off;
        pa_oracle_locate_kv(i, table, block_size, &phys, &off);
        if (phys < 0 || (int64_t)phys >= num_blocks) {
            rc = ORACLE_BAD_BLOCK;
            break;
        }
        const int64_t base = (((int64_t)phys * block_size + off) * num_kv_heads + kv_head) * head_dim;
        for (int j = 0; j < head_dim; ++j) {
            K[(size_t)i * head_dim + j] = cache_elem(k_cache, base + j, cache_dtype, k_scale);
            V[(size_t)i * head_dim + j] = cache_elem(v_cache, base + j, cache_dtype, v_scale);
        }
    }
    if (rc == ORACLE_OK) {
        for (int j = 0; j < head_dim; ++j) qd[j] = decode_elem(q_row[j], dtype);
        /* pass 1: scores and their maximum */
        double m = -INFINITY;
        for (int i = 0; i < ctx; ++i) {
            double dot = 0.0;
            for (int j = 0; j < head_dim; ++j) dot += qd[j] * K[(size_t)i * head_dim + j];
            x[i] = scale * dot;
            if (x[i] > m) m = x[i];
        }
        /* pass 2: normalised weights and the weighted sum of values */
        double denom = 0.0;
        for (int i = 0; i < ctx; ++i) {
            x[i] = exp(x[i] - m);
            denom += x[i];
        }
        for (int i = 0; i < ctx; ++i) {
            const double p = x[i] / denom;
            for (int j = 0; j < head_dim; ++j) out[j] += p * V[(size_t)i * head_dim + j];
        }
    }
    free(K); free(V); free(x); free(qd);
    return rc;
}

/* Decode attention for every (sequence, query head).
 * out: [num_seqs, num_heads, head_dim] float64; q: [num_seqs, num_heads,
 * head_dim]; block_tables: [num_seqs, max_blocks_per_seq].  q holds bit
 * patterns of dtype 0 (binary16) or 1 (bfloat16); the caches hold bit
 * patterns of cache_dtype 0 or 1, or (2) E4M3 bytes whose values are
 * multiplied by k_scale (v_scale).  num_threads <= 0 uses every available
 * thread. */
int pa_oracle_decode(double* out, const uint16_t* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                     int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, double scale, int num_threads, int dtype, int cache_dtype,
                     double k_scale, double v_scale) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || num_heads % num_kv_heads != 0 ||
        (dtype != ORACLE_FP16 && dtype != ORACLE_BF16) || cache_dtype < 0 || cache_dtype > 2)
        return ORACLE_BAD_ARG;
    const int group = num_heads / num_kv_heads;
    const int64_t work = (int64_t)num_seqs * num_heads;
    int rc = ORACLE_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int64_t w = 0; w < work; ++w) {
        const int s = (int)(w / num_heads);
        const int h = (int)(w % num_heads);
        const int r = decode_one(out + w * head_dim, q + w * head_dim, k_cache, v_cache,
                                 block_tables + (int64_t)s * max_blocks_per_seq, max_blocks_per_seq,
                                 context_lens[s], num_kv_heads, h / group, head_dim, block_size,
                                 num_blocks, scale, dtype, cache_dtype, k_scale, v_scale);
        if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            rc = r;
        }
    }
    return rc;
}

/* Paged prefill, whole or chunked.  Sequence s has query rows [qsl[s],
 * qsl[s + 1]) of q and out (qlen rows), and context_lens[s] tokens in its
 * table, the last qlen of which are the queries' own tokens (written to the
 * cache beforehand).  Query row i of the sequence sits at position
 * pos = ctx - qlen + i and attends to positions 0..pos, its own included
 * (the causal order of the prompt; "Efficient Memory Management for LLM
 * Serving with PagedAttention -- in-depth reading", section 5.1, item 5:
 * chunked prefill; "vAttention", the paged prefill kernels it measures).
 * Each (row, head) is therefore decode attention over the first pos + 1
 * tokens of the table, computed by decode_one.
 * out: [total_rows][num_heads][head_dim] float64; q: the same shape in
 * dtype 0 / 1 bit patterns; caches as pa_oracle_decode. */
int pa_oracle_prefill(double* out, const uint16_t* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      const int32_t* query_start_loc, int num_seqs, int num_heads, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, double scale, int num_threads,
                      int dtype, int cache_dtype, double k_scale, double v_scale) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || num_heads % num_kv_heads != 0 ||
        (dtype != ORACLE_FP16 && dtype != ORACLE_BF16) || cache_dtype < 0 || cache_dtype > 2)
        return ORACLE_BAD_ARG;
    if (num_seqs > 0 && query_start_loc[0] != 0) return ORACLE_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        const int qlen = query_start_loc[s + 1] - query_start_loc[s];
        if (qlen < 0 || qlen > context_lens[s]) return ORACLE_BAD_CONTEXT;
    }
    const int group = num_heads / num_kv_heads;
    const int64_t rows = num_seqs > 0 ? query_start_loc[num_seqs] : 0;
    const int64_t work = rows * num_heads;
    int rc = ORACLE_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
#endif
    for (int64_t w = 0; w < work; ++w) {
        const int64_t r = w / num_heads;
        const int h = (int)(w % num_heads);
        int s = 0;  /* the sequence of row r: the last s with query_start_loc[s] <= r */
        while (s + 1 < num_seqs && query_start_loc[s + 1] <= r) ++s;
        const int qlen = query_start_loc[s + 1] - query_start_loc[s];
        const int pos = context_lens[s] - qlen + (int)(r - query_start_loc[s]);
        const int e = decode_one(out + w * head_dim, q + w * head_dim, k_cache, v_cache,
                                 block_tables + (int64_t)s * max_blocks_per_seq, max_blocks_per_seq, pos + 1,
                                 num_kv_heads, h / group, head_dim, block_size, num_blocks, scale, dtype,
                                 cache_dtype, k_scale, v_scale);
        if (e != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            rc = e;
        }
    }
    return rc;
}

/* Threads an OpenMP region of this library would use by default. */
int pa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
