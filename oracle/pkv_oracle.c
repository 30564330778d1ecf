/*
 * CPU oracle for the paged KV cache hot path, plain C, fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library; the CUDA library never calls it and
 * shares no code, header or table with it.
 *
 * Two operations, each the plain definition written out:
 *
 *   oracle_write   -- the reshape_and_cache scatter: each new token's key and
 *                     value rows are copied, bit for bit, into the slot that
 *                     slot_mapping names (block = slot / B, offset = slot % B).
 *                     "[vLLM] PagedAttention: OS 페이징 기법으로 KV 캐시를 관리하는
 *                     방법", PagedAttention 커널 (write_to_paged_cache ->
 *                     ops.reshape_and_cache); slot arithmetic as in "KV Cache와
 *                     PagedAttention 완전 해부", §5단계 and §6단계 (block 42,
 *                     slots 0..5, next token into slot 6).
 *
 *   oracle_copy_blocks -- the copy-on-write block copy (see below).
 *
 *   oracle_decode  -- decode attention of one query token per sequence over its
 *                     first context_lens[s] cached tokens. The cached K and V
 *                     rows are first gathered through the block table into
 *                     contiguous fp64 arrays, then
 *                         x_j = scale * sum_d q[d] * K[j][d]
 *                         w_j = exp(x_j - max x) / sum_i exp(x_i - max x)
 *                         o[d] = sum_j w_j * V[j][d]
 *                     "KV Cache와 PagedAttention 완전 해부", 부록 (Attention =
 *                     softmax(Q K^T / sqrt d) V); "vLLM: LLM 서빙 메모리 최적화의
 *                     교과서", 01 Problem Definition (a_ij, o_i) and eq. (4),
 *                     whose block-wise form gives the same o_i. Subtracting
 *                     max x leaves w unchanged (it cancels in the ratio).
 *                     Query head h reads kv head h / (H / Hkv) (contiguous
 *                     GQA groups). A context of 0 tokens gives o = 0.
 *
 *   oracle_multi_query -- several query tokens per sequence (a chunked-prefill
 *                     chunk or the tokens a speculative step verifies:
 *                     "Sparse Computation and Memory Management for Efficient
 *                     LLM Inference", the chunked prefill paragraph and
 *                     Speculative Decoding). Sequence s has q_len =
 *                     query_start_loc[s+1] - query_start_loc[s] query tokens;
 *                     they are its last q_len context positions, and query
 *                     token i (position p = ctx - q_len + i) attends the
 *                     positions j <= p, as a_ij and o_i are defined over
 *                     j <= i in "vLLM: LLM 서빙 메모리 최적화의 교과서", 01
 *                     Problem Definition. Each output row is oracle_decode's
 *                     formula over the first p + 1 cached tokens.
 *
 * fp16/bf16 inputs are widened to double exactly from their bit patterns. An
 * FP8 (E4M3) cache holds codes of value / scale; its elements are code * scale,
 * computed exactly in double (oracle_write_fp8, oracle_e4m3_*).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double widen_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double widen(uint16_t bits, int dtype) {
    return dtype == 0 ? widen_f16(bits) : widen_bf16(bits);
}

double oracle_widen(uint16_t bits, int dtype) { return widen(bits, dtype); }

/*
 * FP8 E4M3 (the OCP 8-bit format with 4 exponent bits): 1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; the
 * largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the
 * subnormals m/8 * 2^-6.
 */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* Nearest E4M3 value to x, ties to the even mantissa, magnitudes above 448 saturated to 448. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_d = a; /* distance to code 0 (value 0) */
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/*
 * The quantizing cache write of an FP8 cache: code = E4M3(value / scale), the
 * division done in fp32 (correctly rounded) and the result rounded to the
 * nearest E4M3 value with saturation. "[vLLM] PagedAttention: ...",
 * write_to_paged_cache(..., kv_cache_dtype, k_scale, v_scale). Returns the
 * number of tokens written, or -(t + 1) for the first token whose slot lies
 * outside the pool.
 */
long long oracle_write_fp8(const uint16_t* key, const uint16_t* value, uint8_t* key_cache, uint8_t* value_cache,
                           const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                           int block_size, long long num_blocks, int src_dtype, float k_scale, float v_scale) {
    long long written = 0, bad = 0;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            if (!bad) bad = -(long long)(t + 1);
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                float kf = (float)widen(key[src + d], src_dtype);
                float vf = (float)widen(value[src + d], src_dtype);
                key_cache[dst + d] = oracle_e4m3_encode(kf / k_scale);
                value_cache[dst + d] = oracle_e4m3_encode(vf / v_scale);
            }
        }
        ++written;
    }
    return bad ? bad : written;
}

/*
 * Returns the number of tokens written, or -(t + 1) for the first token t
 * whose slot lies outside the pool (nothing is written for that token).
 */
long long oracle_write(const uint16_t* key, const uint16_t* value, uint16_t* key_cache,
                       uint16_t* value_cache, const int64_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size, long long num_blocks) {
    long long written = 0, bad = 0;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token */
        if (slot >= (int64_t)num_blocks * block_size) {
            if (!bad) bad = -(long long)(t + 1);
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            memcpy(key_cache + dst, key + src, sizeof(uint16_t) * head_dim);
            memcpy(value_cache + dst, value + src, sizeof(uint16_t) * head_dim);
        }
        ++written;
    }
    return bad ? bad : written;
}

/*
 * The block copy of copy-on-write: for each pair (src, dst) of block_mapping,
 * every kv head's K and V rows of physical block src are copied, bit for bit,
 * into block dst. "Sparse Computation and Memory Management for Efficient LLM
 * Inference", Copy-on-Write (append_kv_with_cow: fused_block_copy(phys,
 * new_phys) before the write); "KV Cache와 PagedAttention 완전 해부", §9단계.
 * Sources are read as they were before the call. Returns the number of pairs
 * copied, or -(i + 1) for the first pair i naming a block outside the pool
 * (that pair is skipped).
 */
long long oracle_copy_blocks(uint16_t* key_cache, uint16_t* value_cache, const int64_t* block_mapping,
                             int num_pairs, int num_kv_heads, int head_dim, int block_size,
                             long long num_blocks) {
    const size_t per_block = (size_t)num_kv_heads * block_size * head_dim;
    long long copied = 0, bad = 0;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (!bad) bad = -(long long)(i + 1);
            continue;
        }
        memmove(key_cache + dst * per_block, key_cache + src * per_block, sizeof(uint16_t) * per_block);
        memmove(value_cache + dst * per_block, value_cache + src * per_block, sizeof(uint16_t) * per_block);
        ++copied;
    }
    return bad ? bad : copied;
}

/* One (sequence, query head) pair. Returns 0, or -1 on a block id outside the pool. */
/* Cache element j of a pool of 16-bit (cache_dtype 0, 1) or E4M3 (cache_dtype 2) elements, in value units. */
static double cache_value(const void* cache, size_t j, int cache_dtype, double scale) {
    if (cache_dtype == 2) return oracle_e4m3_decode(((const uint8_t*)cache)[j]) * scale;
    return widen(((const uint16_t*)cache)[j], cache_dtype);
}

static int decode_pair(double* out, const uint16_t* query, const void* key_cache,
                       const void* value_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, double scale,
                       int block_size, int num_heads, int num_kv_heads, int head_dim,
                       long long num_blocks, int dtype, int cache_dtype, double k_scale, double v_scale,
                       int s, int h) {
    const int D = head_dim, B = block_size;
    double* o = out + ((size_t)s * num_heads + h) * D;
    int ctx = context_lens[s];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (ctx <= 0) return 0;
    const int group = num_heads / num_kv_heads;
    const int g = h / group;

    /* gather the sequence's K and V rows into contiguous arrays */
    double* K = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    double* x = (double*)malloc(sizeof(double) * (size_t)ctx);
    double* q = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = 0;
    for (int j = 0; j < ctx && !rc; ++j) {
        long long phys = block_tables[(size_t)s * max_blocks_per_seq + j / B];
        if (phys < 0 || phys >= num_blocks) { rc = -1; break; }
        size_t base = (((size_t)phys * num_kv_heads + g) * B + (j % B)) * D;
        for (int d = 0; d < D; ++d) {
            K[(size_t)j * D + d] = cache_value(key_cache, base + d, cache_dtype, k_scale);
            V[(size_t)j * D + d] = cache_value(value_cache, base + d, cache_dtype, v_scale);
        }
    }
    if (!rc) {
        for (int d = 0; d < D; ++d) q[d] = widen(query[((size_t)s * num_heads + h) * D + d], dtype);
        /* scores */
        double mx = -INFINITY;
        for (int j = 0; j < ctx; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)j * D + d];
            x[j] = scale * acc;
            if (x[j] > mx) mx = x[j];
        }
        /* softmax weights */
        double den = 0.0;
        for (int j = 0; j < ctx; ++j) {
            x[j] = exp(x[j] - mx);
            den += x[j];
        }
        /* weighted sum of values */
        for (int j = 0; j < ctx; ++j) {
            double w = x[j] / den;
            for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)j * D + d];
        }
    }
    free(K);
    free(V);
    free(x);
    free(q);
    return rc;
}

/*
 * out: [S][H][D] doubles (only the selected pairs are written).
 * pairs: NULL for every (s, h), else npairs (s, h) int32 pairs.
 * num_threads: <= 0 uses the OpenMP default. Returns 0, or -1 if any block id
 * lies outside the pool.
 */
int oracle_decode(double* out, const uint16_t* query, const void* key_cache,
                  const void* value_cache, const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs, double scale, int block_size,
                  int num_heads, int num_kv_heads, int head_dim, long long num_blocks, int dtype,
                  int cache_dtype, double k_scale, double v_scale,
                  const int32_t* pairs, long long npairs, int num_threads) {
    long long n = pairs ? npairs : (long long)num_seqs * num_heads;
    int rc = 0;
#ifdef _OPENMP
    /* a thread count for this loop only: omp_set_num_threads would outlive the call */
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc) num_threads(nt)
#else
    (void)num_threads;
#endif
    for (long long i = 0; i < n; ++i) {
        int s = pairs ? pairs[2 * i] : (int)(i / num_heads);
        int h = pairs ? pairs[2 * i + 1] : (int)(i % num_heads);
        rc |= decode_pair(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                          context_lens, scale, block_size, num_heads, num_kv_heads, head_dim,
                          num_blocks, dtype, cache_dtype, k_scale, v_scale, s, h);
    }
    return rc ? -1 : 0;
}

/*
 * One (sequence, query head) pair of the multi-query case: all q_len query
 * rows of the sequence. Returns 0, -1 on a block id outside the pool, or -2 if
 * q_len is negative or larger than the context.
 */
static int mq_pair(double* out, const uint16_t* query, const void* key_cache, const void* value_cache,
                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                   const int32_t* query_start_loc, double scale, int block_size, int num_heads,
                   int num_kv_heads, int head_dim, long long num_blocks, int dtype, int cache_dtype,
                   double k_scale, double v_scale, int s, int h) {
    const int D = head_dim, B = block_size;
    const int ctx = context_lens[s];
    const int q0 = query_start_loc[s], q_len = query_start_loc[s + 1] - q0;
    if (q_len < 0 || q_len > ctx) return -2;
    if (q_len == 0) return 0;
    const int group = num_heads / num_kv_heads;
    const int g = h / group;

    /* gather the sequence's K and V rows into contiguous arrays */
    double* K = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    double* x = (double*)malloc(sizeof(double) * (size_t)ctx);
    double* q = (double*)malloc(sizeof(double) * (size_t)D);
    int rc = 0;
    for (int j = 0; j < ctx && !rc; ++j) {
        long long phys = block_tables[(size_t)s * max_blocks_per_seq + j / B];
        if (phys < 0 || phys >= num_blocks) { rc = -1; break; }
        size_t base = (((size_t)phys * num_kv_heads + g) * B + (j % B)) * D;
        for (int d = 0; d < D; ++d) {
            K[(size_t)j * D + d] = cache_value(key_cache, base + d, cache_dtype, k_scale);
            V[(size_t)j * D + d] = cache_value(value_cache, base + d, cache_dtype, v_scale);
        }
    }
    for (int i = 0; i < q_len && !rc; ++i) {
        const size_t row = (size_t)(q0 + i) * num_heads + h;
        double* o = out + row * D;
        const int n = ctx - q_len + i + 1; /* tokens at positions 0 .. ctx - q_len + i */
        for (int d = 0; d < D; ++d) {
            o[d] = 0.0;
            q[d] = widen(query[row * D + d], dtype);
        }
        double mx = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)j * D + d];
            x[j] = scale * acc;
            if (x[j] > mx) mx = x[j];
        }
        double den = 0.0;
        for (int j = 0; j < n; ++j) {
            x[j] = exp(x[j] - mx);
            den += x[j];
        }
        for (int j = 0; j < n; ++j) {
            double w = x[j] / den;
            for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)j * D + d];
        }
    }
    free(K);
    free(V);
    free(x);
    free(q);
    return rc;
}

/*
 * out: [query_start_loc[num_seqs]][H][D] doubles; query likewise (bits).
 * query_start_loc: [num_seqs + 1] int32, non-decreasing, starting at 0.
 * Returns 0, -1 if a block id lies outside the pool, -2 on a bad q_len.
 */
int oracle_multi_query(double* out, const uint16_t* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                       const int32_t* query_start_loc, int num_seqs, double scale, int block_size,
                       int num_heads, int num_kv_heads, int head_dim, long long num_blocks, int dtype,
                       int cache_dtype, double k_scale, double v_scale, int num_threads) {
    long long n = (long long)num_seqs * num_heads;
    int rc1 = 0, rc2 = 0;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc1, rc2) num_threads(nt)
#else
    (void)num_threads;
#endif
    for (long long i = 0; i < n; ++i) {
        int r = mq_pair(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start_loc, scale, block_size, num_heads, num_kv_heads, head_dim, num_blocks,
                        dtype, cache_dtype, k_scale, v_scale, (int)(i / num_heads), (int)(i % num_heads));
        if (r == -1) rc1 = 1;
        if (r == -2) rc2 = 1;
    }
    return rc1 ? -1 : (rc2 ? -2 : 0);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
