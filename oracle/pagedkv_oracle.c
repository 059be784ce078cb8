/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU reference for the decode-step
 * paged KV cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library: it has its own binary16 / bfloat16
 * decoders, its own indexing and its own arithmetic.
 *
 * What it follows (the pages, by title and section):
 *  - "从零手写 vLLM 核心：mini-vllm 项目深度解析", §2 分页KV缓存（PagedAttention）:
 *    the KV cache is cut into fixed 16-token blocks, handed out and released
 *    on demand, and blocks may be shared between sequences (prefix cache,
 *    parallel sampling).
 *  - same page, §关键工程决策 item 3: separate K and V pools, layer-major,
 *    with the block-size axis placed before the KV-head axis, i.e. one
 *    layer's pool is [num_blocks][block_size][num_kv_heads][head_dim].
 *  - same page, §关键工程决策 item 1: every layer reads its own cache length
 *    (context_lens is a per-call input here).
 *  - "micro-vLLM" wiki, execution chain (KVCacheManager): a block table maps
 *    each sequence's logical block i to a physical block id.
 *  - "MinivLLM" page, 使用教程 step 5 and 核心亮点: PagedAttention is the
 *    decode-stage attention over that cache.
 *
 * The decode attention computed here is the plain definition of attention
 * for one query token per sequence over the context gathered through the
 * block table:
 *     z_t   = scale * sum_d q[d] * K_t[d]                 (t < context_len)
 *     w_t   = exp(z_t - max_u z_u) / sum_u exp(z_u - max_u z_u)
 *     out   = sum_t w_t * V_t
 * in fp64 from the exactly decoded 16-bit inputs, with grouped-query heads
 * (query head i reads KV head i / (num_q_heads / num_kv_heads)).  Where the
 * pages are silent (GQA mapping, scale, empty context) the readings are the
 * ones the project's design notes list; an empty context (length 0) yields
 * an all-zero output.
 *
 * Parity pins (checked by the CPU test suite, not by this file): exhaustive
 * decoder comparison against numpy float16 / torch bfloat16 conversion;
 * attention against torch's scaled_dot_product_attention in float64 on a
 * context gathered independently with numpy; brute force in pure Python on
 * tiny inputs; closed forms (length 1, uniform scores, two-token logistic
 * weights); invariants (weights sum to 1, permutation of physical block ids,
 * shared prefix blocks == private copies).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PKO_OK 0
#define PKO_ERR_ARG 1
#define PKO_ERR_BLOCK_ID 2
#define PKO_ERR_SLOT 3
#define PKO_ERR_NOMEM 4

#define PKO_F16 0
#define PKO_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 is zero / subnormal (fraction * 2^-24), exponent 31 is
 * infinity (fraction 0) or NaN. */
double pko_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits.  Exponent 0 is zero / subnormal
 * (fraction * 2^-133), exponent 255 is infinity or NaN. */
double pko_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -133);
    } else if (expo == 255) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(128 + frac), expo - 134);
    }
    return sign ? -mag : mag;
}

static double decode(int dtype, uint16_t v) {
    return dtype == PKO_BF16 ? pko_bf16_to_f64(v) : pko_f16_to_f64(v);
}

/* Decode n 16-bit values into doubles (used by the tests to read GPU
 * outputs and cache contents with the oracle's own decoder). */
void pko_decode_array(int dtype, const uint16_t* src, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = decode(dtype, src[i]);
}

/* Block-table plumbing: the physical slot of the token at position
 * context_len - 1 of each sequence, i.e. the slot the new token of this
 * decode step is written to:
 *     slot = block_tables[s][p / block_size] * block_size + p % block_size.
 * A sequence with context_len <= 0 has no new token and gets slot -1. */
int pko_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int block_size,
                     int num_blocks, int64_t* slot_mapping) {
    if (!block_tables || !context_lens || !slot_mapping || block_size <= 0)
        return PKO_ERR_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int n = context_lens[s];
        if (n <= 0) { slot_mapping[s] = -1; continue; }
        int p = n - 1;
        int logical = p / block_size;
        if (logical >= max_blocks_per_seq) return PKO_ERR_ARG;
        int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + logical];
        if (b < 0 || b >= num_blocks) return PKO_ERR_BLOCK_ID;
        slot_mapping[s] = (int64_t)b * block_size + p % block_size;
    }
    return PKO_OK;
}

/* The KV write: token t's K and V rows ([num_kv_heads][head_dim] each) are
 * copied into slot slot_mapping[t] of one layer's pools.  A negative slot is
 * a padding token and is skipped.  A pure byte copy. */
int pko_reshape_and_cache(const uint16_t* k_new, const uint16_t* v_new,
                          uint16_t* k_cache, uint16_t* v_cache,
                          const int64_t* slot_mapping, int num_tokens,
                          int num_blocks, int block_size, int num_kv_heads,
                          int head_dim) {
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
        return PKO_ERR_ARG;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return PKO_ERR_SLOT;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        int64_t dst = (blk * block_size + off) * row;
        memcpy(k_cache + dst, k_new + (int64_t)t * row, (size_t)row * 2);
        memcpy(v_cache + dst, v_new + (int64_t)t * row, (size_t)row * 2);
    }
    return PKO_OK;
}

/* Decode attention in fp64.
 *  q        [num_seqs][num_q_heads][head_dim]           16-bit
 *  k_cache  [num_blocks][block_size][num_kv_heads][head_dim]
 *  v_cache  same layout as k_cache
 *  block_tables [num_seqs][max_blocks_per_seq] int32
 *  context_lens [num_seqs] int32
 *  out      [num_seqs][num_q_heads][head_dim] double
 *  weights  optional; if non-null, weights[(s*num_q_heads + i)*weights_stride + t]
 *           receives w_t for t < context_len.
 * Two passes per (sequence, query head): scores and their maximum, then the
 * exponentials, their sum and the weighted sum of V rows. */
int pko_decode_attention(int dtype, const uint16_t* q, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens,
                         int num_seqs, int num_q_heads, int num_kv_heads,
                         int head_dim, int num_blocks, int block_size,
                         double scale, double* out, double* weights,
                         int64_t weights_stride) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKO_ERR_ARG;
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0)
        return PKO_ERR_ARG;
    int group = num_q_heads / num_kv_heads;
    int max_len = max_blocks_per_seq * block_size;
    double* z = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!z || !qd) { free(z); free(qd); return PKO_ERR_NOMEM; }
    int rc = PKO_OK;
    for (int s = 0; s < num_seqs && rc == PKO_OK; ++s) {
        int n = context_lens[s];
        if (n < 0 || n > max_len) { rc = PKO_ERR_ARG; break; }
        for (int i = 0; i < num_q_heads; ++i) {
            double* o = out + ((int64_t)s * num_q_heads + i) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n == 0) continue;
            int h = i / group;
            const uint16_t* qi = q + ((int64_t)s * num_q_heads + i) * head_dim;
            for (int d = 0; d < head_dim; ++d) qd[d] = decode(dtype, qi[d]);
            double zmax = -INFINITY;
            for (int t = 0; t < n; ++t) {
                int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                if (b < 0 || b >= num_blocks) { rc = PKO_ERR_BLOCK_ID; break; }
                int64_t row = (((int64_t)b * block_size + t % block_size) * num_kv_heads + h) * head_dim;
                double acc = 0.0;
                for (int d = 0; d < head_dim; ++d) acc += qd[d] * decode(dtype, k_cache[row + d]);
                z[t] = scale * acc;
                if (z[t] > zmax) zmax = z[t];
            }
            if (rc != PKO_OK) break;
            double denom = 0.0;
            for (int t = 0; t < n; ++t) {
                z[t] = exp(z[t] - zmax);
                denom += z[t];
            }
            for (int t = 0; t < n; ++t) {
                int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                int64_t row = (((int64_t)b * block_size + t % block_size) * num_kv_heads + h) * head_dim;
                double w = z[t] / denom;
                if (weights) weights[((int64_t)s * num_q_heads + i) * weights_stride + t] = w;
                for (int d = 0; d < head_dim; ++d) o[d] += w * decode(dtype, v_cache[row + d]);
            }
        }
    }
    free(z);
    free(qd);
    return rc;
}

/* Whole-block copy of one layer's pools (the device half of copy-on-write):
 * block dst[i] receives block src[i] ([block_size][num_kv_heads][head_dim]
 * of K and of V).  A pure byte copy, pair by pair in order. */
int pko_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int32_t* src,
                    const int32_t* dst, int num_pairs, int num_blocks, int block_size,
                    int num_kv_heads, int head_dim) {
    if (!k_cache || !v_cache || !src || !dst) return PKO_ERR_ARG;
    int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks)
            return PKO_ERR_BLOCK_ID;
        memcpy(k_cache + dst[i] * blk, k_cache + src[i] * blk, (size_t)blk * 2);
        memcpy(v_cache + dst[i] * blk, v_cache + src[i] * blk, (size_t)blk * 2);
    }
    return PKO_OK;
}

/* Chunked-prefill attention in fp64 (the prefill stage's attention, here over
 * the paged cache): sequence s contributes q_len[s] query rows, packed from
 * row cu_q_lens[s], at positions context_lens[s] - q_len[s] .. context_lens[s]
 * - 1; their own K/V are already in the cache.  The query at position p
 * attends to the tokens 0..p of its sequence (causal), each head as in
 * decode attention.  q and out are [num_rows][num_q_heads][head_dim]. */
int pko_prefill_attention(int dtype, const uint16_t* q, const uint16_t* k_cache,
                          const uint16_t* v_cache, const int32_t* block_tables,
                          int max_blocks_per_seq, const int32_t* context_lens,
                          const int32_t* cu_q_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int num_blocks, int block_size,
                          double scale, double* out) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !cu_q_lens || !out)
        return PKO_ERR_ARG;
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PKO_ERR_ARG;
    int group = num_q_heads / num_kv_heads;
    int max_len = max_blocks_per_seq * block_size;
    double* z = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!z || !qd) { free(z); free(qd); return PKO_ERR_NOMEM; }
    int rc = PKO_OK;
    for (int s = 0; s < num_seqs && rc == PKO_OK; ++s) {
        int n = context_lens[s];
        int rows = cu_q_lens[s + 1] - cu_q_lens[s];
        if (n < rows || n > max_len || rows < 0) { rc = PKO_ERR_ARG; break; }
        for (int r = 0; r < rows && rc == PKO_OK; ++r) {
            int p = n - rows + r;           /* this query's position */
            int64_t qrow = (int64_t)cu_q_lens[s] + r;
            for (int i = 0; i < num_q_heads; ++i) {
                double* o = out + (qrow * num_q_heads + i) * head_dim;
                const uint16_t* qi = q + (qrow * num_q_heads + i) * head_dim;
                int h = i / group;
                for (int d = 0; d < head_dim; ++d) { qd[d] = decode(dtype, qi[d]); o[d] = 0.0; }
                double zmax = -INFINITY;
                for (int t = 0; t <= p; ++t) {
                    int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                    if (b < 0 || b >= num_blocks) { rc = PKO_ERR_BLOCK_ID; break; }
                    int64_t row = (((int64_t)b * block_size + t % block_size) * num_kv_heads + h) * head_dim;
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d) acc += qd[d] * decode(dtype, k_cache[row + d]);
                    z[t] = scale * acc;
                    if (z[t] > zmax) zmax = z[t];
                }
                if (rc != PKO_OK) break;
                double denom = 0.0;
                for (int t = 0; t <= p; ++t) { z[t] = exp(z[t] - zmax); denom += z[t]; }
                for (int t = 0; t <= p; ++t) {
                    int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                    int64_t row = (((int64_t)b * block_size + t % block_size) * num_kv_heads + h) * head_dim;
                    double w = z[t] / denom;
                    for (int d = 0; d < head_dim; ++d) o[d] += w * decode(dtype, v_cache[row + d]);
                }
            }
        }
    }
    free(z);
    free(qd);
    return rc;
}
