// pkv_cache_ops.cu -- block-table plumbing and the KV write.
//
// Layout ("从零手写 vLLM 核心：mini-vllm 项目深度解析", §关键工程决策 item 3):
// one layer's pool is [num_blocks][16][num_kv_heads][head_dim], so one slot
// (block b, row r) is a contiguous run of num_kv_heads * head_dim elements
// starting at element (b * 16 + r) * num_kv_heads * head_dim.  The write is
// therefore a gather-free scatter of whole rows: each thread moves one 16-byte
// vector, consecutive threads consecutive vectors of a row (coalesced on
// both sides).
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

// Slot of the token at position n - 1 ("mini-vllm 项目深度解析" §2: 16-token
// blocks; "micro-vLLM" wiki: block table), or -1 for an empty / invalid row.
// A bad value is reported in the status word only when `report` is set.
__device__ __forceinline__ int64_t slot_of(const int32_t* block_tables, int max_blocks_per_seq,
                                           int n, int s, int num_blocks, unsigned int* status,
                                           bool report) {
    if (n <= 0) {
        if (n < 0 && report) atomicOr(status, PKV_DEV_BAD_LENGTH);
        return -1;
    }
    if (n > max_blocks_per_seq * PKV_BLOCK_SIZE) {
        if (report) atomicOr(status, PKV_DEV_BAD_LENGTH);
        return -1;
    }
    const int p = n - 1;
    const int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + p / PKV_BLOCK_SIZE];
    if (b < 0 || b >= num_blocks) {
        if (report) atomicOr(status, PKV_DEV_BAD_BLOCK_ID);
        return -1;
    }
    return (int64_t)b * PKV_BLOCK_SIZE + p % PKV_BLOCK_SIZE;
}

__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables,
                                    int max_blocks_per_seq,
                                    const int32_t* __restrict__ context_lens, int num_seqs,
                                    int num_blocks, int64_t* __restrict__ slot_mapping,
                                    unsigned int* status) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= num_seqs) return;
    slot_mapping[s] = slot_of(block_tables, max_blocks_per_seq, context_lens[s], s, num_blocks,
                              status, true);
}

// One thread per 16-byte vector of K or V: idx -> (tensor, token, vector).
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k_new,
                                         const uint4* __restrict__ v_new,
                                         uint4* __restrict__ k_cache,
                                         uint4* __restrict__ v_cache,
                                         const int64_t* __restrict__ slot_mapping,
                                         int num_tokens, int64_t num_slots, int row_vecs,
                                         unsigned int* status) {
    const int64_t per_tensor = (int64_t)num_tokens * row_vecs;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 2 * per_tensor) return;
    const bool is_v = idx >= per_tensor;
    const int64_t r = is_v ? idx - per_tensor : idx;
    const int t = (int)(r / row_vecs);
    const int c = (int)(r % row_vecs);
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (c == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
        return;
    }
    const uint4 v = is_v ? v_new[r] : k_new[r];
    (is_v ? v_cache : k_cache)[slot * row_vecs + c] = v;
}

// Decode-step write: the slot comes from the block table and the length of
// each sequence (one new token per sequence), then the row is copied as in
// reshape_and_cache_kernel.  The first vector's thread records the slot.
__global__ void decode_step_write_kernel(const uint4* __restrict__ k_new,
                                         const uint4* __restrict__ v_new,
                                         uint4* __restrict__ k_cache,
                                         uint4* __restrict__ v_cache,
                                         const int32_t* __restrict__ block_tables,
                                         int max_blocks_per_seq,
                                         const int32_t* __restrict__ context_lens,
                                         int num_seqs, int num_blocks, int row_vecs,
                                         int64_t* __restrict__ slot_out, unsigned int* status) {
    const int64_t per_tensor = (int64_t)num_seqs * row_vecs;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 2 * per_tensor) return;
    const bool is_v = idx >= per_tensor;
    const int64_t r = is_v ? idx - per_tensor : idx;
    const int s = (int)(r / row_vecs);
    const int c = (int)(r % row_vecs);
    const bool reporter = !is_v && c == 0;  // one thread per sequence reports
    const int64_t slot = slot_of(block_tables, max_blocks_per_seq, context_lens[s], s,
                                 num_blocks, status, reporter);
    if (reporter && slot_out) slot_out[s] = slot;
    if (slot < 0) return;
    const uint4 v = is_v ? v_new[r] : k_new[r];
    (is_v ? v_cache : k_cache)[slot * row_vecs + c] = v;
}

// Whole-block copies for copy-on-write: block dst[i] of both pools receives
// block src[i] ([16][Hkv][D] each).  One CTA per pair.  Its threads first
// scan the pair list for a clash: pair i's destination is another pair's
// destination or source, or its source is another pair's destination.  Then
// the result would depend on the order in which the CTAs run, so a pair in
// clash is skipped (its blocks keep their contents) and flagged instead.  A
// pair whose source is its destination copies nothing and clashes with no
// pair on that account.  Then the CTA moves the K and V blocks, one 16-byte
// vector per thread per step.
__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, int num_pairs, int num_blocks, int block_vecs,
    unsigned int* status) {
    const int i = blockIdx.x;
    const int32_t s = src[i], d = dst[i];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (threadIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK_ID);
        return;
    }
    int clash = 0;
    for (int j = threadIdx.x; j < num_pairs; j += blockDim.x) {
        if (j == i) continue;
        const int32_t sj = src[j], dj = dst[j];
        if (dj == d || (sj == d && s != d) || dj == s) clash = 1;
    }
    if (__syncthreads_or(clash)) {
        if (threadIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK_ID);
        return;
    }
    if (s == d) return;
    for (int r = threadIdx.x; r < 2 * block_vecs; r += blockDim.x) {
        const bool is_v = r >= block_vecs;
        const int c = is_v ? r - block_vecs : r;
        uint4* pool = is_v ? v_cache : k_cache;
        pool[(int64_t)d * block_vecs + c] = pool[(int64_t)s * block_vecs + c];
    }
}

}  // namespace

// Launches the decode-step write (used by paged_kv_decode_step).
pkv_status launch_decode_step_write(const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    int num_seqs, int num_blocks, int num_kv_heads, int head_dim,
                                    int64_t* slot_out, cudaStream_t stream) {
    unsigned int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int row_vecs = num_kv_heads * head_dim / 8;
    const int64_t total = 2ll * num_seqs * row_vecs;
    const int grid = (int)((total + kThreads - 1) / kThreads);
    decode_step_write_kernel<<<grid, kThreads, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_tables,
        max_blocks_per_seq, context_lens, num_seqs, num_blocks, row_vecs, slot_out, status);
    return cuda_status(cudaGetLastError());
}

}  // namespace pkv

extern "C" {

pkv_status paged_kv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_blocks,
                                 int64_t* slot_mapping, pkv_stream_t stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables || !context_lens || !slot_mapping) return PKV_ERR_INVALID_ARG;
    unsigned int* status = pkv::status_word();
    if (!status) return PKV_ERR_CUDA;
    const int threads = 128;
    pkv::slot_mapping_kernel<<<(num_seqs + threads - 1) / threads, threads, 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(
        block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks, slot_mapping,
        status);
    return pkv::cuda_status(cudaGetLastError());
}

pkv_status reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, const int64_t* slot_mapping, int num_tokens,
                             int num_blocks, int num_kv_heads, int head_dim, pkv_dtype dtype,
                             pkv_stream_t stream) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || !pkv::aligned16(k_cache) ||
        !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    unsigned int* status = pkv::status_word();
    if (!status) return PKV_ERR_CUDA;
    const int row_vecs = num_kv_heads * head_dim / 8;
    const int64_t total = 2ll * num_tokens * row_vecs;
    const int grid = (int)((total + pkv::kThreads - 1) / pkv::kThreads);
    pkv::reshape_and_cache_kernel<<<grid, pkv::kThreads, 0,
                                    reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, num_tokens,
        (int64_t)num_blocks * PKV_BLOCK_SIZE, row_vecs, status);
    return pkv::cuda_status(cudaGetLastError());
}

pkv_status paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_block_ids,
                                const int32_t* dst_block_ids, int num_pairs, int num_blocks,
                                int num_kv_heads, int head_dim, pkv_dtype dtype,
                                pkv_stream_t stream) {
    if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_block_ids || !dst_block_ids) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k_cache) || !pkv::aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
    unsigned int* status = pkv::status_word();
    if (!status) return PKV_ERR_CUDA;
    const int block_vecs = PKV_BLOCK_SIZE * num_kv_heads * head_dim / 8;
    pkv::copy_blocks_kernel<<<num_pairs, pkv::kThreads, 0,
                              reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src_block_ids,
        dst_block_ids, num_pairs, num_blocks, block_vecs, status);
    return pkv::cuda_status(cudaGetLastError());
}

}  // extern "C"
