/*
 * pagedkv.h -- C ABI of libpagedkv: decode-step PagedAttention over a
 * block-paged KV cache on one GB300 (sm_103a).
 *
 * Sources (page title, section):
 *  [P1] "micro-vLLM" wiki -- execution chain: the KVCacheManager manages
 *       logical blocks, the block table, the prefix cache, and allocation and
 *       release; the ModelRunner owns the physical KV cache.
 *  [P2] "MinivLLM -- 用最小代码读懂 vLLM 推理内核" -- 使用教程 step 5 and
 *       核心亮点: a self-written PagedAttention serves the decode stage.
 *  [P3] "从零手写 vLLM 核心：mini-vllm 项目深度解析" -- §2 分页KV缓存: the cache
 *       is cut into fixed 16-token blocks, allocated and released on demand,
 *       shareable between sequences (prefix cache, parallel sampling), and
 *       correct under pressure through admission control; §关键工程决策
 *       item 1: each layer reads its own cache length; item 3: K and V
 *       pools are separate and layer-major, with the block-size axis before
 *       the KV-head axis, and attention reads views, not strided copies.
 *
 * Conventions shared by every device entry point:
 *  - All pointers to tensors are DEVICE pointers owned by the caller unless a
 *    parameter says "host".  The library never allocates, frees or keeps a
 *    reference to caller memory after the call returns; work is enqueued on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and the call
 *    does not synchronise.
 *  - One layer's pool (K or V) is contiguous [num_blocks][16][num_kv_heads]
 *    [head_dim] of 16-bit elements ([P3] item 3).  A layer-major stack of L
 *    pools is L such arrays back to back; pass the base of one layer.
 *  - q, K, V and out share one dtype (PKV_F16 or PKV_BF16); arithmetic is
 *    fp32 inside the kernels; outputs are rounded to nearest even.
 *  - block_tables [num_seqs][max_blocks_per_seq] int32 map logical block j
 *    of sequence s to a physical block id in [0, num_blocks) ([P1]).  Only
 *    entries j < ceil(context_lens[s] / 16) are read.
 *  - context_lens [num_seqs] int32 count the tokens of each sequence INCLUDING
 *    the token written this step (it sits at position context_len - 1).  A
 *    length of 0 is a padding row whose attention output is all zeros.
 *  - Arguments are validated on the host; a bad argument returns an error
 *    and enqueues nothing.  Values that live on the device (block ids,
 *    lengths, slots) are checked by the kernels themselves: a bad value is
 *    never dereferenced, the affected row is skipped or zero-filled, and a
 *    bit is set in the device status word (pkv_device_status).  No kernel
 *    traps, asserts or spins without a bound.
 *  - The decode partition pass, the merge pass and the host-input staging
 *    kernel are launched as programmatic dependents of the kernel before them
 *    on the stream, so their CTAs are scheduled while it drains.  Each waits
 *    for that kernel to complete (griddepcontrol.wait, which also makes its
 *    stores visible) before it reads or writes any caller memory, whatever
 *    that kernel is.  One exception, internal to a call: in
 *    paged_kv_decode_step_layers the partition pass of layer l > 0 reads
 *    context_lens, block_tables, layer l's q, k_new, v_new and pools, and
 *    writes layer l's pools and out, before that wait: the kernel before it
 *    is layer l - 1's, which touches none of them.  It waits before its
 *    first workspace write (layer l - 1's merge reads the workspace) and
 *    before it ends, so that it never completes before that kernel.  The
 *    TMA partition pass (after its prologue) and the merge pass (once its
 *    partition pass has finished) let the next kernel's CTAs be scheduled
 *    before they end; a dependent of another library must then wait for
 *    them (griddepcontrol.wait) before it reads their outputs, as
 *    programmatic dependent launch requires of any dependent.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (struct CUstream_st*), spelled without CUDA headers. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes */
    PKV_ERR_UNSUPPORTED = 2,   /* a valid shape the library has no kernel for */
    PKV_ERR_NO_BLOCKS = 3,     /* allocator: not enough free blocks (nothing taken) */
    PKV_ERR_BAD_BLOCK_ID = 4,  /* allocator: id out of range or not allocated */
    PKV_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    PKV_ERR_WORKSPACE = 6      /* workspace null or smaller than required */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Tokens per physical block, fixed by [P3] §2. */
#define PKV_BLOCK_SIZE 16

/* Bits of the device status word (see pkv_device_status). */
#define PKV_DEV_BAD_BLOCK_ID 0x1u   /* a table entry outside [0, num_blocks) was skipped */
#define PKV_DEV_BAD_LENGTH   0x2u   /* a context length < 0 or beyond the table / bound */
#define PKV_DEV_BAD_SLOT     0x4u   /* a slot >= num_blocks * 16 was skipped by the write */
#define PKV_DEV_TIMEOUT      0x8u   /* a kernel gave up an internal wait (~2 s) and returned */

/* Library version (major * 10000 + minor * 100 + patch). */
int pkv_version(void);

/* Static text for a status code. */
const char* pkv_status_string(pkv_status status);

/* Bytes of ONE pool (K or V) holding `num_layers` layer-major layers of
 * [num_blocks][block_size][num_kv_heads][head_dim] ([P3] item 3).  Returns 0
 * for a non-positive size or a block_size other than 16. */
size_t pkv_cache_bytes(int num_layers, int num_blocks, int block_size, int num_kv_heads,
                       int head_dim, pkv_dtype dtype);

/* ---------------------------------------------------------------------------
 * Host block allocator ([P1] KVCacheManager; [P3] §2: on-demand allocation
 * and release, sharing through reference counts, admission control).  Plain
 * host memory owned by the handle; not thread-safe (one owner thread).
 * ------------------------------------------------------------------------- */
typedef struct pkv_allocator pkv_allocator;

/* Creates an allocator over block ids [0, num_blocks), all free. */
pkv_status paged_kv_alloc_create(int num_blocks, pkv_allocator** out);
void paged_kv_alloc_destroy(pkv_allocator* a);

/* Takes n free blocks (reference count 1 each) into out_block_ids[n] (host).
 * All or nothing: with fewer than n free blocks nothing is taken and
 * PKV_ERR_NO_BLOCKS is returned, so a scheduler can refuse admission. */
pkv_status paged_kv_alloc(pkv_allocator* a, int n, int32_t* out_block_ids);

/* Adds one reference to each listed allocated block (a sequence starts
 * sharing a prefix block).  All or nothing: PKV_ERR_BAD_BLOCK_ID if any id is
 * out of range or free. */
pkv_status paged_kv_share(pkv_allocator* a, int n, const int32_t* block_ids);

/* Drops one reference from each listed block; a block whose count reaches 0
 * returns to the free list.  All or nothing: PKV_ERR_BAD_BLOCK_ID if any id
 * is out of range or free, or is listed more often than it is referenced. */
pkv_status paged_kv_free(pkv_allocator* a, int n, const int32_t* block_ids);

int paged_kv_num_free(const pkv_allocator* a);

/* Reference count of one block (0 = free or cached), or -1 for an id out of range. */
int paged_kv_refcount(const pkv_allocator* a, int32_t block_id);

/* ---------------------------------------------------------------------------
 * Prefix cache, copy-on-write and rollback ([P1] KVCacheManager: prefix
 * cache; [P3] §2: blocks shared by sequences with a common prefix; [P3]
 * §工程启示: KV rollback for speculative decoding).
 *
 * A full block can be registered under a 64-bit hash of its content and of
 * everything before it (paged_kv_block_hash chains a parent hash with the
 * block's 16 token ids).  When its count drops to 0 a registered block is
 * not freed but kept as "cached": paged_kv_prefix_lookup can revive it for a
 * new sequence with the same prefix, and paged_kv_alloc evicts cached blocks
 * (least recently released first) only once the free blocks run out.
 * paged_kv_num_free counts free and cached blocks alike (both can be taken).
 * ------------------------------------------------------------------------- */

/* Hash of one block: chains `parent_hash` (0 for the first block of a
 * sequence) with the block's token ids (splitmix64 mixing; deterministic
 * across runs and machines). */
uint64_t paged_kv_block_hash(uint64_t parent_hash, const int32_t* tokens, int num_tokens);

/* Registers live block `block_id` as holding the content named by `hash`.
 * If another block already holds that hash, nothing changes (PKV_OK). A
 * block that already carries a different hash gives PKV_ERR_INVALID_ARG; a
 * block that is not live gives PKV_ERR_BAD_BLOCK_ID. */
pkv_status paged_kv_prefix_insert(pkv_allocator* a, int32_t block_id, uint64_t hash);

/* Looks up hashes[0..n) in order and stops at the first miss.  Every hit
 * gains one reference (a cached block becomes live again) and its id goes to
 * out_block_ids[i]; *num_hits receives the number of leading hits. */
pkv_status paged_kv_prefix_lookup(pkv_allocator* a, int n, const uint64_t* hashes,
                                  int32_t* out_block_ids, int* num_hits);

/* Number of blocks registered in the prefix cache (live or cached). */
int paged_kv_num_cached(const pkv_allocator* a);

/* Copy-on-write before writing into live block `block_id`.  If the caller
 * holds the only reference, the block keeps its id (*needs_copy = 0) and
 * leaves the prefix cache (its content is about to change).  Otherwise a new
 * block is taken (*out_block_id, *needs_copy = 1), the caller's reference
 * moves to it, and the caller must copy the block's contents on the device
 * (paged_kv_copy_blocks) before writing.  PKV_ERR_NO_BLOCKS if none can be
 * taken (nothing changes). */
pkv_status paged_kv_cow(pkv_allocator* a, int32_t block_id, int32_t* out_block_id,
                        int* needs_copy);

/* Rollback of a sequence to new_len tokens (e.g. rejected speculative
 * tokens): drops the references of block_table[ceil(new_len/16) ..
 * num_table_blocks) (host table; those entries become -1) and returns the
 * kept block count.  A kept last block that becomes partial leaves the
 * prefix cache when the caller holds its only reference; if it is shared the
 * caller must copy-on-write before writing into it.  All or nothing:
 * PKV_ERR_INVALID_ARG if new_len needs more blocks than the table has,
 * PKV_ERR_BAD_BLOCK_ID if a dropped entry is out of range, free, or listed
 * more often than it is referenced. */
pkv_status paged_kv_rollback(pkv_allocator* a, int32_t* block_table, int num_table_blocks,
                             int new_len, int* new_num_blocks);

/* ---------------------------------------------------------------------------
 * Device operations
 * ------------------------------------------------------------------------- */

/* Block-table plumbing ([P1] block table; [P3] §2 16-token blocks, item 1):
 * for each sequence s with n = context_lens[s] > 0,
 *     slot_mapping[s] = block_tables[s][(n-1)/16] * 16 + (n-1) % 16
 * (the slot of this step's token); n == 0 gives -1.  A length beyond the
 * table or a table entry outside [0, num_blocks) gives -1 and sets a status
 * bit.  slot_mapping: [num_seqs] int64, device. */
pkv_status paged_kv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_blocks,
                                 int64_t* slot_mapping, pkv_stream_t stream);

/* The KV write ([P3] item 3 layout): for each token t with slot =
 * slot_mapping[t] >= 0, copies k_new[t] and v_new[t] ([num_kv_heads][head_dim]
 * each) into row slot % 16 of physical block slot / 16 of one layer's pools.
 * slot < 0 marks a padding token (skipped); slot >= num_blocks * 16 is
 * skipped and flagged.  Slots must be unique within a call.  Bit-exact copy.
 * k_new, v_new: [num_tokens][num_kv_heads][head_dim]; k_cache, v_cache: one
 * layer's pools; head_dim * 2 bytes must be a multiple of 16. */
pkv_status reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, const int64_t* slot_mapping, int num_tokens,
                             int num_blocks, int num_kv_heads, int head_dim, pkv_dtype dtype,
                             pkv_stream_t stream);

/* Whole-block copies in both pools of one layer (the device half of
 * copy-on-write): block dst_block_ids[i] receives block src_block_ids[i]
 * ([16][num_kv_heads][head_dim] of K and of V), for i < num_pairs.  Both id
 * arrays are device int32; an id outside [0, num_blocks) skips that pair and
 * sets PKV_DEV_BAD_BLOCK_ID.  The destinations must be distinct and none may
 * be the source of another pair (a pair with src == dst copies nothing):
 * otherwise the outcome would depend on the order in which the copies run,
 * so every pair in such a clash is skipped, its blocks left as they were, and
 * PKV_DEV_BAD_BLOCK_ID is set; the other pairs are copied.  num_pairs is at
 * most 2^31 - 1.  Bit-exact copy. */
pkv_status paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_block_ids,
                                const int32_t* dst_block_ids, int num_pairs, int num_blocks,
                                int num_kv_heads, int head_dim, pkv_dtype dtype,
                                pkv_stream_t stream);

/* Workspace (bytes) paged_attention_decode needs for these sizes: the
 * split-context partials (running max, running sum and unnormalised output
 * per partition and query head, fp32) plus partition offsets.  The caller
 * allocates it (device, 256-byte aligned) and may reuse it across calls on
 * the same stream; its contents need no initialisation. */
size_t paged_attention_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                       int max_context_len);

/* Decode attention ([P2] step 5; [P3] §2, items 1 and 3): for each sequence s
 * and query head i, with n = context_lens[s] and KV head h = i / (num_q_heads
 * / num_kv_heads), over the n tokens found through block_tables[s]:
 *     z_t = scale * <q[s][i], K_t[h]>,  w = softmax(z),  out[s][i] = sum_t w_t V_t[h].
 * The work is cut into pieces processed in parallel, each keeping a running
 * max and sum (online softmax); a merge kernel combines the pieces of a
 * sequence by log-sum-exp.  With a table of 64 or more blocks the (sequence,
 * KV-head group, block) units are split evenly over the persistent CTAs;
 * shorter tables are cut into partitions of near-equal size.
 *  q, out:     [num_seqs][num_q_heads][head_dim], dtype.
 *  k_cache, v_cache: one layer's pools, dtype.
 *  max_context_len: host upper bound on every context_lens[s] (sizes grids
 *              and the workspace); a device length above it (or above
 *              max_blocks_per_seq * 16, or negative) is flagged and its output
 *              row is written as zeros.
 *  workspace:  >= paged_attention_workspace_bytes(num_seqs, num_q_heads,
 *              head_dim, max_context_len) bytes, else PKV_ERR_WORKSPACE.
 * Supported: head_dim 64 or 128, num_q_heads / num_kv_heads in 1..8,
 * num_seqs <= 8192; else PKV_ERR_UNSUPPORTED. */
pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int max_context_len,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int num_blocks, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream);

/* As paged_attention_decode, with the partition length fixed by the caller:
 * a sequence of n blocks is cut into ceil(n / partition_blocks) partitions
 * of near-equal size (at most partition_blocks physical blocks of 16 tokens
 * each); 0 picks the length from the device-side lengths as
 * paged_attention_decode does.
 * The result does not depend on the partition length beyond fp32 rounding.
 * partition_blocks must be >= paged_attention_min_partition_blocks(
 * max_context_len) so that the workspace bound holds. */
pkv_status paged_attention_decode_partitioned(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream);

/* Smallest partition length (blocks) the workspace bound allows. */
int paged_attention_min_partition_blocks(int max_context_len);

/* The two passes of paged_attention_decode_partitioned, enqueued separately
 * (same arguments, same workspace, same partition_blocks; call the partition
 * pass first).  The partition pass computes, per piece (a partition, or with
 * partition_blocks = 0 and a table of 64 or more blocks a CTA's share of a
 * sequence and KV-head group), the running max, running sum and unnormalised
 * output of each query head, and writes sequences held by one piece straight
 * to `out`; the merge pass combines the pieces of the other sequences by
 * log-sum-exp:
 *     M = max_p m_p,  L = sum_p l_p e^(m_p - M),  out = sum_p o_p e^(m_p - M) / L.
 * The merge pass enqueues nothing when no sequence can span two partitions. */
pkv_status paged_attention_partition_pass(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream);
pkv_status paged_attention_merge_pass(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream);

/* The write half of a decode step ([P3] §2 and item 1): for each sequence
 * with n = context_lens[s] > 0, copies k_new[s] and v_new[s]
 * ([num_seqs][num_kv_heads][head_dim]) to the slot of position n - 1
 * (as paged_kv_slot_mapping computes it) in one layer's pools.  An empty or
 * invalid row writes nothing (invalid values are flagged).  slot_mapping_out
 * may be NULL. */
pkv_status paged_kv_write_new_tokens(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* context_lens,
                                     int num_seqs, int num_blocks, int num_kv_heads,
                                     int head_dim, int64_t* slot_mapping_out, pkv_dtype dtype,
                                     pkv_stream_t stream);

/* One decode step of one layer ([P3] §2 and item 1: write, then attend):
 * the result of paged_kv_write_new_tokens followed by paged_attention_decode.
 * The write is fused into the partition pass: the warp that reads a
 * sequence's last block takes the new token's row from k_new / v_new and
 * stores it into its slot, so one kernel writes and attends, and the merge
 * pass follows. Within the call, nothing reads the new rows back from the cache.
 * slot_mapping_out may be NULL; if not, it receives the slots ([num_seqs]
 * int64, device). */
pkv_status paged_kv_decode_step(const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int max_context_len, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int num_blocks, float scale,
                                void* out, int64_t* slot_mapping_out, void* workspace,
                                size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Cascade decode for a shared prefix ([P3] §2: blocks shared between
 * sequences, prefix cache / parallel sampling).  Precondition: the first
 * num_prefix_blocks entries of EVERY sequence's block table name the same
 * physical blocks, and those blocks are full (16 tokens each).  Then the
 * prefix is attended once for all sharers: a prefix pass puts query vectors
 * of several sequences side by side against each prefix K/V row, the
 * partition pass covers each sequence's own blocks after the prefix, and the
 * merge combines them by log-sum-exp.  A sequence shorter than the prefix
 * sees only its own length of it.  The result is that of
 * paged_attention_decode (up to fp32 rounding); only the reads change.
 * ------------------------------------------------------------------------- */
size_t paged_attention_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                               int max_context_len, int num_prefix_blocks);

pkv_status paged_attention_decode_cascade(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int max_context_len, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int num_blocks,
                                          int num_prefix_blocks, float scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          pkv_dtype dtype, pkv_stream_t stream);

/* paged_kv_decode_step with the cascade: every sequence's new token must lie
 * past the shared prefix (context_len - 1 >= 16 * num_prefix_blocks); a
 * sequence whose token would land in a shared block is flagged
 * (PKV_DEV_BAD_LENGTH) and its token is not written. */
pkv_status paged_kv_decode_step_cascade(const void* q, const void* k_new, const void* v_new,
                                        void* k_cache, void* v_cache,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* context_lens, int max_context_len,
                                        int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int num_blocks, int num_prefix_blocks,
                                        float scale, void* out, int64_t* slot_mapping_out,
                                        void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                                        pkv_stream_t stream);

/* Chunked-prefill attention over the paged cache ([P2] 使用教程 step 4 and
 * 核心亮点: a self-written FlashAttention serves the prefill stage; [P3]
 * §关键工程决策 item 2: prefill chunks are batched with decode).  Sequence s
 * contributes q_len[s] = cu_q_lens[s+1] - cu_q_lens[s] query rows (packed:
 * rows cu_q_lens[s] .. cu_q_lens[s+1] of q and out, [rows][num_q_heads]
 * [head_dim]) at positions context_lens[s] - q_len[s] .. context_lens[s] - 1.
 * Their K/V must already be in the cache (reshape_and_cache with their
 * slots).  The query at position p attends to tokens 0..p of its sequence
 * (causal), query head i reading KV head i / (num_q_heads / num_kv_heads).
 * cu_q_lens: [num_seqs + 1] int32, device; max_q_len: host bound on every
 * q_len; num_q_rows: the rows of q and out.  A sequence whose rows fall
 * outside [0, num_q_rows), whose q_len exceeds max_q_len or its context_len,
 * or whose context_len exceeds max_blocks_per_seq * 16 is flagged
 * (PKV_DEV_BAD_LENGTH) and skipped: no row outside q and out is touched.
 * Supported: head_dim 64 or 128, num_q_heads / num_kv_heads up to 16. */
pkv_status paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* cu_q_lens,
                                   int num_seqs, int max_q_len, int num_q_rows, int num_q_heads,
                                   int num_kv_heads, int head_dim, int num_blocks, float scale,
                                   void* out, pkv_dtype dtype, pkv_stream_t stream);

/* The first of the two kernels of paged_kv_decode_step: the fused write
 * and partition pass.  paged_attention_merge_pass with partition_blocks = 0
 * and the same arguments completes the step. */
pkv_status paged_kv_decode_step_partition_pass(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int num_blocks, float scale, void* out, int64_t* slot_mapping_out, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream);

/* One decode step of every layer of a layer-major stack ([P3] item 3: pools
 * are layer-major; item 1: every layer reads its cache through the same
 * per-sequence lengths here): for l < num_layers, paged_kv_decode_step on
 *   q + l*[B][Hq][D], k_new / v_new + l*[B][Hkv][D], the pools' layer l
 *   (k_cache / v_cache + l*[num_blocks][16][Hkv][D]) and out + l*[B][Hq][D],
 * in order on `stream`, sharing block_tables, context_lens and the workspace.
 * out must not overlap q, k_new, v_new or the pools (a later layer's pass
 * runs beside the previous layer's merge).
 * The call neither allocates nor synchronises, so a caller may capture it
 * into a CUDA graph (stream capture) and replay the whole step. */
pkv_status paged_kv_decode_step_layers(const void* q, const void* k_new, const void* v_new,
                                       void* k_cache, void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_dim, int num_blocks,
                                       int num_layers, float scale, void* out, void* workspace,
                                       size_t workspace_bytes, pkv_dtype dtype,
                                       pkv_stream_t stream);

/* Device staging bytes paged_kv_decode_step_host needs: device copies of q,
 * k_new, v_new, block_tables, context_lens and out, each 256-byte aligned. */
size_t paged_kv_decode_step_staging_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int max_blocks_per_seq);

/* paged_kv_decode_step with the step's inputs and its output in HOST memory
 * (page-locked): q_host, k_new_host, v_new_host, block_tables_host and
 * context_lens_host are brought into the caller's device `staging` buffer on
 * `stream`, the step runs on the device-resident pools, and the attention
 * output lands in out_host.  Host buffers that have a device mapping
 * (page-locked memory under unified addressing) are read by one staging
 * kernel and the output is written to out_host by the attention kernels
 * themselves; a buffer without one is moved by cudaMemcpyAsync.  The host
 * buffers must stay unchanged until the stream reaches the step, as for any
 * asynchronous copy.  The call returns once everything is enqueued:
 * synchronise `stream` before reading out_host.  Shapes and dtypes as for
 * paged_kv_decode_step; staging_bytes must be at least
 * paged_kv_decode_step_staging_bytes(...). */
pkv_status paged_kv_decode_step_host(const void* q_host, const void* k_new_host,
                                     const void* v_new_host, const int32_t* block_tables_host,
                                     const int32_t* context_lens_host, void* out_host,
                                     void* staging, size_t staging_bytes, void* k_cache,
                                     void* v_cache, int max_blocks_per_seq, int max_context_len,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int num_blocks, float scale, void* workspace,
                                     size_t workspace_bytes, pkv_dtype dtype,
                                     pkv_stream_t stream);

/* Size of the static scratch used by paged_attention_decode_noalloc (32 MiB
 * per GPU that loads the library, held until the process exits). */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* PKV_NOALLOC_SCRATCH_BYTES as the library was built with it (for bindings
 * that do not read this header). */
size_t paged_attention_noalloc_scratch_bytes(void);

/* paged_attention_decode for callers that cannot allocate device memory (a
 * plug-in inside a framework that owns all device memory; a runtime whose
 * memory plan is fixed at start-up and that must not call cudaMalloc, which
 * synchronises the device and can fail mid-request).  There is no workspace
 * argument: the split-context partials go to a static device array of
 * PKV_NOALLOC_SCRATCH_BYTES inside the library.  The caller still passes all
 * inputs and the output, as for paged_attention_decode.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 *  - The first call on a device performs a one-time set-up there (it looks up
 *    the array's device address); make that first call before any stream
 *    capture.
 *  - A problem whose paged_attention_workspace_bytes(num_seqs, num_q_heads,
 *    head_dim, max_context_len) exceeds PKV_NOALLOC_SCRATCH_BYTES is rejected
 *    with PKV_ERR_WORKSPACE and nothing is enqueued.
 *  - Every call shares the one array and leaves its partials there; nothing in
 *    it needs to start at zero.  Calls that overlap on the GPU (other streams,
 *    other threads) race on it: serialise them.
 * The pages have no counterpart to this entry point; it exists for the callers
 * above.  Same semantics, shapes and errors as paged_attention_decode
 * otherwise. */
pkv_status paged_attention_decode_noalloc(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int max_context_len, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int num_blocks,
                                          float scale, void* out, pkv_dtype dtype,
                                          pkv_stream_t stream);

/* Device status word of the current device: returns (in *flags) the
 * PKV_DEV_* bits set by kernels since the last reset, and clears them if
 * `reset` is non-zero.  Synchronises the device. */
pkv_status pkv_device_status(unsigned int* flags, int reset);

/* The status word as a status code, for one stream: waits for `stream`,
 * reads and clears the word, and returns PKV_ERR_CUDA if a kernel timed out
 * (PKV_DEV_TIMEOUT) or the stream holds a CUDA error, else PKV_ERR_BAD_BLOCK_ID
 * if a table entry was out of range, else PKV_ERR_INVALID_ARG if a length or a
 * slot was, else PKV_OK.  The word is per device, so bits set by work on other
 * streams of the device are read (and cleared) too.  The pages define no such
 * call: it reports the device-side checks every kernel here makes instead of
 * trapping. */
pkv_status paged_kv_last_error(pkv_stream_t stream);

/* Diagnostic of the bounded waits: launches one warp on `stream` that waits
 * on an mbarrier nothing arrives on, with the same bounded wait every kernel
 * here uses, limited to about 0.1 s.  The wait gives up, sets
 * PKV_DEV_TIMEOUT in the device status word and the kernel returns; the
 * context stays usable.  The pages have no counterpart: this exercises the
 * failure path that replaces trapping or hanging. */
pkv_status pkv_selftest_bounded_wait(pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
