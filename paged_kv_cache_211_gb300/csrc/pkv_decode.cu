// pkv_decode.cu -- decode-step PagedAttention: split-context partition pass
// and log-sum-exp merge.
//
// What is computed ("MinivLLM" 使用教程 step 5 / 核心亮点: PagedAttention for
// the decode stage; "从零手写 vLLM 核心：mini-vllm 项目深度解析" §2: 16-token
// blocks reached through a block table; §关键工程决策 item 1: per-layer
// lengths; item 3: [num_blocks][16][num_kv_heads][head_dim] pools): for every
// sequence s and query head i (KV head h = i / g, g = Hq / Hkv)
//     out[s][i] = sum_t softmax_t(scale * <q[s][i], K_t[h]>) * V_t[h]
// over the t < context_lens[s] tokens of the sequence.
//
// Work decomposition.  A sequence's logical blocks are cut into partitions
// of PB blocks; a work item is (partition, KV head).  Each CTA of the
// persistent partition kernel walks items with a grid stride.  Inside an
// item, warp w takes the item's blocks w, w + 4, w + 8, ... and keeps an
// online softmax (running max m, running sum l, unnormalised output o) for
// the g query heads of its KV head; the four warps are combined through
// shared memory at the end of the item.  A sequence with one partition gets
// its output written directly; otherwise the item leaves (m, l, o) in the
// workspace and the merge kernel combines the partitions by log-sum-exp.
//
// Per 16-token block and KV head, a warp does the two contractions on the
// tensor cores with mma.sync m16n8k16 (fp32 accumulate):
//   scores  S^T[16 tok x 8 heads] = K[16 tok x D] . Q^T[D x 8 heads]
//   output  O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 tok x 8 heads]
// The g <= 8 query heads of the group form the n = 8 side, so each K/V row
// is read from HBM once per KV head, not once per query head.  K and V are
// loaded straight from global memory into the MMA operand registers with
// 16-byte loads: lane (r = lane/4, c = lane%4) reads, for K, rows r and r+8
// of the block (16-byte chunks 4j + c) and, for V, rows 2c, 2c+1, 2c+8, 2c+9
// (chunks r and r + 8).  The reduction index D of the score MMA may be
// permuted freely as long as q uses the same permutation, which is what
// makes the K chunks usable as-is; V rows are paired into token pairs with
// byte permutes, and P is brought from the score layout to the operand
// layout of the second MMA with two 8x8 movmatrix transposes.  Loads of the
// next block are issued before the current block is computed (two register
// stages).
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "pkv_internal.cuh"
#include "pkv_tma.cuh"

namespace pkv {

pkv_status launch_decode_step_write(const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    int num_seqs, int num_blocks, int num_kv_heads, int head_dim,
                                    int64_t* slot_out, cudaStream_t stream);

namespace {

constexpr int kWarps = 4;                 // warps per CTA of the partition kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxGroup = 8;              // query heads per KV head (the MMA's n = 8)
constexpr int kMaxSeqs = 8192;            // per call (lengths and offsets live in smem)
constexpr int kMaxPartitionsPerSeq = 64;  // bounds the workspace
constexpr int kAdaptiveMinBlocks = 8;     // adaptive partitions are at least this long
constexpr int kAdaptiveMaxBlocks = 512;
constexpr int kItemsPerCta = 4;           // adaptive partitioning aims at this many per CTA
constexpr float kLog2e = 1.4426950408889634f;

int ceil_div(int a, int b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

int min_partition_blocks(int max_context_len) {
    const int mb = ceil_div(std::max(max_context_len, 0), PKV_BLOCK_SIZE);
    return std::max(1, ceil_div(mb, kMaxPartitionsPerSeq));
}

struct WsLayout {
    size_t offsets, m, l, o, total;
    size_t rows;  // partial rows (m, l and o of one query head) it holds
};

// Largest grid of the even-split partition pass; its workspace holds two rows
// of every query head per CTA.
constexpr int kMaxEvenGrid = 256;
// Shortest table bound (in blocks) for which the TMA pass splits evenly.
constexpr int kEvenMinBlocks = 64;
// Most query heads one even-split slot holds (heads per item x group); the
// workspace reserves two slots of that many rows per CTA.
constexpr int kEvenMaxHeads = 16;

WsLayout ws_layout(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                   int extra_rows_per_seq = 0) {
    const int mb = ceil_div(std::max(max_context_len, 0), PKV_BLOCK_SIZE);
    const int parts =
        std::max(1, ceil_div(mb, min_partition_blocks(max_context_len))) + extra_rows_per_seq;
    size_t rows = (size_t)num_seqs * parts * num_q_heads;
    // the even split (bounds of kEvenMinBlocks blocks or more, no cascade)
    // keeps two slots of up to kEvenMaxHeads query-head rows per CTA
    if (extra_rows_per_seq == 0 && mb >= kEvenMinBlocks)
        rows = std::max(rows, (size_t)2 * kMaxEvenGrid * std::min(num_q_heads, kEvenMaxHeads));
    WsLayout w;
    w.rows = rows;
    w.offsets = 0;
    w.m = align256((size_t)(num_seqs + 1) * 4);
    w.l = w.m + align256(rows * 4);
    w.o = w.l + align256(rows * 4);
    w.total = w.o + align256(rows * head_dim * 4);
    return w;
}

struct DecodeParams {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    int* ws_offsets;
    float* ws_m;
    float* ws_l;
    float* ws_o;
    unsigned int* status;
    // optional fused KV write of the step's token (all null for plain decode)
    const void* k_new;          // [num_seqs][num_kv_heads][D]
    const void* v_new;
    void* k_cache_w;            // the same pools, written through these
    void* v_cache_w;
    int64_t* slot_out;          // [num_seqs] or null
    int num_seqs, num_q_heads, num_kv_heads, group;
    int max_blocks_per_seq, num_blocks, len_bound;
    int partition_blocks;      // > 0: fixed partition length (blocks)
    int skip_blocks;           // cascade: leading shared blocks handled by the prefix pass
    int prefix_parts;          // cascade: 1 (the prefix pass writes workspace row s of
                               // sequence s), else 0
    int item_row0;             // first workspace row of the items (num_seqs in a cascade)
    int even_row0;             // TMA pass, even split: first workspace row of the slots
                               // (a cascade's whole suffixes keep rows item_row0 + s)
    long long ws_rows;         // host: partial rows the workspace holds
    int min_partition_blocks;  // lower bound of the adaptive choice
    int target_items;
    int even_split;            // TMA pass: cut the (sequence, head group, block) units evenly
    int trigger_merge;         // register-pipelined pass: a merge pass follows in this call
                               // (let it launch early)
    int no_wait;               // TMA pass of a cascade: the previous kernel is this call's
                               // prefix pass, which runs beside it on disjoint memory and
                               // itself started after everything before it: no
                               // griddepcontrol.wait at all
    int early_reads;           // TMA pass: the previous kernel on the stream is this
                               // library's, launched in the same call, and touches none of
                               // the lengths, tables, this layer's inputs, pools or out:
                               // read and write them before griddepcontrol.wait (which
                               // comes before the first workspace write)
    float scale_log2;          // scale * log2(e): scores live in base 2
};

// Sum over the CTA of NW warps; every thread gets the result.
template <int NW = kWarps>
__device__ __forceinline__ int cta_sum(int v, int* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) t += red[w];
    return t;
}

// Exclusive prefix sum over the CTA of NW warps (thread order); *total gets the sum.
template <int NW = kWarps>
__device__ __forceinline__ int cta_exclusive_scan(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) before += red[w];
        all += red[w];
    }
    *total = all;
    return before + incl - v;
}

// Partition-pass items of one sequence.  Normally its blocks in partitions
// of pb (an empty sequence keeps one empty partition, which writes zeros).
// In cascade mode the first `skip` blocks belong to the prefix pass, which
// writes the sequence's prefix workspace row; the items cover the remaining
// blocks only, and may be none.
__device__ __forceinline__ int item_parts(int n, int pb, int skip, int prefix_parts) {
    const int nblk = (n + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
    if (prefix_parts == 0) return nblk == 0 ? 1 : (nblk + pb - 1) / pb;
    const int rest = nblk > skip ? nblk - skip : 0;
    return (rest + pb - 1) / pb;
}

// Operand registers of one 16-token block for one lane (see the file comment).
template <int D>
struct BlockFrag {
    static constexpr int KC = D / 32;  // K: 16-byte chunks per row (rows r and r+8)
    static constexpr int VC = D / 64;  // V: 16-byte chunks per token (4 tokens)
    uint4 k[2][KC];
    uint4 v[VC][4];
    bool bad;
    int rnew;     // row of this step's new token in this block, or -1
    size_t blk;   // first row of the physical block
};

// Loads one block's K/V fragments.  With rnew >= 0 the block holds this
// step's token at row rnew, which is not in the cache yet: that row is taken
// from knew / vnew ([D] each, this KV head) instead.
template <typename T, int D>
__device__ __forceinline__ void fetch_block(BlockFrag<D>& f, const T* kbase, const T* vbase,
                                            int id, size_t row_stride, int gid, int tig,
                                            int rnew, const T* knew, const T* vnew) {
    f.bad = id < 0;
    f.rnew = f.bad ? -1 : rnew;
    const size_t blk = (size_t)(f.bad ? 0 : id) * PKV_BLOCK_SIZE;
    f.blk = blk;
    const T* kr0 = gid == f.rnew ? knew : kbase + (blk + gid) * row_stride;
    const T* kr1 = gid + 8 == f.rnew ? knew : kbase + (blk + gid + 8) * row_stride;
#pragma unroll
    for (int j = 0; j < BlockFrag<D>::KC; ++j) {
        f.k[0][j] = ld_stream(kr0 + (4 * j + tig) * 8);
        f.k[1][j] = ld_stream(kr1 + (4 * j + tig) * 8);
    }
#pragma unroll
    for (int c = 0; c < BlockFrag<D>::VC; ++c) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int tok = 2 * tig + (t & 1) + (t >> 1) * 8;
            const T* src = tok == f.rnew ? vnew : vbase + (blk + tok) * row_stride;
            f.v[c][t] = ld_stream(src + (gid + 8 * c) * 8);
        }
    }
}

// The KV write fused into the decode step: the lanes that hold the new row
// (taken from k_new / v_new by fetch_block) store it into its cache slot.
template <typename T, int D>
__device__ __forceinline__ void store_new_row(const BlockFrag<D>& f, T* kbase_w, T* vbase_w,
                                              size_t row_stride, int gid, int tig) {
    const int r = f.rnew;
#pragma unroll
    for (int j = 0; j < BlockFrag<D>::KC; ++j) {
        if (gid == r)
            *reinterpret_cast<uint4*>(kbase_w + (f.blk + r) * row_stride + (4 * j + tig) * 8) =
                f.k[0][j];
        if (gid + 8 == r)
            *reinterpret_cast<uint4*>(kbase_w + (f.blk + r) * row_stride + (4 * j + tig) * 8) =
                f.k[1][j];
    }
#pragma unroll
    for (int c = 0; c < BlockFrag<D>::VC; ++c) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int tok = 2 * tig + (t & 1) + (t >> 1) * 8;
            if (tok == r)
                *reinterpret_cast<uint4*>(vbase_w + (f.blk + r) * row_stride +
                                          (gid + 8 * c) * 8) = f.v[c][t];
        }
    }
}

template <typename T, int D>
struct WarpState {
    static constexpr int NT = D / 16;  // 16-row tiles of the output's D axis
    float m0, m1;                      // running max (base 2) of heads 2c, 2c+1
    float l0, l1;                      // this lane's share of the running sums
    float o[NT][4];                    // O^T accumulator fragments
};

template <typename T, int D>
__device__ __forceinline__ void compute_block(WarpState<T, D>& st, BlockFrag<D>& f,
                                              const uint4 (&qf)[D / 32], int nv, float scale_log2,
                                              int gid, int tig) {
    using E = Elem<T>;
    constexpr int KC = BlockFrag<D>::KC;
    constexpr int NT = WarpState<T, D>::NT;
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
    float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KC; ++j) {
        E::mma(sa, f.k[0][j].x, f.k[1][j].x, f.k[0][j].y, f.k[1][j].y, qf[j].x, qf[j].y);
        E::mma(sb, f.k[0][j].z, f.k[1][j].z, f.k[0][j].w, f.k[1][j].w, qf[j].z, qf[j].w);
    }
    // rows: token gid (s0, s1) and gid + 8 (s2, s3); columns: heads 2*tig, 2*tig + 1
    float s0 = (sa[0] + sb[0]) * scale_log2;
    float s1 = (sa[1] + sb[1]) * scale_log2;
    float s2 = (sa[2] + sb[2]) * scale_log2;
    float s3 = (sa[3] + sb[3]) * scale_log2;
    if (nv < PKV_BLOCK_SIZE) {  // last (partial) block or a skipped bad block: select, never weight
        if (gid >= nv) s0 = s1 = -INFINITY;
        if (gid + 8 >= nv) s2 = s3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < BlockFrag<D>::VC; ++c) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int tok = 2 * tig + (t & 1) + (t >> 1) * 8;
                if (tok >= nv) f.v[c][t] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float ms0 = mn0 == -INFINITY ? 0.f : mn0;  // all-masked so far: keep everything 0
    const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
    const float c0 = fast_exp2(st.m0 - ms0), c1 = fast_exp2(st.m1 - ms1);
    const float p0 = fast_exp2(s0 - ms0), p1 = fast_exp2(s1 - ms1);
    const float p2 = fast_exp2(s2 - ms0), p3 = fast_exp2(s3 - ms1);
    st.l0 = st.l0 * c0 + p0 + p2;
    st.l1 = st.l1 * c1 + p1 + p3;
    st.m0 = mn0;
    st.m1 = mn1;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        st.o[i][0] *= c0;
        st.o[i][1] *= c1;
        st.o[i][2] *= c0;
        st.o[i][3] *= c1;
    }
    // P^T operand: lane (gid, tig) needs head gid at tokens 2tig, 2tig+1 (+8)
    const uint32_t pt = movmatrix_trans(E::pack(p0, p1));
    const uint32_t pb = movmatrix_trans(E::pack(p2, p3));
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int c = i >> 2, w = i & 3;
        const uint32_t x0 = word_of(f.v[c][0], w), x1 = word_of(f.v[c][1], w);
        const uint32_t x2 = word_of(f.v[c][2], w), x3 = word_of(f.v[c][3], w);
        E::mma(st.o[i], __byte_perm(x0, x1, 0x5410), __byte_perm(x0, x1, 0x7632),
               __byte_perm(x2, x3, 0x5410), __byte_perm(x2, x3, 0x7632), pt, pb);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) decode_partition_kernel(const DecodeParams p) {
    constexpr int KC = BlockFrag<D>::KC;
    constexpr int VC = BlockFrag<D>::VC;
    constexpr int NT = WarpState<T, D>::NT;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int red[kWarps];
    const int B = p.num_seqs;
    float* sm_o = reinterpret_cast<float*>(smem_raw);  // [kWarps][8][D]
    float* sm_m = sm_o + kWarps * kMaxGroup * D;        // [kWarps][8]
    float* sm_l = sm_m + kWarps * kMaxGroup;            // [kWarps][8]
    int* sm_len = reinterpret_cast<int*>(sm_l + kWarps * kMaxGroup);  // [B]
    int* sm_off = sm_len + B;                                          // [B + 1]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3;

    // (1) validated lengths and the total number of blocks
    int my_blocks = 0;
    for (int s = tid; s < B; s += kThreads) {
        int n = p.context_lens[s];
        if (n < 0 || n > p.len_bound) {
            if (blockIdx.x == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            n = 0;  // the row is written as zeros
        }
        // cascade: the step's token must land past the shared prefix
        if (n > 0 && p.prefix_parts && p.k_new && (n - 1) / PKV_BLOCK_SIZE < p.skip_blocks) {
            if (blockIdx.x == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            if (p.slot_out && blockIdx.x == 0) p.slot_out[s] = -1;
        }
        sm_len[s] = n;
        if (n == 0 && p.slot_out && blockIdx.x == 0) p.slot_out[s] = -1;  // nothing written
        my_blocks += (n + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
    }
    const int total_blocks = cta_sum(my_blocks, red);
    // a merge pass of this call may be launched now (it waits for this grid's
    // results); nothing else may start early: the next call's kernels could
    // overwrite the inputs this pass still reads
    if (p.trigger_merge) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // (2) partition length: fixed, or enough items for every CTA
    int PB = p.partition_blocks;
    if (PB <= 0) {
        const long long want =
            ((long long)total_blocks * p.num_kv_heads + p.target_items - 1) / p.target_items;
        const long long lo = p.min_partition_blocks;
        const long long hi = kAdaptiveMaxBlocks > lo ? kAdaptiveMaxBlocks : lo;
        PB = (int)(want < lo ? lo : (want > hi ? hi : want));
    }

    // (3) partitions per sequence and their exclusive prefix sum
    const int chunk = (B + kThreads - 1) / kThreads;
    const int s_lo = min(B, tid * chunk), s_hi = min(B, s_lo + chunk);
    int mine = 0;
    for (int s = s_lo; s < s_hi; ++s) mine += item_parts(sm_len[s], PB, p.skip_blocks, p.prefix_parts);
    int total_parts = 0;
    int run = cta_exclusive_scan(mine, red, &total_parts);
    for (int s = s_lo; s < s_hi; ++s) {
        sm_off[s] = run;
        run += item_parts(sm_len[s], PB, p.skip_blocks, p.prefix_parts);
    }
    if (tid == 0) sm_off[B] = total_parts;
    __syncthreads();
    if (blockIdx.x == 0) {
        // workspace rows of sequence s: its prefix rows, then one per item
        for (int s = tid; s <= B; s += kThreads) p.ws_offsets[s] = sm_off[s];
    }

    const T* __restrict__ q = static_cast<const T*>(p.q);
    const T* __restrict__ kc = static_cast<const T*>(p.k_cache);
    const T* __restrict__ vc = static_cast<const T*>(p.v_cache);
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, g = p.group;
    const size_t row_stride = (size_t)Hkv * D;
    const int total_items = total_parts * Hkv;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int gp = item / Hkv;
        const int h = item - gp * Hkv;
        int a = 0, b = B - 1;  // the sequence owning global partition gp
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (sm_off[mid] <= gp) a = mid; else b = mid - 1;
        }
        const int s = a;
        const int part = gp - sm_off[s];
        const int nparts = sm_off[s + 1] - sm_off[s] + p.prefix_parts;  // workspace rows of s
        const int ws_row = p.item_row0 + gp;                            // this item's row
        const int n = sm_len[s];
        const int nblk = (n + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
        const int blk_lo = p.skip_blocks + part * PB;
        const int blk_hi = min(nblk, blk_lo + PB);

        // query fragment: column gid of the score MMA is query head h*g + gid
        uint4 qf[KC];
        {
            const bool live = gid < g;
            const T* qrow = q + ((size_t)s * Hq + (size_t)h * g + (live ? gid : 0)) * D;
#pragma unroll
            for (int j = 0; j < KC; ++j)
                qf[j] = live ? *reinterpret_cast<const uint4*>(qrow + (4 * j + tig) * 8)
                             : make_uint4(0u, 0u, 0u, 0u);
        }

        WarpState<T, D> st;
        st.m0 = st.m1 = -INFINITY;
        st.l0 = st.l1 = 0.f;
#pragma unroll
        for (int i = 0; i < NT; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;

        const T* kbase = kc + (size_t)h * D;
        const T* vbase = vc + (size_t)h * D;
        // this step's token (position n-1) lives in the sequence's last block
        const bool writes = p.k_new != nullptr && n > 0;
        const int last_blk = writes ? nblk - 1 : -1;
        const int rnew = (n - 1) & (PKV_BLOCK_SIZE - 1);
        const T* knew = writes ? static_cast<const T*>(p.k_new) + ((size_t)s * Hkv + h) * D : kbase;
        const T* vnew = writes ? static_cast<const T*>(p.v_new) + ((size_t)s * Hkv + h) * D : vbase;
        const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
        // physical ids of this warp's blocks, 32 at a time (lane l: block j0 + l*kWarps)
        auto load_ids = [&](int j0) {
            const int j = j0 + lane * kWarps;
            int id = -1;
            if (j < blk_hi) {
                id = table[j];
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                    id = -1;  // never dereferenced; its tokens are masked out
                }
            }
            return id;
        };
        int j = blk_lo + warp;
        int k = 0;  // index of block j among this warp's blocks
        int ids = 0;
        BlockFrag<D> fa, fb;
        T* kbase_w = static_cast<T*>(p.k_cache_w) + (size_t)h * D;
        T* vbase_w = static_cast<T*>(p.v_cache_w) + (size_t)h * D;
        // the step's token: write it (lanes holding it) and record its slot (head 0)
        auto finish_new_row = [&](const BlockFrag<D>& f) {
            if (f.rnew >= 0) store_new_row<T, D>(f, kbase_w, vbase_w, row_stride, gid, tig);
            if (p.slot_out && h == 0 && lane == 0)
                p.slot_out[s] = f.bad ? -1 : (int64_t)f.blk + rnew;
        };
        if (j < blk_hi) {
            ids = load_ids(j);
            fetch_block<T, D>(fa, kbase, vbase, __shfl_sync(0xffffffffu, ids, 0), row_stride,
                              gid, tig, j == last_blk ? rnew : -1, knew, vnew);
        }
        while (j < blk_hi) {
            int jn = j + kWarps;
            if (jn < blk_hi) {
                if (((k + 1) & 31) == 0) ids = load_ids(jn);
                fetch_block<T, D>(fb, kbase, vbase, __shfl_sync(0xffffffffu, ids, (k + 1) & 31),
                                  row_stride, gid, tig, jn == last_blk ? rnew : -1, knew, vnew);
            }
            if (j == last_blk) finish_new_row(fa);
            compute_block<T, D>(st, fa, qf, fa.bad ? 0 : min(PKV_BLOCK_SIZE, n - j * 16),
                                p.scale_log2, gid, tig);
            j = jn;
            ++k;
            if (j >= blk_hi) break;
            jn = j + kWarps;
            if (jn < blk_hi) {
                if (((k + 1) & 31) == 0) ids = load_ids(jn);
                fetch_block<T, D>(fa, kbase, vbase, __shfl_sync(0xffffffffu, ids, (k + 1) & 31),
                                  row_stride, gid, tig, jn == last_blk ? rnew : -1, knew, vnew);
            }
            if (j == last_blk) finish_new_row(fb);
            compute_block<T, D>(st, fb, qf, fb.bad ? 0 : min(PKV_BLOCK_SIZE, n - j * 16),
                                p.scale_log2, gid, tig);
            j = jn;
            ++k;
        }

        // full sums over the eight token rows of the fragment
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
            st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
        }
        // this warp's (m, l, o) -> shared memory; lane holds heads 2tig, 2tig+1 at
        // d = 8*(gid + 8c) + e, e = 0..7, from tiles 4c .. 4c+3
        float* mo = sm_o + warp * kMaxGroup * D;
#pragma unroll
        for (int c = 0; c < VC; ++c) {
            const int d0 = 8 * (gid + 8 * c);
            float* r0 = mo + (2 * tig) * D + d0;
            float* r1 = mo + (2 * tig + 1) * D + d0;
            *reinterpret_cast<float4*>(r0) =
                make_float4(st.o[4 * c][0], st.o[4 * c][2], st.o[4 * c + 1][0], st.o[4 * c + 1][2]);
            *reinterpret_cast<float4*>(r0 + 4) = make_float4(
                st.o[4 * c + 2][0], st.o[4 * c + 2][2], st.o[4 * c + 3][0], st.o[4 * c + 3][2]);
            *reinterpret_cast<float4*>(r1) =
                make_float4(st.o[4 * c][1], st.o[4 * c][3], st.o[4 * c + 1][1], st.o[4 * c + 1][3]);
            *reinterpret_cast<float4*>(r1 + 4) = make_float4(
                st.o[4 * c + 2][1], st.o[4 * c + 2][3], st.o[4 * c + 3][1], st.o[4 * c + 3][3]);
        }
        if (gid == 0) {
            sm_m[warp * kMaxGroup + 2 * tig] = st.m0;
            sm_m[warp * kMaxGroup + 2 * tig + 1] = st.m1;
            sm_l[warp * kMaxGroup + 2 * tig] = st.l0;
            sm_l[warp * kMaxGroup + 2 * tig + 1] = st.l1;
        }
        __syncthreads();

        // combine the warps: one thread per (query head of the group, 8-wide slice of D)
        constexpr int SL = D / 8;
        for (int x = tid; x < g * SL; x += kThreads) {
            const int hh = x / SL, d0 = (x - hh * SL) * 8;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + hh]);
            const float Ms = M == -INFINITY ? 0.f : M;
            float L = 0.f;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float e = fast_exp2(sm_m[w * kMaxGroup + hh] - Ms);
                L += e * sm_l[w * kMaxGroup + hh];
                const float* src = sm_o + (w * kMaxGroup + hh) * D + d0;
                const float4 u = *reinterpret_cast<const float4*>(src);
                const float4 v = *reinterpret_cast<const float4*>(src + 4);
                acc[0] += e * u.x; acc[1] += e * u.y; acc[2] += e * u.z; acc[3] += e * u.w;
                acc[4] += e * v.x; acc[5] += e * v.y; acc[6] += e * v.z; acc[7] += e * v.w;
            }
            const int qh = h * g + hh;
            if (nparts == 1) {
                const float inv = L > 0.f ? 1.f / L : 0.f;
                uint4 packed;
                packed.x = Elem<T>::pack(acc[0] * inv, acc[1] * inv);
                packed.y = Elem<T>::pack(acc[2] * inv, acc[3] * inv);
                packed.z = Elem<T>::pack(acc[4] * inv, acc[5] * inv);
                packed.w = Elem<T>::pack(acc[6] * inv, acc[7] * inv);
                *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)s * Hq + qh) * D +
                                          d0) = packed;
            } else {
                const size_t row = (size_t)ws_row * Hq + qh;
                float* dst = p.ws_o + row * D + d0;
                *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                if (d0 == 0) {
                    p.ws_m[row] = M;
                    p.ws_l[row] = L;
                }
            }
        }
        __syncthreads();  // shared buffers are reused by the next item
    }
}


// ============================================================================
// Partition pass, TMA version (the default).
//
// One persistent CTA per SM with eight consumer warps, each doing the
// arithmetic of the kernel above on its share of the blocks.  Every consumer
// keeps a ring of shared-memory stages, each holding the 16 rows x D K and V
// tiles of one block of its KV head.  The tiles arrive by
// cp.async.bulk.tensor copies of boxes of 16 rows x 64 elements with the
// 128-byte swizzle, each stage tracked by a "full" mbarrier; the consumer
// reads its fragments with ldmatrix (.trans for V), conflict-free under the
// swizzle.  Three feeds fill the rings (compile-time variants):
//  - producer warp (items of one or two KV heads: long contexts): a ninth
//    warp walks the same items as the consumers and issues every copy, in
//    lane-parallel batches; a consumer releases a stage through its "empty"
//    mbarrier once its fragments are in registers.  With one head per item
//    the CTA has 12 warps and setmaxnreg moves the producer warpgroup's
//    registers to the consumers (which spilled at nine warps' 168);
//  - self-feeding consumers (items of four or more heads: short contexts):
//    no producer warp; each consumer walks its blocks twice, once to load and
//    once to consume, and lane 0 refills a stage with the block one ring
//    ahead as soon as the stage's fragments are in registers;
//  - stream producer (a cascade's suffixes, split over the consumer warps):
//    12 warps; lane v of the producer warp walks consumer v's own stream and
//    refills each of its slots once released, and setmaxnreg moves registers
//    from the producer's warpgroup to the consumers.
// With warp items each consumer warp works alone, every block of its piece's
// head, and writes the piece's result itself: no combine across the
// consumers and no CTA-wide barrier.  Its pieces are whole one-head items
// (many short items: large batches of short contexts, self-feeding) or, for
// a cascade's suffixes, an equal run of the (sequence, KV head, block) units.
// Either way every slot but the one being read is in flight, across item
// boundaries.  Every mbarrier wait is bounded: on a time-out the kernel sets
// PKV_DEV_TIMEOUT, stops issuing and waiting, lets every copy it issued land,
// and returns.
// ============================================================================
constexpr int kTmaConsumers = 8;
// threads of the TMA partition kernel: 8 consumer warps, plus the producer
// warp unless the consumers feed themselves; the stream-producer and wide
// producer builds have 12 (the producer warp's warpgroup gives its registers
// to the consumers)
__host__ __device__ constexpr int tma_threads(bool self_feed, bool stream = false,
                                              bool wide = false) {
    return stream || wide ? 12 * 32 : (kTmaConsumers + (self_feed ? 0 : 1)) * 32;
}
// Register shares of the stream-producer build (12 warps launched at 168):
// warps 8-11 (the producer warp and three that leave) and the consumers.
constexpr int kStreamLaunchRegs = 168;
constexpr int kStreamProducerRegs = 72;
constexpr int kStreamConsumerRegs = 216;
static_assert(128 * kStreamProducerRegs + 256 * kStreamConsumerRegs <= 384 * kStreamLaunchRegs,
              "register shares exceed the launch total");
constexpr int kTmaItemsPerCta = 8;
constexpr int kTmaMaxStages = 8;
// The ring's full / empty barriers (one arrival each) and use counts, one
// slot per thread side by side (a separate function: inlined, it changed how
// the kernel's registers are allocated).
__device__ __noinline__ void init_ring(uint64_t* full, uint64_t* empty, int* last_use, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], 1);
        last_use[i] = -1;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
}

template <typename T, int D, bool kOneHead, bool kSelfFeed, int kHPC = 1, bool kWarpItems = false,
          bool kStream = false, bool kWide = false>
__global__ void __launch_bounds__(tma_threads(kSelfFeed, kStream, kWide), 1)
    decode_partition_tma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                                const __grid_constant__ CUtensorMap tmap_v, int nstages,
                                int heads_per_item) {
    // kHPC: KV heads each consumer warp serves per block.  2 (D = 64 items of
    // two heads, producer warp only): a stage holds both heads' tiles, so a
    // consumer step moves 8 KB, as one head does at D = 128.
    static_assert(kHPC == 1 || (kHPC == 2 && !kSelfFeed && !kOneHead), "two heads per consumer");
    // kWarpItems: consumer warp w of CTA c takes items c * 8 + w, then every
    // (8 * gridDim.x)-th item after it (item mode only, one head per item)
    static_assert(!kWarpItems || ((kSelfFeed || kStream) && kOneHead && kHPC == 1), "warp items");
    // kStream: warp items fed by a producer warp whose lane v walks consumer
    // v's stream (the consumers do not issue their own copies)
    static_assert(!kStream || (kWarpItems && !kSelfFeed), "stream producer");
    // kWide: the producer warp (one head per item) in a CTA of 12 warps, whose
    // warpgroup gives its registers to the consumers (setmaxnreg), as the
    // stream producer's does: the consumers no longer spill
    static_assert(!kWide || (kOneHead && kHPC == 1 && !kSelfFeed && !kStream && !kWarpItems),
                  "wide producer");
    using E = Elem<T>;
    constexpr int NC = kTmaConsumers;
    constexpr int HALVES = D / 64;
    constexpr int TILE = 16 * D * 2;      // one K or V tile: 16 rows x D
    constexpr int STAGE = 2 * kHPC * TILE;  // K tiles of the consumer's heads, then V tiles
    constexpr int KS = D / 16;         // k-steps of the score MMA = row tiles of O^T
    constexpr int DP = D + 4;          // padded rows of the merge buffer
    extern __shared__ unsigned char smem_raw[];
    const int B = p.num_seqs;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-B aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)NC * nstages * STAGE);
    uint64_t* empty = full + NC * nstages;
    int* stage_id = reinterpret_cast<int*>(empty + NC * nstages);     // block id per slot
    int* last_use = stage_id + NC * nstages;                           // last use issued per slot
    const int g = p.group;
    float* sm_o = reinterpret_cast<float*>(last_use + NC * nstages);   // [NC][g][DP]
    float* sm_m = sm_o + NC * g * DP;                                  // [NC][8]
    float* sm_l = sm_m + NC * kMaxGroup;                               // [NC][8]
    constexpr int NT = tma_threads(kSelfFeed, kStream, kWide), NW = NT / 32;  // threads, warps
    int* red = reinterpret_cast<int*>(sm_l + NC * kMaxGroup);          // [NC + 1]
    volatile int* abort_flag = red + 2 * NC + 1;                       // red: up to 2 NC + 1 warps
    int* sm_len = red + NC + 2 + NC;                                   // [B]
    int* sm_off = sm_len + B;                                          // [B + 1]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    init_ring(full, empty, last_use, NC * nstages);
    if (tid == 0) *abort_flag = 0;

    // This grid is a programmatic dependent of the previous kernel on the
    // stream and may start before it ends.  Only when that kernel is this
    // library's own, launched by the same call on other memory (a previous
    // layer of paged_kv_decode_step_layers), do the lengths, the tables and
    // the cache get read before the consumers' griddepcontrol.wait below;
    // otherwise every thread waits here first, since any earlier kernel may
    // have written them and only the wait makes its stores visible.
    if (!p.early_reads && !p.no_wait) asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // validated lengths, partition length, partitions per sequence (all warps)
    int my_blocks = 0;
    for (int s = tid; s < B; s += NT) {
        int n = p.context_lens[s];
        if (n < 0 || n > p.len_bound) {
            if (blockIdx.x == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            n = 0;
        }
        if (n > 0 && p.prefix_parts && p.k_new && (n - 1) / PKV_BLOCK_SIZE < p.skip_blocks) {
            if (blockIdx.x == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        }
        sm_len[s] = n;
        my_blocks += (n + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
    }
    const int total_blocks = cta_sum<NW>(my_blocks, red);
    const bool even = p.even_split != 0;  // uniform over the grid
    int PB = p.partition_blocks;
    if (!even && PB <= 0) {
        const int groups0 = p.num_kv_heads / (kOneHead ? 1 : heads_per_item);
        if ((long long)B * groups0 >= 4ll * gridDim.x * (kWarpItems ? NC : 1)) {
            // enough items without splitting: one partition per sequence
            int my_max = 0;
            for (int s = tid; s < B; s += NT) {
                const int nb = (sm_len[s] + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE - p.skip_blocks;
                my_max = max(my_max, nb);
            }
            for (int o = 16; o > 0; o >>= 1) my_max = max(my_max, __shfl_xor_sync(0xffffffffu, my_max, o));
            __syncthreads();
            if (lane == 0) red[warp] = my_max;
            __syncthreads();
            int mx = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) mx = max(mx, red[w]);
            PB = max(mx, p.min_partition_blocks);
        } else {
            // items cover heads_per_item KV heads of their blocks: aim at target_items
            // 32-bit: blocks x groups stays below 2^31 (8192 sequences, a table
            // of int32 entries, at most 8 groups)
            const unsigned want =
                ((unsigned)total_blocks * groups0 + p.target_items - 1) / (unsigned)p.target_items;
            const int lo = p.min_partition_blocks;
            const int hi = kAdaptiveMaxBlocks > lo ? kAdaptiveMaxBlocks : lo;
            PB = (int)want < lo ? lo : ((int)want > hi ? hi : (int)want);
        }
    }
    const int chunk = (B + NT - 1) / NT;
    const int s_lo = min(B, tid * chunk), s_hi = min(B, s_lo + chunk);
    // item mode: partitions per sequence; even split: blocks per sequence
    auto units_of = [&](int s) {  // (a cascade's shared prefix is not the items')
        return even ? max((sm_len[s] + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE - p.skip_blocks, 0)
                    : item_parts(sm_len[s], PB, p.skip_blocks, p.prefix_parts);
    };
    int mine = 0;
    for (int s = s_lo; s < s_hi; ++s) mine += units_of(s);
    int total_parts = 0;
    int run = cta_exclusive_scan<NW>(mine, red, &total_parts);
    for (int s = s_lo; s < s_hi; ++s) {
        sm_off[s] = run;
        run += units_of(s);
    }
    if (tid == 0) sm_off[B] = total_parts;
    __syncthreads();
    // The next kernel on the stream (the merge pass, or the next call's first
    // kernel) may be scheduled now, so that its CTAs start as this grid's
    // leave the SMs.  Each of this library's dependents waits for this grid
    // (griddepcontrol.wait) before it touches what this grid reads or
    // writes; only the next layer's partition pass of a multi-layer step
    // reads early, and then only its own layer's pools, the lengths and the
    // tables, which this grid never writes.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const size_t row_stride = (size_t)Hkv * D;
    // An item is one partition of one sequence and a group of HPI KV heads
    // (HPI = 1: one head; HPI = Hkv: all heads, so a block's heads -- one
    // contiguous run of the pool -- are fetched together).  Consumer warp w
    // serves heads hg*HPI + (w % CPB)*kHPC + e, e < kHPC, of the item and every
    // CPH-th block of it, CPB = HPI / kHPC, CPH = NC / CPB.
    const int HPI = kOneHead ? 1 : heads_per_item;  // a constant in the one-head build
    const int groups = Hkv / HPI;
    const int total_items = total_parts * groups;
    // consumers per block: one per kHPC heads of the item (warp items: the
    // item's one consumer), and a consumer takes every CPH-th block of it
    const int CPB = kWarpItems ? 1 : HPI / kHPC;
    const int CPH = kWarpItems ? 1 : NC / CPB;
    // A work item: blocks [lo, hi) of sequence s for head group hg.  dest < 0:
    // the item is the whole of its (sequence, group) and writes the output;
    // else its partials go to workspace rows dest + (query head within group).
    struct Item {
        int s, hg, n, nblk, lo, hi, dest;
    };
    // Item mode (caller-fixed partition length, cascade suffixes): partition gp
    // of every group, items dealt round-robin to the CTAs.
    auto item_of = [&](int item) {
        Item it;
        const int gp = item / groups;
        it.hg = item - gp * groups;
        int a = 0, b = B - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (sm_off[mid] <= gp) a = mid; else b = mid - 1;
        }
        it.s = a;
        const int nparts = sm_off[a + 1] - sm_off[a] + p.prefix_parts;  // workspace rows of s
        const int ws_row = p.item_row0 + gp;                            // this item's row
        it.dest = nparts == 1 ? -1 : ws_row * Hq + it.hg * HPI * g;
        it.n = sm_len[a];
        it.nblk = (it.n + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
        // the k partitions of a sequence split its blocks evenly (sizes differ
        // by at most one, none above PB): a ragged last partition would leave
        // the CTAs that draw it idle at the end of the pass
        const int k = sm_off[a + 1] - sm_off[a], i = gp - sm_off[a];
        const int rest = max(it.nblk - p.skip_blocks, 0);
        it.lo = p.skip_blocks + (int)((long long)i * rest / k);
        it.hi = p.skip_blocks + (int)((long long)(i + 1) * rest / k);
        return it;
    };
    // Even split: the U = groups * (total blocks) units, ordered (sequence,
    // group, block), are cut into one range of equal size per worker (a CTA;
    // with warp items, a consumer warp: worker c * 8 + w); a worker's range is
    // a run of segments, each a whole (sequence, group) written straight to
    // the output except possibly the first and the last, which leave partials
    // in workspace slots 2c and 2c + 1 (c = the worker; rows from even_row0).
    // In a cascade the blocks are those past the shared prefix, and a whole
    // segment leaves its partials in row item_row0 + s instead, for the merge.
    const long long U = even ? (long long)groups * sm_off[B] : 0;
    // this thread's worker: its CTA, or with warp items its consumer warp (a
    // stream producer's lane v walks consumer v's range)
    const int worker =
        kWarpItems ? (int)blockIdx.x * NC + ((kStream && warp >= NC) ? (lane < NC ? lane : 0) : warp)
                   : (int)blockIdx.x;
    const int workers = kWarpItems ? (int)gridDim.x * NC : (int)gridDim.x;
    const long long u_begin = U * worker / workers;
    const long long u_end = U * (worker + 1) / workers;
    struct Cursor {
        int item, s;
        long long u;
    };
    auto cursor_begin = [&]() {
        Cursor c;
        c.item = worker;
        c.u = u_begin;
        c.s = 0;
        if (even && u_begin < u_end) {  // the sequence holding unit u_begin
            int a = 0, b = B - 1;
            while (a < b) {
                const int mid = (a + b + 1) >> 1;
                if ((long long)groups * sm_off[mid] <= u_begin) a = mid; else b = mid - 1;
            }
            c.s = a;
        }
        return c;
    };
    auto next_item = [&](Cursor& c, Item& it) -> bool {
        if (!even) {
            if (c.item >= total_items) return false;
            it = item_of(c.item);
            c.item += kWarpItems ? (int)gridDim.x * NC : (int)gridDim.x;
            return true;
        }
        if (c.u >= u_end) return false;
        const int s = c.s;
        const int nb = sm_off[s + 1] - sm_off[s];
        const long long r = c.u - (long long)groups * sm_off[s];
        const int hg = (int)(r / nb);
        const int b0 = (int)(r - (long long)hg * nb);
        const long long left = u_end - c.u;
        const int len = (long long)(nb - b0) < left ? nb - b0 : (int)left;
        it.s = s;
        it.hg = hg;
        it.n = sm_len[s];
        it.nblk = p.skip_blocks + nb;  // blocks of the sequence (the last holds the new token)
        it.lo = p.skip_blocks + b0;
        it.hi = p.skip_blocks + b0 + len;
        if (b0 == 0 && len == nb)
            it.dest = p.prefix_parts ? (p.item_row0 + s) * Hq + hg * HPI * g : -1;
        else
            it.dest = p.even_row0 + (2 * worker + (c.u == u_begin ? 0 : 1)) * (HPI * g);
        c.u += len;
        if (b0 + len == nb && hg == groups - 1) {  // on to the next sequence with blocks
            int t = s + 1;
            while (t < B && sm_off[t + 1] == sm_off[t]) ++t;
            c.s = t;
        }
        return true;
    };

    if constexpr (kStream) {
        if (warp >= NC) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kStreamProducerRegs));
            if (warp == NC) {
                // ------------------------------------------------ stream producer
                // Lane v (< 8) walks consumer v's stream of (item, block) in the
                // consumer's order and refills each of its ring slots as soon as
                // the consumer releases it (one non-blocking poll per lane and
                // pass): the consumers only wait, read their fragments and
                // release.  (A self-feeding consumer spent ~750 cycles of a
                // ~3000-cycle stage issuing its own refill.)
                const bool mine = lane < NC;
                Cursor pc = cursor_begin();
                Item pit;
                bool live = mine && next_item(pc, pit);
                int pj = live ? pit.lo : 0;
                while (live && pj >= pit.hi) {  // pieces with no block
                    live = next_item(pc, pit);
                    if (live) pj = pit.lo;
                }
                // the table entry of the next refill, loaded one refill ahead
                auto entry = [&]() {
                    return live ? p.block_tables[(size_t)pit.s * p.max_blocks_per_seq + pj] : 0;
                };
                int id_next = entry();
                int nf = 0, slot = 0;
                uint32_t ph = 1u;  // parity of the empty phase the next refill waits for
                long long t_last = clock64();
                while (__any_sync(0xffffffffu, live)) {
                    if (!live) continue;
                    if (*abort_flag) {
                        live = false;
                        continue;
                    }
                    const int k = lane * nstages + slot;
                    if (!mbar_test_wait(&empty[k], ph)) {
                        if (clock64() - t_last > kWaitCycles) {
                            *abort_flag = 1;
                            atomicOr(p.status, PKV_DEV_TIMEOUT);
                            live = false;
                        }
                        continue;
                    }
                    int id = id_next;
                    if (id < 0 || id >= p.num_blocks) {
                        atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                        id = -1;  // block 0 is fetched and fully masked
                    }
                    stage_id[k] = id;
                    last_use[k] = nf;
                    mbar_arrive_expect_tx(&full[k], STAGE);
                    unsigned char* st = ring + (size_t)k * STAGE;
                    const int row = (id < 0 ? 0 : id) * PKV_BLOCK_SIZE;
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh) {
                        tma_load_rows(st + hh * 2048, &tmap_k, &full[k], hh * 64, pit.hg, row);
                        tma_load_rows(st + TILE + hh * 2048, &tmap_v, &full[k], hh * 64, pit.hg,
                                      row);
                    }
                    ++nf;
                    if (++slot == nstages) {
                        slot = 0;
                        ph ^= 1u;
                    }
                    ++pj;
                    while (live && pj >= pit.hi) {
                        live = next_item(pc, pit);
                        if (live) pj = pit.lo;
                    }
                    id_next = entry();
                    t_last = clock64();
                }
                // every copy issued must land before the CTA may exit
                __syncwarp();
                for (int k = lane; k < NC * nstages; k += 32) {
                    const int use = last_use[k];
                    if (use >= 0) mbar_drain(&full[k], (use / nstages) & 1, p.status);
                }
            }
            return;
        }
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kStreamConsumerRegs));
    }

    constexpr bool self_feed = kSelfFeed;
    auto lockstep_producer = [&]() {
        // ------------------------------------------------------------ producer
        // Batches of BB blocks x CPB consumers' heads, lane t issuing (block
        // jb + t / CPB, heads slot t % CPB of the group) for consumer t % CPB +
        // CPB * ((block - lo) % CPH).  A batch gives each consumer at most
        // min(4, nstages) blocks, so no lane ever waits for a slot another lane
        // of this warp has yet to fill: every wait is on a consumer warp, never
        // on a diverged lane of this one.
        const int per = min(4, nstages);
        const int BB = CPH * per;               // blocks per batch (a multiple of CPH)
        // lane-constant roles (no division inside the loops)
        const int bi = lane / CPB;              // this lane's block in a batch
        const int hl = lane - bi * CPB;         // and heads slot within the group
        const int wl = hl + CPB * (bi % CPH);   // the consumer it feeds
        const int uoff = bi / CPH;              // its stage offset within the batch
        int pc[NC], subv[NC];  // stages issued so far per consumer; consumer's block phase
#pragma unroll
        for (int v = 0; v < NC; ++v) {
            pc[v] = 0;
            subv[v] = v / CPB;
        }
        // table entry of this lane's block in the batch starting at jb (-1: none / bad)
        auto lane_id = [&](const int32_t* table, int jb, int hi) {
            if (jb + bi >= hi) return -1;
            const int id = table[jb + bi];
            if (id < 0 || id >= p.num_blocks) {
                if (hl == 0) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                return -1;  // never read: block 0 is fetched and fully masked
            }
            return id;
        };
        Cursor cur = cursor_begin();
        Item it;
        while (next_item(cur, it)) {
            const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks_per_seq;
            const int h = it.hg * HPI + hl * kHPC;  // the lane's first head
            int id_cur = bi < BB ? lane_id(table, it.lo, it.hi) : -1;
            for (int jb = it.lo; jb < it.hi; jb += BB) {
                const int cnt = min(BB, it.hi - jb);   // blocks in this batch
                // the next batch's table entries are loaded one batch ahead
                const int id_next = bi < BB ? lane_id(table, jb + BB, it.hi) : -1;
                if (bi < cnt && !*abort_flag) {
                    const int id = id_cur;
                    const int w = wl;
                    int base = 0;
#pragma unroll
                    for (int v = 0; v < NC; ++v)
                        if (v == w) base = pc[v];
                    const int use = base + uoff;
                    const int k = w * nstages + use % nstages;
                    if (mbar_wait(&empty[k], ((use / nstages) & 1) ^ 1, abort_flag, p.status)) {
                        stage_id[k] = id;
                        last_use[k] = use;
                        mbar_arrive_expect_tx(&full[k], STAGE);
                        unsigned char* st = ring + (size_t)k * STAGE;
                        const int row = (id < 0 ? 0 : id) * PKV_BLOCK_SIZE;
#pragma unroll
                        for (int e = 0; e < kHPC; ++e) {
#pragma unroll
                            for (int hh = 0; hh < HALVES; ++hh) {
                                tma_load_rows(st + e * TILE + hh * 2048, &tmap_k, &full[k],
                                              hh * 64, h + e, row);
                                tma_load_rows(st + (kHPC + e) * TILE + hh * 2048, &tmap_v,
                                              &full[k], hh * 64, h + e, row);
                            }
                        }
                    }
                }
                id_cur = id_next;
                if (cnt == BB) {  // a full batch gives every consumer `per` stages
#pragma unroll
                    for (int v = 0; v < NC; ++v) pc[v] += per;
                } else {          // blocks of the batch with bi % CPH == subv[v]
#pragma unroll
                    for (int v = 0; v < NC; ++v)
                        pc[v] += cnt > subv[v] ? (cnt - subv[v] + CPH - 1) / CPH : 0;
                }
                __syncwarp();
            }
        }
        // every copy issued must land before the CTA may exit: wait for the
        // last use issued into each slot (earlier uses completed before reuse)
        __syncwarp();
        for (int k = lane; k < NC * nstages; k += 32) {
            const int use = last_use[k];
            if (use >= 0) mbar_drain(&full[k], (use / nstages) & 1, p.status);
        }
    };
    if constexpr (kWide) {
        if (warp >= NC) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kStreamProducerRegs));
            if (warp == NC) lockstep_producer();
            return;
        }
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kStreamConsumerRegs));
    } else if (!self_feed && warp == NC) {
        lockstep_producer();
        return;
    }

    // -------------------------------------------------------------- consumers
    // Self-feeding (measured faster when items carry 4 or more heads, i.e. few
    // consumers per head and short per-head runs): every warp feeds its own
    // ring of nstages slots, lane 0 issuing the TMA copies of the block
    // nstages ahead of the one the warp consumes as soon as the consumed
    // stage's fragments are in registers.  Two walks over the same sequence of
    // (item, block) give the blocks to fetch and the blocks to consume.
    // Otherwise the producer warp above fills the rings.
    const int w = warp;
    // this consumer's heads slot in the group, and block phase
    const int hl = w % CPB, sub = kWarpItems ? 0 : w / CPB;
    struct Stream {
        Cursor c;
        Item it;
        int j;
        bool live;
    };
    Stream fs;  // the fetch walk: this warp's next block to load
    fs.live = false;
    fs.j = 0;
    auto skip_done = [&](Stream& st) {  // past items this warp has no (more) block in
        while (st.live && st.j >= st.it.hi) {
            st.live = next_item(st.c, st.it);
            if (st.live) st.j = st.it.lo + sub;
        }
    };
    // lane t holds the table entry of the fetch walk's block t steps (of CPH
    // blocks) on within its item, from one parallel load per item (or per 32
    // steps): a refill never waits on a table load issued by the refill before
    // it (a chain of one dependent global load per stage held long walks to
    // 1.5 us a stage)
    int fs_tab = 0;  // this lane's entry
    int fs_t = 0;    // the lane holding the next block's entry
    auto load_tab = [&]() {  // whole warp
        const int jl = fs.j + lane * CPH;
        fs_tab = fs.live && jl < fs.it.hi
                     ? p.block_tables[(size_t)fs.it.s * p.max_blocks_per_seq + jl]
                     : 0;
        fs_t = 0;
    };
    int nfetch = 0;        // stages issued by this warp
    int fslot = 0;         // its ring slot (nfetch mod nstages, kept without a division)
    bool feeding = true;   // false after a wait gave up: issue nothing more
    auto fetch_next = [&]() {  // whole warp; lane 0 issues
        if (!fs.live || !feeding) return;
        const int k = w * nstages + fslot;
        int id = __shfl_sync(0xffffffffu, fs_tab, fs_t);
        if (lane == 0) {
            if (id < 0 || id >= p.num_blocks) {
                atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                id = -1;  // block 0 is fetched and fully masked
            }
            stage_id[k] = id;
            last_use[k] = nfetch;
            mbar_arrive_expect_tx(&full[k], STAGE);
            unsigned char* st = ring + (size_t)k * STAGE;
            const int row = (id < 0 ? 0 : id) * PKV_BLOCK_SIZE;
            const int h = fs.it.hg * HPI + hl;
#pragma unroll
            for (int hh = 0; hh < HALVES; ++hh) {
                tma_load_rows(st + hh * 2048, &tmap_k, &full[k], hh * 64, h, row);
                tma_load_rows(st + TILE + hh * 2048, &tmap_v, &full[k], hh * 64, h, row);
            }
        }
        ++nfetch;
        if (++fslot == nstages) fslot = 0;
        fs.j += CPH;
        if (fs.j >= fs.it.hi) {  // on to the next item this warp has a block in
            skip_done(fs);
            load_tab();
        } else if (++fs_t == 32) {
            load_tab();
        }
    };
    // the first nstages blocks (before griddepcontrol.wait only with
    // early_reads: then the previous kernel writes nothing read here)
    if constexpr (kSelfFeed) {
        fs.c = cursor_begin();
        fs.live = next_item(fs.c, fs.it);
        fs.j = fs.live ? fs.it.lo + sub : 0;
        skip_done(fs);
        load_tab();
        for (int t = 0; t < nstages; ++t) fetch_next();
    }

    // q, k_new, v_new and every output may belong to the previous kernel:
    // wait for it (a cascade's partition pass has nothing to wait for).  A
    // later layer of a multi-layer step (early_reads) reads nothing that the
    // kernel before it (the previous layer's merge) writes, and writes only
    // the shared workspace that this merge reads: it waits just before its
    // first workspace write instead, so that its blocks up to then overlap
    // that merge.  Every consumer thread waits before it ends, so that this
    // grid never completes before the kernel it depends on.  (A repeated
    // wait returns at once.)
    // The map of workspace rows the merge pass reads is the same for every
    // layer of a multi-layer step (same lengths, tables and launch shape), so
    // only the first layer writes it.
    if (!p.early_reads && !p.no_wait) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (blockIdx.x == 0 && !p.early_reads)
        for (int s = tid; s <= B; s += NC * 32) p.ws_offsets[s] = sm_off[s];
    if (blockIdx.x == 0) {
        if (p.slot_out) {
            // no slot for an empty or invalid sequence, nor for a cascade
            // token that would land in a shared block
            for (int s = tid; s < B; s += NC * 32) {
                const int n = sm_len[s];
                if (n == 0 || (p.prefix_parts && p.k_new && (n - 1) / PKV_BLOCK_SIZE < p.skip_blocks))
                    p.slot_out[s] = -1;
            }
        }
    }
    if (even && !p.prefix_parts) {
        // empty (or invalid) sequences have no units: their rows are zeros
        // (a cascade's merge writes every row)
        for (int s = blockIdx.x; s < B; s += gridDim.x) {
            if (sm_len[s] != 0) continue;
            uint4* o = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (size_t)s * Hq * D);
            for (int x = tid; x < Hq * D / 8; x += NC * 32) o[x] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    const int gid = lane >> 2, tig = lane & 3;
    const T* __restrict__ q = static_cast<const T*>(p.q);
    // the ring slot this warp consumes next and its phase parity (the stage
    // count mod nstages and the parity of its quotient, kept without a
    // division: two integer divisions a stage by the runtime ring depth cost
    // more than the score MMAs)
    int cslot = 0;
    uint32_t cphase = 0;
    const int kbase = w * nstages;
    Cursor cur = cursor_begin();
    Item it;
    while (next_item(cur, it)) {
        const int s = it.s, n = it.n;
        const int h = it.hg * HPI + hl * kHPC;  // this consumer's first head
        // q fragments: column gid of head e's score MMA is query head (h+e)*g + gid
        uint32_t qf[kHPC][KS][2];
#pragma unroll
        for (int e = 0; e < kHPC; ++e) {
            const bool live = gid < g;
            const T* qrow = q + ((size_t)s * Hq + (size_t)(h + e) * g + (live ? gid : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qf[e][ks][0] =
                    live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tig) : 0u;
                qf[e][ks][1] =
                    live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tig) : 0u;
            }
        }
        float m0[kHPC], m1[kHPC], l0[kHPC], l1[kHPC];
        float o[kHPC][KS][4];
#pragma unroll
        for (int e = 0; e < kHPC; ++e) {
            m0[e] = m1[e] = -INFINITY;
            l0[e] = l1[e] = 0.f;
#pragma unroll
            for (int i = 0; i < KS; ++i) o[e][i][0] = o[e][i][1] = o[e][i][2] = o[e][i][3] = 0.f;
        }

        const bool writes = p.k_new != nullptr && n > 0;
        const int last_blk = writes ? it.nblk - 1 : -1;
        const int rnew = (n - 1) & (PKV_BLOCK_SIZE - 1);
        T* kbase_w = static_cast<T*>(p.k_cache_w) + (size_t)h * D;
        T* vbase_w = static_cast<T*>(p.v_cache_w) + (size_t)h * D;

        for (int j = it.lo + sub; j < it.hi; j += CPH) {
            const int k = kbase + cslot;
            const uint32_t parity = cphase;
            if (++cslot == nstages) {
                cslot = 0;
                cphase ^= 1u;
            }
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait(&full[k], parity, abort_flag, p.status));
            unsigned char* st = ring + (size_t)k * STAGE;
            const int id = ok ? stage_id[k] : -1;
            const int nv = id < 0 ? 0 : min(PKV_BLOCK_SIZE, n - j * PKV_BLOCK_SIZE);
            if (j == last_blk) {
                // this step's token: not in the cache yet; patch it into the
                // stage from k_new / v_new and store it into its slot (lane:
                // head e, K or V, 16-byte chunk c)
                if (id >= 0) {
                    constexpr int CH = D / 8;
                    static_assert(2 * CH * kHPC <= 32, "one lane per chunk");
                    if (lane < 2 * CH * kHPC) {
                        const int e = lane / (2 * CH), r2 = lane - e * 2 * CH;
                        const bool isv = r2 >= CH;
                        const int c = isv ? r2 - CH : r2;
                        const T* src = static_cast<const T*>(isv ? p.v_new : p.k_new) +
                                       ((size_t)s * Hkv + h + e) * D + c * 8;
                        const uint4 v = *reinterpret_cast<const uint4*>(src);
                        *reinterpret_cast<uint4*>(st + ((isv ? kHPC : 0) + e) * TILE +
                                                  swz(rnew, c)) = v;
                        T* dst = (isv ? vbase_w : kbase_w) +
                                 ((size_t)id * PKV_BLOCK_SIZE + rnew) * row_stride + e * D + c * 8;
                        *reinterpret_cast<uint4*>(dst) = v;
                    }
                    // the stage is refilled by the async proxy after release
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    __syncwarp();
                }
                if (p.slot_out && h == 0 && lane == 0)
                    p.slot_out[s] = id >= 0 ? (int64_t)id * PKV_BLOCK_SIZE + rnew : -1;
            }
            // the softmax and P V of head e from its scaled scores s0..s3 and
            // its V fragments
            auto head_tail = [&](int e, float s0, float s1, float s2, float s3,
                                 uint32_t (&vf)[KS][4]) {
                if (nv < PKV_BLOCK_SIZE) {  // partial last block: select, never weight
                    if (gid >= nv) s0 = s1 = -INFINITY;
                    if (gid + 8 >= nv) s2 = s3 = -INFINITY;
                    const uint32_t mlo = (2 * tig < nv ? 0x0000ffffu : 0u) |
                                         (2 * tig + 1 < nv ? 0xffff0000u : 0u);
                    const uint32_t mhi = (2 * tig + 8 < nv ? 0x0000ffffu : 0u) |
                                         (2 * tig + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        vf[i][0] &= mlo;
                        vf[i][1] &= mlo;
                        vf[i][2] &= mhi;
                        vf[i][3] &= mhi;
                    }
                }
                float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m0[e], mx0), mn1 = fmaxf(m1[e], mx1);
                const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
                const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
                const float c0 = fast_exp2(m0[e] - ms0), c1 = fast_exp2(m1[e] - ms1);
                const float p0 = fast_exp2(s0 - ms0), p1 = fast_exp2(s1 - ms1);
                const float p2 = fast_exp2(s2 - ms0), p3 = fast_exp2(s3 - ms1);
                l0[e] = l0[e] * c0 + p0 + p2;
                l1[e] = l1[e] * c1 + p1 + p3;
                m0[e] = mn0;
                m1[e] = mn1;
#pragma unroll
                for (int i = 0; i < KS; ++i) {
                    o[e][i][0] *= c0;
                    o[e][i][1] *= c1;
                    o[e][i][2] *= c0;
                    o[e][i][3] *= c1;
                }
                const uint32_t pt = movmatrix_trans(E::pack(p0, p1));
                const uint32_t pbt = movmatrix_trans(E::pack(p2, p3));
#pragma unroll
                for (int i = 0; i < KS; ++i)
                    E::mma(o[e][i], vf[i][0], vf[i][1], vf[i][2], vf[i][3], pt, pbt);
            };
            // head by head: its fragments into registers, then (after the last
            // head's) the slot goes back to the producer or is refilled with the
            // block nstages ahead (the async-proxy copy after the warp's reads)
#pragma unroll
            for (int e = 0; e < kHPC; ++e) {
                uint32_t kf[KS][4], vf[KS][4];
                if (ok) {
                    const uint32_t kt = smem_addr(st) + e * TILE;
                    const uint32_t vt = smem_addr(st) + (kHPC + e) * TILE;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int row = lane & 15;
                        ldsm_x4(kf[ks], kt + swz(row, 2 * ks + (lane >> 4)));
                        const int mi = lane >> 3;
                        const int tok = (lane & 7) + 8 * (mi >> 1);
                        ldsm_x4_trans(vf[ks], vt + swz(tok, 2 * ks + (mi & 1)));
                    }
                }
                if (e == kHPC - 1) {
                    if constexpr (kSelfFeed) {
                        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                        __syncwarp();
                        if (ok) fetch_next(); else feeding = false;
                    } else {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[k]);
                    }
                }
                if (!ok || nv == 0) continue;

                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KS; ks += 2) {
                    E::mma(sa, kf[ks][0], kf[ks][1], kf[ks][2], kf[ks][3], qf[e][ks][0],
                           qf[e][ks][1]);
                    E::mma(sb, kf[ks + 1][0], kf[ks + 1][1], kf[ks + 1][2], kf[ks + 1][3],
                           qf[e][ks + 1][0], qf[e][ks + 1][1]);
                }
                float s0 = (sa[0] + sb[0]) * p.scale_log2, s1 = (sa[1] + sb[1]) * p.scale_log2;
                float s2 = (sa[2] + sb[2]) * p.scale_log2, s3 = (sa[3] + sb[3]) * p.scale_log2;
                head_tail(e, s0, s1, s2, s3, vf);
            }
        }

        // combine the consumer warps of this item (named barrier: consumers
        // only), one round per head a consumer serves
#pragma unroll
        for (int e = 0; e < kHPC; ++e) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0[e] += __shfl_xor_sync(0xffffffffu, l0[e], off);
                l1[e] += __shfl_xor_sync(0xffffffffu, l1[e], off);
            }
            float* mo = sm_o + w * g * DP;  // rows of the g live query heads only
            const bool live0 = 2 * tig < g, live1 = 2 * tig + 1 < g;
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                if (live0) {
                    mo[(2 * tig) * DP + 16 * i + gid] = o[e][i][0];
                    mo[(2 * tig) * DP + 16 * i + 8 + gid] = o[e][i][2];
                }
                if (live1) {
                    mo[(2 * tig + 1) * DP + 16 * i + gid] = o[e][i][1];
                    mo[(2 * tig + 1) * DP + 16 * i + 8 + gid] = o[e][i][3];
                }
            }
            if (gid == 0) {
                sm_m[w * kMaxGroup + 2 * tig] = m0[e];
                sm_m[w * kMaxGroup + 2 * tig + 1] = m1[e];
                sm_l[w * kMaxGroup + 2 * tig] = l0[e];
                sm_l[w * kMaxGroup + 2 * tig + 1] = l1[e];
            }
            if constexpr (kWarpItems) __syncwarp();
            else asm volatile("bar.sync 1, %0;\n" ::"r"(NC * 32) : "memory");
            if (p.early_reads && it.dest >= 0)  // uniform over the item's consumers
                asm volatile("griddepcontrol.wait;\n" ::: "memory");
            constexpr int SL = D / 8;
            // one thread per (KV head of this round, query head of its group,
            // 8-wide slice of D), merging the CPH consumers that hold that head:
            // consumer v holds heads hg*HPI + (v % CPB)*kHPC + e (warp items:
            // the lanes of the item's one consumer, w)
            constexpr int XS = kWarpItems ? 32 : NC * 32;
            for (int x = kWarpItems ? lane : tid; x < CPB * g * SL; x += XS) {
                const int slot = x / (g * SL);  // heads slot within the group
                const int hk = slot * kHPC + e;  // head within the group
                const int hh = (x / SL) % g, d0 = (x % SL) * 8;
                auto holder = [&](int c) { return kWarpItems ? w : slot + CPB * c; };
                float M = -INFINITY;
                for (int c = 0; c < CPH; ++c) M = fmaxf(M, sm_m[holder(c) * kMaxGroup + hh]);
                const float Ms = M == -INFINITY ? 0.f : M;
                float L = 0.f;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int c = 0; c < CPH; ++c) {
                    const int v = holder(c);
                    const float ew = fast_exp2(sm_m[v * kMaxGroup + hh] - Ms);
                    L += ew * sm_l[v * kMaxGroup + hh];
                    const float* src = sm_o + (v * g + hh) * DP + d0;
                    const float4 u = *reinterpret_cast<const float4*>(src);
                    const float4 u2 = *reinterpret_cast<const float4*>(src + 4);
                    acc[0] += ew * u.x; acc[1] += ew * u.y; acc[2] += ew * u.z; acc[3] += ew * u.w;
                    acc[4] += ew * u2.x; acc[5] += ew * u2.y; acc[6] += ew * u2.z; acc[7] += ew * u2.w;
                }
                const int qh = (it.hg * HPI + hk) * g + hh;
                if (it.dest < 0) {
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    uint4 packed;
                    packed.x = E::pack(acc[0] * inv, acc[1] * inv);
                    packed.y = E::pack(acc[2] * inv, acc[3] * inv);
                    packed.z = E::pack(acc[4] * inv, acc[5] * inv);
                    packed.w = E::pack(acc[6] * inv, acc[7] * inv);
                    *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)s * Hq + qh) * D +
                                              d0) = packed;
                } else {
                    const size_t row = (size_t)it.dest + hk * g + hh;
                    float* dst = p.ws_o + row * D + d0;
                    *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    if (d0 == 0) {
                        p.ws_m[row] = M;
                        p.ws_l[row] = L;
                    }
                }
            }
            if constexpr (kWarpItems) __syncwarp();
            else asm volatile("bar.sync 1, %0;\n" ::"r"(NC * 32) : "memory");
        }
    }
    // A cascade's suffix pass (no_wait) waits here for the prefix pass it ran
    // beside, so that its merge, a programmatic dependent of this grid, sees
    // both passes complete once this grid is
    if (p.early_reads || p.no_wait) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // every copy this warp issued must land before the CTA may exit: wait for
    // the last use issued into each of its slots (normally already consumed)
    __syncwarp();
    if (kSelfFeed && lane == 0) {
        for (int k = w * nstages; k < (w + 1) * nstages; ++k) {
            const int use = last_use[k];
            if (use >= 0) mbar_drain(&full[k], (use / nstages) & 1, p.status);
        }
    }
}


constexpr int kMergeThreads = 128;

struct MergeParams {
    const int* ws_offsets;
    const float* ws_m;
    const float* ws_l;
    const float* ws_o;
    void* out;
    int num_seqs, num_q_heads;
    int min_rows;  // merge sequences with at least this many workspace rows
    int prefix_rows;  // cascade: 1 (row s holds sequence s's prefix partials), else 0
    int item_row0;    // first workspace row of the items
    int even_row0;    // first workspace row of the even split's slots
    // even split of the TMA pass (even_grid > 0): ws_offsets holds block
    // offsets, and the CTAs that covered a (sequence, group) left its partials
    // in their slots (two per CTA, even_heads query heads each)
    int even_grid, even_heads, groups;
};

// Log-sum-exp merge of one (sequence, query head)'s partitions by one warp:
//   M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  out = sum_p o_p 2^(m_p - M) / L.
template <typename T, int D>
__device__ __forceinline__ void merge_one(const MergeParams& p, int wg, int lane) {
    constexpr int PER = D / 32;
    const int Hq = p.num_q_heads;
    const int s = wg / Hq, qh = wg - s * Hq;
    // the workspace rows of (s, qh): np of them, row(i) for i < np (-1: none)
    int np;
    size_t base = 0;
    int c0 = 0, lq = 0;
    long long U = 0, start = 0;
    const long long G = p.even_grid;  // even split: its workers (CTAs or consumer warps)
    int ne = 0;                       // even split: workers that covered (s, qh)'s group
    if (G > 0) {
        const int nb = p.ws_offsets[s + 1] - p.ws_offsets[s];
        if (nb > 0) {
            U = (long long)p.groups * p.ws_offsets[p.num_seqs];
            const int hg = qh / p.even_heads;
            lq = qh - hg * p.even_heads;
            start = (long long)p.groups * p.ws_offsets[s] + (long long)hg * nb;
            // worker holding unit u: the largest c with floor(c * U / G) <= u
            auto cta_of = [&](long long u) { return (int)(((u + 1) * G + U - 1) / U - 1); };
            c0 = cta_of(start);
            ne = cta_of(start + nb - 1) - c0 + 1;
        }
        // no blocks (zeros) or one worker: the partition pass wrote the
        // output, unless a cascade's prefix row is still to be merged
        if (ne < 2 && p.prefix_rows == 0) return;
        np = ne + p.prefix_rows;
    } else {
        const int off = p.ws_offsets[s];
        np = p.ws_offsets[s + 1] - off + p.prefix_rows;
        if (np < p.min_rows) return;  // a one-row sequence was written by the partition pass
        base = ((size_t)p.item_row0 + off) * Hq + qh;
    }
    // row i of (s, qh), -1 for none (rows fit in 32 bits: the workspace is
    // sized from int arguments)
    auto row_of = [&](int i) -> int {
        if (G == 0) {
            if (p.prefix_rows == 0) return (int)(base + (size_t)i * Hq);
            // cascade: the prefix row first, then the items
            return i == 0 ? s * Hq + qh : (int)(base + (size_t)(i - 1) * Hq);
        }
        if (p.prefix_rows) {  // cascade: the prefix row first, then the suffix's rows
            if (i == 0) return s * Hq + qh;
            --i;
            if (ne == 1) return (p.item_row0 + s) * Hq + qh;  // a whole suffix
        }
        const long long c = c0 + i;
        const long long b = c * U / G;
        if (b == (c + 1) * U / G) return -1;  // a worker with no units (U < G)
        const long long slot = (i == 0 && b < start) ? 2 * c + 1 : 2 * c;
        return (int)(p.even_row0 + slot * p.even_heads + lq);
    };
    // Two dependent rounds of loads after the offsets: lane i finds row i and
    // loads its m and l while every lane loads its slice of the first kPre
    // rows' partial outputs (row numbers passed by shuffle); then M, the
    // weights and the sums (rows past kPre, and past 32, in further rounds).
    using V = typename std::conditional<PER == 4, float4, float2>::type;
    constexpr int kPre = 4;
    const int rl = lane < np ? row_of(lane) : -1;  // lane i: row i (i < 32)
    V pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int r = __shfl_sync(0xffffffffu, rl, k);
        if (r >= 0) pre[k] = *reinterpret_cast<const V*>(p.ws_o + (size_t)r * D + lane * PER);
    }
    float mi = -INFINITY, li = 0.f;
    if (rl >= 0) {
        mi = p.ws_m[rl];
        li = p.ws_l[rl];
    }
    float M = mi;
    for (int i = lane + 32; i < np; i += 32) {
        const int r = row_of(i);
        if (r >= 0) M = fmaxf(M, p.ws_m[r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Ms = M == -INFINITY ? 0.f : M;
    const float wi = mi == -INFINITY ? 0.f : fast_exp2(mi - Ms);  // lane i: row i's weight
    float L = wi * li;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    auto add = [&](float w, const V& u) {
        if constexpr (PER == 4) {
            acc[0] += w * u.x; acc[1] += w * u.y; acc[2] += w * u.z; acc[3] += w * u.w;
        } else {
            acc[0] += w * u.x; acc[1] += w * u.y;
        }
    };
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const float w = __shfl_sync(0xffffffffu, wi, k);
        // rows past np, and rows with no units, carry weight 0 and a load
        // never issued: select, never multiply an unset register
        if (w != 0.f) add(w, pre[k]);
    }
    for (int i = kPre; i < np; ++i) {
        const int r = i < 32 ? __shfl_sync(0xffffffffu, rl, i) : row_of(i);
        if (r < 0) continue;
        float w;
        if (i < 32) {
            w = __shfl_sync(0xffffffffu, wi, i);
        } else {
            w = fast_exp2(p.ws_m[r] - Ms);
            if (lane == 0) L += w * p.ws_l[r];
        }
        add(w, *reinterpret_cast<const V*>(p.ws_o + (size_t)r * D + lane * PER));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    T* dst = static_cast<T*>(p.out) + ((size_t)s * Hq + qh) * D + lane * PER;
    if constexpr (PER == 4) {
        uint2 packed;
        packed.x = Elem<T>::pack(acc[0] * inv, acc[1] * inv);
        packed.y = Elem<T>::pack(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = packed;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = Elem<T>::pack(acc[0] * inv, acc[1] * inv);
    }
}

// The merge pass: warp w of the grid merges (sequence, query head) pairs w,
// w + 4 * gridDim.x, ...  The grid may be smaller than one warp per pair, so
// that every CTA fits beside a partition CTA on its SM (see merge_grid_cap).
template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads, 8) decode_merge_kernel(const MergeParams p) {
    // launched early (programmatic dependent launch).  The next grid may be
    // scheduled at once: its CTAs take the SMs the partition pass leaves
    // (the next layer's partition pass of a multi-layer step starts on its
    // own layer there; any other dependent waits for this grid first).
    // Then wait for the partition pass.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    constexpr int WPC = kMergeThreads / 32;
    const int lane = threadIdx.x & 31;
    const int pairs = p.num_seqs * p.num_q_heads;
    for (int wg = blockIdx.x * WPC + (threadIdx.x >> 5); wg < pairs; wg += gridDim.x * WPC)
        merge_one<T, D>(p, wg, lane);
}

size_t partition_smem_bytes(int head_dim, int num_seqs) {
    return (size_t)kWarps * kMaxGroup * head_dim * 4 + 2 * kWarps * kMaxGroup * 4 +
           (size_t)(2 * num_seqs + 1) * 4;
}

constexpr int kPassPartition = 1;
constexpr int kPassMerge = 2;
// A cascade's prefix pass takes at most 1 / kCascadePrefixShare of the SMs
// (PKV_PREFIX_CTAS=<n> overrides, for comparison runs); the partition pass
// over the sequences' own blocks takes the rest.
constexpr int kCascadePrefixShare = 8;
int cascade_prefix_ctas(int sms) {
    static const int forced = [] {
        const char* v = std::getenv("PKV_PREFIX_CTAS");
        return v ? std::atoi(v) : 0;
    }();
    if (forced > 0) return std::min(forced, std::max(1, sms - 1));
    return std::max(1, sms / kCascadePrefixShare);
}

template <typename T, int D>
pkv_status launch_decode(const DecodeParams& prm_in, const MergeParams& mp, int pb_lower,
                         int max_blocks, bool need_merge, int passes, bool plain_merge,
                         cudaStream_t stream) {
    DecodeParams prm = prm_in;
    auto kern = decode_partition_kernel<T, D>;
    const size_t smem = partition_smem_bytes(D, prm.num_seqs);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess)
        return PKV_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    const long long parts_upper = (long long)prm.num_seqs * std::max(1, ceil_div(max_blocks, pb_lower));
    const long long items_upper = parts_upper * prm.num_kv_heads;
    const int grid = (int)std::max<long long>(1, std::min<long long>(items_upper, (long long)std::max(occ, 1) * sms));
    prm.target_items = grid * kItemsPerCta;
    prm.trigger_merge = (passes & kPassMerge) && need_merge;
    if (passes & kPassPartition) {
        kern<<<grid, kThreads, smem, stream>>>(prm);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    if ((passes & kPassMerge) && need_merge) {
        // programmatic dependent launch: the merge grid is scheduled while the
        // partition grid drains and waits (griddepcontrol.wait) for its results
        constexpr int WPC = kMergeThreads / 32;
        const int pairs = prm.num_seqs * prm.num_q_heads;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((pairs + WPC - 1) / WPC));
        cfg.blockDim = dim3(kMergeThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = plain_merge ? 0 : 1;
        if (cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, D>, mp) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return PKV_OK;
}


// ---------------------------------------------------------------------------
// Host side of the TMA partition pass.
// ---------------------------------------------------------------------------
int smem_optin_bytes() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    return v;
}

// Registers a kernel's CTA of `threads` holds (allocated per warp in units of
// 256), cached per kernel.
int cta_registers(const void* fn, int threads) {
    static std::mutex mu;
    static const void* keys[16];
    static int regs[16];
    static int n = 0;
    std::lock_guard<std::mutex> lk(mu);
    int r = -1;
    for (int i = 0; i < n; ++i)
        if (keys[i] == fn) r = regs[i];
    if (r < 0) {
        cudaFuncAttributes a;
        if (cudaFuncGetAttributes(&a, fn) != cudaSuccess) return -1;
        r = a.numRegs;
        if (n < 16) {
            keys[n] = fn;
            regs[n++] = r;
        }
    }
    return (r * 32 + 255) / 256 * 256 * ((threads + 31) / 32);
}

// Merge CTAs that fit on one SM beside one partition CTA (registers, shared
// memory and threads; at least 1).  The merge pass is launched while its
// partition pass runs; capped at this many CTAs per SM, every merge CTA is
// resident from the start, and none lands on an SM the partition pass leaves,
// where it would keep out the next layer's partition CTA.
int merge_ctas_beside(const void* part, int part_threads, size_t part_smem, const void* merge) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int regs_sm = 0, smem_sm = 0, smem_res = 0, threads_sm = 0;
    if (cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&smem_res, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) !=
            cudaSuccess)
        return 1;
    const long long pr = cta_registers(part, part_threads);
    const long long mr = cta_registers(merge, kMergeThreads);
    if (pr <= 0 || mr <= 0) return 1;
    long long k = (regs_sm - pr) / mr;
    k = std::min<long long>(
        k, ((long long)smem_sm - (long long)part_smem - 2ll * smem_res) / std::max(1, smem_res));
    k = std::min<long long>(k, (threads_sm - part_threads) / kMergeThreads);
    return (int)std::max<long long>(1, k);
}

size_t tma_fixed_smem(int head_dim, int num_seqs, int group) {
    return 1024 + (size_t)kTmaConsumers * group * (head_dim + 4) * 4 +
           2 * kTmaConsumers * kMaxGroup * 4 + (2 * kTmaConsumers + 2) * 4 +
           (size_t)(2 * num_seqs + 1) * 4;
}

size_t tma_stage_smem(int head_dim, int heads_per_consumer = 1) {
    // K and V tiles of the consumer's heads, two mbarriers, a block id and a
    // use count, per consumer
    return (size_t)kTmaConsumers *
           (2 * (size_t)heads_per_consumer * 16 * head_dim * 2 + 2 * 8 + 4 + 4);
}

// Stages per consumer ring that fit in the opt-in shared memory (0 if < 2).
int tma_stages(int head_dim, int num_seqs, int group, int heads_per_consumer = 1) {
    const long long room =
        (long long)smem_optin_bytes() - (long long)tma_fixed_smem(head_dim, num_seqs, group);
    const long long ns = room / (long long)tma_stage_smem(head_dim, heads_per_consumer);
    return ns < 2 ? 0 : (int)std::min<long long>(ns, kTmaMaxStages);
}

// Consumers serve two heads per block (kHPC = 2) for items of two D = 64 heads
// on the producer warp, unless PKV_TWO_HEADS=0 (one head each, kept for
// comparison runs).
bool two_heads_per_consumer() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_TWO_HEADS");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

// KV heads per TMA item.  One head per item keeps each consumer's share of a
// partition long and the partials few; several heads per item fetch more of a
// block's contiguous run at once and keep consumers busy when contexts are
// short.  Rule, from sweeps of 1/2/4/8 heads per item on five workloads:
// under an even split, the fewest heads that fetch 256 bytes of each row;
// else one head when unsplit (sequence, head) items already give every SM 4
// of them, or when there are no more of them than SMs; otherwise the fewest
// heads that make max_blocks * heads >= 256, i.e. at least 32 blocks per
// consumer of a longest sequence (28-layer steps with 2..32-block contexts ran
// 1.12x faster at 8 heads per item than at 1).
// PKV_HEADS_PER_ITEM=<n> or =all overrides.
int tma_heads_per_item(int num_seqs, int max_blocks, int num_kv_heads, int head_dim,
                       bool even) {
    // consumers split evenly over the heads of an item, so a valid count
    // divides both the KV heads and the consumer warps
    auto valid = [&](int h) { return h >= 1 && num_kv_heads % h == 0 && kTmaConsumers % h == 0; };
    static const int forced = [] {
        const char* v = std::getenv("PKV_HEADS_PER_ITEM");
        if (!v) return 0;
        return std::strcmp(v, "all") == 0 ? -1 : std::atoi(v);
    }();
    if (forced == -1) {
        int h = std::min(num_kv_heads, kTmaConsumers);
        while (!valid(h)) --h;
        return h;
    }
    if (forced > 0) return valid(forced) ? forced : 1;
    if (even) {
        // an even split walks one head group of a sequence at a time: fetch
        // at least 256 contiguous bytes of each row (one D = 64 head is 128;
        // measured 1.17x faster with two heads per item there; four heads, the
        // whole row, measured no faster)
        int h = std::max(1, 128 / head_dim);
        while (h < num_kv_heads && !valid(h)) ++h;
        return valid(h) ? h : 1;
    }
    if ((long long)num_seqs * num_kv_heads >= 4ll * sm_count()) return 1;
    // so few (sequence, head) pairs that one head per item still leaves SMs
    // idle: one head, so that each sequence's blocks spread over a CTA's eight
    // consumers (4 sequences x 8 heads: 12.3 us a step against 19.5 at 8 heads)
    if ((long long)num_seqs * num_kv_heads <= sm_count()) return 1;
    int hpi = 1;
    for (int h = 2; h <= kTmaConsumers; ++h) {
        if ((long long)max_blocks * hpi >= 32ll * kTmaConsumers) break;
        if (valid(h)) hpi = h;
    }
    return hpi;
}

// Consumer warps take whole one-head items of their own (warp items) when
// the (sequence, KV head) pairs give every consumer warp of the grid half an
// item or more, unless PKV_WARP_ITEMS=0 (kept for comparison runs).
bool warp_items_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_WARP_ITEMS");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

// Adaptive partitioning aims at this many items per CTA (PKV_TMA_ITEMS overrides).
int tma_items_per_cta(int heads_per_item) {
    static const int forced = [] {
        const char* v = std::getenv("PKV_TMA_ITEMS");
        return v ? std::atoi(v) : 0;
    }();
    if (forced > 0) return forced;
    return heads_per_item == 1 ? kTmaItemsPerCta : kTmaItemsPerCta / 2;
}

// The stream-producer build feeds a cascade's suffix pass unless
// PKV_STREAM_FEED=0 (the self-feeding warps, kept for comparison runs).
bool stream_feed_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_STREAM_FEED");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

// One-head items on the producer warp run the 12-warp build unless
// PKV_WIDE=0 (the 9-warp build, kept for comparison runs).
bool wide_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_WIDE");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

// Its register shares (setmaxnreg) add up only at its 168-register launch.
template <typename T, int D>
bool wide_regs_ok() {
    static const bool ok = [] {
        cudaFuncAttributes a;
        return cudaFuncGetAttributes(&a, decode_partition_tma_kernel<T, D, true, false, 1, false,
                                                                     false, true>) ==
                   cudaSuccess &&
               a.numRegs == kStreamLaunchRegs;
    }();
    return ok;
}

// Its register shares (setmaxnreg) add up only at its 168-register launch.
template <typename T, int D>
bool stream_regs_ok() {
    static const bool ok = [] {
        cudaFuncAttributes a;
        return cudaFuncGetAttributes(&a, decode_partition_tma_kernel<T, D, true, false, 1, true,
                                                                     true>) == cudaSuccess &&
               a.numRegs == kStreamLaunchRegs;
    }();
    return ok;
}

template <typename T, int D>
pkv_status launch_decode_tma(const DecodeParams& prm_in, const MergeParams& mp_in, int pb_lower,
                             int max_blocks, bool need_merge, int passes, int nstages,
                             int sm_cap, bool plain_merge, cudaStream_t stream,
                             bool feeds_next = false) {
    DecodeParams prm = prm_in;
    MergeParams mp = mp_in;
    int sms = sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    if (sm_cap > 0) sms = std::min(sms, sm_cap);  // the other SMs run a cascade's prefix pass
    // The adaptive, non-cascade pass over long contexts splits the work
    // evenly over the CTAs (measured: CTAs of the round-robin item split
    // finished up to 17 % apart on lognormal lengths).  Short contexts (under
    // kEvenMinBlocks blocks) keep items: cut evenly, nearly every sequence
    // would span CTAs and need a merge (measured 1.2x slower on 2..32-block
    // contexts).  A caller-fixed partition length or a cascade suffix keeps
    // items of whole partitions.
    bool even = prm.prefix_parts == 0 && prm.partition_blocks <= 0 &&
                max_blocks >= kEvenMinBlocks;
    // items cover `hpi` KV heads of one partition
    int hpi = tma_heads_per_item(prm.num_seqs, max_blocks, prm.num_kv_heads, D, even);
    if (even && hpi * prm.group > kEvenMaxHeads) {
        // more query heads per slot than the workspace keeps (only through
        // the heads-per-item override): items instead
        even = false;
        hpi = tma_heads_per_item(prm.num_seqs, max_blocks, prm.num_kv_heads, D, false);
    }
    // A cascade's suffixes (each sequence is merged with its prefix row
    // anyway) are split evenly over the grid's consumer warps: each warp
    // streams an equal run of (sequence, KV head, block) units.  A warp's
    // time is set by its blocks (a stage costs a third of a copy's round
    // trip), and items dealt whole left the longest suffix's warp running
    // alone at the end (cascade step 56.8 -> see the measurements).  Needs
    // 2 B Hq rows (prefix, whole suffixes) plus two slots of g rows per warp.
    bool warp_even = false;
    if (prm.prefix_parts > 0 && prm.partition_blocks <= 0 && warp_items_enabled() &&
        prm.group <= kEvenMaxHeads) {
        const long long rows = 2ll * prm.num_seqs * prm.num_q_heads +
                               2ll * sms * kTmaConsumers * prm.group;
        warp_even = rows <= prm.ws_rows;
    }
    if (warp_even) {
        even = true;
        hpi = 1;
    }
    const int groups = prm.num_kv_heads / hpi;
    int grid;
    if (even) {
        const long long units_upper = (long long)prm.num_seqs * groups * std::max(1, max_blocks);
        grid = (int)std::max<long long>(1, std::min<long long>(units_upper,
                                                              std::min(sms, kMaxEvenGrid)));
        if (warp_even) grid = std::min(sms, kMaxEvenGrid);
        prm.even_split = 1;
        mp.even_grid = warp_even ? grid * kTmaConsumers : grid;  // workers
        mp.even_heads = hpi * prm.group;
        mp.groups = groups;
        if (warp_even) {
            prm.even_row0 = 2 * prm.num_seqs * prm.num_q_heads;
            mp.even_row0 = prm.even_row0;
        } else {
            need_merge = max_blocks > 1;  // a one-block (sequence, group) is never cut
        }
    } else {
        const long long items_upper =
            (long long)prm.num_seqs * std::max(1, ceil_div(max_blocks, pb_lower)) * groups;
        grid = (int)std::max<long long>(1, std::min<long long>(items_upper, sms));
        // per-head items: 8 per CTA; all-heads items carry Hkv heads each: 4 per CTA
        prm.target_items = grid * tma_items_per_cta(hpi);
    }
    const bool warp_items = warp_even || (!even && hpi == 1 && warp_items_enabled() &&
                                          (long long)prm.num_seqs * prm.num_kv_heads >=
                                              (long long)kTmaConsumers * sms / 2);
    if (warp_items && !even) prm.target_items = grid * kTmaConsumers * 2;  // two items per warp

    int merge_cap = 0;  // merge CTAs that fit beside this pass's partition CTAs
    if (passes & kPassPartition) {
        CUtensorMap tmk, tmv;
        const pkv_dtype dt = std::is_same<T, __nv_bfloat16>::value ? PKV_BF16 : PKV_F16;
        if (!make_pool_map(&tmk, prm.k_cache, prm.num_blocks, prm.num_kv_heads, D, dt) ||
            !make_pool_map(&tmv, prm.v_cache, prm.num_blocks, prm.num_kv_heads, D, dt))
            return PKV_ERR_CUDA;
        // consumers that feed themselves measured faster with 4 or more heads
        // per item (short contexts: 28-layer steps 8 % faster), the producer
        // warp with 1 or 2 (long contexts: 10 % faster)
        // two D = 64 heads per consumer step (8 KB, as one head at D = 128),
        // fed by the producer warp: the even split's items of two heads
        const int ns2 = (D == 64 && even && hpi == 2 && two_heads_per_consumer())
                            ? tma_stages(D, prm.num_seqs, prm.group, 2)
                            : 0;
        const int hpc = ns2 >= 2 ? 2 : 1;
        if (hpc == 2) nstages = ns2;
        // a cascade's suffixes split over the consumer warps: their rings are
        // filled by a stream-producer warp (unless PKV_STREAM_FEED=0, or the
        // build does not launch at the register count its shares assume)
        const bool stream_feed = warp_even && stream_feed_enabled() && stream_regs_ok<T, D>();
        const bool self_feed = !stream_feed && ((hpi >= 4 && hpc == 1) || warp_items);
        // (the two-head build exists at D = 64 only)
        constexpr int kTwo = D == 64 ? 2 : 1;
        // one-head items on the producer warp run in 12 warps, their consumers
        // given more registers (long-context step 172.5 -> 171.9 us; two-head
        // items measured no faster)
        const bool wide = !stream_feed && !self_feed && hpi == 1 && wide_enabled() &&
                          wide_regs_ok<T, D>();
        auto kern = stream_feed ? decode_partition_tma_kernel<T, D, true, false, 1, true, true>
                    : warp_items ? decode_partition_tma_kernel<T, D, true, true, 1, true>
                    : self_feed ? decode_partition_tma_kernel<T, D, false, true>
                    : hpi == 1  ? (wide ? decode_partition_tma_kernel<T, D, true, false, 1, false,
                                                                       false, true>
                                        : decode_partition_tma_kernel<T, D, true, false>)
                    : hpc == 2 ? decode_partition_tma_kernel<T, D, false, false, kTwo>
                               : decode_partition_tma_kernel<T, D, false, false>;
        const size_t smem = tma_fixed_smem(D, prm.num_seqs, prm.group) +
                            (size_t)nstages * tma_stage_smem(D, hpc);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        // programmatic dependent launch: the CTAs are scheduled while the
        // previous kernel drains; with early_reads the prologue and the first
        // cache loads overlap a previous layer's merge pass (see the kernel)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(tma_threads(self_feed, stream_feed, wide));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, prm, tmk, tmv, nstages, hpi) != cudaSuccess)
            return PKV_ERR_CUDA;
        merge_cap = sms * merge_ctas_beside(reinterpret_cast<const void*>(kern),
                                            tma_threads(self_feed, stream_feed, wide), smem,
                                            reinterpret_cast<const void*>(
                                                decode_merge_kernel<T, D>));
    }
    if ((passes & kPassMerge) && need_merge) {
        constexpr int WPC = kMergeThreads / 32;
        const int pairs = prm.num_seqs * prm.num_q_heads;
        int mgrid = (pairs + WPC - 1) / WPC;
        // When the next kernel is the next layer's partition pass, the merge
        // fits beside a partition CTA on every SM (else its CTAs, landing on
        // the SMs this pass leaves, would hold that layer's CTAs off them
        // until the merge ends: 1.3x slower 28-layer steps).  Otherwise it
        // takes as many CTAs as it has pairs / 4 (capped, 8192 pairs of
        // D = 64 merged 8 % slower).
        if (feeds_next && !plain_merge && merge_cap > 0) mgrid = std::min(mgrid, merge_cap);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)mgrid);
        cfg.blockDim = dim3(kMergeThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = plain_merge ? 0 : 1;
        if (cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, D>, mp) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return PKV_OK;
}


// Which partition kernel runs: the TMA pipeline unless PKV_DECODE_KERNEL=ldg
// selects the register-pipelined kernel (kept for comparison).
bool use_tma_kernel() {
    static const bool tma = [] {
        const char* v = std::getenv("PKV_DECODE_KERNEL");
        return !(v && std::strcmp(v, "ldg") == 0);
    }();
    return tma;
}

pkv_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int max_context_len, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                       float scale, void* out, void* workspace, size_t workspace_bytes,
                       int partition_blocks, pkv_dtype dtype, int passes,
                       cudaStream_t stream, const void* k_new = nullptr,
                       const void* v_new = nullptr, int64_t* slot_out = nullptr,
                       int prefix_blocks = 0, bool chained = false, bool feeds_next = false) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 ||
        partition_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    const int g = num_q_heads / num_kv_heads;
    if (g > kMaxGroup || (head_dim != 64 && head_dim != 128) || num_seqs > kMaxSeqs)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    const int prefix_parts = prefix_blocks > 0 ? 1 : 0;  // the cascade's prefix row
    const WsLayout ws =
        ws_layout(num_seqs, num_q_heads, head_dim, max_context_len, prefix_parts);
    if (!workspace || workspace_bytes < ws.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_WORKSPACE;
    const int min_pb = min_partition_blocks(max_context_len);
    if (partition_blocks > 0 && partition_blocks < min_pb) return PKV_ERR_INVALID_ARG;
    unsigned int* status = status_word();
    if (!status) return PKV_ERR_CUDA;

    const int len_bound = (int)std::min<long long>(max_context_len,
                                                   (long long)max_blocks_per_seq * PKV_BLOCK_SIZE);
    const int max_blocks = ceil_div(len_bound, PKV_BLOCK_SIZE);
    const int pb_lower =
        partition_blocks > 0 ? partition_blocks : std::max(min_pb, kAdaptiveMinBlocks);
    // a cascade merges every sequence (its prefix rows plus its suffix items)
    const bool need_merge = prefix_parts > 0 || max_blocks > pb_lower;

    char* wsb = static_cast<char*>(workspace);
    DecodeParams prm;
    prm.q = q;
    prm.k_cache = k_cache;
    prm.v_cache = v_cache;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.out = out;
    prm.ws_offsets = reinterpret_cast<int*>(wsb + ws.offsets);
    prm.ws_m = reinterpret_cast<float*>(wsb + ws.m);
    prm.ws_l = reinterpret_cast<float*>(wsb + ws.l);
    prm.ws_o = reinterpret_cast<float*>(wsb + ws.o);
    prm.status = status;
    prm.k_new = k_new;
    prm.v_new = v_new;
    prm.k_cache_w = const_cast<void*>(k_cache);
    prm.v_cache_w = const_cast<void*>(v_cache);
    prm.slot_out = k_new ? slot_out : nullptr;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = g;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.len_bound = len_bound;
    prm.partition_blocks = partition_blocks;
    prm.skip_blocks = prefix_blocks;
    prm.prefix_parts = prefix_parts;
    prm.item_row0 = num_seqs * prefix_parts;  // rows 0 .. num_seqs - 1: the prefix partials
    prm.even_row0 = 0;
    prm.ws_rows = (long long)ws.rows;
    prm.no_wait = 0;
    prm.min_partition_blocks = pb_lower;
    prm.target_items = 0;
    prm.even_split = 0;
    prm.trigger_merge = 0;
    prm.early_reads = chained ? 1 : 0;
    prm.scale_log2 = scale * kLog2e;

    MergeParams mp;
    mp.ws_offsets = prm.ws_offsets;
    mp.ws_m = prm.ws_m;
    mp.ws_l = prm.ws_l;
    mp.ws_o = prm.ws_o;
    mp.out = out;
    mp.num_seqs = num_seqs;
    mp.num_q_heads = num_q_heads;
    mp.min_rows = prefix_parts > 0 ? 1 : 2;
    mp.prefix_rows = prefix_parts;
    mp.item_row0 = prm.item_row0;
    mp.even_row0 = 0;
    mp.even_grid = 0;  // the TMA pass sets the even-split fields
    mp.even_heads = 0;
    mp.groups = 0;

    // partition kernel (TMA pipeline or register pipeline) and merge kernel
    // the TMA kernel maps its 8 consumer warps onto the KV heads (Hkv must divide 8)
    const int nstages = use_tma_kernel() && kTmaConsumers % num_kv_heads == 0
                            ? tma_stages(head_dim, num_seqs, g)
                            : 0;
    const int grid_blocks = std::max(1, max_blocks - prefix_blocks);  // blocks items can cover
    auto run = [&](int pass_mask, int sm_cap, bool plain_merge) -> pkv_status {
        if (nstages > 0) {
            if (dtype == PKV_BF16)
                return head_dim == 128
                           ? launch_decode_tma<__nv_bfloat16, 128>(prm, mp, pb_lower, grid_blocks,
                                                                   need_merge, pass_mask, nstages,
                                                                   sm_cap, plain_merge, stream,
                                                                   feeds_next)
                           : launch_decode_tma<__nv_bfloat16, 64>(prm, mp, pb_lower, grid_blocks,
                                                                  need_merge, pass_mask, nstages,
                                                                  sm_cap, plain_merge, stream,
                                                                  feeds_next);
            return head_dim == 128
                       ? launch_decode_tma<__half, 128>(prm, mp, pb_lower, grid_blocks, need_merge,
                                                        pass_mask, nstages, sm_cap, plain_merge,
                                                        stream, feeds_next)
                       : launch_decode_tma<__half, 64>(prm, mp, pb_lower, grid_blocks, need_merge,
                                                       pass_mask, nstages, sm_cap, plain_merge,
                                                       stream, feeds_next);
        }
        if (dtype == PKV_BF16)
            return head_dim == 128
                       ? launch_decode<__nv_bfloat16, 128>(prm, mp, pb_lower, grid_blocks,
                                                           need_merge, pass_mask, plain_merge,
                                                           stream)
                       : launch_decode<__nv_bfloat16, 64>(prm, mp, pb_lower, grid_blocks,
                                                          need_merge, pass_mask, plain_merge,
                                                          stream);
        return head_dim == 128 ? launch_decode<__half, 128>(prm, mp, pb_lower, grid_blocks,
                                                            need_merge, pass_mask, plain_merge,
                                                            stream)
                               : launch_decode<__half, 64>(prm, mp, pb_lower, grid_blocks,
                                                           need_merge, pass_mask, plain_merge,
                                                           stream);
    };
    if (prefix_parts == 0) return run(passes, 0, false);

    // Cascade.  The shared prefix for all sharers runs first on the tensor
    // cores, on a few SMs (an ordinary launch: it waits for everything before
    // it).  The partition pass over the sequences' own blocks is its
    // programmatic dependent and runs beside it on the other SMs: the two
    // share nothing they write (prefix rows vs item rows, the new tokens
    // land past the prefix), so the TMA pass waits for it only before it
    // ends (the register-pipelined pass waits at its start).
    // The suffix pass runs on the SMs the prefix pass leaves; its merge is
    // planned for the same SM count (an even split's workers).  The merge is
    // the suffix pass's programmatic dependent: the suffix pass's threads wait
    // for the prefix pass before they end, so the merge's wait covers both.
    const int sms = sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    const int prefix_ctas = cascade_prefix_ctas(sms);
    const int suffix_sms =
        std::max(1, sms - cascade_prefix_grid(num_seqs, num_q_heads, num_kv_heads, prefix_ctas));
    if (passes & kPassPartition) {
        int pgrid = 0;
        pkv_status rc = launch_cascade_prefix(
            q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, len_bound,
            num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, prefix_blocks,
            prm.scale_log2, prm.ws_m, prm.ws_l, prm.ws_o, dtype, prefix_ctas, &pgrid, stream);
        if (rc != PKV_OK) return rc;
        prm.no_wait = 1;
        rc = run(kPassPartition, suffix_sms, true);
        if (rc != PKV_OK) return rc;
    }
    return (passes & kPassMerge) ? run(kPassMerge, suffix_sms, !(passes & kPassPartition))
                                 : PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

int paged_attention_min_partition_blocks(int max_context_len) {
    return pkv::min_partition_blocks(max_context_len);
}

size_t paged_attention_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                       int max_context_len) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    return pkv::ws_layout(num_seqs, num_q_heads, head_dim, max_context_len).total;
}

size_t paged_attention_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                               int max_context_len, int num_prefix_blocks) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        num_prefix_blocks < 0)
        return 0;
    return pkv::ws_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                          num_prefix_blocks > 0 ? 1 : 0)
        .total;
}

pkv_status paged_attention_decode_cascade(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int max_context_len, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int num_blocks,
                                          int num_prefix_blocks, float scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          pkv_dtype dtype, pkv_stream_t stream) {
    if (num_prefix_blocks <= 0) return PKV_ERR_INVALID_ARG;
    return pkv::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, out, workspace, workspace_bytes, 0, dtype,
                            pkv::kPassPartition | pkv::kPassMerge,
                            reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr,
                            num_prefix_blocks);
}

pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int max_context_len,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int num_blocks, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
    return pkv::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, out, workspace, workspace_bytes, 0, dtype,
                            pkv::kPassPartition | pkv::kPassMerge,
                            reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_attention_decode_partitioned(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream) {
    return pkv::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, out, workspace, workspace_bytes, partition_blocks,
                            dtype, pkv::kPassPartition | pkv::kPassMerge,
                            reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_attention_partition_pass(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream) {
    return pkv::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, out, workspace, workspace_bytes, partition_blocks,
                            dtype, pkv::kPassPartition, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_attention_merge_pass(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, float scale, void* out,
    void* workspace, size_t workspace_bytes, int partition_blocks, pkv_dtype dtype,
    pkv_stream_t stream) {
    return pkv::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            num_blocks, scale, out, workspace, workspace_bytes, partition_blocks,
                            dtype, pkv::kPassMerge, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_kv_write_new_tokens(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* context_lens,
                                     int num_seqs, int num_blocks, int num_kv_heads,
                                     int head_dim, int64_t* slot_mapping_out, pkv_dtype dtype,
                                     pkv_stream_t stream) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || !pkv::aligned16(k_cache) ||
        !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    return pkv::launch_decode_step_write(k_new, v_new, k_cache, v_cache, block_tables,
                                         max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                                         num_kv_heads, head_dim, slot_mapping_out,
                                         reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pkv {
namespace {

pkv_status decode_step_impl(const void* q, const void* k_new, const void* v_new, void* k_cache,
                            void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                            float scale, void* out, int64_t* slot_mapping_out, void* workspace,
                            size_t workspace_bytes, pkv_dtype dtype, int passes,
                            cudaStream_t stream, int prefix_blocks = 0,
                            bool chained = false, bool feeds_next = false) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       num_blocks, scale, out, workspace, workspace_bytes, 0, dtype, passes,
                       stream, k_new, v_new, slot_mapping_out, prefix_blocks, chained,
                       feeds_next);
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status paged_kv_decode_step(const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int max_context_len, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int num_blocks, float scale,
                                void* out, int64_t* slot_mapping_out, void* workspace,
                                size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
    return pkv::decode_step_impl(q, k_new, v_new, k_cache, v_cache, block_tables,
                                 max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                 num_q_heads, num_kv_heads, head_dim, num_blocks, scale, out,
                                 slot_mapping_out, workspace, workspace_bytes, dtype,
                                 pkv::kPassPartition | pkv::kPassMerge,
                                 reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_kv_decode_step_layers(const void* q, const void* k_new, const void* v_new,
                                       void* k_cache, void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_dim, int num_blocks,
                                       int num_layers, float scale, void* out, void* workspace,
                                       size_t workspace_bytes, pkv_dtype dtype,
                                       pkv_stream_t stream) {
    if (num_layers < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_layers == 0 || num_seqs == 0) return PKV_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !out) return PKV_ERR_INVALID_ARG;
    const size_t q_layer = (size_t)num_seqs * num_q_heads * head_dim * 2;
    const size_t new_layer = (size_t)num_seqs * num_kv_heads * head_dim * 2;
    const size_t pool_layer = (size_t)num_blocks * PKV_BLOCK_SIZE * num_kv_heads * head_dim * 2;
    for (int l = 0; l < num_layers; ++l) {
        const pkv_status rc = pkv::decode_step_impl(
            static_cast<const char*>(q) + l * q_layer, static_cast<const char*>(k_new) + l * new_layer,
            static_cast<const char*>(v_new) + l * new_layer, static_cast<char*>(k_cache) + l * pool_layer,
            static_cast<char*>(v_cache) + l * pool_layer, block_tables, max_blocks_per_seq,
            context_lens, max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
            num_blocks, scale, static_cast<char*>(out) + l * q_layer, nullptr, workspace,
            workspace_bytes, dtype, pkv::kPassPartition | pkv::kPassMerge,
            reinterpret_cast<cudaStream_t>(stream), 0,
            /*chained=*/l > 0,   // layer l-1's kernels write only layer l-1's pools
            /*feeds_next=*/l + 1 < num_layers);
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

pkv_status paged_kv_decode_step_cascade(const void* q, const void* k_new, const void* v_new,
                                        void* k_cache, void* v_cache,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* context_lens, int max_context_len,
                                        int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int num_blocks, int num_prefix_blocks,
                                        float scale, void* out, int64_t* slot_mapping_out,
                                        void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                                        pkv_stream_t stream) {
    if (num_prefix_blocks <= 0) return PKV_ERR_INVALID_ARG;
    return pkv::decode_step_impl(q, k_new, v_new, k_cache, v_cache, block_tables,
                                 max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                 num_q_heads, num_kv_heads, head_dim, num_blocks, scale, out,
                                 slot_mapping_out, workspace, workspace_bytes, dtype,
                                 pkv::kPassPartition | pkv::kPassMerge,
                                 reinterpret_cast<cudaStream_t>(stream), num_prefix_blocks);
}

pkv_status paged_kv_decode_step_partition_pass(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int num_blocks, float scale, void* out, int64_t* slot_mapping_out, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, pkv_stream_t stream) {
    return pkv::decode_step_impl(q, k_new, v_new, k_cache, v_cache, block_tables,
                                 max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                 num_q_heads, num_kv_heads, head_dim, num_blocks, scale, out,
                                 slot_mapping_out, workspace, workspace_bytes, dtype,
                                 pkv::kPassPartition, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
