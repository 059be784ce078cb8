// pkv_prefill.cu -- chunked-prefill attention over the paged cache.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "pkv_internal.cuh"
#include "pkv_tc.cuh"
#include "pkv_tma.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ============================================================================
// Chunked prefill over the paged cache ("MinivLLM" 使用教程 step 4 / 核心亮点:
// FlashAttention for the prefill stage; "mini-vllm 项目深度解析"
// §关键工程决策 item 2: prefill chunks batched with decode).
//
// Sequence s has q_len = cu_q_lens[s+1] - cu_q_lens[s] query rows (already
// written to the cache) at positions n - q_len .. n - 1, n = context_lens[s];
// the row at position p attends to tokens 0..p.  A CTA takes one sequence,
// one KV head and a tile of 64 rows of (query token, query head of the
// group) pairs, so every K/V block it loads serves all g query heads.  A
// producer warp stages the head's blocks 0 .. (tile's causal bound) into a
// 4-stage ring with the same tensor-map TMA copies as the decode pass; four
// consumer warps of 16 rows each run S = Q K^T and O += P V on mma.sync with
// K (ldmatrix) and V (ldmatrix.trans) as the B operands, P going from the
// score accumulators straight into the A operand, and an online softmax per
// row.  Waits are bounded as in the decode pass.
// ============================================================================
constexpr int kPrefillConsumers = 4;
constexpr int kPrefillThreads = (kPrefillConsumers + 1) * 32;
constexpr int kPrefillRows = kPrefillConsumers * 16;
constexpr int kPrefillStages = 4;

struct PrefillParams {
    const void* q;
    void* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* cu_q_lens;
    unsigned int* status;
    int num_seqs, num_q_heads, num_kv_heads, group, max_blocks_per_seq, num_blocks;
    int max_q_len, num_q_rows;  // host bounds: longest chunk, rows of q and out
    int tiles_per_seq;  // ceil(max_q_len * group / kPrefillRows)
    float scale_log2;
    // Cascade prefix mode of the tensor-core kernel (prefix_tokens > 0): the
    // query rows are every sequence's decode query (row r of a KV head's rows:
    // sequence r / group, query head r % group of that KV head), the keys are
    // the shared prefix (the first prefix_tokens / 16 entries of block-table
    // row 0), a row sees min(its length, prefix_tokens) of them, and each
    // row's unnormalised result (m, l, o; base-2 scores) goes to workspace
    // row sequence * num_q_heads + query head.
    int prefix_tokens, len_bound;
    float* ws_m;
    float* ws_l;
    float* ws_o;
};

// A sequence's chunk is usable if its rows lie inside q/out, it is no longer
// than the host bound the grid was sized for, and it fits its context and the
// table.  qlen == 0 is a valid empty chunk (skipped without a flag).
__device__ __forceinline__ bool prefill_lengths_ok(const PrefillParams& p, int q0, int qlen,
                                                   int n) {
    return qlen > 0 && q0 >= 0 && q0 <= p.num_q_rows - qlen && qlen <= p.max_q_len &&
           n >= qlen && n <= p.max_blocks_per_seq * PKV_BLOCK_SIZE;
}

template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads)
    prefill_tma_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v) {
    using E = Elem<T>;
    constexpr int NS = kPrefillStages;
    constexpr int HALVES = D / 64;
    constexpr int TILE = 16 * D * 2;
    constexpr int STAGE = 2 * TILE;
    constexpr int KS = D / 16;   // k-steps over D
    constexpr int DN = D / 8;    // 8-wide column tiles of O
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * STAGE);
    uint64_t* empty = full + NS;
    int* stage_ok = reinterpret_cast<int*>(empty + NS);
    volatile int* abort_flag = stage_ok + NS;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x % p.tiles_per_seq;
    const int h = (blockIdx.x / p.tiles_per_seq) % p.num_kv_heads;
    const int s = blockIdx.x / (p.tiles_per_seq * p.num_kv_heads);
    const int g = p.group, Hq = p.num_q_heads;
    const int q0 = p.cu_q_lens[s], qlen = p.cu_q_lens[s + 1] - q0;
    const int n = p.context_lens[s];
    if (!prefill_lengths_ok(p, q0, qlen, n)) {
        if (tid == 0 && tile == 0 && h == 0 && qlen != 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        return;
    }
    const int row0 = tile * kPrefillRows;      // first (token, head) row of the tile
    if (row0 >= qlen * g) return;              // beyond this sequence's chunk
    const int tok_last = min(qlen, (row0 + kPrefillRows + g - 1) / g) - 1;
    const int p_last = n - qlen + tok_last;    // the tile's largest query position
    const int nblk = p_last / PKV_BLOCK_SIZE + 1;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kPrefillConsumers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == kPrefillConsumers) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
            int issued = 0;
            for (int j = 0; j < nblk && !*abort_flag; ++j) {
                const int k = j % NS;
                if (!mbar_wait(&empty[k], ((j / NS) & 1) ^ 1, abort_flag, p.status)) break;
                int id = table[j];
                const bool ok = id >= 0 && id < p.num_blocks;
                if (!ok) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                    id = 0;  // fetched but never used
                }
                stage_ok[k] = ok;
                mbar_arrive_expect_tx(&full[k], STAGE);
                unsigned char* st = ring + k * STAGE;
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh) {
                    tma_load_rows(st + hh * 2048, &tmap_k, &full[k], hh * 64, h, id * PKV_BLOCK_SIZE);
                    tma_load_rows(st + TILE + hh * 2048, &tmap_v, &full[k], hh * 64, h,
                                  id * PKV_BLOCK_SIZE);
                }
                issued = j + 1;
            }
            for (int j = max(0, issued - NS); j < issued; ++j)
                mbar_drain(&full[j % NS], (j / NS) & 1, p.status);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int gid = lane >> 2, tig = lane & 3;
    // this lane's two rows of the tile: warp*16 + gid and + 8
    int rpos[2];   // query position of each row (-1: padding row)
    const T* qrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int R = row0 + warp * 16 + gid + 8 * r;
        const int t = R / g, hq = h * g + R % g;
        const bool live = t < qlen;
        rpos[r] = live ? n - qlen + t : -1;
        qrow[r] = static_cast<const T*>(p.q) + ((size_t)(q0 + (live ? t : 0)) * Hq + hq) * D;
    }
    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = rpos[0] >= 0 ? *reinterpret_cast<const uint32_t*>(qrow[0] + 16 * ks + 2 * tig) : 0u;
        qa[ks][1] = rpos[1] >= 0 ? *reinterpret_cast<const uint32_t*>(qrow[1] + 16 * ks + 2 * tig) : 0u;
        qa[ks][2] = rpos[0] >= 0 ? *reinterpret_cast<const uint32_t*>(qrow[0] + 16 * ks + 8 + 2 * tig) : 0u;
        qa[ks][3] = rpos[1] >= 0 ? *reinterpret_cast<const uint32_t*>(qrow[1] + 16 * ks + 8 + 2 * tig) : 0u;
    }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[DN][4];
#pragma unroll
    for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int j = 0; j < nblk; ++j) {
        const int k = j % NS;
        const bool got = mbar_wait(&full[k], (j / NS) & 1, abort_flag, p.status);
        const bool ok = got && stage_ok[k];
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        uint32_t vb[KS][4];
        if (ok) {
            const uint32_t kt = smem_addr(ring + k * STAGE), vt = kt + TILE;
            const int mi = lane >> 3;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t kb[4];  // b0, b1 of tokens 0-7, then of tokens 8-15
                ldsm_x4(kb, kt + swz((lane & 7) + 8 * (mi >> 1), 2 * ks + (mi & 1)));
                E::mma(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kb[0], kb[1]);
                E::mma(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kb[2], kb[3]);
                // V: b0, b1 of D columns 16ks..+7, then of 16ks+8..+15
                ldsm_x4_trans(vb[ks], vt + swz((lane & 7) + 8 * (mi & 1), 2 * ks + (mi >> 1)));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[k]);
        if (!ok) continue;
        // slots past the context (the tail of its last block) hold no token:
        // select them out of V, never weight them by zero (0 x NaN = NaN)
        if ((j + 1) * PKV_BLOCK_SIZE > n) {
            const int t0 = j * PKV_BLOCK_SIZE + 2 * tig;
            const uint32_t mlo = (t0 < n ? 0x0000ffffu : 0u) | (t0 + 1 < n ? 0xffff0000u : 0u);
            const uint32_t mhi = (t0 + 8 < n ? 0x0000ffffu : 0u) | (t0 + 9 < n ? 0xffff0000u : 0u);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                vb[ks][0] &= mlo;
                vb[ks][1] &= mhi;
                vb[ks][2] &= mlo;
                vb[ks][3] &= mhi;
            }
        }
        // scores of rows (gid, gid+8) x tokens 16j + 8nt + 2tig + {0,1}; causal mask
        float sv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t0 = j * PKV_BLOCK_SIZE + 8 * nt + 2 * tig;
            sv[nt][0] = t0 <= rpos[0] ? sc[nt][0] * p.scale_log2 : -INFINITY;
            sv[nt][1] = t0 + 1 <= rpos[0] ? sc[nt][1] * p.scale_log2 : -INFINITY;
            sv[nt][2] = t0 <= rpos[1] ? sc[nt][2] * p.scale_log2 : -INFINITY;
            sv[nt][3] = t0 + 1 <= rpos[1] ? sc[nt][3] * p.scale_log2 : -INFINITY;
        }
        float mx[2] = {fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1])),
                       fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]))};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float corr[2], ms[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float mn = fmaxf(m[r], mx[r]);
            ms[r] = mn == -INFINITY ? 0.f : mn;
            corr[r] = fast_exp2(m[r] - ms[r]);
            m[r] = mn;
        }
        float pv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pv[nt][0] = fast_exp2(sv[nt][0] - ms[0]);
            pv[nt][1] = fast_exp2(sv[nt][1] - ms[0]);
            pv[nt][2] = fast_exp2(sv[nt][2] - ms[1]);
            pv[nt][3] = fast_exp2(sv[nt][3] - ms[1]);
        }
        l[0] = l[0] * corr[0] + pv[0][0] + pv[0][1] + pv[1][0] + pv[1][1];
        l[1] = l[1] * corr[1] + pv[0][2] + pv[0][3] + pv[1][2] + pv[1][3];
#pragma unroll
        for (int i = 0; i < DN; ++i) {
            o[i][0] *= corr[0];
            o[i][1] *= corr[0];
            o[i][2] *= corr[1];
            o[i][3] *= corr[1];
        }
        // P as the A operand (rows x 16 tokens) straight from the score layout
        const uint32_t pa0 = E::pack(pv[0][0], pv[0][1]), pa1 = E::pack(pv[0][2], pv[0][3]);
        const uint32_t pa2 = E::pack(pv[1][0], pv[1][1]), pa3 = E::pack(pv[1][2], pv[1][3]);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            E::mma(o[2 * ks], pa0, pa1, pa2, pa3, vb[ks][0], vb[ks][1]);
            E::mma(o[2 * ks + 1], pa0, pa1, pa2, pa3, vb[ks][2], vb[ks][3]);
        }
    }
    // normalise and store rows (gid: o[.][0..1], gid+8: o[.][2..3]) at columns 8i + 2tig
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float lr = l[r];
        lr += __shfl_xor_sync(0xffffffffu, lr, 1);
        lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        if (rpos[r] < 0) continue;
        const float inv = lr > 0.f ? 1.f / lr : 0.f;
        const int R = row0 + warp * 16 + gid + 8 * r;
        T* dst = static_cast<T*>(p.out) + ((size_t)(q0 + R / g) * Hq + h * g + R % g) * D;
#pragma unroll
        for (int i = 0; i < DN; ++i)
            *reinterpret_cast<uint32_t*>(dst + 8 * i + 2 * tig) =
                E::pack(o[i][2 * r] * inv, o[i][2 * r + 1] * inv);
    }
}

// ============================================================================
// Chunked prefill on the 5th-generation tensor cores (the default).
//
// Work item: one sequence, one KV head and a tile of 128 (query token, query
// head) rows; key tiles of 128 tokens (8 paged blocks).  A persistent CTA per
// SM walks the items heaviest first (last query rows: longest causal range),
// and its pipelines run on across items:
//   warp 0   TMA-loads the K blocks of each key tile into a 2-stage ring,
//   warp 3   the V blocks into another (and marks blocks with bad ids),
//   warp 2   owns tensor memory and copies each item's Q rows (cp.async)
//            into one of two Q buffers while the previous item computes,
//   warp 1   (one thread) issues S(J) = Q K(J)^T into one of two tensor-memory
//            score buffers, two key tiles ahead of O += P(J) V(J) into the
//            tensor-memory output, each as tcgen05.mma over 128-byte swizzled
//            shared memory (Q, K, P K-major; V MN-major), with completion
//            signalled through mbarriers,
//   warps 4-7 (one thread per row) read S(J) from tensor memory, mask it
//            (causal, bad blocks) where needed, run the online softmax, write
//            P(J) as 16-bit values into shared memory, and at the end of an
//            item read O, hand it back for the next item and store O / l.
// O is rescaled only when a row's running maximum grows by more than 2^8 (P
// then stays <= 256; O / l is unchanged), so most key tiles never touch O.  V
// rows no row of the tile may see (past the causal bound, in a bad block, or
// never loaded) are zeroed before P V so that no 0 x NaN reaches O.  Every
// wait is bounded.
// ============================================================================
constexpr int kTcThreads = 384;

// Two-wide fp32 arithmetic and the three-input maximum of this architecture
// (PTX fma/add .f32x2 on packed register pairs, max.f32 with three sources):
// half the instructions of the softmax's inner loop.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// One 32-byte store (a whole L2 sector; the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(ptr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
constexpr int kTcRows = 128;     // (query token, query head) rows per tile
constexpr int kTcKeys = 128;     // keys per key tile
constexpr float kTcRescale = 8.f;  // log2 of the largest P before O is rescaled

// One work item of the tensor-core prefill.
struct TcItem {
    int s, h, q0, qlen, n, row0, p_last, nblk, nkv;
};

// Item i of the heaviest-first order; false if it holds no rows (or its
// sequence's lengths are invalid: flagged once, by the item of tile 0, head 0).
__device__ __forceinline__ bool tc_item(const PrefillParams& p, int i, bool flag, TcItem& it) {
    const int per_tile = p.num_seqs * p.num_kv_heads;
    const int tile = p.tiles_per_seq - 1 - i / per_tile;
    const int rem = i - (i / per_tile) * per_tile;
    it.s = rem / p.num_kv_heads;
    it.h = rem - it.s * p.num_kv_heads;
    it.q0 = p.cu_q_lens[it.s];
    it.qlen = p.cu_q_lens[it.s + 1] - it.q0;
    it.n = p.context_lens[it.s];
    if (!prefill_lengths_ok(p, it.q0, it.qlen, it.n)) {
        if (flag && tile == 0 && it.h == 0 && it.qlen != 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        return false;
    }
    const int g = p.group;
    it.row0 = tile * kTcRows;
    if (it.row0 >= it.qlen * g) return false;
    const int tok_last = min(it.qlen, (it.row0 + kTcRows + g - 1) / g) - 1;
    it.p_last = it.n - it.qlen + tok_last;
    it.nblk = it.p_last / PKV_BLOCK_SIZE + 1;
    it.nkv = (it.nblk + 7) / 8;
    return true;
}

// Item i of the cascade prefix mode: KV head i % num_kv_heads, tile
// i / num_kv_heads of that head's num_seqs * group rows; every item reads all
// prefix blocks.
__device__ __forceinline__ bool tc_prefix_item(const PrefillParams& p, int i, TcItem& it) {
    it.h = i % p.num_kv_heads;
    it.row0 = (i / p.num_kv_heads) * kTcRows;
    it.s = 0;                    // the prefix's blocks: block-table row 0
    it.q0 = 0;                   // decode queries: row t of q is sequence t
    it.qlen = p.num_seqs;
    it.n = p.prefix_tokens;
    if (it.row0 >= p.num_seqs * p.group) return false;
    it.p_last = p.prefix_tokens - 1;
    it.nblk = p.prefix_tokens / PKV_BLOCK_SIZE;
    it.nkv = (it.nblk + 7) / 8;
    return true;
}

template <bool kPrefix>
__device__ __forceinline__ bool tc_next(const PrefillParams& p, int i, bool flag, TcItem& it) {
    if constexpr (kPrefix) return tc_prefix_item(p, i, it);
    return tc_item(p, i, flag, it);
}

template <typename T, int D, bool kPrefix>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_q, int q_tma, int num_items) {
    using E = Elem<T>;
    constexpr int HALVES = D / 64;
    constexpr int REG = kTcRows * 128;     // one 64-element half of 128 rows: 16 KB
    constexpr int TILE = HALVES * REG;     // a Q tile, or one K or V key tile
    constexpr int HK = kTcKeys / 2;        // keys per softmax group
    constexpr uint32_t kCols = 512;        // S0, S1 (128 columns each), O_0, O_1 (128 each)
    constexpr uint32_t kOCol = 256;        // O of group q at kOCol + 128 q
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* sq = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 2 Q buffers
    unsigned char* sk = sq + 2 * TILE;      // 2 stages
    unsigned char* sv = sk + 2 * TILE;      // 2 stages
    uint64_t* bars = reinterpret_cast<uint64_t*>(sv + 2 * TILE);
    uint64_t* k_full = bars + 0;
    uint64_t* k_empty = bars + 2;
    uint64_t* v_full = bars + 4;
    uint64_t* v_empty = bars + 6;
    uint64_t* s_full = bars + 8;
    uint64_t* q_full = bars + 12;
    uint64_t* q_empty = bars + 14;
    uint64_t* p_full = bars + 16;          // [group]
    uint64_t* pv_done = bars + 18;         // [group]
    uint64_t* o_ready = bars + 20;         // an item's last P V done (both groups)
    uint64_t* o_free = bars + 21;          // group 1 has read both O halves of an item
    uint64_t* xchg = bars + 22;            // [lane quarter]: group 0's (m, l) written
    uint64_t* xfree = bars + 26;           // [lane quarter]: ... and read by group 1
    uint64_t* mma_idle = bars + 30;
    int* vbad = reinterpret_cast<int*>(bars + 31);           // [2] bad-block bits per V stage
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vbad + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* xml = reinterpret_cast<float*>(tmem_slot + 2);    // [2][128]: group 0's m, l per row

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = p.group, Hq = p.num_q_heads;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&xchg[i], 32);
            mbar_init(&xfree[i], 32);
        }
        mbar_init(o_ready, 1);
        mbar_init(o_free, 4);
        mbar_init(mma_idle, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 2) tc_alloc(tmem_slot, kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the cascade's partition pass may be scheduled beside this grid now:
    // the two touch disjoint memory, and the merge after them is an ordinary
    // launch that waits for both
    if constexpr (kPrefix) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------ K (warp 0) / V (warp 3) producers
        const bool isk = warp == 0;
        const CUtensorMap* map = isk ? &tmap_k : &tmap_v;
        uint64_t* full = isk ? k_full : v_full;
        uint64_t* empty = isk ? k_empty : v_empty;
        unsigned char* ring = isk ? sk : sv;
        int J = 0;  // key tiles issued by this CTA
        bool live = true;
        for (int i = blockIdx.x; i < num_items && live; i += gridDim.x) {
            TcItem it;
            if (!tc_next<kPrefix>(p, i, isk && lane == 0, it)) continue;
            const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks_per_seq;
            for (int j = 0; j < it.nkv; ++j, ++J) {
                const int b = J & 1, ph = (J >> 1) & 1;
                live = __all_sync(0xffffffffu, mbar_wait(&empty[b], ph ^ 1, abort_flag, p.status));
                if (!live) break;
                const int nb = min(8, it.nblk - 8 * j);
                int id = 0;
                bool bad = false;
                if (lane < nb) {
                    id = table[8 * j + lane];
                    bad = id < 0 || id >= p.num_blocks;
                    if (bad) id = 0;  // fetched, then masked and zeroed
                }
                const unsigned badm = __ballot_sync(0xffffffffu, bad);
                if (lane == 0) {
                    if (isk && badm) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                    if (!isk) vbad[b] = (int)badm;
                    mbar_arrive_expect_tx(&full[b], (uint32_t)(nb * HALVES * 2048));
                }
                __syncwarp();
                if (lane < nb) {
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh)
                        tma_load_rows(ring + b * TILE + hh * REG + lane * 2048, map, &full[b],
                                      hh * 64, it.h, id * PKV_BLOCK_SIZE);
                }
            }
        }
        // every copy issued must land before the CTA may exit
        if (lane == 0)
            for (int j = max(0, J - 2); j < J; ++j) mbar_drain(&full[j & 1], (j >> 1) & 1, p.status);
    } else if (warp == 2 && q_tma) {
        // ----------------------- Q tile of each item by tensor copies (lane 0)
        // Rows row0.. of an item are 128 / g query rows (tokens of its chunk,
        // or sequences in the prefix mode) x the g query heads of KV head h,
        // one box per 64-element half; rows past q read as zeros, rows of
        // the next chunk see no key and are never stored.  The CTA's next
        // item's tile is fetched into L2 meanwhile.
        if (lane == 0) {
            int I = 0;
            for (int i = blockIdx.x; i < num_items; i += gridDim.x) {
                TcItem it;
                if (!tc_next<kPrefix>(p, i, false, it)) continue;
                const int qbuf = I & 1;
                if (!mbar_wait(&q_empty[qbuf], ((I >> 1) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&q_full[qbuf], (uint32_t)TILE);
#pragma unroll
                for (int hh = 0; hh < HALVES; ++hh)
                    tma_load_rows(sq + qbuf * TILE + hh * REG, &tmap_q, &q_full[qbuf], hh * 64,
                                  it.h * g, it.q0 + it.row0 / g);
                for (int i2 = i + gridDim.x; i2 < num_items; i2 += gridDim.x) {
                    TcItem nx;
                    if (!tc_next<kPrefix>(p, i2, false, nx)) continue;
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh)
                        tma_prefetch_rows(&tmap_q, hh * 64, nx.h * g, nx.q0 + nx.row0 / g);
                    break;
                }
                ++I;
            }
            // every copy issued must land before the CTA may exit: the last
            // tile issued into each buffer
            for (int b2 = 0; b2 < 2; ++b2) {
                const int uses = (I - b2 + 1) / 2;
                if (uses > 0) mbar_drain(&q_full[b2], (uses - 1) & 1, p.status);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // --------------------------------------- Q rows of each item (cp.async)
        const T* qb = static_cast<const T*>(p.q);
        constexpr int CH = D / 8;  // 16-byte chunks per row
        int I = 0;
        for (int i = blockIdx.x; i < num_items; i += gridDim.x) {
            TcItem it;
            if (!tc_next<kPrefix>(p, i, false, it)) continue;
            const int qbuf = I & 1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&q_empty[qbuf], ((I >> 1) & 1) ^ 1, abort_flag, p.status)))
                break;
            unsigned char* dstb = sq + qbuf * TILE;
            for (int x = lane; x < kTcRows * CH; x += 32) {
                const int r = x / CH, c = x - r * CH;
                const int R = it.row0 + r, t = R / g;
                const bool live_row = t < it.qlen;
                const T* src = qb + ((size_t)(it.q0 + (live_row ? t : 0)) * Hq + it.h * g +
                                     (R - t * g)) * D + c * 8;
                const uint32_t dst =
                    smem_addr(dstb + (c >> 3) * REG + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                // rows past the chunk are zero-filled (source size 0)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
                             "l"(src), "r"(live_row ? 16 : 0)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;\n" ::: "memory");
            asm volatile("cp.async.wait_all;\n" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full[qbuf]);
            ++I;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t id_s = tc_idesc_f16(kBf16, kTcRows, kTcKeys, 0, 0);
            const uint32_t id_pv = tc_idesc_f16(kBf16, kTcRows, D, 0, 1);
            const uint32_t aq = smem_addr(sq), ak = smem_addr(sk), av = smem_addr(sv);
            // Two cursors over the same sequence of key tiles (items in order,
            // key tiles within each): scores run two tiles ahead of P V.
            struct Cur {
                int i, I, j, J, nkv;  // item index, items seen, key tile in item, global tile
            };
            auto advance = [&](Cur& c) -> bool {  // to the next key tile; false at the end
                if (c.i >= 0 && ++c.j < c.nkv) {
                    ++c.J;
                    return true;
                }
                for (c.i = c.i < 0 ? (int)blockIdx.x : c.i + (int)gridDim.x; c.i < num_items;
                     c.i += gridDim.x) {
                    TcItem it;
                    if (!tc_next<kPrefix>(p, c.i, false, it)) continue;
                    c.nkv = it.nkv;
                    c.j = 0;
                    ++c.I;
                    ++c.J;
                    return true;
                }
                return false;
            };
            // S(J) overwrites score buffer J % 2, which held S(J-2) and then
            // P(J-2): P(J-2) V(J-2) was issued before it by this thread, and
            // one thread's tcgen05.mma run in issue order
            auto issue_s = [&](const Cur& c) -> bool {
                const int b = c.J & 1, ph = (c.J >> 1) & 1, qbuf = c.I & 1;
                if (!mbar_wait(&k_full[b], ph, abort_flag, p.status)) return false;
                if (c.j == 0 && !mbar_wait(&q_full[qbuf], (c.I >> 1) & 1, abort_flag, p.status))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc_mma(tmem + b * kTcKeys,
                           tc_smem_desc(aq + qbuf * TILE + (ks >> 2) * REG + (ks & 3) * 32, 16, 1024),
                           tc_smem_desc(ak + b * TILE + (ks >> 2) * REG + (ks & 3) * 32, 16, 1024),
                           id_s, ks > 0);
                tc_commit(&s_full[b]);
                tc_commit(&k_empty[b]);
                if (c.j == c.nkv - 1) tc_commit(&q_empty[qbuf]);  // the item's last use of Q
                return true;
            };
            // O_q += P_q V_q over key half q of the tile (q = softmax group);
            // P_q sits in tensor memory over the first 32 columns of the
            // group's half of score buffer J % 2
            auto issue_pv = [&](const Cur& c) -> bool {
                const int b = c.J & 1;
                if (!mbar_wait(&v_full[b], (c.J >> 1) & 1, abort_flag, p.status)) return false;
                // the item's first P V overwrites O: the last item's must have been read
                if (c.j == 0 && c.I >= 1 && !mbar_wait(o_free, (c.I - 1) & 1, abort_flag, p.status))
                    return false;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (!mbar_wait(&p_full[q], c.J & 1, abort_flag, p.status)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < HK / 16; ++kk)
                        tc_mma_tmem_a(tmem + kOCol + 128 * q, tmem + b * kTcKeys + HK * q + 8 * kk,
                                      tc_smem_desc(av + b * TILE + (q * (HK / 16) + kk) * 2048, REG,
                                                   1024),
                                      id_pv, c.j > 0 || kk > 0);
                    tc_commit(&pv_done[q]);
                }
                tc_commit(&v_empty[b]);
                if (c.j == c.nkv - 1) tc_commit(o_ready);  // O of the item is complete
                return true;
            };
            Cur cs = {-1, -1, 0, -1, 0}, cp = {-1, -1, 0, -1, 0};
            bool live = true, more_s = advance(cs);
            for (int k = 0; k < 2 && more_s && live; ++k) {
                live = issue_s(cs);
                more_s = advance(cs);
            }
            while (live && advance(cp)) {
                live = issue_pv(cp);
                if (live && more_s) {
                    live = issue_s(cs);
                    more_s = advance(cs);
                }
            }
            // nothing of this thread's may still run when tensor memory is freed
            tc_commit(mma_idle);
            mbar_drain(mma_idle, 0, p.status);
        }
        __syncwarp();
    } else {
        // ------------------------- softmax: two groups of four warps, one thread per
        // (row, key half); each group runs its own online softmax over its half of
        // every key tile into its own O, and the halves merge at the end of an item
        const int q = (warp - 4) >> 2;                       // group: key half
        const int wq = warp & 3;                             // tensor-memory lane quarter
        const int r = 32 * wq + lane;                        // row of the tile
        const uint32_t trow = tmem + ((uint32_t)(32 * wq) << 16);
        const uint32_t ocol = kOCol + 128 * q;
        const float sl2 = p.scale_log2;
        int J = 0, I = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < num_items && ok; i += gridDim.x) {
            TcItem it;
            if (!tc_next<kPrefix>(p, i, false, it)) continue;
            const int R = it.row0 + r, t = R / g;
            const bool live_row = t < it.qlen;
            int pos = live_row ? it.n - it.qlen + t : -1;         // keys 0..pos are visible
            if constexpr (kPrefix) {
                // sequence t sees the prefix up to its own length (an invalid
                // length, flagged by the partition pass, sees nothing)
                int n = live_row ? p.context_lens[t] : 0;
                if (n < 0 || n > p.len_bound) n = 0;
                pos = min(n, p.prefix_tokens) - 1;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nkv; ++j, ++J) {
                const int b = J & 1, ph = (J >> 1) & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], ph, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
                float sc[HK];
#pragma unroll
                for (int c = 0; c < HK / 32; ++c)
                    tc_ld32(trow + b * kTcKeys + HK * q + 32 * c,
                            reinterpret_cast<uint32_t(&)[32]>(sc[32 * c]));
                tc_wait_ld();
                ok = __all_sync(0xffffffffu, mbar_wait(&v_full[b], ph, abort_flag, p.status));
                if (!ok) break;
                const unsigned bad = ((unsigned)vbad[b] >> (4 * q)) & 0xFu;  // this half's blocks
                const int key0 = kTcKeys * j + HK * q;
                // Halves below every row's causal bound with no bad block (most of
                // them) need no mask: max over the raw scores, and the scale goes
                // into the exponent's fma.  Others: select (never scale garbage
                // into use), then the same exponent with a unit multiplier.
                const bool plain = __all_sync(0xffffffffu, key0 + HK - 1 <= pos) && bad == 0u &&
                                   sl2 > 0.f;
                // eight independent partial maxima / sums: no long dependency chain
                float mxp[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mxp[e] = -INFINITY;
                float mul = sl2;
                if (plain) {
#pragma unroll
                    for (int c = 0; c < HK; c += 2)
                        mxp[(c >> 1) & 7] = max3(mxp[(c >> 1) & 7], sc[c], sc[c + 1]);
                } else {
                    mul = 1.f;
#pragma unroll
                    for (int c = 0; c < HK; ++c) {
                        const bool vis = key0 + c <= pos && !((bad >> (c >> 4)) & 1u);
                        sc[c] = vis ? sc[c] * sl2 : -INFINITY;
                        mxp[c & 7] = fmaxf(mxp[c & 7], sc[c]);
                    }
                }
                float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                 fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
                if (plain) mx *= sl2;
                const float m_new = fmaxf(m_used, mx);
                // lazy rescale: only when the maximum grew by more than 2^kTcRescale
                const bool grow = m_used != -INFINITY && m_new > m_used + kTcRescale;
                const float f = grow ? fast_exp2(m_used - m_new) : 1.f;
                if (m_used == -INFINITY || grow) m_used = m_new;
                const float ms = m_used == -INFINITY ? 0.f : m_used;
                // P in registers first: none of this waits on the tensor core
                uint32_t pk[HK / 2];
                const uint64_t mul2 = f2(mul, mul), nms2 = f2(-ms, -ms);
                uint64_t acc2[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < HK / 2; ++c) {
                    float a0, a1;
                    f2_split(f2_fma(f2(sc[2 * c], sc[2 * c + 1]), mul2, nms2), a0, a1);
                    const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
                    acc2[c & 3] = f2_add(acc2[c & 3], f2(p0, p1));
                    pk[c] = E::pack(p0, p1);
                }
                float psp[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_split(acc2[e], psp[2 * e], psp[2 * e + 1]);
                const float psum = ((psp[0] + psp[1]) + (psp[2] + psp[3])) +
                                   ((psp[4] + psp[5]) + (psp[6] + psp[7]));
                // P(J-1) V(J-1) done: O may be rescaled below, and waiting
                // here, before P(J) is released, keeps every wait on pv_done at
                // most one phase behind (after the release P(J) V(J) could
                // complete first and make the parity ambiguous).  It has almost
                // always completed by now.
                if (J >= 1) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&pv_done[q], (J - 1) & 1, abort_flag, p.status));
                    if (!ok) break;
                    tc_fence_after();
                }
                // P over the scores just read (tensor memory, this group's half)
                tc_st32(trow + b * kTcKeys + HK * q, reinterpret_cast<uint32_t(&)[32]>(pk[0]));
                if (__any_sync(0xffffffffu, grow)) {
                    // O_q holds P(J-1) V(J-1): scale it (whole warp: tensor-memory
                    // access is warp-wide)
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tc_ld32(trow + ocol + 32 * c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tc_st32(trow + ocol + 32 * c, o);
                    }
                }
                tc_wait_st();
                l = l * f + psum;
                // V rows of this half no row may see must be finite zeros before
                // P V (0 x NaN = NaN)
                if (j == it.nkv - 1 || bad) {
                    unsigned char* vt = sv + b * TILE;
                    for (int x = r; x < HK * 8 * HALVES; x += 128) {
                        const int kq = x / (8 * HALVES), rest = x - kq * (8 * HALVES);
                        if (key0 + kq <= it.p_last && !((bad >> (kq >> 4)) & 1u)) continue;
                        *reinterpret_cast<uint4*>(vt + (rest >> 3) * REG + (HK * q + kq) * 128 +
                                                  ((rest & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                tc_fence_before();  // P and a rescaled O are ordered before the next MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[q]);
            }
            if (!ok) break;
            // epilogue: group 0 hands its (m, l) to group 1, which stores
            // (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) / (l_0 2^(m_0 - M) + l_1 2^(m_1 - M))
            if (q == 0) {
                if (I >= 1 && !__all_sync(0xffffffffu, mbar_wait(&xfree[wq], (I - 1) & 1,
                                                                 abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                xml[r] = m_used;
                xml[128 + r] = l;
                mbar_arrive(&xchg[wq]);
                ++I;
                continue;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(&xchg[wq], I & 1, abort_flag, p.status));
            if (!ok) break;
            const float m0 = xml[r], l0 = xml[128 + r];
            mbar_arrive(&xfree[wq]);
            const float M = fmaxf(m0, m_used);
            const float Ms = M == -INFINITY ? 0.f : M;
            const float w0 = fast_exp2(m0 - Ms), w1 = fast_exp2(m_used - Ms);
            const float L = l0 * w0 + l * w1;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            ok = __all_sync(0xffffffffu, mbar_wait(o_ready, I & 1, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const size_t orow = (size_t)(it.q0 + (live_row ? t : 0)) * Hq + it.h * g + (R - t * g);
            T* dst = static_cast<T*>(p.out) + orow * D;
            // rows start 2 D (out) or 4 D (ws_o) bytes apart: 32-byte aligned with the base
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
            const bool ws32 = (reinterpret_cast<uintptr_t>(p.ws_o) & 31u) == 0;
            if constexpr (kPrefix) {
                // partials of this row for the cascade's merge: o relative to M
                if (live_row) {
                    p.ws_m[orow] = M;
                    p.ws_l[orow] = L;
                }
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o0[32], o1[32];
                tc_ld32(trow + kOCol + 32 * c, o0);
                tc_ld32(trow + kOCol + 128 + 32 * c, o1);
                tc_wait_ld();
                // rows as 32-byte stores (whole L2 sectors) when the base is
                // 32-byte aligned, else 16-byte ones
                if constexpr (kPrefix) {
                    if (live_row) {
                        float* od = p.ws_o + orow * D + 32 * c;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t w[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                w[u] = __float_as_uint(__uint_as_float(o0[8 * e + u]) * w0 +
                                                       __uint_as_float(o1[8 * e + u]) * w1);
                            if (ws32) {
                                st_global_v8(od + 8 * e, w);
                            } else {
                                *reinterpret_cast<uint4*>(od + 8 * e) = make_uint4(w[0], w[1], w[2], w[3]);
                                *reinterpret_cast<uint4*>(od + 8 * e + 4) =
                                    make_uint4(w[4], w[5], w[6], w[7]);
                            }
                        }
                    }
                } else if (live_row) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        uint32_t w[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            w[u] = E::pack((__uint_as_float(o0[16 * e + 2 * u]) * w0 +
                                            __uint_as_float(o1[16 * e + 2 * u]) * w1) * inv,
                                           (__uint_as_float(o0[16 * e + 2 * u + 1]) * w0 +
                                            __uint_as_float(o1[16 * e + 2 * u + 1]) * w1) * inv);
                        if (out32) {
                            st_global_v8(dst + 32 * c + 16 * e, w);
                        } else {
                            *reinterpret_cast<uint4*>(dst + 32 * c + 16 * e) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4*>(dst + 32 * c + 16 * e + 8) =
                                make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            ++I;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tc_dealloc(tmem, kCols);
    }
}

// ============================================================================
// Chunked prefill on the tensor cores, two query tiles per CTA.
//
// Work item: one sequence, one KV head and a pair of 128-row query tiles A
// and B (256 consecutive (query token, query head) rows); key tiles of 128
// tokens (8 paged blocks), the pair's key range (that of its last live row)
// for both tiles.  A persistent CTA per SM walks the items heaviest first.
//   warp 0   TMA-loads the K blocks of each key tile into a 2-stage ring,
//   warp 3   the V blocks into another (and marks blocks with bad ids),
//   warp 2   owns tensor memory and copies each tile's Q rows (cp.async) as
//            soon as the previous item's last S of that tile is done,
//   warp 1   (one thread) issues, per key tile J, S_A(J), S_B(J) into the
//            tiles' score buffers and O_X += P_X(J) V(J) into their outputs
//            in the order ... P V_A(J), S_A(J+1), P V_B(J), S_B(J+1) ..., so
//            the tensor core works on one tile while the other's softmax runs,
//   warps 4-7 / 8-11: the softmax of tile A / B, one thread per row holding
//            the whole key tile: a first pass over the scores in tensor
//            memory finds the row maximum, a second computes P and writes it
//            as 16-bit values over the scores already read.
// Tensor memory: S_A, S_B (128 columns each), O_A, O_B (D each).  One
// thread issues every MMA and they run in issue order, so S_X(J) completes
// after P V_X(J-1): when the softmax sees S_X(J), O_X holds every earlier
// tile and may be rescaled without another wait.  O is rescaled only when a
// row's running maximum grows by more than 2^8.  V rows no row may see (past
// the pair's bound, in a bad block, never loaded) are zeroed before P V.
// Every wait is bounded.
// ============================================================================
constexpr int kTc2Threads = 384;
constexpr int kTc2Rows = 2 * kTcRows;   // rows per item: tiles A and B
// Registers a thread: the block is launched at kTc2LaunchRegs (the host
// checks the build); the load / MMA warpgroup then gives up registers and the
// two softmax warpgroups take them (setmaxnreg), so that a softmax thread
// holds a whole 128-key row of scores.  The shares add up to the launch total.
constexpr int kTc2LaunchRegs = 168;
constexpr int kTc2OtherRegs = 88;
constexpr int kTc2SoftmaxRegs = 208;
static_assert(128 * kTc2OtherRegs + 256 * kTc2SoftmaxRegs <= kTc2Threads * kTc2LaunchRegs,
              "register shares exceed the launch total");

struct Tc2Item {
    int s, h, q0, qlen, n, row0, p_last, nkv;
};

// Item i of the heaviest-first order (pairs from the end of each chunk);
// false if it holds no rows or its sequence's lengths are invalid (flagged
// once, by the item of pair 0, head 0).
__device__ __forceinline__ bool tc2_item(const PrefillParams& p, int i, bool flag, Tc2Item& it) {
    const int per_pair = p.num_seqs * p.num_kv_heads;
    const int pair = p.tiles_per_seq - 1 - i / per_pair;
    const int rem = i - (i / per_pair) * per_pair;
    it.s = rem / p.num_kv_heads;
    it.h = rem - it.s * p.num_kv_heads;
    it.q0 = p.cu_q_lens[it.s];
    it.qlen = p.cu_q_lens[it.s + 1] - it.q0;
    it.n = p.context_lens[it.s];
    if (!prefill_lengths_ok(p, it.q0, it.qlen, it.n)) {
        if (flag && pair == 0 && it.h == 0 && it.qlen != 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        return false;
    }
    const int g = p.group;
    it.row0 = pair * kTc2Rows;
    if (it.row0 >= it.qlen * g) return false;
    const int tok_last = min(it.qlen, (it.row0 + kTc2Rows + g - 1) / g) - 1;
    it.p_last = it.n - it.qlen + tok_last;
    it.nkv = (it.p_last / PKV_BLOCK_SIZE + 1 + 7) / 8;
    return true;
}

// The item this CTA takes in round r: rounds alternate direction over the
// CTAs (snake order), so that the heaviest-first items even out (Llama-7B-
// shaped 8 x 2048: the busiest CTA 6.5 % above the mean dealt round-robin,
// 0.4 % in snake order).  Past num_items in the last round: no item.
__device__ __forceinline__ int tc2_round_item(int r) {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? G - 1 - c : c);
}

template <typename T, int D>
__global__ void __launch_bounds__(kTc2Threads, 1)
    prefill_tc2_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_q, int q_tma, int num_items) {
    using E = Elem<T>;
    constexpr int HALVES = D / 64;
    constexpr int REG = kTcRows * 128;     // one 64-element half of 128 rows: 16 KB
    constexpr int TILE = HALVES * REG;     // a Q tile, or one K or V key tile
    constexpr uint32_t kCols = 512;
    constexpr uint32_t kOCol = 2 * kTcKeys;  // O_A at kOCol, O_B at kOCol + D
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* sq = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // Q_A, Q_B
    unsigned char* sk = sq + 2 * TILE;      // 2 stages
    unsigned char* sv = sk + 2 * TILE;      // 2 stages
    uint64_t* bars = reinterpret_cast<uint64_t*>(sv + 2 * TILE);
    uint64_t* k_full = bars + 0;            // [stage]
    uint64_t* k_empty = bars + 2;
    uint64_t* v_full = bars + 4;
    uint64_t* v_empty = bars + 6;
    uint64_t* q_full = bars + 8;            // [tile]
    uint64_t* q_empty = bars + 10;
    uint64_t* s_full = bars + 12;           // [tile]: S_X(J) written
    uint64_t* p_full = bars + 14;           // [tile]: its 4 softmax warps wrote P_X(J)
    uint64_t* o_ready = bars + 16;          // [tile]: an item's last P V_X done
    uint64_t* o_free = bars + 18;           // [tile]: its softmax warps read O_X
    uint64_t* mma_idle = bars + 20;
    int* vbad = reinterpret_cast<int*>(bars + 21);           // [2] bad-block bits per V stage
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vbad + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = p.group, Hq = p.num_q_heads;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_ready[i], 1);
            mbar_init(&o_free[i], 4);
        }
        mbar_init(mma_idle, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 2) tc_alloc(tmem_slot, kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // whole warpgroups: warps 0-3 release registers, 4-11 take them
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kTc2OtherRegs));
    if (warp == 0 || warp == 3) {
        // ------------------------------------------------ K (warp 0) / V (warp 3) producers
        const bool isk = warp == 0;
        const CUtensorMap* map = isk ? &tmap_k : &tmap_v;
        uint64_t* full = isk ? k_full : v_full;
        uint64_t* empty = isk ? k_empty : v_empty;
        unsigned char* ring = isk ? sk : sv;
        int J = 0;  // key tiles issued by this CTA
        bool live = true;
        for (int rd = 0; rd * (int)gridDim.x < num_items && live; ++rd) {
            const int i = tc2_round_item(rd);
            Tc2Item it;
            if (i >= num_items || !tc2_item(p, i, isk && lane == 0, it)) continue;
            const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks_per_seq;
            const int nblk = it.p_last / PKV_BLOCK_SIZE + 1;
            for (int j = 0; j < it.nkv; ++j, ++J) {
                const int b = J & 1, ph = (J >> 1) & 1;
                live = __all_sync(0xffffffffu, mbar_wait(&empty[b], ph ^ 1, abort_flag, p.status));
                if (!live) break;
                const int nb = min(8, nblk - 8 * j);
                int id = 0;
                bool bad = false;
                if (lane < nb) {
                    id = table[8 * j + lane];
                    bad = id < 0 || id >= p.num_blocks;
                    if (bad) id = 0;  // fetched, then masked and zeroed
                }
                const unsigned badm = __ballot_sync(0xffffffffu, bad);
                if (lane == 0) {
                    if (isk && badm) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
                    if (!isk) vbad[b] = (int)badm;
                    mbar_arrive_expect_tx(&full[b], (uint32_t)(nb * HALVES * 2048));
                }
                __syncwarp();
                if (lane < nb) {
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh)
                        tma_load_rows(ring + b * TILE + hh * REG + lane * 2048, map, &full[b],
                                      hh * 64, it.h, id * PKV_BLOCK_SIZE);
                }
            }
        }
        // every copy issued must land before the CTA may exit
        if (lane == 0)
            for (int j = max(0, J - 2); j < J; ++j) mbar_drain(&full[j & 1], (j >> 1) & 1, p.status);
    } else if (warp == 2 && q_tma) {
        // ------------------------- Q tiles of each item by tensor copies (lane 0)
        // Tile X of an item is rows row0 + 128 X .. of the chunk: 128 / g
        // tokens x the g query heads of KV head h, one box per 64-element
        // half.  Rows past the chunk belong to the next chunk (or read as
        // zeros past q): their rows see no key and are never stored.  The
        // CTA's next item's tiles are fetched into L2 meanwhile, so that
        // the copy at the item boundary finds them there.
        if (lane == 0) {
            const int g = p.group;
            int I = 0;
            int issued[2] = {0, 0};  // copies issued into Q_X
            for (int rd = 0; rd * (int)gridDim.x < num_items; ++rd) {
                const int i = tc2_round_item(rd);
                Tc2Item it;
                if (i >= num_items || !tc2_item(p, i, false, it)) continue;
                bool live = true;
                for (int X = 0; X < 2 && live; ++X) {
                    live = mbar_wait(&q_empty[X], (I & 1) ^ 1, abort_flag, p.status);
                    if (!live) break;
                    ++issued[X];
                    mbar_arrive_expect_tx(&q_full[X], (uint32_t)TILE);
                    const int row = it.q0 + (it.row0 + X * kTcRows) / g;
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh)
                        tma_load_rows(sq + X * TILE + hh * REG, &tmap_q, &q_full[X], hh * 64,
                                      it.h * g, row);
                }
                if (!live) break;
                for (int r2 = rd + 1; r2 * (int)gridDim.x < num_items; ++r2) {
                    const int i2 = tc2_round_item(r2);
                    Tc2Item nx;
                    if (i2 >= num_items || !tc2_item(p, i2, false, nx)) continue;
#pragma unroll
                    for (int X = 0; X < 2; ++X)
#pragma unroll
                        for (int hh = 0; hh < HALVES; ++hh)
                            tma_prefetch_rows(&tmap_q, hh * 64, nx.h * g,
                                              nx.q0 + (nx.row0 + X * kTcRows) / g);
                    break;
                }
                ++I;
            }
            // every copy issued must land before the CTA may exit
            for (int X = 0; X < 2; ++X)
                if (issued[X] > 0) mbar_drain(&q_full[X], (issued[X] - 1) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------ Q rows of each item's two tiles (cp.async)
        const T* qb = static_cast<const T*>(p.q);
        constexpr int CH = D / 8;  // 16-byte chunks per row
        int I = 0;
        bool live = true;
        for (int rd = 0; rd * (int)gridDim.x < num_items && live; ++rd) {
            const int i = tc2_round_item(rd);
            Tc2Item it;
            if (i >= num_items || !tc2_item(p, i, false, it)) continue;
            for (int X = 0; X < 2 && live; ++X) {
                live = __all_sync(0xffffffffu, mbar_wait(&q_empty[X], (I & 1) ^ 1, abort_flag,
                                                         p.status));
                if (!live) break;
                unsigned char* dstb = sq + X * TILE;
                for (int x = lane; x < kTcRows * CH; x += 32) {
                    const int r = x / CH, c = x - r * CH;
                    const int R = it.row0 + X * kTcRows + r, t = R / g;
                    const bool live_row = t < it.qlen;
                    const T* src = qb + ((size_t)(it.q0 + (live_row ? t : 0)) * Hq + it.h * g +
                                         (live_row ? R - t * g : 0)) * D + c * 8;
                    const uint32_t dst =
                        smem_addr(dstb + (c >> 3) * REG + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                    // rows past the chunk are zero-filled (source size 0)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
                                 "l"(src), "r"(live_row ? 16 : 0)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;\n" ::: "memory");
                asm volatile("cp.async.wait_all;\n" ::: "memory");
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[X]);
            }
            ++I;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t id_s = tc_idesc_f16(kBf16, kTcRows, kTcKeys, 0, 0);
            const uint32_t id_pv = tc_idesc_f16(kBf16, kTcRows, D, 0, 1);
            const uint32_t aq = smem_addr(sq), ak = smem_addr(sk), av = smem_addr(sv);
            // a cursor over the key tiles of this CTA's items, in order
            struct Cur {
                int r, I, j, J, nkv;  // round, items seen, key tile in item, global tile
            };
            auto advance = [&](Cur& c) -> bool {
                if (c.r >= 0 && ++c.j < c.nkv) {
                    ++c.J;
                    return true;
                }
                for (++c.r; c.r * (int)gridDim.x < num_items; ++c.r) {
                    const int i = tc2_round_item(c.r);
                    Tc2Item it;
                    if (i >= num_items || !tc2_item(p, i, false, it)) continue;
                    c.nkv = it.nkv;
                    c.j = 0;
                    ++c.I;
                    ++c.J;
                    return true;
                }
                return false;
            };
            // S_X(c) = Q_X K(c)^T into tile X's score buffer.  S_X(J) overwrites
            // P_X(J-1), whose P V was issued before it by this thread (in order).
            auto issue_s = [&](const Cur& c, int X) -> bool {
                const int b = c.J & 1;
                if (X == 0 && !mbar_wait(&k_full[b], (c.J >> 1) & 1, abort_flag, p.status))
                    return false;
                if (c.j == 0 && !mbar_wait(&q_full[X], c.I & 1, abort_flag, p.status))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc_mma(tmem + X * kTcKeys,
                           tc_smem_desc(aq + X * TILE + (ks >> 2) * REG + (ks & 3) * 32, 16, 1024),
                           tc_smem_desc(ak + b * TILE + (ks >> 2) * REG + (ks & 3) * 32, 16, 1024),
                           id_s, ks > 0);
                tc_commit(&s_full[X]);
                if (X == 1) tc_commit(&k_empty[b]);                 // both tiles read K(J)
                if (c.j == c.nkv - 1) tc_commit(&q_empty[X]);      // the item's last use of Q_X
                return true;
            };
            // O_X += P_X(c) V(c): P_X over the first 64 columns of its score buffer
            auto issue_pv = [&](const Cur& c, int X) -> bool {
                const int b = c.J & 1;
                if (X == 0 && !mbar_wait(&v_full[b], (c.J >> 1) & 1, abort_flag, p.status))
                    return false;
                // the item's first P V overwrites O_X: the last item's must have been read
                if (c.j == 0 && c.I >= 1 &&
                    !mbar_wait(&o_free[X], (c.I - 1) & 1, abort_flag, p.status))
                    return false;
                if (!mbar_wait(&p_full[X], c.J & 1, abort_flag, p.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk)
                    tc_mma_tmem_a(tmem + kOCol + X * D, tmem + X * kTcKeys + 8 * kk,
                                  tc_smem_desc(av + b * TILE + kk * 2048, REG, 1024), id_pv,
                                  c.j > 0 || kk > 0);
                if (X == 1) tc_commit(&v_empty[b]);                 // both tiles read V(J)
                if (c.j == c.nkv - 1) tc_commit(&o_ready[X]);      // O_X of the item complete
                return true;
            };
            Cur cs = {-1, -1, 0, -1, 0}, cp = {-1, -1, 0, -1, 0};
            bool live = true;
            bool more = advance(cs);
            if (more) live = issue_s(cs, 0) && issue_s(cs, 1);
            while (live && advance(cp)) {
                more = advance(cs);
                live = issue_pv(cp, 0);
                if (live && more) live = issue_s(cs, 0);
                if (live) live = issue_pv(cp, 1);
                if (live && more) live = issue_s(cs, 1);
            }
            // nothing of this thread's may still run when tensor memory is freed
            tc_commit(mma_idle);
            mbar_drain(mma_idle, 0, p.status);
        }
        __syncwarp();
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kTc2SoftmaxRegs));
        // ---------------- softmax of tile X (warps 4-7: A, 8-11: B), one thread per row
        const int X = (warp - 4) >> 2;
        const int wq = warp & 3;                             // tensor-memory lane quarter
        const int r = 32 * wq + lane;                        // row of the tile
        const uint32_t trow = tmem + ((uint32_t)(32 * wq) << 16);
        const uint32_t sx = trow + X * kTcKeys;              // this tile's scores / P
        const uint32_t ox = trow + kOCol + X * D;            // this tile's O
        const float sl2 = p.scale_log2;
        // rows start 2 D bytes apart: 32-byte aligned whenever out is
        const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
        int J = 0, I = 0;
        bool ok = true;
        for (int rd = 0; rd * (int)gridDim.x < num_items && ok; ++rd) {
            const int i = tc2_round_item(rd);
            Tc2Item it;
            if (i >= num_items || !tc2_item(p, i, false, it)) continue;
            const int R = it.row0 + X * kTcRows + r, t = R / g;
            const bool live_row = t < it.qlen;
            const int pos = live_row ? it.n - it.qlen + t : -1;   // keys 0..pos are visible
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nkv; ++j, ++J) {
                const int b = J & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], J & 1, abort_flag, p.status));
                if (!ok) break;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&v_full[b], (J >> 1) & 1, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
                const unsigned bad = (unsigned)vbad[b];              // 8 blocks of the tile
                const int key0 = kTcKeys * j;
                // tiles with no bad block keep the raw scores (the scale goes into
                // the exponent); at the causal bound the keys past a row's
                // position read as -inf (a select); tiles below every row's
                // bound need no mask at all
                const bool plain = bad == 0u && sl2 > 0.f;
                const bool whole = __all_sync(0xffffffffu, key0 + kTcKeys - 1 <= pos);
                const float mul = plain ? sl2 : 1.f;
                // scaled score of key key0 + c (masked: -inf); raw for a plain tile
                auto masked = [&](float v, int c) {
                    const bool vis = key0 + c <= pos && !((bad >> (c >> 4)) & 1u);
                    return vis ? v * sl2 : -INFINITY;
                };
                // the whole 128-key row of scores in registers: one round trip
                // to tensor memory per key tile
                float sc[kTcKeys];
#pragma unroll
                for (int q4 = 0; q4 < kTcKeys / 32; ++q4)
                    tc_ld32(sx + 32 * q4, reinterpret_cast<uint32_t(&)[32]>(sc[32 * q4]));
                tc_wait_ld();
                float mxp[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mxp[e] = -INFINITY;
                if (plain) {
                    if (!whole) {
                        const int lim = pos - key0;  // keys 0..lim of the tile are visible
#pragma unroll
                        for (int c = 0; c < kTcKeys; ++c) sc[c] = c <= lim ? sc[c] : -INFINITY;
                    }
#pragma unroll
                    for (int c = 0; c < kTcKeys; c += 2)
                        mxp[(c >> 1) & 7] = max3(mxp[(c >> 1) & 7], sc[c], sc[c + 1]);
                } else {
#pragma unroll
                    for (int c = 0; c < kTcKeys; ++c) {
                        sc[c] = masked(sc[c], c);
                        mxp[c & 7] = fmaxf(mxp[c & 7], sc[c]);
                    }
                }
                float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                 fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
                if (plain) mx *= sl2;
                const float m_new = fmaxf(m_used, mx);
                // lazy rescale: only when the maximum grew by more than 2^kTcRescale
                const bool grow = m_used != -INFINITY && m_new > m_used + kTcRescale;
                const float f = grow ? fast_exp2(m_used - m_new) : 1.f;
                if (m_used == -INFINITY || grow) m_used = m_new;
                const float ms = m_used == -INFINITY ? 0.f : m_used;
                if (__any_sync(0xffffffffu, grow)) {
                    // O_X holds every earlier tile (S_X(J) completed after P V_X(J-1)):
                    // scale it (whole warp: tensor-memory access is warp-wide)
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tc_ld32(ox + 32 * c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tc_st32(ox + 32 * c, o);
                    }
                }
                // P, written as 16-bit pairs over the first 64 columns: P of keys
                // 32c.. lands on columns 16c.. (every score is in registers)
                const uint64_t mul2 = f2(mul, mul), nms2 = f2(-ms, -ms);
                uint64_t acc2[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int c4 = 0; c4 < kTcKeys / 32; ++c4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float a0, a1;
                        f2_split(f2_fma(f2(sc[32 * c4 + 2 * e], sc[32 * c4 + 2 * e + 1]), mul2,
                                        nms2),
                                 a0, a1);
                        const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
                        acc2[e & 3] = f2_add(acc2[e & 3], f2(p0, p1));
                        pk[e] = E::pack(p0, p1);
                    }
                    tc_st16(sx + 16 * c4, pk);
                }
                float psp[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_split(acc2[e], psp[2 * e], psp[2 * e + 1]);
                const float psum = ((psp[0] + psp[1]) + (psp[2] + psp[3])) +
                                   ((psp[4] + psp[5]) + (psp[6] + psp[7]));
                tc_wait_st();
                l = l * f + psum;
                // V rows no row of the pair may see must be finite zeros before
                // P V (0 x NaN = NaN); both tiles zero the same rows
                if (j == it.nkv - 1 || bad) {
                    unsigned char* vt = sv + b * TILE;
                    for (int x = r; x < kTcKeys * 8 * HALVES; x += kTcRows) {
                        const int kq = x / (8 * HALVES), rest = x - kq * (8 * HALVES);
                        if (key0 + kq <= it.p_last && !((bad >> (kq >> 4)) & 1u)) continue;
                        *reinterpret_cast<uint4*>(vt + (rest >> 3) * REG + kq * 128 +
                                                  ((rest & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                tc_fence_before();  // P and a rescaled O are ordered before the next MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[X]);
            }
            if (!ok) break;
            // epilogue: O_X / l for the live rows
            const float inv = l > 0.f ? 1.f / l : 0.f;
            ok = __all_sync(0xffffffffu, mbar_wait(&o_ready[X], I & 1, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            T* dst = static_cast<T*>(p.out) +
                     ((size_t)(it.q0 + (live_row ? t : 0)) * Hq + it.h * g +
                      (live_row ? R - t * g : 0)) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc_ld32(ox + 32 * c, o);
                tc_wait_ld();
                if (live_row) {
                    uint32_t w[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        w[u] = E::pack(__uint_as_float(o[2 * u]) * inv,
                                       __uint_as_float(o[2 * u + 1]) * inv);
                    if (out32) {
                        // 32-byte stores: each fills a whole L2 sector
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t w8[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) w8[u] = w[8 * h + u];
                            st_global_v8(dst + 32 * c + 16 * h, w8);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * e) =
                                make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[X]);
            ++I;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tc_dealloc(tmem, kCols);
    }
}

template <int D>
size_t prefill_tc_smem() {
    // 2 Q buffers, 2 K and 2 V stages, barriers and the (m, l) hand-over
    // (under 2 KB); 1 KB alignment slack
    return 1024 + (size_t)6 * (D / 64) * kTcRows * 128 + 2048;
}

// Which prefill kernel runs: the tcgen05 kernel with two query tiles per CTA,
// unless PKV_PREFILL_KERNEL selects one kept for comparison: =tc1 the
// tcgen05 kernel with one query tile and two softmax groups per key tile
// (also the cascade's prefix pass), =mma the mma.sync kernel.  Returns 1
// for two tiles, 2 for one tile, 0 for mma.sync.
int prefill_kernel_choice() {
    static const int k = [] {
        const char* v = std::getenv("PKV_PREFILL_KERNEL");
        if (v && std::strcmp(v, "mma") == 0) return 0;
        if (v && std::strcmp(v, "tc1") == 0) return 2;
        return 1;
    }();
    return k;
}

template <typename T, int D>
pkv_status launch_prefill(const PrefillParams& prm_in, const void* k_cache, const void* v_cache,
                          int num_blocks, int num_kv_heads, int max_q_len, pkv_dtype dtype,
                          cudaStream_t stream) {
    CUtensorMap tmk, tmv;
    if (!make_pool_map(&tmk, k_cache, num_blocks, num_kv_heads, D, dtype) ||
        !make_pool_map(&tmv, v_cache, num_blocks, num_kv_heads, D, dtype))
        return PKV_ERR_CUDA;
    PrefillParams prm = prm_in;
    int choice = prefill_kernel_choice();
    // the two-tile kernel's register shares assume its launch count; any other
    // build takes the one-tile kernel
    static const bool tc2_regs_ok = [] {
        cudaFuncAttributes a;
        return cudaFuncGetAttributes(&a, prefill_tc2_kernel<T, D>) == cudaSuccess &&
               a.numRegs == kTc2LaunchRegs;
    }();
    if (choice == 1 && !tc2_regs_ok) choice = 2;
    if (choice == 1) {
        prm.tiles_per_seq = ceil_div(max_q_len * prm.group, kTc2Rows);  // pairs of tiles
        auto kern = prefill_tc2_kernel<T, D>;
        const size_t smem = prefill_tc_smem<D>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        const long long items = (long long)prm.num_seqs * num_kv_heads * prm.tiles_per_seq;
        if (items > 0x7fffffffll) return PKV_ERR_UNSUPPORTED;
        const int sms = sm_count();
        if (sms <= 0) return PKV_ERR_CUDA;
        const int grid = (int)std::min<long long>(items, sms);  // persistent: one CTA per SM
        // Q tiles by tensor copies when the group divides the tile's 128 rows
        CUtensorMap tmq = tmk;
        const int q_tma =
            make_q_tile_map(&tmq, prm.q, prm.num_q_rows, prm.num_q_heads, D, prm.group, dtype)
                ? 1
                : 0;
        if (!q_tma) tmq = tmk;  // unused
        kern<<<grid, kTc2Threads, smem, stream>>>(prm, tmk, tmv, tmq, q_tma, (int)items);
        return cuda_status(cudaGetLastError());
    }
    if (choice == 2) {
        prm.tiles_per_seq = ceil_div(max_q_len * prm.group, kTcRows);
        auto kern = prefill_tc_kernel<T, D, false>;
        const size_t smem = prefill_tc_smem<D>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        const long long items = (long long)prm.num_seqs * num_kv_heads * prm.tiles_per_seq;
        if (items > 0x7fffffffll) return PKV_ERR_UNSUPPORTED;
        const int sms = sm_count();
        if (sms <= 0) return PKV_ERR_CUDA;
        const int grid = (int)std::min<long long>(items, sms);  // persistent: one CTA per SM
        CUtensorMap tmq = tmk;
        const int q_tma =
            make_q_tile_map(&tmq, prm.q, prm.num_q_rows, prm.num_q_heads, D, prm.group, dtype)
                ? 1
                : 0;
        if (!q_tma) tmq = tmk;  // unused
        kern<<<grid, kTcThreads, smem, stream>>>(prm, tmk, tmv, tmq, q_tma, (int)items);
        return cuda_status(cudaGetLastError());
    }
    prm.tiles_per_seq = ceil_div(max_q_len * prm.group, kPrefillRows);
    auto kern = prefill_tma_kernel<T, D>;
    const size_t smem = 1024 + (size_t)kPrefillStages * (2 * 16 * D * 2) + kPrefillStages * 20 + 16;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    const long long grid = (long long)prm.num_seqs * num_kv_heads * prm.tiles_per_seq;
    if (grid > 0x7fffffffll) return PKV_ERR_UNSUPPORTED;
    kern<<<(unsigned)grid, kPrefillThreads, smem, stream>>>(prm, tmk, tmv);
    return cuda_status(cudaGetLastError());
}

template <typename T, int D>
pkv_status launch_prefix_tc(const PrefillParams& prm, const void* k_cache, const void* v_cache,
                            int num_items, int grid, pkv_dtype dtype, cudaStream_t stream) {
    CUtensorMap tmk, tmv;
    if (!make_pool_map(&tmk, k_cache, prm.num_blocks, prm.num_kv_heads, D, dtype) ||
        !make_pool_map(&tmv, v_cache, prm.num_blocks, prm.num_kv_heads, D, dtype))
        return PKV_ERR_CUDA;
    auto kern = prefill_tc_kernel<T, D, true>;
    const size_t smem = prefill_tc_smem<D>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    // decode queries [num_seqs][Hq][D]: row t of a KV head's rows is sequence t / g
    CUtensorMap tmq = tmk;
    const int q_tma =
        make_q_tile_map(&tmq, prm.q, prm.num_seqs, prm.num_q_heads, D, prm.group, dtype) ? 1 : 0;
    if (!q_tma) tmq = tmk;  // unused
    kern<<<grid, kTcThreads, smem, stream>>>(prm, tmk, tmv, tmq, q_tma, num_items);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int cascade_prefix_grid(int num_seqs, int num_q_heads, int num_kv_heads, int max_ctas) {
    // one CTA per (KV head, row tile of the sharers' query rows), at most max_ctas
    const long long items =
        (long long)num_kv_heads * ceil_div(num_seqs * (num_q_heads / num_kv_heads), kTcRows);
    return (int)std::max<long long>(1, std::min<long long>(items, max_ctas));
}

pkv_status launch_cascade_prefix(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int len_bound, int num_seqs,
                                 int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                 int prefix_blocks, float scale_log2, float* ws_m, float* ws_l,
                                 float* ws_o, pkv_dtype dtype, int max_ctas, int* grid_out,
                                 cudaStream_t stream) {
    unsigned int* status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int g = num_q_heads / num_kv_heads;
    const long long items = (long long)num_kv_heads * ceil_div(num_seqs * g, kTcRows);
    const int grid = cascade_prefix_grid(num_seqs, num_q_heads, num_kv_heads, max_ctas);
    *grid_out = grid;
    PrefillParams prm = {};
    prm.q = q;
    prm.out = nullptr;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.cu_q_lens = nullptr;
    prm.status = status;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = g;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.scale_log2 = scale_log2;
    prm.prefix_tokens = prefix_blocks * PKV_BLOCK_SIZE;
    prm.len_bound = len_bound;
    prm.ws_m = ws_m;
    prm.ws_l = ws_l;
    prm.ws_o = ws_o;
    if (dtype == PKV_BF16)
        return head_dim == 128 ? launch_prefix_tc<__nv_bfloat16, 128>(prm, k_cache, v_cache,
                                                                     (int)items, grid, dtype,
                                                                     stream)
                               : launch_prefix_tc<__nv_bfloat16, 64>(prm, k_cache, v_cache,
                                                                    (int)items, grid, dtype,
                                                                    stream);
    return head_dim == 128
               ? launch_prefix_tc<__half, 128>(prm, k_cache, v_cache, (int)items, grid, dtype,
                                               stream)
               : launch_prefix_tc<__half, 64>(prm, k_cache, v_cache, (int)items, grid, dtype,
                                              stream);
}

}  // namespace pkv

extern "C" {

pkv_status paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* cu_q_lens,
                                   int num_seqs, int max_q_len, int num_q_rows, int num_q_heads,
                                   int num_kv_heads, int head_dim, int num_blocks, float scale,
                                   void* out, pkv_dtype dtype, pkv_stream_t stream) {
    if (num_seqs < 0 || max_q_len < 0 || num_q_rows < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    const int g = num_q_heads / num_kv_heads;
    if (g > 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_q_len == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !cu_q_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) ||
        !pkv::aligned16(out))
        return PKV_ERR_INVALID_ARG;
    unsigned int* status = pkv::status_word();
    if (!status) return PKV_ERR_CUDA;
    pkv::PrefillParams prm;
    prm.q = q;
    prm.out = out;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.cu_q_lens = cu_q_lens;
    prm.status = status;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = g;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.max_q_len = max_q_len;
    prm.num_q_rows = num_q_rows;
    prm.tiles_per_seq = 0;  // set by the launcher for the kernel it picks
    prm.scale_log2 = scale * pkv::kLog2e;
    prm.prefix_tokens = 0;  // prefill, not the cascade's prefix pass
    prm.len_bound = 0;
    prm.ws_m = prm.ws_l = prm.ws_o = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == PKV_BF16)
        return head_dim == 128
                   ? pkv::launch_prefill<__nv_bfloat16, 128>(prm, k_cache, v_cache, num_blocks,
                                                            num_kv_heads, max_q_len, dtype, st)
                   : pkv::launch_prefill<__nv_bfloat16, 64>(prm, k_cache, v_cache, num_blocks,
                                                           num_kv_heads, max_q_len, dtype, st);
    return head_dim == 128 ? pkv::launch_prefill<__half, 128>(prm, k_cache, v_cache, num_blocks,
                                                              num_kv_heads, max_q_len, dtype, st)
                           : pkv::launch_prefill<__half, 64>(prm, k_cache, v_cache, num_blocks,
                                                             num_kv_heads, max_q_len, dtype, st);
}

}  // extern "C"
