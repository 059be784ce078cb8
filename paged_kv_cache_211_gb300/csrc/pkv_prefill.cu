// pkv_prefill.cu -- chunked-prefill attention over the paged cache.
#include <cmath>

#include "pkv_internal.cuh"
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
    int tiles_per_seq;  // ceil(max_q_len * group / kPrefillRows)
    float scale_log2;
};

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
    if (qlen <= 0 || n < qlen || n > p.max_blocks_per_seq * PKV_BLOCK_SIZE) {
        if (tid == 0 && tile == 0 && h == 0 && (qlen < 0 || n < qlen ||
                                                 n > p.max_blocks_per_seq * PKV_BLOCK_SIZE))
            atomicOr(p.status, PKV_DEV_BAD_LENGTH);
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

template <typename T, int D>
pkv_status launch_prefill(const PrefillParams& prm, const void* k_cache, const void* v_cache,
                          int num_blocks, int num_kv_heads, pkv_dtype dtype, cudaStream_t stream) {
    CUtensorMap tmk, tmv;
    if (!make_pool_map(&tmk, k_cache, num_blocks, num_kv_heads, D, dtype) ||
        !make_pool_map(&tmv, v_cache, num_blocks, num_kv_heads, D, dtype))
        return PKV_ERR_CUDA;
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

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* cu_q_lens,
                                   int num_seqs, int max_q_len, int num_q_heads,
                                   int num_kv_heads, int head_dim, int num_blocks, float scale,
                                   void* out, pkv_dtype dtype, pkv_stream_t stream) {
    if (num_seqs < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
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
    prm.tiles_per_seq = pkv::ceil_div(max_q_len * g, pkv::kPrefillRows);
    prm.scale_log2 = scale * pkv::kLog2e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == PKV_BF16)
        return head_dim == 128
                   ? pkv::launch_prefill<__nv_bfloat16, 128>(prm, k_cache, v_cache, num_blocks,
                                                            num_kv_heads, dtype, st)
                   : pkv::launch_prefill<__nv_bfloat16, 64>(prm, k_cache, v_cache, num_blocks,
                                                           num_kv_heads, dtype, st);
    return head_dim == 128 ? pkv::launch_prefill<__half, 128>(prm, k_cache, v_cache, num_blocks,
                                                              num_kv_heads, dtype, st)
                           : pkv::launch_prefill<__half, 64>(prm, k_cache, v_cache, num_blocks,
                                                             num_kv_heads, dtype, st);
}

}  // extern "C"
