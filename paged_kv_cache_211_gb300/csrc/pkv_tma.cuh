// pkv_tma.cuh -- TMA, mbarrier and ldmatrix primitives (inline PTX) and the
// tensor map of a paged pool, shared by the decode and prefill kernels.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)

#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

// How long a kernel waits on an mbarrier before it gives up (~2 s at 2 GHz).
constexpr long long kWaitCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of the same phase (never suspends the thread): for a
// warp whose lanes poll different barriers.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with parity `parity`.  Returns false without
// waiting once *abort is set, and sets *abort and the status bit when the
// wait exceeds `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status, long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!*abort) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) {
            *abort = 1;
            atomicOr(status, PKV_DEV_TIMEOUT);
            return false;
        }
    }
    return false;
}

// A bounded wait that ignores the abort flag (used to let issued copies land).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, unsigned int* status) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(status, PKV_DEV_TIMEOUT);
            return;
        }
    }
}

// 16 rows x 64 elements of one KV head: tensor coordinates (element x, head, row).
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int x, int head, int row) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(head), "r"(row)
        : "memory");
}

// Fetch the same box into L2 only (no shared memory, no barrier): a later
// tma_load_rows of it then finds the rows in L2.
__device__ __forceinline__ void tma_prefetch_rows(const CUtensorMap* map, int x, int head, int row) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(head), "r"(row)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// Byte offset of 16-byte chunk c (of D/8) of row `row` in a swizzled tile of
// 64-element boxes: box c/8 (2 KB each), 128-byte row, chunk (c%8) ^ (row%8).
__device__ __forceinline__ uint32_t swz(int row, int c) {
    return (uint32_t)((c >> 3) * 2048 + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}


// ---------------------------------------------------------------------------
// Host side: the tensor map of one layer's pool.
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, fetched through the runtime (no link against the
// driver library).  nullptr if unavailable.
inline EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// A pool [NB][16][Hkv][D] viewed as (element, head, row) with boxes of
// 64 elements x 1 head x 16 rows and the 128-byte swizzle.
inline bool make_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads,
                   int head_dim, pkv_dtype dtype) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads,
                                (cuuint64_t)num_blocks * PKV_BLOCK_SIZE};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2,
                                   (cuuint64_t)num_kv_heads * head_dim * 2};
    const cuuint32_t box[3] = {64, 1, PKV_BLOCK_SIZE};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, 3, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Query rows [num_rows][num_q_heads][D] viewed as (element, head, row) with
// boxes of 64 elements x `group` heads x (128 / group) rows and the 128-byte
// swizzle: one box is one 64-element half of a 128-row tile whose row r is
// (row r / group, head r % group), the layout the tensor-core kernels read.
// Rows past num_rows read as zeros.  Needs group to divide 128.
inline bool make_q_tile_map(CUtensorMap* map, const void* q, int num_rows, int num_q_heads,
                            int head_dim, int group, pkv_dtype dtype) {
    if (group <= 0 || 128 % group != 0 || num_rows <= 0) return false;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads,
                                (cuuint64_t)num_rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2,
                                   (cuuint64_t)num_q_heads * head_dim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, 3, const_cast<void*>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace pkv
