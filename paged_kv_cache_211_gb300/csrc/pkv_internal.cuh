// pkv_internal.cuh -- shared internals of libpagedkv (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pagedkv.h"

namespace pkv {

// Device address of the status word on the current device (set-up once per
// device, see pkv_api.cu).  Returns nullptr if CUDA fails.
unsigned int* status_word();

// Multiprocessor count of the current device (cached per device).
int sm_count();

inline pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// The cascade's prefix pass on the tensor cores (pkv_prefill.cu): every
// sequence's decode query against the first prefix_blocks blocks of
// block-table row 0, shared by all sequences; writes the unnormalised
// partials (m, l, o, base-2 scores) of query head i of sequence s to
// workspace row s * num_q_heads + i.  A persistent grid of at most max_ctas
// CTAs (its size goes to *grid_out); an ordinary launch that lets the next
// kernel on the stream start beside it.
// CTAs of a cascade's prefix pass for these shapes, at most max_ctas.
int cascade_prefix_grid(int num_seqs, int num_q_heads, int num_kv_heads, int max_ctas);
pkv_status launch_cascade_prefix(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int len_bound, int num_seqs,
                                 int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                 int prefix_blocks, float scale_log2, float* ws_m, float* ws_l,
                                 float* ws_o, pkv_dtype dtype, int max_ctas, int* grid_out,
                                 cudaStream_t stream);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// 16-bit element types and their warp-level tensor-core contraction
// (mma.sync m16n8k16, fp32 accumulate; A row-major 16x16, B column-major 16x8).
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // two fp32 -> packed pair, round to nearest even; `lo` in bits 0..15
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

template <>
struct Elem<__half> {
    static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

// Transpose of an 8x8 matrix of 16-bit values held one row per lane quad.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// 2^x with the hardware approximation (ex2.approx; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte read-only streaming load: K/V rows are touched once per call, so
// they bypass L1.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

}  // namespace pkv
