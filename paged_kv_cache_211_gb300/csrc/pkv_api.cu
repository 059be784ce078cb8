// pkv_api.cu -- library-wide entry points: version, status text, pool sizing,
// the device status word, and the host-buffer decode step.
#include <algorithm>
#include <mutex>

#include "pkv_internal.cuh"
#include "pkv_tma.cuh"

namespace {

// Sticky flags set by kernels that met a bad device-side value (see the
// PKV_DEV_* bits in pagedkv.h).  One word per device (module memory).
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace pkv {

unsigned int* status_word() {
    int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_status_ptr[dev];
}

int sm_count() {
    int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace pkv

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape";
        case PKV_ERR_NO_BLOCKS: return "not enough free blocks";
        case PKV_ERR_BAD_BLOCK_ID: return "bad block id";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t pkv_cache_bytes(int num_layers, int num_blocks, int block_size, int num_kv_heads,
                       int head_dim, pkv_dtype dtype) {
    if (num_layers <= 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    if (block_size != PKV_BLOCK_SIZE) return 0;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return 0;
    return (size_t)num_layers * (size_t)num_blocks * (size_t)block_size *
           (size_t)num_kv_heads * (size_t)head_dim * 2u;
}

pkv_status pkv_device_status(unsigned int* flags, int reset) {
    if (!flags) return PKV_ERR_INVALID_ARG;
    unsigned int* p = pkv::status_word();
    if (!p) return PKV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemcpy(flags, p, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (reset && cudaMemset(p, 0, sizeof(unsigned int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (reset && cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

pkv_status paged_kv_last_error(pkv_stream_t stream) {
    unsigned int* p = pkv::status_word();
    if (!p) return PKV_ERR_CUDA;
    unsigned int flags = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemcpyAsync(&flags, p, sizeof(unsigned int), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemsetAsync(p, 0, sizeof(unsigned int), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (flags & PKV_DEV_TIMEOUT) return PKV_ERR_CUDA;
    if (flags & PKV_DEV_BAD_BLOCK_ID) return PKV_ERR_BAD_BLOCK_ID;
    if (flags & (PKV_DEV_BAD_LENGTH | PKV_DEV_BAD_SLOT)) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

size_t paged_kv_decode_step_staging_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int max_blocks_per_seq) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    const size_t B = (size_t)num_seqs;
    size_t total = 0;
    total += align_up(B * num_q_heads * head_dim * 2, 256);          // q
    total += 2 * align_up(B * num_kv_heads * head_dim * 2, 256);     // k_new, v_new
    total += align_up(B * (size_t)max_blocks_per_seq * 4, 256);      // block_tables
    total += align_up(B * 4, 256);                                   // context_lens
    total += align_up(B * num_q_heads * head_dim * 2, 256);          // out
    return total;
}

namespace {

// Up to five host-to-device copies done by one kernel that reads page-locked
// host memory through its device mapping: one launch instead of one copy
// engine transfer per input (each of which costs a few microseconds of set-up
// at these sizes).
struct StageJobs {
    const void* src[5];
    void* dst[5];
    size_t bytes[5];
    int n;
};

__global__ void __launch_bounds__(256) stage_inputs_kernel(const StageJobs jobs) {
    // launched as a programmatic dependent: the previous kernel on the stream
    // may still run (and may still read the staging buffers or write the
    // host inputs); wait for it before touching either
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int j = 0; j < jobs.n; ++j) {
        const size_t bytes = jobs.bytes[j];
        const bool vec = ((reinterpret_cast<uintptr_t>(jobs.src[j]) |
                           reinterpret_cast<uintptr_t>(jobs.dst[j])) & 15u) == 0;
        size_t done = 0;
        if (vec) {
            const uint4* s = static_cast<const uint4*>(jobs.src[j]);
            uint4* d = static_cast<uint4*>(jobs.dst[j]);
            const size_t n16 = bytes / 16;
            for (size_t i = t0; i < n16; i += stride) d[i] = s[i];
            done = n16 * 16;
        }
        // the rest in 4-byte words (every size here is a multiple of 4)
        const uint32_t* s4 = static_cast<const uint32_t*>(jobs.src[j]);
        uint32_t* d4 = static_cast<uint32_t*>(jobs.dst[j]);
        for (size_t i = done / 4 + t0; i < bytes / 4; i += stride) d4[i] = s4[i];
    }
}

// One warp waits on an mbarrier that nothing arrives on, with the bounded wait
// every kernel of the library uses (here limited to `limit` cycles): it must
// give up, set PKV_DEV_TIMEOUT and return.
__global__ void bounded_wait_selftest_kernel(unsigned int* status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        pkv::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncwarp();
    pkv::mbar_wait(&bar, 0, &abort_flag, status, limit);
}

// The device address of page-locked host memory, or null if the pointer has
// none (not page-locked, or not mapped into the device's address space).
const void* mapped_host(const void* host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        (void)cudaGetLastError();  // clear the error a plain pointer may leave
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
    return a.devicePointer;
}

}  // namespace

pkv_status pkv_selftest_bounded_wait(pkv_stream_t stream) {
    unsigned int* status = pkv::status_word();
    if (!status) return PKV_ERR_CUDA;
    // ~0.1 s at the GB300's 2 GHz SM clock
    bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        status, 200000000ll);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status paged_kv_decode_step_host(const void* q_host, const void* k_new_host,
                                     const void* v_new_host, const int32_t* block_tables_host,
                                     const int32_t* context_lens_host, void* out_host,
                                     void* staging, size_t staging_bytes, void* k_cache,
                                     void* v_cache, int max_blocks_per_seq, int max_context_len,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int num_blocks, float scale, void* workspace,
                                     size_t workspace_bytes, pkv_dtype dtype,
                                     pkv_stream_t stream) {
    if (!q_host || !k_new_host || !v_new_host || !block_tables_host || !context_lens_host ||
        !out_host || !staging)
        return PKV_ERR_INVALID_ARG;
    const size_t need = paged_kv_decode_step_staging_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                           head_dim, max_blocks_per_seq);
    if (need == 0) return PKV_ERR_INVALID_ARG;
    if (staging_bytes < need || (reinterpret_cast<uintptr_t>(staging) & 255u))
        return PKV_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t B = (size_t)num_seqs;
    const size_t q_bytes = B * num_q_heads * head_dim * 2;
    const size_t kv_bytes = B * num_kv_heads * head_dim * 2;
    const size_t bt_bytes = B * (size_t)max_blocks_per_seq * 4;
    char* p = static_cast<char*>(staging);
    void* q_d = p;                p += align_up(q_bytes, 256);
    void* kn_d = p;               p += align_up(kv_bytes, 256);
    void* vn_d = p;               p += align_up(kv_bytes, 256);
    int32_t* bt_d = reinterpret_cast<int32_t*>(p);  p += align_up(bt_bytes, 256);
    int32_t* cl_d = reinterpret_cast<int32_t*>(p);  p += align_up(B * 4, 256);
    void* out_d = p;
    // inputs with a device mapping are staged by one kernel, the others by
    // one cudaMemcpyAsync each
    const void* srcs[5] = {q_host, k_new_host, v_new_host, block_tables_host, context_lens_host};
    void* dsts[5] = {q_d, kn_d, vn_d, bt_d, cl_d};
    const size_t sizes[5] = {q_bytes, kv_bytes, kv_bytes, bt_bytes, B * 4};
    StageJobs jobs;
    jobs.n = 0;
    for (int i = 0; i < 5; ++i) {
        const void* mapped = mapped_host(srcs[i]);
        if (mapped && (reinterpret_cast<uintptr_t>(mapped) & 3u) == 0) {
            jobs.src[jobs.n] = mapped;
            jobs.dst[jobs.n] = dsts[i];
            jobs.bytes[jobs.n] = sizes[i];
            ++jobs.n;
        } else if (cudaMemcpyAsync(dsts[i], srcs[i], sizes[i], cudaMemcpyHostToDevice, st) !=
                   cudaSuccess) {
            return PKV_ERR_CUDA;
        }
    }
    if (jobs.n > 0) {
        size_t total = 0;
        for (int i = 0; i < jobs.n; ++i) total += jobs.bytes[i];
        const int blocks = (int)std::min<size_t>(128, (total / 16 + 255) / 256 + 1);
        // programmatic dependent launch: the grid is scheduled while the
        // previous kernel drains and waits for it (griddepcontrol.wait) before
        // it reads or writes anything; it never lets its own dependents start
        // early, and the partition pass after it waits for it as well
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, stage_inputs_kernel, jobs) != cudaSuccess) return PKV_ERR_CUDA;
    }
    // the kernels only store to `out`: with a device mapping of out_host they
    // write the result there directly, else into staging and one copy back
    void* out_mapped = const_cast<void*>(mapped_host(out_host));
    const bool direct = out_mapped && (reinterpret_cast<uintptr_t>(out_mapped) & 15u) == 0;
    pkv_status rc = paged_kv_decode_step(q_d, kn_d, vn_d, k_cache, v_cache, bt_d,
                                         max_blocks_per_seq, cl_d, max_context_len, num_seqs,
                                         num_q_heads, num_kv_heads, head_dim, num_blocks, scale,
                                         direct ? out_mapped : out_d, nullptr, workspace,
                                         workspace_bytes, dtype, stream);
    if (rc != PKV_OK) return rc;
    if (!direct &&
        cudaMemcpyAsync(out_host, out_d, q_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // extern "C"
