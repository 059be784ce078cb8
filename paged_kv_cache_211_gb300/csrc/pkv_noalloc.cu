// pkv_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// paged_attention_decode needs a caller-provided workspace for the partials
// of its split-context pass.  Some callers have no way to provide one:
//  - a plug-in or custom operator living inside a host framework that owns
//    all device memory and hands the library nothing but the tensors of the
//    call;
//  - a runtime that fixes its whole memory plan at start-up and forbids
//    allocation on the serving path, because cudaMalloc synchronises the
//    device (a stall in a latency-critical decode loop) and can fail late,
//    in the middle of a request, when memory is fragmented or full.
// For them this entry point uses scratch memory that lives in the library
// itself: a file-scope device array of a fixed size, reserved when the
// library's device code is loaded on a GPU and held until the process exits.
// It allocates nothing per call.
#include <mutex>

#include "pkv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Host code must not use this name as a device
// address: on the host it denotes a stand-in object, not GPU memory.  The
// device address is looked up with cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device.  Looked up once per
// device, with that device current; nullptr if CUDA reports an error.
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

size_t paged_attention_noalloc_scratch_bytes(void) { return kScratchBytes; }

pkv_status paged_attention_decode_noalloc(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int max_context_len, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int num_blocks,
                                          float scale, void* out, pkv_dtype dtype,
                                          pkv_stream_t stream) {
    const size_t need =
        paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len);
    if (need > kScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the static scratch
    void* scratch = scratch_address();
    if (!scratch) return PKV_ERR_CUDA;
    return paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, max_context_len, num_seqs, num_q_heads,
                                  num_kv_heads, head_dim, num_blocks, scale, out, scratch,
                                  kScratchBytes, dtype, stream);
}

}  // extern "C"
