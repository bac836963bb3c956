// pa_decode_noalloc.cu - pa_decode for callers that cannot allocate device memory.
//
// pa_decode asks its caller for a workspace.  Some callers cannot provide one:
// a serving engine that has already reserved nearly all of HBM for its KV-cache
// pool and admits no further allocations, a host program that only receives
// device pointers from another runtime and owns no allocator, or a per-token
// decode loop that cannot afford cudaMalloc/cudaFree (both may synchronise the
// device).  This entry point runs the same decode with a fixed scratch area
// that lives in this library's own device image instead.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.  Every
// GPU that loads the library holds it until the process exits.  Host code only
// sees a host-side stand-in for the array's name, so its device address is
// looked up once per device (with that device current) by cudaGetSymbolAddress
// and cached.  Every call on a device shares the array.
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
pa_status scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_decode_noalloc(void *out, const void *q, const void *kv_cache, int num_blocks,
                            int block_size, int num_heads, int num_kv_heads, int head_size,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                            pa_stream_t stream) {
    if (num_seqs > 0 && num_heads > 0 && num_kv_heads > 0 && head_size > 0 &&
        pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size) >
            kNoAllocScratchBytes)
        return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (num_seqs > 0) {
        pa_status st = scratch_on_current_device(&scratch);
        if (st != PA_OK) return st;
    }
    return pa_decode(out, q, kv_cache, num_blocks, block_size, num_heads, num_kv_heads,
                     head_size, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     max_seq_len, scale, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
