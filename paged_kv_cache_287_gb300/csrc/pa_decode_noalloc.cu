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
// looked up by cudaGetSymbolAddress with the device current, and cached per CUDA
// context (by the context's unique id): a context created later on the same
// device (after cudaDeviceReset, or one made through the driver API and made
// current) gets its own lookup, so no call uses an address of a context that is
// gone.  Every call within one context shares the array.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxContexts = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
struct Entry {
    unsigned long long ctx_id;
    void *ptr;
};
Entry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long *);

template <typename F>
F driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

// Unique id of the context current on this thread (0 if there is none or it
// cannot be read).
unsigned long long current_context_id() {
    static CtxGetCurrent get_current = driver_fn<CtxGetCurrent>("cuCtxGetCurrent");
    static CtxGetId get_id = driver_fn<CtxGetId>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current context.
pa_status scratch_in_current_context(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (id != 0)
        for (int i = 0; i < g_scratch_n; ++i)
            if (g_scratch[i].ctx_id == id) {
                *out = g_scratch[i].ptr;
                return PA_OK;
            }
    // Not seen yet (or no context bound yet: the lookup binds the device's primary
    // context, whose id is read again afterwards).
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    if (id == 0) id = current_context_id();
    if (id != 0 && g_scratch_n < kMaxContexts) g_scratch[g_scratch_n++] = Entry{id, p};
    *out = p;
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
        pa_status st = scratch_in_current_context(&scratch);
        if (st != PA_OK) return st;
    }
    return pa_decode(out, q, kv_cache, num_blocks, block_size, num_heads, num_kv_heads,
                     head_size, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     max_seq_len, scale, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
