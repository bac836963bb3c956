// pa_api.cu - the C ABI declared in include/pa.h: host-side argument checks,
// launch configuration and the device error word.  Allocates nothing.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

int device_sm_count() {
    static std::atomic<int> known[64];  // per device; 0 until read
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && (sms = known[dev].load(std::memory_order_relaxed)) > 0) return sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    if (sms <= 0) return 1;
    if (dev >= 0 && dev < 64) known[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

namespace {

// Encoded maps of recent pools: the map is a pure function of the key.
struct MapEntry {
    const void *pool;
    KvGeom g;
    int box_rows, fp8;
    CUtensorMap map;
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_maps_n = 0, g_maps_next = 0;

bool same(const MapEntry &e, const void *pool, const KvGeom &g, int box_rows, int fp8) {
    return e.pool == pool && e.g.num_blocks == g.num_blocks && e.g.block_size == g.block_size &&
           e.g.num_kv_heads == g.num_kv_heads && e.g.head_size == g.head_size &&
           e.box_rows == box_rows && e.fp8 == fp8;
}

bool cached_map(CUtensorMap *map, const void *pool, const KvGeom &g, int box_rows, int fp8) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_maps_n; ++i)
        if (same(g_maps[i], pool, g, box_rows, fp8)) {
            *map = g_maps[i].map;
            return true;
        }
    return false;
}

void keep_map(const CUtensorMap &map, const void *pool, const KvGeom &g, int box_rows, int fp8) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry &e = g_maps[g_maps_next];
    e.pool = pool;
    e.g = g;
    e.box_rows = box_rows;
    e.fp8 = fp8;
    e.map = map;
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_n < kMapCache) ++g_maps_n;
}

}  // namespace

bool encode_kv_map(CUtensorMap *map, const void *kv_cache, const KvGeom &g, int box_rows) {
    if (cached_map(map, kv_cache, g, box_rows, 0)) return true;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t rows =
        (cuuint64_t)g.num_blocks * 2u * (cuuint64_t)g.num_kv_heads * (cuuint64_t)g.block_size;
    cuuint64_t dims[2] = {(cuuint64_t)g.head_size, rows};
    cuuint64_t strides[1] = {(cuuint64_t)g.head_size * 2u};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(kv_cache), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keep_map(*map, kv_cache, g, box_rows, 0);
    return true;
}

bool encode_kv_map_fp8(CUtensorMap *map, const void *kv_cache, const KvGeom &g, int box_rows) {
    if (g.head_size != 128) return false;
    if (cached_map(map, kv_cache, g, box_rows, 1)) return true;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t rows =
        (cuuint64_t)g.num_blocks * 2u * (cuuint64_t)g.num_kv_heads * (cuuint64_t)g.block_size;
    cuuint64_t dims[2] = {(cuuint64_t)g.head_size, rows};
    cuuint64_t strides[1] = {(cuuint64_t)g.head_size};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(kv_cache), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keep_map(*map, kv_cache, g, box_rows, 1);
    return true;
}

}  // namespace pa

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks common to every entry point that reads the pool.
pa_status check_pool(const void *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                     int head_size) {
    if (!kv_cache || !aligned(kv_cache, 16)) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_size != 64 && head_size != 128) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (num_kv_heads > 255) return PA_ERR_UNSUPPORTED;
    // Pool rows must fit the signed 32-bit TMA row coordinate.
    const long long rows = (long long)num_blocks * 2 * num_kv_heads * block_size;
    if (rows >= (1LL << 30)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

pa_status check_heads(int num_heads, int num_kv_heads) {
    if (num_heads <= 0 || num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (group > 8) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

pa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

bool good_scale(float s) { return s == s && s > 0.f && s < 3.0e38f; }

}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_OOB: return "PA_ERR_OOB";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_PRECONDITION: return "PA_ERR_PRECONDITION";
    }
    return "PA_ERR_UNKNOWN";
}

size_t pa_kv_block_bytes(int block_size, int num_kv_heads, int head_size) {
    if (block_size <= 0 || num_kv_heads <= 0 || head_size <= 0) return 0;
    return (size_t)2 * (size_t)block_size * (size_t)num_kv_heads * (size_t)head_size * 2u;
}

// pa_cache_write's checks (and pa_cache_write_fp8's, with kv8 and its scales);
// PA_OK with *nothing_to_do set for an empty batch.
static pa_status write_checks(const void *kv_cache, int num_blocks, int block_size,
                              int num_kv_heads, int head_size, const void *k_new,
                              const void *v_new, int64_t new_row_stride,
                              const int32_t *slot_mapping, int num_tokens, bool kv8, float k_scale,
                              float v_scale, bool *nothing_to_do) {
    *nothing_to_do = false;
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (kv8 && (!good_scale(k_scale) || !good_scale(v_scale))) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) {
        *nothing_to_do = true;
        return PA_OK;
    }
    if (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(slot_mapping, 4))
        return PA_ERR_INVALID_ARG;
    if (new_row_stride < (int64_t)num_kv_heads * head_size || new_row_stride % 8 != 0)
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status pa_cache_write(void *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                         int head_size, const void *k_new, const void *v_new,
                         int64_t new_row_stride, const int32_t *slot_mapping, int num_tokens,
                         pa_stream_t stream) {
    bool none = false;
    pa_status st = write_checks(kv_cache, num_blocks, block_size, num_kv_heads, head_size, k_new,
                                v_new, new_row_stride, slot_mapping, num_tokens, false, 1.f, 1.f,
                                &none);
    if (st != PA_OK || none) return st;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_cache_write(kv_cache, g, k_new, v_new, new_row_stride,
                                            slot_mapping, num_tokens,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

size_t pa_kv_block_bytes_dtype(int block_size, int num_kv_heads, int head_size,
                               int dtype_num_bytes) {
    if (block_size <= 0 || num_kv_heads <= 0 || head_size <= 0 || dtype_num_bytes <= 0) return 0;
    return (size_t)2 * (size_t)block_size * (size_t)num_kv_heads * (size_t)head_size *
           (size_t)dtype_num_bytes;
}

pa_status pa_cache_write_fp8(void *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                             int head_size, const void *k_new, const void *v_new,
                             int64_t new_row_stride, const int32_t *slot_mapping, int num_tokens,
                             float k_scale, float v_scale, pa_stream_t stream) {
    bool none = false;
    pa_status st = write_checks(kv_cache, num_blocks, block_size, num_kv_heads, head_size, k_new,
                                v_new, new_row_stride, slot_mapping, num_tokens, true, k_scale,
                                v_scale, &none);
    if (st != PA_OK || none) return st;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_cache_write_fp8(kv_cache, g, k_new, v_new, new_row_stride,
                                                slot_mapping, num_tokens, k_scale, v_scale,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_fp8(void *out, const void *q, const void *kv_cache, int num_blocks,
                        int block_size, int num_heads, int num_kv_heads, int head_size,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                        float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                        pa_stream_t stream) {
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if ((st = check_heads(num_heads, num_kv_heads)) != PA_OK) return st;
    if (head_size != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return PA_ERR_INVALID_ARG;
    if (!good_scale(k_scale) || !good_scale(v_scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !block_tables || !seq_lens || !aligned(out, 16) || !aligned(q, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (max_seq_len > max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
    if (num_seqs > pa::decode_max_seqs(head_size, num_heads / num_kv_heads, true))
        return PA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * num_kv_heads * (((long long)max_seq_len + 15) / 16) >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    const size_t need = pa::decode_workspace_bytes(num_seqs, head_size, pa::device_sm_count());
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_decode_fp8(out, q, kv_cache, g, num_heads, block_tables,
                                           max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                                           scale, k_scale, v_scale, workspace,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_size) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0) return 0;
    if (num_heads % num_kv_heads != 0) return 0;
    return pa::decode_workspace_bytes(num_seqs, head_size, pa::device_sm_count());
}

// pa_decode's checks of everything but the workspace; PA_OK with
// *nothing_to_do set for an empty batch.
static pa_status decode_checks(const void *out, const void *q, const void *kv_cache, int num_blocks,
                        int block_size, int num_heads, int num_kv_heads, int head_size,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                        bool *nothing_to_do, bool kv8 = false) {
    *nothing_to_do = false;
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if ((st = check_heads(num_heads, num_kv_heads)) != PA_OK) return st;
    if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) {
        *nothing_to_do = true;
        return PA_OK;
    }
    if (!out || !q || !block_tables || !seq_lens || !aligned(out, 16) || !aligned(q, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (max_seq_len > max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
    if (kv8 && head_size != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs > pa::decode_max_seqs(head_size, num_heads / num_kv_heads, kv8))
        return PA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * num_kv_heads * (((long long)max_seq_len + 15) / 16) >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// pa_prefill_chunk's checks; PA_OK with *nothing_to_do set for an empty batch.
static pa_status prefill_checks(const void *out, const void *q, const int32_t *cu_q_lens,
                         int num_chunks, int max_q_len, const void *kv_cache, int num_blocks,
                         int block_size, int num_heads, int num_kv_heads, int head_size,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, float scale, bool *nothing_to_do) {
    *nothing_to_do = false;
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if ((st = check_heads(num_heads, num_kv_heads)) != PA_OK) return st;
    if (num_chunks < 0 || max_q_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return PA_ERR_INVALID_ARG;
    if (num_chunks == 0 || max_q_len == 0) {
        *nothing_to_do = true;
        return PA_OK;
    }
    if (!out || !q || !cu_q_lens || !block_tables || !seq_lens || !aligned(out, 16) ||
        !aligned(q, 16) || !aligned(cu_q_lens, 4) || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (num_chunks > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

pa_status pa_decode(void *out, const void *q, const void *kv_cache, int num_blocks,
                    int block_size, int num_heads, int num_kv_heads, int head_size,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                    void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    bool none = false;
    pa_status st = decode_checks(out, q, kv_cache, num_blocks, block_size, num_heads,
                                 num_kv_heads, head_size, block_tables, max_blocks_per_seq,
                                 seq_lens, num_seqs, max_seq_len, scale, &none);
    if (st != PA_OK || none) return st;
    const size_t need = pa::decode_workspace_bytes(num_seqs, head_size, pa::device_sm_count());
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_decode(out, q, kv_cache, g, num_heads, block_tables,
                                       max_blocks_per_seq, seq_lens, num_seqs, max_seq_len, scale,
                                       workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pa_decode_cascade_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                         int head_size, int shared_len) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || shared_len < 0)
        return 0;
    const int sms = pa::device_sm_count();
    const int splits = pa::prefix_splits(num_seqs, num_heads, num_kv_heads, shared_len, sms);
    return pa::decode_workspace_bytes(num_seqs, head_size, sms) +
           pa::prefix_partial_bytes(splits, num_seqs, num_heads, head_size) +
           (splits > 0 ? pa::cascade_whole_bytes(num_seqs, num_kv_heads, head_size) : 0);
}

int pa_decode_cascade_kernels(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                              int block_size, int max_seq_len, int shared_len, int kv8) {
    if (num_seqs < 0 || max_seq_len < 0 || shared_len < 0 || shared_len > max_seq_len) return -1;
    if (check_heads(num_heads, num_kv_heads) != PA_OK || num_kv_heads > 255) return -1;
    if (head_size != 64 && head_size != 128) return -1;
    if (block_size != 8 && block_size != 16 && block_size != 32) return -1;
    if (num_seqs == 0) return 0;
    if (shared_len == 0)  // pa_decode: one CTA per segment, or the split kernel and its merge
        return pa::decode_seg_ctas(num_seqs, num_kv_heads, max_seq_len, pa::device_sm_count())
                   ? 1
                   : 2;
    const pa::KvGeom g{1, block_size, num_kv_heads, head_size};
    return pa::cascade_one_launch_ctas(num_seqs, num_heads, g, max_seq_len, shared_len, kv8 != 0,
                                       pa::device_sm_count()) > 0
               ? 2
               : 3;
}

// pa_decode_cascade and pa_decode_cascade_fp8 (kv8: an FP8 pool, head size 128).
static pa_status cascade_impl(void *out, const void *q, const void *kv_cache, int num_blocks,
                              int block_size, int num_heads, int num_kv_heads, int head_size,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int num_seqs, int max_seq_len,
                              int shared_len, float scale, bool kv8, float k_scale, float v_scale,
                              void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if ((st = check_heads(num_heads, num_kv_heads)) != PA_OK) return st;
    if (kv8 && head_size != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (shared_len < 0 || shared_len > max_seq_len) return PA_ERR_INVALID_ARG;
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return PA_ERR_INVALID_ARG;
    if (kv8 && (!good_scale(k_scale) || !good_scale(v_scale))) return PA_ERR_INVALID_ARG;
    if (shared_len % 16 != 0 || shared_len % block_size != 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !block_tables || !seq_lens || !aligned(out, 16) || !aligned(q, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (max_seq_len > max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
    if (num_seqs > pa::decode_max_seqs(head_size, num_heads / num_kv_heads, kv8))
        return PA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * num_kv_heads * (((long long)max_seq_len + 15) / 16) >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    const int sms = pa::device_sm_count();
    const int splits = pa::prefix_splits(num_seqs, num_heads, num_kv_heads, shared_len, sms);
    const size_t dec = pa::decode_workspace_bytes(num_seqs, head_size, sms);
    const size_t pre = pa::prefix_partial_bytes(splits, num_seqs, num_heads, head_size);
    const size_t need =
        dec + pre + (splits > 0 ? pa::cascade_whole_bytes(num_seqs, num_kv_heads, head_size) : 0);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PA_ERR_WORKSPACE;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *pre_ml = nullptr, *pre_acc = nullptr;
    void *whole = nullptr;  // after the prefix partials
    if (splits > 0) {
        whole = static_cast<uint8_t *>(workspace) + dec + pre;
        // Prefix partials: (m, l) records, then O rows (room for `splits` splits).
        uint8_t *base = static_cast<uint8_t *>(workspace) + dec;
        const size_t rows = (size_t)splits * num_seqs * num_heads;
        pre_ml = reinterpret_cast<float *>(base);
        pre_acc = reinterpret_cast<float *>(base + (rows * 2 * 4 + 255) / 256 * 256);
        const cudaError_t one = pa::launch_cascade_one(
            out, q, kv_cache, g, num_heads, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
            max_seq_len, shared_len, scale, workspace, pre_ml, pre_acc, whole, kv8, k_scale,
            v_scale, s);
        if (one != cudaErrorNotSupported) return from_cuda(one);
        cudaError_t e = pa::launch_prefix_partials(q, kv_cache, g, num_heads, block_tables,
                                                   max_blocks_per_seq, num_seqs, shared_len,
                                                   scale, splits, pre_ml, pre_acc, kv8, k_scale,
                                                   v_scale, s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    return from_cuda(pa::launch_decode_suffix(out, q, kv_cache, g, num_heads, block_tables,
                                              max_blocks_per_seq, seq_lens, num_seqs,
                                              max_seq_len, shared_len, scale, workspace, pre_ml,
                                              pre_acc, splits, whole, kv8, k_scale, v_scale, s));
}

pa_status pa_decode_cascade(void *out, const void *q, const void *kv_cache, int num_blocks,
                            int block_size, int num_heads, int num_kv_heads, int head_size,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int num_seqs, int max_seq_len,
                            int shared_len, float scale, void *workspace,
                            size_t workspace_bytes, pa_stream_t stream) {
    return cascade_impl(out, q, kv_cache, num_blocks, block_size, num_heads, num_kv_heads,
                        head_size, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                        max_seq_len, shared_len, scale, false, 1.f, 1.f, workspace,
                        workspace_bytes, stream);
}

pa_status pa_decode_cascade_fp8(void *out, const void *q, const void *kv_cache, int num_blocks,
                                int block_size, int num_heads, int num_kv_heads, int head_size,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *seq_lens, int num_seqs, int max_seq_len,
                                int shared_len, float scale, float k_scale, float v_scale,
                                void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    return cascade_impl(out, q, kv_cache, num_blocks, block_size, num_heads, num_kv_heads,
                        head_size, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                        max_seq_len, shared_len, scale, true, k_scale, v_scale, workspace,
                        workspace_bytes, stream);
}

pa_status pa_prefill_chunk(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                           int max_q_len, const void *kv_cache, int num_blocks, int block_size,
                           int num_heads, int num_kv_heads, int head_size,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, float scale, pa_stream_t stream) {
    bool none = false;
    pa_status st = prefill_checks(out, q, cu_q_lens, num_chunks, max_q_len, kv_cache, num_blocks,
                                  block_size, num_heads, num_kv_heads, head_size, block_tables,
                                  max_blocks_per_seq, seq_lens, scale, &none);
    if (st != PA_OK || none) return st;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_prefill(out, q, cu_q_lens, num_chunks, max_q_len, kv_cache, g,
                                        num_heads, block_tables, max_blocks_per_seq, seq_lens,
                                        scale, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pa_attention_varlen_workspace_bytes(int num_seqs, int num_prefills, int num_heads,
                                           int num_kv_heads, int head_size) {
    if (num_prefills < 0 || num_prefills > num_seqs) return 0;
    const size_t dec =
        pa_decode_workspace_bytes(num_seqs - num_prefills, num_heads, num_kv_heads, head_size);
    if (dec == 0 || head_size <= 0) return dec;
    return pa::mixed_workspace_bytes(num_seqs - num_prefills, head_size, pa::device_sm_count());
}

// pa_attention_varlen over a bf16 pool, or (kv8) pa_attention_varlen_fp8.  Every
// host check (the write's, the chunks', the decode tokens' and the workspace's)
// runs before anything is enqueued, so a host-checkable fault leaves the pool
// untouched.
static pa_status varlen_impl(void *out, const void *q, const void *k_new, const void *v_new,
                             const int32_t *slot_mapping, const int32_t *cu_q_lens, int num_seqs,
                             int num_prefills, int num_prefill_tokens, int max_prefill_q_len,
                             void *kv_cache, int num_blocks, int block_size, int num_heads,
                             int num_kv_heads, int head_size, const int32_t *block_tables,
                             int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                             float scale, bool kv8, float k_scale, float v_scale,
                             void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    pa_status st = check_pool(kv_cache, num_blocks, block_size, num_kv_heads, head_size);
    if (st != PA_OK) return st;
    if ((st = check_heads(num_heads, num_kv_heads)) != PA_OK) return st;
    if (num_seqs < 0 || num_prefills < 0 || num_prefills > num_seqs || num_prefill_tokens < 0 ||
        max_prefill_q_len < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_prefills > 0 && num_prefill_tokens < num_prefills) return PA_ERR_INVALID_ARG;
    if (num_prefills == 0 && num_prefill_tokens != 0) return PA_ERR_INVALID_ARG;
    if (kv8 && head_size != 128) return PA_ERR_UNSUPPORTED;
    if (kv8 && (!good_scale(k_scale) || !good_scale(v_scale))) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    const int num_decodes = num_seqs - num_prefills;
    const int64_t rows = (int64_t)num_prefill_tokens + num_decodes;
    if (rows > INT32_MAX) return PA_ERR_UNSUPPORTED;
    const int64_t row_elems = (int64_t)num_heads * head_size;
    const size_t off = (size_t)num_prefill_tokens * (size_t)row_elems * 2;
    const int32_t *dec_tables = block_tables ? block_tables + (size_t)num_prefills *
                                                                  max_blocks_per_seq
                                             : nullptr;
    const int32_t *dec_lens = seq_lens ? seq_lens + num_prefills : nullptr;
    void *dec_out = out ? static_cast<uint8_t *>(out) + off : nullptr;
    const void *dec_q = q ? static_cast<const uint8_t *>(q) + off : nullptr;
    // 1. The write's checks.
    bool none_w = true;
    if (slot_mapping) {
        st = write_checks(kv_cache, num_blocks, block_size, num_kv_heads, head_size, k_new, v_new,
                          (int64_t)num_kv_heads * head_size, slot_mapping, (int)rows, kv8,
                          k_scale, v_scale, &none_w);
        if (st != PA_OK) return st;
    }
    // 2. The chunks' checks.
    bool none_p = true;
    if (num_prefills > 0) {
        st = prefill_checks(out, q, cu_q_lens, num_prefills, max_prefill_q_len, kv_cache,
                            num_blocks, block_size, num_heads, num_kv_heads, head_size,
                            block_tables, max_blocks_per_seq, seq_lens, scale, &none_p);
        if (st != PA_OK) return st;
    }
    // 3. The decode tokens' checks.
    bool none_d = true;
    if (num_decodes > 0) {
        st = decode_checks(dec_out, dec_q, kv_cache, num_blocks, block_size, num_heads,
                           num_kv_heads, head_size, dec_tables, max_blocks_per_seq, dec_lens,
                           num_decodes, max_seq_len, scale, &none_d, kv8);
        if (st != PA_OK) return st;
    }
    // 4. The workspace: the one launch's, or the separate decode's.
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    const int sms = pa::device_sm_count();
    const bool one = !none_p && !none_d && pa::mixed_supported(num_decodes, num_heads, g, kv8);
    if (!none_d) {
        const size_t need = one ? pa::mixed_workspace_bytes(num_decodes, head_size, sms)
                                : pa::decode_workspace_bytes(num_decodes, head_size, sms);
        if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
            return PA_ERR_WORKSPACE;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // With chunks and decode tokens in one launch, the split of its SMs is
    // computed by one extra block of the write's launch.
    pa::MixPlanArgs plan_job;
    const bool plan_in_write =
        one && !none_w && pa::mixed_plan_args(&plan_job, cu_q_lens, num_prefills, g, num_heads,
                                              max_blocks_per_seq, seq_lens, num_seqs, workspace,
                                              kv8);
    // The step's new K/V into their slots (one row per query row).
    if (!none_w) {
        const pa::MixPlanArgs *job = plan_in_write ? &plan_job : nullptr;
        const cudaError_t e =
            kv8 ? pa::launch_cache_write_fp8(kv_cache, g, k_new, v_new,
                                             (int64_t)num_kv_heads * head_size, slot_mapping,
                                             (int)rows, k_scale, v_scale, s, job)
                : pa::launch_cache_write(kv_cache, g, k_new, v_new,
                                         (int64_t)num_kv_heads * head_size, slot_mapping,
                                         (int)rows, s, job);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    // Chunks and decode tokens in one launch when both are present: side by side
    // on disjoint SMs.
    if (one)
        return from_cuda(pa::launch_mixed(out, q, cu_q_lens, num_prefills, num_prefill_tokens,
                                          max_prefill_q_len, kv_cache, g, num_heads,
                                          block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                          scale, workspace, kv8, k_scale, v_scale, s,
                                          plan_in_write, !none_w));
    // Otherwise one part at a time: the chunks (sequences [0, num_prefills), query
    // rows [0, num_prefill_tokens)), then the decode tokens (one row each).
    if (!none_p) {
        const cudaError_t e =
            kv8 ? pa::launch_prefill_fp8(out, q, cu_q_lens, num_prefills, max_prefill_q_len,
                                         kv_cache, g, num_heads, block_tables, max_blocks_per_seq,
                                         seq_lens, scale, k_scale, v_scale, s)
                : pa::launch_prefill(out, q, cu_q_lens, num_prefills, max_prefill_q_len, kv_cache,
                                     g, num_heads, block_tables, max_blocks_per_seq, seq_lens,
                                     scale, s);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    if (!none_d) {
        // Right after the write (no chunks between): the decode's set-up overlaps it.
        const bool after_write = !none_w && none_p;
        const cudaError_t e =
            kv8 ? pa::launch_decode_fp8(dec_out, dec_q, kv_cache, g, num_heads, dec_tables,
                                        max_blocks_per_seq, dec_lens, num_decodes, max_seq_len,
                                        scale, k_scale, v_scale, workspace, s, after_write)
                : pa::launch_decode(dec_out, dec_q, kv_cache, g, num_heads, dec_tables,
                                    max_blocks_per_seq, dec_lens, num_decodes, max_seq_len, scale,
                                    workspace, s, after_write);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

pa_status pa_attention_varlen(void *out, const void *q, const void *k_new, const void *v_new,
                              const int32_t *slot_mapping, const int32_t *cu_q_lens,
                              int num_seqs, int num_prefills, int num_prefill_tokens,
                              int max_prefill_q_len, void *kv_cache, int num_blocks,
                              int block_size, int num_heads, int num_kv_heads, int head_size,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int max_seq_len, float scale,
                              void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    return varlen_impl(out, q, k_new, v_new, slot_mapping, cu_q_lens, num_seqs, num_prefills,
                       num_prefill_tokens, max_prefill_q_len, kv_cache, num_blocks, block_size,
                       num_heads, num_kv_heads, head_size, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, scale, false, 1.f, 1.f, workspace, workspace_bytes,
                       stream);
}

pa_status pa_attention_varlen_fp8(void *out, const void *q, const void *k_new,
                                  const void *v_new, const int32_t *slot_mapping,
                                  const int32_t *cu_q_lens, int num_seqs, int num_prefills,
                                  int num_prefill_tokens, int max_prefill_q_len, void *kv_cache,
                                  int num_blocks, int block_size, int num_heads,
                                  int num_kv_heads, int head_size, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *seq_lens,
                                  int max_seq_len, float scale, float k_scale, float v_scale,
                                  void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    return varlen_impl(out, q, k_new, v_new, slot_mapping, cu_q_lens, num_seqs, num_prefills,
                       num_prefill_tokens, max_prefill_q_len, kv_cache, num_blocks, block_size,
                       num_heads, num_kv_heads, head_size, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, scale, true, k_scale, v_scale, workspace,
                       workspace_bytes, stream);
}

size_t pa_varlen_args_bytes(void) { return sizeof(pa_varlen_args); }

pa_status pa_attention_varlen_packed(const pa_varlen_args *a) {
    if (!a) return PA_ERR_INVALID_ARG;
    return varlen_impl(a->out, a->q, a->k_new, a->v_new, a->slot_mapping, a->cu_q_lens,
                       a->num_seqs, a->num_prefills, a->num_prefill_tokens, a->max_prefill_q_len,
                       a->kv_cache, a->num_blocks, a->block_size, a->num_heads, a->num_kv_heads,
                       a->head_size, a->block_tables, a->max_blocks_per_seq, a->seq_lens,
                       a->max_seq_len, a->scale, a->kv8 != 0, a->k_scale, a->v_scale,
                       a->workspace, a->workspace_bytes, a->stream);
}

pa_status pa_prefill_chunk_fp8(void *out, const void *q, const int32_t *cu_q_lens,
                               int num_chunks, int max_q_len, const void *kv_cache,
                               int num_blocks, int block_size, int num_heads, int num_kv_heads,
                               int head_size, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, float scale,
                               float k_scale, float v_scale, pa_stream_t stream) {
    bool none = false;
    pa_status st = prefill_checks(out, q, cu_q_lens, num_chunks, max_q_len, kv_cache, num_blocks,
                                  block_size, num_heads, num_kv_heads, head_size, block_tables,
                                  max_blocks_per_seq, seq_lens, scale, &none);
    if (st != PA_OK) return st;
    if (head_size != 128) return PA_ERR_UNSUPPORTED;
    if (!good_scale(k_scale) || !good_scale(v_scale)) return PA_ERR_INVALID_ARG;
    if (none) return PA_OK;
    pa::KvGeom g{num_blocks, block_size, num_kv_heads, head_size};
    return from_cuda(pa::launch_prefill_fp8(out, q, cu_q_lens, num_chunks, max_q_len, kv_cache,
                                            g, num_heads, block_tables, max_blocks_per_seq,
                                            seq_lens, scale, k_scale, v_scale,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_error_check(pa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    unsigned bits = 0, b = 0;
    if (pa::take_error_cache_write(&b) != cudaSuccess) return PA_ERR_CUDA;
    bits |= b;
    if (pa::take_error_decode(&b) != cudaSuccess) return PA_ERR_CUDA;
    bits |= b;
    if (pa::take_error_prefill(&b) != cudaSuccess) return PA_ERR_CUDA;
    bits |= b;
    if (bits & 2u) return PA_ERR_TIMEOUT;
    if (bits & 1u) return PA_ERR_OOB;
    if (bits & 4u) return PA_ERR_PRECONDITION;
    return PA_OK;
}

}  // extern "C"
