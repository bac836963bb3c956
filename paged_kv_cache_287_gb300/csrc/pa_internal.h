// pa_internal.h - declarations shared by the translation units of libpagedattn.
// Not part of the public ABI (include/pa.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace pa {

// Raise kernel Kern's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute call is made only when this (kernel, device)
// has not yet been given that much: a launch path's per-call host cost is then
// the launch itself.
template <auto Kern>
cudaError_t ensure_smem(size_t bytes) {
    static std::atomic<int> granted[64];  // per device; zero at start
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const bool tracked = dev >= 0 && dev < 64;
    if (tracked && granted[dev].load(std::memory_order_acquire) >= (int)bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && tracked) {
        int cur = granted[dev].load(std::memory_order_relaxed);
        while (cur < (int)bytes && !granted[dev].compare_exchange_weak(cur, (int)bytes)) {
        }
    }
    return e;
}

// Geometry of the KV pool [num_blocks][2][num_kv_heads][block_size][head_size].
struct KvGeom {
    int num_blocks;
    int block_size;
    int num_kv_heads;
    int head_size;
};

// Each translation unit owns a device error word; these read and clear it.
cudaError_t take_error_cache_write(unsigned *bits);
cudaError_t take_error_decode(unsigned *bits);
cudaError_t take_error_prefill(unsigned *bits);

// Encode a 2-D TMA map over the pool viewed as rows of head_size bf16 elements,
// box = 64 elements x box_rows rows, 128-byte swizzle.  False on failure.  Maps
// are kept in a small cache keyed by (pool address, geometry, element type, box),
// so a pool used call after call is encoded once.
bool encode_kv_map(CUtensorMap *map, const void *kv_cache, const KvGeom &g, int box_rows);
// The same over an FP8 pool (rows of head_size bytes), box = 128 bytes x box_rows.
bool encode_kv_map_fp8(CUtensorMap *map, const void *kv_cache, const KvGeom &g, int box_rows);

int device_sm_count();

// Inputs of the device-side split of a mixed launch's SMs (pa_plan.cuh).
struct MixPlanArgs {
    const int32_t *seq_lens;   // all sequences, chunks first
    const int32_t *cu_q_lens;  // chunk row offsets [num_prefills + 1]
    int num_prefills, num_seqs, sms, max_len;
    float dec_bytes_per_token;  // K+V bytes per decode token: 2 * Hkv * D * element bytes
    float pre_flops_per_pair;   // flops per visible (query, key) pair: 4 * Hq * D
    float dec_sm_gbs, hbm_gbs, pre_sm_tflops;  // rates of the two parts
    int dec_warps;               // decode warps per decode CTA
    int *plan;                   // out: {decode CTAs, decode warps}
};

// plan_job (optional): the split of the mixed launch that follows, computed by
// one extra block of the same launch (no block waits on another).
cudaError_t launch_cache_write(void *kv_cache, const KvGeom &g, const void *k_new,
                               const void *v_new, int64_t new_row_stride,
                               const int32_t *slot_mapping, int num_tokens, cudaStream_t stream,
                               const MixPlanArgs *plan_job = nullptr);

// Whether pa_decode (no shared prefix) over this shape runs one CTA per segment
// and merges in place: one launch instead of the split kernel and its merge.
bool decode_seg_ctas(int num_seqs, int num_kv_heads, int max_seq_len, int sm_count);
// Decode workspace bytes for num_seqs sequences on a device with sm_count SMs.
size_t decode_workspace_bytes(int num_seqs, int head_size, int sm_count);
// Largest num_seqs the decode kernel's shared-memory tables hold (kv8: FP8 pool).
int decode_max_seqs(int head_size, int group, bool kv8 = false);

// FP8 pool (OCP e4m3 codes; real K/V = code value * k_scale / v_scale); head_size 128.
cudaError_t launch_cache_write_fp8(void *kv_cache, const KvGeom &g, const void *k_new,
                                   const void *v_new, int64_t new_row_stride,
                                   const int32_t *slot_mapping, int num_tokens, float k_scale,
                                   float v_scale, cudaStream_t stream,
                                   const MixPlanArgs *plan_job = nullptr);
cudaError_t launch_decode_fp8(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                              int num_heads, const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                              float k_scale, float v_scale, void *workspace, cudaStream_t stream,
                              bool after_write = false);

// after_write: the launch just before on the stream is launch_cache_write(_fp8)
// of this pool; the decode then starts as its programmatic dependent (its set-up
// overlaps the write, its reads of the pool wait for the write to complete).
cudaError_t launch_decode(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                          int num_heads, const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                          void *workspace, cudaStream_t stream, bool after_write = false);

// Shared-prefix (cascade) decode.  The first shared_len tokens of every sequence
// sit in sequence 0's first blocks.  The prefix pass computes, per key-range split,
// the unnormalised (m, l, O) of every (sequence, query head) over those tokens.
// kv8: an FP8 pool (head size 128), real K/V = code * k_scale / v_scale.
int prefix_splits(int num_seqs, int num_heads, int num_kv_heads, int shared_len, int sm_count);
cudaError_t launch_prefix_partials(const void *q, const void *kv_cache, const KvGeom &g,
                                   int num_heads, const int32_t *block_tables,
                                   int max_blocks_per_seq, int num_seqs, int shared_len,
                                   float scale, int splits, float *part_ml, float *part_acc,
                                   bool kv8, float k_scale, float v_scale, cudaStream_t stream);
// Bytes of prefix partials for `splits` splits.
size_t prefix_partial_bytes(int splits, int num_seqs, int num_heads, int head_size);
// The shared-prefix decode as one launch (prefix pass and own tokens side by side
// on disjoint SMs, one key split) plus the cascade merge kernel;
// cudaErrorNotSupported (nothing launched) when the separate launches suit the
// shape better.  pre_ml / pre_acc: room for one split's partials; whole:
// cascade_whole_bytes.
cudaError_t launch_cascade_one(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                               int num_heads, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                               int max_seq_len, int shared_len, float scale, void *workspace,
                               float *pre_ml, float *pre_acc, void *whole, bool kv8,
                               float k_scale, float v_scale, cudaStream_t stream);
// Decode CTAs of that one launch for these shapes on `sms` SMs, or 0 when the
// separate launches are used; *splits (if given): its prefix key splits.
int cascade_one_launch_ctas(int num_seqs, int num_heads, const KvGeom &g, int max_seq_len,
                            int shared_len, bool kv8, int sms, int *splits = nullptr);
// Bytes of the per-segment records of segments one decode warp finishes whole.
size_t cascade_whole_bytes(int num_seqs, int num_kv_heads, int head_size);
// Decode over each sequence's tokens [shared_len, seq_len), then the cascade
// merge kernel, which merges every segment with the prefix partials (pre_splits
// of them at pre_ml / pre_acc).  whole: cascade_whole_bytes of workspace.
cudaError_t launch_decode_suffix(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                                 int num_heads, const int32_t *block_tables,
                                 int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                                 int max_seq_len, int shared_len, float scale, void *workspace,
                                 const float *pre_ml, const float *pre_acc, int pre_splits,
                                 void *whole, bool kv8, float k_scale, float v_scale,
                                 cudaStream_t stream);

// One launch for a flattened mixed batch (chunks first, then decode sequences):
// decode and chunked prefill side by side on disjoint SMs, split on the device.
// mixed_supported: whether the decode part's shared memory fits the launch.
size_t mixed_workspace_bytes(int num_decodes, int head_size, int sm_count);
bool mixed_supported(int num_decodes, int num_heads, const KvGeom &g, bool kv8);
// The split's inputs for launch_mixed's batch (false: no mixed launch for it).
bool mixed_plan_args(MixPlanArgs *pl, const int32_t *cu_q_lens, int num_prefills,
                     const KvGeom &g, int num_heads, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_seqs, void *workspace, bool kv8);
// plan_done: a launch earlier on the stream ran mixed_plan_args' job (the cache
// write's extra block), so no plan kernel is launched here.  after_write: the
// launch just before on the stream is launch_cache_write(_fp8) of this pool; the
// attention launch then starts as its programmatic dependent.
cudaError_t launch_mixed(void *out, const void *q, const int32_t *cu_q_lens, int num_prefills,
                         int num_prefill_tokens, int max_prefill_q_len, const void *kv_cache,
                         const KvGeom &g, int num_heads, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                         float scale, void *workspace, bool kv8, float k_scale, float v_scale,
                         cudaStream_t stream, bool plan_done = false, bool after_write = false);

// Chunked prefill over an FP8 pool (head_size 128).
cudaError_t launch_prefill_fp8(void *out, const void *q, const int32_t *cu_q_lens,
                               int num_chunks, int max_q_len, const void *kv_cache,
                               const KvGeom &g, int num_heads, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, float scale,
                               float k_scale, float v_scale, cudaStream_t stream);

cudaError_t launch_prefill(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                           int max_q_len, const void *kv_cache, const KvGeom &g, int num_heads,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, float scale, cudaStream_t stream);

}  // namespace pa
