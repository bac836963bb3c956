// pa_cache_write.cu - scatter new tokens' K/V rows into their pool slots.
//
// "Inside vLLM: Anatomy of a High-Throughput LLM Inference System", §Engine core:
// each token's KV lives in a block its sequence was given; slot_mapping names
// block*block_size + offset for every new token.  A pure HBM-bound bit copy of
// 16-byte vectors.
#include <algorithm>
#include <cmath>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_plan.cuh"

namespace pa {
namespace {

__device__ unsigned g_err_cache_write;

// Work split shared by both kernels: a grid-stride loop over tokens, kTok tokens
// per step (the loads of all of them are issued before any is stored, for more
// bytes in flight); the block's threads cover a token's K and V rows, one
// 16-byte output vector each, consecutive threads on consecutive bytes of one
// head's row on both sides.  A slot and its block are read and divided once per
// token, in 32 bits (slots are int32).  Slots < 0 are padding; slots past the
// pool are skipped and flagged.  With a plan job the grid has one block more,
// the last, which computes the split of the mixed launch that follows and
// writes no token.
constexpr int kTok = 2;

struct TokenSlot {
    int blk, off;  // blk < 0: nothing to write
};

__device__ __forceinline__ TokenSlot token_slot(const int32_t *slots, int tok, int num_tokens,
                                                int block_size, int64_t num_slots) {
    if (tok >= num_tokens) return {-1, 0};
    const int slot = slots[tok];
    if (slot < 0) return {-1, 0};
    if ((int64_t)slot >= num_slots) {
        if (threadIdx.x == 0) atomicOr(&g_err_cache_write, kErrOob);
        return {-1, 0};
    }
    const int blk = (int)((unsigned)slot / (unsigned)block_size);
    return {blk, slot - blk * block_size};
}

// Output vector index in the pool of vector v (of 2 * vec_per_side) of a token.
template <int kVecPerHead>
__device__ __forceinline__ int64_t pool_vec(TokenSlot ts, int v, int vec_per_side,
                                            int num_kv_heads, int block_size) {
    const int side = v >= vec_per_side ? 1 : 0;  // 0 = K, 1 = V
    const int r = v - side * vec_per_side;
    const int head = r / kVecPerHead, c = r % kVecPerHead;
    return ((((int64_t)ts.blk * 2 + side) * num_kv_heads + head) * block_size + ts.off) *
               kVecPerHead + c;
}

// Tokens of a bf16 pool: the grid's first nb blocks.
template <int D>
__device__ __forceinline__ void write_rows(uint4 *__restrict__ kv, const uint4 *__restrict__ k_new,
                                           const uint4 *__restrict__ v_new,
                                           int64_t row_stride_vec,
                                           const int32_t *__restrict__ slots, int num_tokens,
                                           int block_size, int num_kv_heads, int64_t num_slots,
                                           int nb) {
    // A decode launched as this grid's programmatic dependent may start its set-up
    // now; it reads the pool only once this grid has completed.
    asm volatile("griddepcontrol.launch_dependents;" :::);
    constexpr int kVecPerHead = D / 8;  // 16-byte vectors in one head row
    const int vec_per_side = num_kv_heads * kVecPerHead;
    auto src = [&](int tok, int v) {
        const int side = v >= vec_per_side ? 1 : 0;
        return (side ? v_new : k_new) + (int64_t)tok * row_stride_vec + (v - side * vec_per_side);
    };
    for (int t0 = blockIdx.x; t0 < num_tokens; t0 += kTok * nb) {
        TokenSlot ts[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i)
            ts[i] = token_slot(slots, t0 + i * nb, num_tokens, block_size, num_slots);
        for (int v = threadIdx.x; v < 2 * vec_per_side; v += blockDim.x) {
            uint4 x[kTok];
#pragma unroll
            for (int i = 0; i < kTok; ++i)
                if (ts[i].blk >= 0) x[i] = *src(t0 + i * nb, v);
#pragma unroll
            for (int i = 0; i < kTok; ++i)
                if (ts[i].blk >= 0)
                    kv[pool_vec<kVecPerHead>(ts[i], v, vec_per_side, num_kv_heads, block_size)] =
                        x[i];
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256) cache_write_kernel(uint4 *__restrict__ kv,
                                                          const uint4 *__restrict__ k_new,
                                                          const uint4 *__restrict__ v_new,
                                                          int64_t row_stride_vec,
                                                          const int32_t *__restrict__ slots,
                                                          int num_tokens, int block_size,
                                                          int num_kv_heads, int64_t num_slots) {
    write_rows<D>(kv, k_new, v_new, row_stride_vec, slots, num_tokens, block_size, num_kv_heads,
                  num_slots, (int)gridDim.x);
}

// The same with the plan job in the last block.
template <int D>
__global__ void __launch_bounds__(256) cache_write_plan_kernel(
    uint4 *__restrict__ kv, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    int64_t row_stride_vec, const int32_t *__restrict__ slots, int num_tokens, int block_size,
    int num_kv_heads, int64_t num_slots, const MixPlanArgs job) {
    const int nb = (int)gridDim.x - 1;
    if ((int)blockIdx.x == nb) {
        mix_plan_block(job);
        return;
    }
    write_rows<D>(kv, k_new, v_new, row_stride_vec, slots, num_tokens, block_size, num_kv_heads,
                  num_slots, nb);
}

// FP8 pool (one OCP e4m3 code per element, same layout): each element x of a
// new row is stored as the e4m3 code nearest to x / scale (binary32 division,
// ties to even, saturating at +-448).  One thread writes one 16-byte vector of
// codes from 32 bytes of bf16 input.  kPow2: the scale is a power of two whose
// reciprocal r is a normal binary32 number; then x * r is the same real number
// as x / scale, so its rounding is the same, and the division's slow path is
// skipped (sc holds r).
template <bool kPow2>
__device__ __forceinline__ float div_scale(float x, float sc) {
    return kPow2 ? x * sc : __fdiv_rn(x, sc);
}

template <bool kPow2>
__device__ __forceinline__ uint4 e4m3_vec(const uint4 *src, float sc) {
    const uint4 in[2] = {src[0], src[1]};
    const uint32_t *w = reinterpret_cast<const uint32_t *>(in);
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = pack_e4m3x2(div_scale<kPow2>(bf16_lo(w[2 * k]), sc),
                                        div_scale<kPow2>(bf16_hi(w[2 * k]), sc));
        const uint32_t hi = pack_e4m3x2(div_scale<kPow2>(bf16_lo(w[2 * k + 1]), sc),
                                        div_scale<kPow2>(bf16_hi(w[2 * k + 1]), sc));
        q[k] = lo | (hi << 16);
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
}

// Tokens of an FP8 pool: the grid's first nb blocks.
template <int D, bool kPow2>
__device__ __forceinline__ void write_rows_fp8(uint4 *__restrict__ kv,
                                               const uint4 *__restrict__ k_new,
                                               const uint4 *__restrict__ v_new,
                                               int64_t row_stride_vec,
                                               const int32_t *__restrict__ slots, int num_tokens,
                                               int block_size, int num_kv_heads,
                                               int64_t num_slots, float k_scale, float v_scale,
                                               int nb) {
    asm volatile("griddepcontrol.launch_dependents;" :::);  // as in write_rows
    constexpr int kVecPerHead = D / 16;  // 16-byte vectors of codes in one head row
    const int vec_per_side = num_kv_heads * kVecPerHead;
    for (int t0 = blockIdx.x; t0 < num_tokens; t0 += kTok * nb) {
        TokenSlot ts[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i)
            ts[i] = token_slot(slots, t0 + i * nb, num_tokens, block_size, num_slots);
        for (int v = threadIdx.x; v < 2 * vec_per_side; v += blockDim.x) {
            const int side = v >= vec_per_side ? 1 : 0;
            const int r = v - side * vec_per_side;
            const uint4 *base = (side ? v_new : k_new) + 2 * r;
            const float sc = side ? v_scale : k_scale;
            uint4 x[kTok][2];
#pragma unroll
            for (int i = 0; i < kTok; ++i)
                if (ts[i].blk >= 0) {
                    const uint4 *p = base + (int64_t)(t0 + i * nb) * row_stride_vec;
                    x[i][0] = p[0];
                    x[i][1] = p[1];
                }
#pragma unroll
            for (int i = 0; i < kTok; ++i)
                if (ts[i].blk >= 0)
                    kv[pool_vec<kVecPerHead>(ts[i], v, vec_per_side, num_kv_heads, block_size)] =
                        e4m3_vec<kPow2>(x[i], sc);
        }
    }
}

template <int D, bool kPow2>
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    uint4 *__restrict__ kv, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    int64_t row_stride_vec, const int32_t *__restrict__ slots, int num_tokens, int block_size,
    int num_kv_heads, int64_t num_slots, float k_scale, float v_scale) {
    write_rows_fp8<D, kPow2>(kv, k_new, v_new, row_stride_vec, slots, num_tokens, block_size,
                             num_kv_heads, num_slots, k_scale, v_scale, (int)gridDim.x);
}

template <int D, bool kPow2>
__global__ void __launch_bounds__(256) cache_write_fp8_plan_kernel(
    uint4 *__restrict__ kv, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    int64_t row_stride_vec, const int32_t *__restrict__ slots, int num_tokens, int block_size,
    int num_kv_heads, int64_t num_slots, float k_scale, float v_scale, const MixPlanArgs job) {
    const int nb = (int)gridDim.x - 1;
    if ((int)blockIdx.x == nb) {
        mix_plan_block(job);
        return;
    }
    write_rows_fp8<D, kPow2>(kv, k_new, v_new, row_stride_vec, slots, num_tokens, block_size,
                             num_kv_heads, num_slots, k_scale, v_scale, nb);
}

}  // namespace

cudaError_t take_error_cache_write(unsigned *bits) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_err_cache_write, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_cache_write, &zero, sizeof(unsigned));
    return e;
}

namespace {

// Threads per block: a token's output vectors rounded up to whole warps, at most
// 256; token blocks: kTok tokens each, at most eight blocks of 256 threads per
// SM; one block more for a plan job.
void token_grid(int num_tokens, int vecs_per_token, bool plan_job, int *threads, int *blocks) {
    *threads = std::min(256, (vecs_per_token + 31) / 32 * 32);
    const long long cap = (long long)device_sm_count() * 8 * 256 / *threads;
    *blocks = (int)std::max(1LL, std::min<long long>((num_tokens + kTok - 1) / kTok, cap)) +
              (plan_job ? 1 : 0);
}

// 1 / s when s is a power of two and 1 / s a normal binary32 number (then exact),
// else 0.
float pow2_reciprocal(float s) {
    int e;
    if (!(s > 0.f) || std::frexp(s, &e) != 0.5f) return 0.f;
    // s = 2^(e-1); 1/s = 2^(1-e) is normal for 1 - e in [-126, 127].
    if (1 - e < -126 || 1 - e > 127) return 0.f;
    return std::ldexp(1.0f, 1 - e);
}

}  // namespace

cudaError_t launch_cache_write(void *kv_cache, const KvGeom &g, const void *k_new,
                               const void *v_new, int64_t new_row_stride,
                               const int32_t *slot_mapping, int num_tokens, cudaStream_t stream,
                               const MixPlanArgs *plan_job) {
    int threads, blocks;
    token_grid(num_tokens, 2 * g.num_kv_heads * (g.head_size / 8), plan_job != nullptr,
               &threads, &blocks);
    const int64_t num_slots = (int64_t)g.num_blocks * g.block_size;
    const int64_t stride_vec = new_row_stride / 8;
    uint4 *kv = static_cast<uint4 *>(kv_cache);
    const uint4 *kn = static_cast<const uint4 *>(k_new), *vn = static_cast<const uint4 *>(v_new);
    const bool d128 = g.head_size == 128;
    if (plan_job)
        (d128 ? cache_write_plan_kernel<128> : cache_write_plan_kernel<64>)
            <<<(unsigned)blocks, threads, 0, stream>>>(kv, kn, vn, stride_vec, slot_mapping,
                                                       num_tokens, g.block_size, g.num_kv_heads,
                                                       num_slots, *plan_job);
    else
        (d128 ? cache_write_kernel<128> : cache_write_kernel<64>)
            <<<(unsigned)blocks, threads, 0, stream>>>(kv, kn, vn, stride_vec, slot_mapping,
                                                       num_tokens, g.block_size, g.num_kv_heads,
                                                       num_slots);
    return cudaGetLastError();
}

cudaError_t launch_cache_write_fp8(void *kv_cache, const KvGeom &g, const void *k_new,
                                   const void *v_new, int64_t new_row_stride,
                                   const int32_t *slot_mapping, int num_tokens, float k_scale,
                                   float v_scale, cudaStream_t stream,
                                   const MixPlanArgs *plan_job) {
    int threads, blocks;
    token_grid(num_tokens, 2 * g.num_kv_heads * (g.head_size / 16), plan_job != nullptr,
               &threads, &blocks);
    const int64_t num_slots = (int64_t)g.num_blocks * g.block_size;
    const int64_t stride_vec = new_row_stride / 8;  // 16-byte bf16 vectors per token row
    // Both scales powers of two with normal reciprocals: multiply by those.
    const float rk = pow2_reciprocal(k_scale), rv = pow2_reciprocal(v_scale);
    const bool pow2 = rk > 0.f && rv > 0.f;
    const float ks = pow2 ? rk : k_scale, vs = pow2 ? rv : v_scale;
    uint4 *kv = static_cast<uint4 *>(kv_cache);
    const uint4 *kn = static_cast<const uint4 *>(k_new), *vn = static_cast<const uint4 *>(v_new);
    const bool d128 = g.head_size == 128;
    if (plan_job)
        (d128 ? (pow2 ? cache_write_fp8_plan_kernel<128, true>
                      : cache_write_fp8_plan_kernel<128, false>)
              : (pow2 ? cache_write_fp8_plan_kernel<64, true>
                      : cache_write_fp8_plan_kernel<64, false>))
            <<<(unsigned)blocks, threads, 0, stream>>>(kv, kn, vn, stride_vec, slot_mapping,
                                                       num_tokens, g.block_size, g.num_kv_heads,
                                                       num_slots, ks, vs, *plan_job);
    else
        (d128 ? (pow2 ? cache_write_fp8_kernel<128, true> : cache_write_fp8_kernel<128, false>)
              : (pow2 ? cache_write_fp8_kernel<64, true> : cache_write_fp8_kernel<64, false>))
            <<<(unsigned)blocks, threads, 0, stream>>>(kv, kn, vn, stride_vec, slot_mapping,
                                                       num_tokens, g.block_size, g.num_kv_heads,
                                                       num_slots, ks, vs);
    return cudaGetLastError();
}

}  // namespace pa
