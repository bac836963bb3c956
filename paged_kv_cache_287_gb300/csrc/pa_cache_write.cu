// pa_cache_write.cu - scatter new tokens' K/V rows into their pool slots.
//
// "Inside vLLM: Anatomy of a High-Throughput LLM Inference System", §Engine core:
// each token's KV lives in a block its sequence was given; slot_mapping names
// block*block_size + offset for every new token.  A pure HBM-bound bit copy of
// 16-byte vectors.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned g_err_cache_write;

// Work split shared by both kernels: a grid-stride loop over tokens, two tokens
// per step (the loads of both are issued before either is stored, for more
// bytes in flight); the block's threads cover a token's K and V rows, one
// 16-byte output vector each, consecutive threads on consecutive bytes of one
// head's row on both sides.  A slot and its block are read and divided once per
// token, in 32 bits (slots are int32).  Slots < 0 are padding; slots past the
// pool are skipped and flagged.
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

template <int D>
__global__ void __launch_bounds__(256) cache_write_kernel(uint4 *__restrict__ kv,
                                                          const uint4 *__restrict__ k_new,
                                                          const uint4 *__restrict__ v_new,
                                                          int64_t row_stride_vec,
                                                          const int32_t *__restrict__ slots,
                                                          int num_tokens, int block_size,
                                                          int num_kv_heads, int64_t num_slots) {
    constexpr int kVecPerHead = D / 8;  // 16-byte vectors in one head row
    const int vec_per_side = num_kv_heads * kVecPerHead;
    auto src = [&](int tok, int v) {
        const int side = v >= vec_per_side ? 1 : 0;
        return (side ? v_new : k_new) + (int64_t)tok * row_stride_vec + (v - side * vec_per_side);
    };
    for (int t0 = blockIdx.x; t0 < num_tokens; t0 += 2 * gridDim.x) {
        const int t1 = t0 + gridDim.x;
        const TokenSlot a = token_slot(slots, t0, num_tokens, block_size, num_slots);
        const TokenSlot b = token_slot(slots, t1, num_tokens, block_size, num_slots);
        for (int v = threadIdx.x; v < 2 * vec_per_side; v += blockDim.x) {
            uint4 x0, x1;
            if (a.blk >= 0) x0 = *src(t0, v);
            if (b.blk >= 0) x1 = *src(t1, v);
            if (a.blk >= 0) kv[pool_vec<kVecPerHead>(a, v, vec_per_side, num_kv_heads, block_size)] = x0;
            if (b.blk >= 0) kv[pool_vec<kVecPerHead>(b, v, vec_per_side, num_kv_heads, block_size)] = x1;
        }
    }
}

// FP8 pool (one OCP e4m3 code per element, same layout): each element x of a
// new row is stored as the e4m3 code nearest to x / scale (binary32 division,
// ties to even, saturating at +-448).  One thread writes one 16-byte vector of
// codes from 32 bytes of bf16 input.
__device__ __forceinline__ uint4 e4m3_vec(const uint4 *src, float sc) {
    const uint4 in[2] = {src[0], src[1]};
    const uint32_t *w = reinterpret_cast<const uint32_t *>(in);
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = pack_e4m3x2(__fdiv_rn(bf16_lo(w[2 * k]), sc),
                                        __fdiv_rn(bf16_hi(w[2 * k]), sc));
        const uint32_t hi = pack_e4m3x2(__fdiv_rn(bf16_lo(w[2 * k + 1]), sc),
                                        __fdiv_rn(bf16_hi(w[2 * k + 1]), sc));
        q[k] = lo | (hi << 16);
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
}

template <int D>
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    uint4 *__restrict__ kv, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    int64_t row_stride_vec, const int32_t *__restrict__ slots, int num_tokens, int block_size,
    int num_kv_heads, int64_t num_slots, float k_scale, float v_scale) {
    constexpr int kVecPerHead = D / 16;  // 16-byte vectors of codes in one head row
    const int vec_per_side = num_kv_heads * kVecPerHead;
    for (int t0 = blockIdx.x; t0 < num_tokens; t0 += 2 * gridDim.x) {
        const int t1 = t0 + gridDim.x;
        const TokenSlot a = token_slot(slots, t0, num_tokens, block_size, num_slots);
        const TokenSlot b = token_slot(slots, t1, num_tokens, block_size, num_slots);
        for (int v = threadIdx.x; v < 2 * vec_per_side; v += blockDim.x) {
            const int side = v >= vec_per_side ? 1 : 0;
            const int r = v - side * vec_per_side;
            const uint4 *base = side ? v_new : k_new;
            const float sc = side ? v_scale : k_scale;
            if (a.blk >= 0)
                kv[pool_vec<kVecPerHead>(a, v, vec_per_side, num_kv_heads, block_size)] =
                    e4m3_vec(base + (int64_t)t0 * row_stride_vec + 2 * r, sc);
            if (b.blk >= 0)
                kv[pool_vec<kVecPerHead>(b, v, vec_per_side, num_kv_heads, block_size)] =
                    e4m3_vec(base + (int64_t)t1 * row_stride_vec + 2 * r, sc);
        }
    }
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
// 256; blocks: two tokens each, at most eight blocks of 256 threads per SM.
void token_grid(int num_tokens, int vecs_per_token, int *threads, int *blocks) {
    *threads = std::min(256, (vecs_per_token + 31) / 32 * 32);
    const long long cap = (long long)device_sm_count() * 8 * 256 / *threads;
    *blocks = (int)std::max(1LL, std::min<long long>((num_tokens + 1) / 2, cap));
}

}  // namespace

cudaError_t launch_cache_write(void *kv_cache, const KvGeom &g, const void *k_new,
                               const void *v_new, int64_t new_row_stride,
                               const int32_t *slot_mapping, int num_tokens,
                               cudaStream_t stream) {
    int threads, blocks;
    token_grid(num_tokens, 2 * g.num_kv_heads * (g.head_size / 8), &threads, &blocks);
    const int64_t num_slots = (int64_t)g.num_blocks * g.block_size;
    const int64_t stride_vec = new_row_stride / 8;
    if (g.head_size == 128)
        cache_write_kernel<128><<<(unsigned)blocks, threads, 0, stream>>>(
            static_cast<uint4 *>(kv_cache), static_cast<const uint4 *>(k_new),
            static_cast<const uint4 *>(v_new), stride_vec, slot_mapping, num_tokens,
            g.block_size, g.num_kv_heads, num_slots);
    else
        cache_write_kernel<64><<<(unsigned)blocks, threads, 0, stream>>>(
            static_cast<uint4 *>(kv_cache), static_cast<const uint4 *>(k_new),
            static_cast<const uint4 *>(v_new), stride_vec, slot_mapping, num_tokens,
            g.block_size, g.num_kv_heads, num_slots);
    return cudaGetLastError();
}

cudaError_t launch_cache_write_fp8(void *kv_cache, const KvGeom &g, const void *k_new,
                                   const void *v_new, int64_t new_row_stride,
                                   const int32_t *slot_mapping, int num_tokens, float k_scale,
                                   float v_scale, cudaStream_t stream) {
    int threads, blocks;
    token_grid(num_tokens, 2 * g.num_kv_heads * (g.head_size / 16), &threads, &blocks);
    const int64_t num_slots = (int64_t)g.num_blocks * g.block_size;
    const int64_t stride_vec = new_row_stride / 8;  // 16-byte bf16 vectors per token row
    if (g.head_size == 128)
        cache_write_fp8_kernel<128><<<(unsigned)blocks, threads, 0, stream>>>(
            static_cast<uint4 *>(kv_cache), static_cast<const uint4 *>(k_new),
            static_cast<const uint4 *>(v_new), stride_vec, slot_mapping, num_tokens,
            g.block_size, g.num_kv_heads, num_slots, k_scale, v_scale);
    else
        cache_write_fp8_kernel<64><<<(unsigned)blocks, threads, 0, stream>>>(
            static_cast<uint4 *>(kv_cache), static_cast<const uint4 *>(k_new),
            static_cast<const uint4 *>(v_new), stride_vec, slot_mapping, num_tokens,
            g.block_size, g.num_kv_heads, num_slots, k_scale, v_scale);
    return cudaGetLastError();
}

}  // namespace pa
