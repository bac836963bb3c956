// pa_cache_write.cu - scatter new tokens' K/V rows into their pool slots.
//
// "Inside vLLM: Anatomy of a High-Throughput LLM Inference System", §Engine core:
// each token's KV lives in a block its sequence was given; slot_mapping names
// block*block_size + offset for every new token.  A pure HBM-bound bit copy: one
// thread moves one 16-byte vector, consecutive threads cover one head's row of
// head_size*2 contiguous bytes on both sides.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned g_err_cache_write;

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
    const int64_t total = (int64_t)num_tokens * 2 * vec_per_side;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int tok = (int)(i / (2 * vec_per_side));
        const int rem = (int)(i - (int64_t)tok * 2 * vec_per_side);
        const int side = rem / vec_per_side;  // 0 = K, 1 = V
        const int r = rem - side * vec_per_side;
        const int head = r / kVecPerHead;
        const int c = r - head * kVecPerHead;
        const int64_t slot = slots[tok];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0 && side == 0) atomicOr(&g_err_cache_write, kErrOob);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const int64_t dst =
            (((blk * 2 + side) * num_kv_heads + head) * block_size + off) * kVecPerHead + c;
        const uint4 *src = side ? v_new : k_new;
        kv[dst] = src[(int64_t)tok * row_stride_vec + r];
    }
}

// FP8 pool (one OCP e4m3 code per element, same layout): each element x of a
// new row is stored as the e4m3 code nearest to x / scale (binary32 division,
// ties to even, saturating at +-448).  One thread writes one 16-byte vector of
// codes from 32 bytes of bf16 input.
template <int D>
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    uint4 *__restrict__ kv, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    int64_t row_stride_vec, const int32_t *__restrict__ slots, int num_tokens, int block_size,
    int num_kv_heads, int64_t num_slots, float k_scale, float v_scale) {
    constexpr int kVecPerHead = D / 16;  // 16-byte vectors of codes in one head row
    const int vec_per_side = num_kv_heads * kVecPerHead;
    const int64_t total = (int64_t)num_tokens * 2 * vec_per_side;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int tok = (int)(i / (2 * vec_per_side));
        const int rem = (int)(i - (int64_t)tok * 2 * vec_per_side);
        const int side = rem / vec_per_side;  // 0 = K, 1 = V
        const int r = rem - side * vec_per_side;
        const int head = r / kVecPerHead;
        const int c = r - head * kVecPerHead;
        const int64_t slot = slots[tok];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0 && side == 0) atomicOr(&g_err_cache_write, kErrOob);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const uint4 *src = (side ? v_new : k_new) + (int64_t)tok * row_stride_vec + 2 * r;
        const float sc = side ? v_scale : k_scale;
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
        const int64_t dst =
            (((blk * 2 + side) * num_kv_heads + head) * block_size + off) * kVecPerHead + c;
        kv[dst] = make_uint4(q[0], q[1], q[2], q[3]);
    }
}

}  // namespace

cudaError_t take_error_cache_write(unsigned *bits) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_err_cache_write, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_cache_write, &zero, sizeof(unsigned));
    return e;
}

cudaError_t launch_cache_write(void *kv_cache, const KvGeom &g, const void *k_new,
                               const void *v_new, int64_t new_row_stride,
                               const int32_t *slot_mapping, int num_tokens,
                               cudaStream_t stream) {
    const int64_t total = (int64_t)num_tokens * 2 * g.num_kv_heads * (g.head_size / 8);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
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
    const int64_t total = (int64_t)num_tokens * 2 * g.num_kv_heads * (g.head_size / 16);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
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
