// pa_prefill.cu - chunked-prefill attention over a paged KV cache.
//
// Chunked prefill ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
// System", advanced features: a long prompt is split into chunks interleaved with
// generation): a chunk of q_len new tokens, whose K/V were just written to the
// pool, attends causally to its sequence's cached context and to itself.  The
// batch is flattened (§Generate function): chunk s owns query rows
// cu_q_lens[s] .. cu_q_lens[s+1]-1.
//
// Design: one CTA per (query tile, KV head, chunk).  The CTA's rows are the
// query tile's tokens for every query head of the KV head's GQA group, so each
// K/V tile is fetched once for the whole group.  A producer warp streams 64-key
// K/V tiles through the block table with 128B-swizzled 2-D TMA copies into a
// 3-stage ring (full/empty mbarriers); up to 8 consumer warps each own 16 rows
// and run QK^T, an fp32 online softmax and PV on bf16 warp MMAs with P kept in
// registers.  Keys past a row's position are masked; tiles past the CTA's
// causal limit are never fetched.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned g_err_prefill;

constexpr int kKeys = 64;         // keys per K/V tile
constexpr int kStages = 3;
constexpr int kMaxWarps = 8;      // consumer warps

template <int D>
struct PLay {
    static constexpr int kPanels = D / 64;
    static constexpr int kPanelBytes = kKeys * 128;   // 64 rows of one 128-byte panel
    static constexpr int kTileBytes = kPanels * kPanelBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
};

struct PrefillArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const int32_t *cu_q_lens;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int num_heads, num_kv_heads, group;
    int block_size, max_blocks, num_blocks;
    int q_tile;        // query tokens per CTA (16 * (8 / group))
    int warps;         // consumer warps = group * q_tile / 16
    float scale_log2;
};

template <int D>
constexpr size_t prefill_smem_bytes() {
    return 1024 + (size_t)kStages * PLay<D>::kStageBytes + 2 * kStages * 8;
}

__device__ __forceinline__ int prefill_row(int blk, int h, int off, const PrefillArgs &a) {
    if (blk < 0 || blk >= a.num_blocks) {
        atomicOr(&g_err_prefill, kErrOob);
        return -(1 << 30);
    }
    return ((blk * 2) * a.num_kv_heads + h) * a.block_size + off;
}

template <int D>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const PrefillArgs a) {
    using L = PLay<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<size_t>(smem_raw) + 1023) & ~static_cast<size_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * L::kStageBytes);
    uint64_t *empty = full + kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.z, h = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
    const int q0 = a.cu_q_lens[s];
    const int q_len = a.cu_q_lens[s + 1] - q0;
    const int t0 = qt * a.q_tile;
    if (t0 >= q_len) return;
    int len = a.seq_lens[s];
    const int max_len = a.max_blocks * a.block_size;
    if (len < q_len || len > max_len) {
        if (threadIdx.x == 0) atomicOr(&g_err_prefill, kErrOob);
        len = std::min(std::max(len, q_len), max_len);
    }
    const int ctx = len - q_len;
    const int t_last = std::min(t0 + a.q_tile, q_len) - 1;   // last valid token of the tile
    const int n_keys = ctx + t_last + 1;                      // keys any row of the CTA sees
    const int n_kt = (n_keys + kKeys - 1) / kKeys;
    const int G = a.group;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kv_map);
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], a.warps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == a.warps) {
        // ------------------------------------------------------------ producer warp
        const int bs = a.block_size;
        const int box_rows = bs >= 16 ? 16 : bs;
        const int boxes = kKeys / box_rows;   // 4 or 8
        const int32_t *bt = a.block_tables + (size_t)s * a.max_blocks;
        const int v_off = a.num_kv_heads * bs;
        const uint32_t box_bytes = (uint32_t)box_rows * 128u;
        const uint64_t policy = policy_evict_first();
        auto box_row = [&](int kt) {
            int r = -1;
            const int tok = kt * kKeys + lane * box_rows;
            if (lane < boxes && tok < len) r = prefill_row(bt[tok / bs], h, tok % bs, a);
            return r;
        };
        int nxt = box_row(0);
        for (int kt = 0; kt < n_kt; ++kt) {
            const int cur = nxt;
            if (kt + 1 < n_kt) nxt = box_row(kt + 1);
            const int st = kt % kStages;
            if (kt >= kStages) {
                if (!mbar_wait_bounded(&empty[st], (uint32_t)((kt / kStages) - 1) & 1u)) {
                    if (lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
                    return;  // consumers time out on the full barrier in turn
                }
            }
            const unsigned have = __ballot_sync(0xffffffffu, cur != -1);
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st],
                                      (uint32_t)__popc(have) * 2u * L::kPanels * box_bytes);
            __syncwarp();
            if (cur != -1) {
                uint8_t *stg = smem + (size_t)st * L::kStageBytes;
#pragma unroll
                for (int p = 0; p < L::kPanels; ++p) {
                    tma_load_2d_hint(stg + p * L::kPanelBytes + lane * box_rows * 128, &kv_map,
                                     &full[st], 64 * p, cur, policy);
                    tma_load_2d_hint(stg + L::kTileBytes + p * L::kPanelBytes +
                                         lane * box_rows * 128,
                                     &kv_map, &full[st], 64 * p, cur + v_off, policy);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int sub = a.q_tile / 16;           // 16-token sub-tiles per query tile
    const int gh = warp / sub;               // query head inside the group
    const int ts = warp - gh * sub;
    const int hq = h * G + gh;
    const int tw = t0 + ts * 16;             // first token of this warp's rows
    const int r0 = lane >> 2;                // rows r0 and r0+8 of the warp
    // Causal limit of row r: min(ctx + tw + r, len - 1).
    const int lim0 = std::min(ctx + tw + r0, len - 1);
    const int lim1 = std::min(ctx + tw + r0 + 8, len - 1);
    const int warp_lo = std::min(ctx + tw, len - 1);
    const int warp_hi = std::min(ctx + tw + 15, len - 1);

    uint32_t qf[D / 16][4];
    {
        const int ta = tw + r0, tb = tw + r0 + 8;
        const __nv_bfloat16 *qa = a.q + ((size_t)(q0 + ta) * a.num_heads + hq) * D;
        const __nv_bfloat16 *qb = a.q + ((size_t)(q0 + tb) * a.num_heads + hq) * D;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const int d = 16 * k + 2 * (lane & 3);
            qf[k][0] = ta < q_len ? *reinterpret_cast<const uint32_t *>(qa + d) : 0u;
            qf[k][1] = tb < q_len ? *reinterpret_cast<const uint32_t *>(qb + d) : 0u;
            qf[k][2] = ta < q_len ? *reinterpret_cast<const uint32_t *>(qa + d + 8) : 0u;
            qf[k][3] = tb < q_len ? *reinterpret_cast<const uint32_t *>(qb + d + 8) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int st = kt % kStages;
        if (!mbar_wait_bounded(&full[st], (uint32_t)(kt / kStages) & 1u)) {
            if (lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
            return;
        }
        const int k0 = kt * kKeys;
        if (k0 <= warp_hi) {
            const uint32_t kb = smem_u32(smem + (size_t)st * L::kStageBytes);
            const uint32_t vb = kb + L::kTileBytes;
            float sacc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t panel = kb + (k >> 2) * L::kPanelBytes;
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int mi = lane >> 3;
                    const int row = np * 16 + (lane & 7) + (mi >> 1) * 8;
                    const int chunk = 2 * (k & 3) + (mi & 1);
                    uint32_t bf[4];
                    ldsm_x4(bf, swz128(panel, row, chunk));
                    mma_bf16(sacc[2 * np], qf[k], bf[0], bf[1]);
                    mma_bf16(sacc[2 * np + 1], qf[k], bf[2], bf[3]);
                }
            }
            const bool need_mask = (k0 + kKeys - 1 > warp_lo);
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int key = k0 + nt * 8 + 2 * (lane & 3);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float x0 = sacc[nt][e] * a.scale_log2;
                    float x1 = sacc[nt][2 + e] * a.scale_log2;
                    if (need_mask) {
                        x0 = key + e <= lim0 ? x0 : -INFINITY;
                        x1 = key + e <= lim1 ? x1 : -INFINITY;
                    }
                    sacc[nt][e] = x0;
                    sacc[nt][2 + e] = x1;
                    mx0 = fmaxf(mx0, x0);
                    mx1 = fmaxf(mx1, x1);
                }
            }
#pragma unroll
            for (int o_ = 1; o_ < 4; o_ <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float cr0 = fast_exp2(m0 - mn0), cr1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            uint32_t pa[4][4];
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const uint32_t lo = pack_bf16(fast_exp2(sacc[nt][0] - mn0),
                                              fast_exp2(sacc[nt][1] - mn0));
                const uint32_t hi = pack_bf16(fast_exp2(sacc[nt][2] - mn1),
                                              fast_exp2(sacc[nt][3] - mn1));
                rs0 += bf16_lo(lo) + bf16_hi(lo);
                rs1 += bf16_lo(hi) + bf16_hi(hi);
                pa[nt >> 1][(nt & 1) * 2 + 0] = lo;
                pa[nt >> 1][(nt & 1) * 2 + 1] = hi;
            }
#pragma unroll
            for (int o_ = 1; o_ < 4; o_ <<= 1) {
                rs0 += __shfl_xor_sync(0xffffffffu, rs0, o_);
                rs1 += __shfl_xor_sync(0xffffffffu, rs1, o_);
            }
            l0 = l0 * cr0 + rs0;
            l1 = l1 * cr1 + rs1;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= cr0;
                o[i][1] *= cr0;
                o[i][2] *= cr1;
                o[i][3] *= cr1;
            }
            // Keys at or past the sequence end (stale rows, unfetched boxes): their V
            // must contribute exactly zero even if the stale data is not finite.
            const int kv_valid = len - k0;  // keys of this tile inside the sequence
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const uint32_t panel = vb + (dp >> 2) * L::kPanelBytes;
                    const int mi = lane >> 3;
                    const int row = kk * 16 + (lane & 7) + (mi & 1) * 8;
                    const int chunk = 2 * (dp & 3) + (mi >> 1);
                    uint32_t bf[4];
                    ldsm_x4_t(bf, swz128(panel, row, chunk));
                    if (kv_valid < kKeys) {
                        const int kr = kk * 16 + 2 * (lane & 3);
                        const uint32_t m_lo = (kr < kv_valid ? 0xffffu : 0u) |
                                              (kr + 1 < kv_valid ? 0xffff0000u : 0u);
                        const uint32_t m_hi = (kr + 8 < kv_valid ? 0xffffu : 0u) |
                                              (kr + 9 < kv_valid ? 0xffff0000u : 0u);
                        bf[0] &= m_lo;
                        bf[1] &= m_hi;
                        bf[2] &= m_lo;
                        bf[3] &= m_hi;
                    }
                    mma_bf16(o[2 * dp], pa[kk], bf[0], bf[1]);
                    mma_bf16(o[2 * dp + 1], pa[kk], bf[2], bf[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    // Normalise and store the rows this warp owns.
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    const int ta = tw + r0, tb = tw + r0 + 8;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int d = i * 8 + 2 * (lane & 3);
        if (ta < q_len)
            *reinterpret_cast<uint32_t *>(a.out + ((size_t)(q0 + ta) * a.num_heads + hq) * D + d) =
                pack_bf16(o[i][0] * i0, o[i][1] * i0);
        if (tb < q_len)
            *reinterpret_cast<uint32_t *>(a.out + ((size_t)(q0 + tb) * a.num_heads + hq) * D + d) =
                pack_bf16(o[i][2] * i1, o[i][3] * i1);
    }
}

template <int D>
cudaError_t launch_prefill_d(const PrefillArgs &a, const CUtensorMap &map, dim3 grid,
                             cudaStream_t stream) {
    const size_t smem = prefill_smem_bytes<D>();
    auto kern = prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, (a.warps + 1) * 32, smem, stream>>>(map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t take_error_prefill(unsigned *bits) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_err_prefill, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_prefill, &zero, sizeof(unsigned));
    return e;
}

cudaError_t launch_prefill(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                           int max_q_len, const void *kv_cache, const KvGeom &g, int num_heads,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, float scale, cudaStream_t stream) {
    CUtensorMap map;
    if (!encode_kv_map(&map, kv_cache, g, g.block_size >= 16 ? 16 : g.block_size))
        return cudaErrorInvalidValue;
    PrefillArgs a;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.cu_q_lens = cu_q_lens;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_heads = num_heads;
    a.num_kv_heads = g.num_kv_heads;
    a.group = num_heads / g.num_kv_heads;
    a.block_size = g.block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = g.num_blocks;
    a.q_tile = 16 * (kMaxWarps / a.group);
    a.warps = a.group * (a.q_tile / 16);
    a.scale_log2 = scale * 1.4426950408889634f;
    dim3 grid((unsigned)((max_q_len + a.q_tile - 1) / a.q_tile), (unsigned)g.num_kv_heads,
              (unsigned)num_chunks);
    if (g.head_size == 128) return launch_prefill_d<128>(a, map, grid, stream);
    return launch_prefill_d<64>(a, map, grid, stream);
}

}  // namespace pa
