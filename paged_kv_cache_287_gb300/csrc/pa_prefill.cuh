// pa_prefill.cuh - chunked-prefill attention over a paged KV cache.
//
// Chunked prefill ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
// System", advanced features: a long prompt is split into chunks interleaved with
// generation): a chunk of q_len new tokens, whose K/V were just written to the
// pool, attends causally to its sequence's cached context and to itself.  The
// batch is flattened (§Generate function): chunk s owns query rows
// cu_q_lens[s] .. cu_q_lens[s+1]-1.
//
// Design (tcgen05): one CTA per (two 128-row query tiles, KV head, chunk); a
// tile's rows are its tokens times the G query heads of the KV head, so each K/V
// tile is fetched once for 256 rows of the whole GQA group.
//   warp 0     streams 128-key K/V tiles through the block table with
//              128B-swizzled 2-D TMA copies into a 3-slot K ring and a 2-slot
//              V ring;
//   warps 1, 10  issue tcgen05.mma, one warp per query tile (warp 1 also owns
//              the tensor memory): S_t = Q_t.K^T (A and B K-major from shared
//              memory) and O_t += P_t.V (P from tensor memory, V MN-major);
//   warps 2-5  and 6-9: one warpgroup per query tile, one thread per row: the
//              softmax, P (bf16) written into tensor memory over its own
//              scores, and the final normalisation of O.
// Tensor memory (512 columns x 128 lanes): S_0/P_0 [0,128), S_1/P_1 [128,256),
// O_0 [256,384), O_1 [384,512).  Per K/V tile and query tile: S = Q.K^T as one
// N = 128 product (a 64-key product costs nearly as much: each k step re-reads
// the 128-row A operand), the softmax over all 128 keys (P overwrites the first
// 64 columns of its own scores), and O += P.V in two 64-key parts, the first
// issued while the softmax still works on keys 64-127.  A tile's next scores
// are issued once its P.V is done (P sits where they are written), so each
// tile is a chain scores -> softmax -> P.V -> scores whose length, set mostly
// by the latency of a group of dependent MMAs, bounds the kernel; the other
// tile's chain fills the tensor cores meanwhile.  The two tiles' softmaxes take
// turns (a token passed between the warpgroups): one tile's softmax runs under
// the other tile's products instead of sharing the exponential units with the
// other softmax.  Keys past a row's position are masked; tiles past the CTA's
// causal limit are never fetched.
#pragma once

#include <algorithm>
#include <cmath>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned g_err_prefill;

// The softmax reference max is raised only when a row max exceeds it by more
// than this (log2 units): P stays <= 2^8 and O is rescaled rarely.
constexpr float kTcRescaleSlack = 8.0f;

constexpr int kTcRows = 128;    // query rows per tile (the MMA's M)
constexpr int kTcTiles = 2;     // query tiles per CTA
constexpr int kTcKeys = 128;    // keys per K/V tile
constexpr int kKSlots = 3;      // K ring: a slot frees once both Q.K^T products are done
constexpr int kVSlots = 2;      // V ring: a slot frees once both P.V products are done
// warp 0: TMA producer; warps 2..9: softmax warpgroups; warps 1 and 10: one MMA
// issuer per query tile.  With 11 warps one scheduler holds three, which caps a
// thread at 168 registers.
constexpr int kTcWarps = 3 + 4 * kTcTiles;
constexpr int kTcThreads = kTcWarps * 32;
constexpr uint32_t kTmemCols = 512, kColO = 256;
// Chunks are taken longest cached context first (ranked on the device) when
// there are at most this many; more keep the order of the batch.
constexpr int kRankMax = 256;

struct PrefillArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const int32_t *cu_q_lens;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int num_heads, num_kv_heads, group;
    int block_size, max_blocks, num_blocks;
    int q_tile;        // query tokens per 128-row tile: floor(128 / group)
    int negate_q;      // 1 if the softmax scale is negative (Q is negated instead)
    float scale_log2;  // |scale| * log2(e), at least 1e-30
    // Shared-prefix mode (part_ml != nullptr): the "chunk" is the whole decode
    // batch (row = sequence), every row sees every key of the shared prefix
    // [0, shared_len) held by sequence 0's blocks, split over blockIdx.z in
    // ranges of split_tiles K/V tiles; the unnormalised (m, l, O) of each
    // (split, sequence, query head) go to part_ml / part_acc.
    float *part_ml;    // [splits][num_seqs][num_heads][2]: m (log2 units), l
    float *part_acc;   // [splits][num_seqs][num_heads][D]
    int shared_len, split_tiles, prefix_rows;  // prefix_rows: the batch's sequences
    float k_scale, v_scale;  // FP8 pool: real K/V = e4m3 value * scale (1 for bf16)
};

template <int D>
struct TcLay {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kTcRows * 128;     // 16 KB: one 64-dim panel of a tile
    static constexpr int kQTile = kPanels * kQPanel;
    static constexpr int kQBytes = kTcTiles * kQTile;
    static constexpr int kKvPanel = kTcKeys * 128;
    static constexpr int kKBytes = kPanels * kKvPanel;  // one K (or V) tile
    static constexpr int kOperands = kQBytes + (kKSlots + kVSlots) * kKBytes;
    static constexpr size_t kSmem = 1024 + (size_t)kOperands + 32 * 8;  // + barriers, TMEM slot
};

__device__ __forceinline__ int prefill_row(int blk, int h, int off, const PrefillArgs &a) {
    if (blk < 0 || blk >= a.num_blocks) {
        atomicOr(&g_err_prefill, kErrOob);
        return -(1 << 30);  // wholly outside the map: TMA fills zeros, nothing is read
    }
    return ((blk * 2) * a.num_kv_heads + h) * a.block_size + off;
}

// Bounded wait whose outcome is the same on every lane of the warp (the warp's
// later tcgen05.ld/st are warp-collective, so a timeout must be warp-uniform).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

// One prefill CTA at (virtual) block index bid of a grid of size grid; called by
// prefill_tc_kernel and by the mixed-batch kernel (whose CTAs may have more warps
// than kTcWarps: the extra warps only take part in the CTA-wide barriers).
// KV8: an FP8 (e4m3) pool.  Each K/V tile then lands by TMA in the upper half of
// its ring slot, and the extra warp kTcWarps converts it in place to f16 (every
// e4m3 value is an f16 value), one row per lane: a row's f16 output overwrites
// only that row's codes.  The products run as f16 MMAs; each query row is scaled
// by a power of two into f16 range, and the scores are scaled back with k_scale;
// P is f16, and v_scale multiplies the normalised output.
template <int D, bool KV8 = false>
__device__ __forceinline__ void prefill_body(const CUtensorMap &kv_map, const PrefillArgs &a,
                                             const uint3 bid, const uint3 grid) {
    using L = TcLay<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<size_t>(smem_raw) + 1023) & ~static_cast<size_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sK = smem + L::kQBytes;
    uint8_t *sV = sK + kKSlots * L::kKBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOperands);
    uint64_t *k_full = bars, *k_empty = bars + 3, *v_full = bars + 6, *v_empty = bars + 8;
    // Per query tile t: scores ready, P of keys 0-63 written, P.V done, softmax done (the
    // turn token), P of keys 64-127 written.
    uint64_t *s_full = bars + 10, *p_full = bars + 12, *pv_done = bars + 14, *sm_turn = bars + 16;
    uint64_t *p_hi = bars + 18;
    uint64_t *q_full = bars + 22;  // [2]
    uint64_t *drain = bars + 24;   // [2], one per issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 26);
    // FP8 pool: a tile's codes have landed in its slot's upper half.
    uint64_t *k_staged = bars + 27, *v_staged = bars + 30;
    static_assert(kKSlots <= 3 && kVSlots <= 2 && kTcTiles <= 2,
                  "the fixed barrier offsets above hold 3 K slots, 2 V slots and 2 tiles");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grid (query tile, head, chunk rank): CTAs are dispatched in that order, so
    // the chunk with the longest cached context, and within a chunk the latest
    // query tiles, start first (longest work first keeps the tail short).
    __shared__ int s_ctx[kRankMax];
    __shared__ int s_pick;
    const bool prefix = a.part_ml != nullptr;
    int s = prefix ? 0 : (int)bid.z;
    const int nchunks = grid.z;
    if (!prefix && nchunks <= kRankMax) {
        for (int i = threadIdx.x; i < nchunks; i += blockDim.x)
            s_ctx[i] = a.seq_lens[i] - (a.cu_q_lens[i + 1] - a.cu_q_lens[i]);
        __syncthreads();
        for (int i = threadIdx.x; i < nchunks; i += blockDim.x) {
            const int ci = s_ctx[i];
            int rank = 0;
            for (int k = 0; k < nchunks; ++k) {
                const int ck = s_ctx[k];
                rank += (ck > ci) || (ck == ci && k < i);
            }
            if (rank == (int)bid.z) s_pick = i;
        }
        __syncthreads();
        s = s_pick;
    }
    const int h = bid.y;
    const int qt = grid.x - 1 - bid.x;  // latest query tiles first
    const int q0 = prefix ? 0 : a.cu_q_lens[s];
    const int q_len = prefix ? a.prefix_rows : a.cu_q_lens[s + 1] - q0;
    const int QT = a.q_tile, G = a.group;
    const int t0 = qt * kTcTiles * QT;
    if (t0 >= q_len) return;
    const bool has1 = t0 + QT < q_len;  // the second tile holds at least one token
    // Keys [key0, key0 + len) of the sequence are this CTA's; key indices below
    // are relative to key0.
    int len, ctx, key0 = 0, n_kt;
    if (!prefix) {
        len = a.seq_lens[s];
        const int max_len = a.max_blocks * a.block_size;
        if (len < q_len || len > max_len) {
            if (threadIdx.x == 0) atomicOr(&g_err_prefill, kErrOob);
            len = std::min(std::max(len, q_len), max_len);
        }
        ctx = len - q_len;
        const int t_last = std::min(t0 + kTcTiles * QT, q_len) - 1;
        n_kt = (ctx + t_last + 1 + kTcKeys - 1) / kTcKeys;
    } else {
        key0 = (int)bid.z * a.split_tiles * kTcKeys;
        len = std::min(a.shared_len - key0, a.split_tiles * kTcKeys);
        ctx = len;  // no causal limit: every row sees the whole range
        n_kt = (len + kTcKeys - 1) / kTcKeys;
        if (len <= 0) return;
    }

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kv_map);
        // A K or V slot is free once every active issuer has committed its
        // products that read it.
        const uint32_t issuers = has1 ? 2u : 1u;
        for (int i = 0; i < kKSlots; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], issuers);
        }
        for (int i = 0; i < kVSlots; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], issuers);
        }
        for (int i = 0; i < kTcTiles; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
            mbar_init(&sm_turn[i], 4);
            mbar_init(&p_hi[i], 4);
        }
        for (int i = 0; i < kTcTiles; ++i) {
            mbar_init(&q_full[i], 4);
            mbar_init(&drain[i], 1);
        }
        if (KV8) {
            for (int i = 0; i < kKSlots; ++i) mbar_init(&k_staged[i], 1);
            for (int i = 0; i < kVSlots; ++i) mbar_init(&v_staged[i], 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const int bs = a.block_size;
        const int box_rows = bs >= 16 ? 16 : bs;
        const int nbox = kTcKeys / box_rows;  // 8 or 16 boxes per tile
        const int32_t *bt = a.block_tables + (size_t)s * a.max_blocks;
        const int v_off = a.num_kv_heads * bs;
        const uint64_t policy = policy_evict_first();
        auto box_row = [&](int kt) {
            const int tok = kt * kTcKeys + lane * box_rows;
            if (lane >= nbox) return 0;
            if (tok >= len) return -(1 << 30);  // past the range: TMA fills zeros
            return prefill_row(bt[(key0 + tok) / bs], h, (key0 + tok) % bs, a);
        };
        int nxt = box_row(0);
        int issued = 0;
        // As a programmatic dependent of the cache write that fills the pool (the
        // mixed launch of a step), the set-up above overlapped that write; the
        // pool is read only after it has completed (a no-op in any other launch).
        asm volatile("griddepcontrol.wait;" ::: "memory");
        auto load = [&](uint8_t *dst, uint64_t *bar, int row) {
            if constexpr (KV8) {
                // The tile's codes (128 bytes per key) into the slot's upper half.
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(kTcKeys * 128));
                __syncwarp();
                if (lane < nbox)
                    tma_load_2d_hint(dst + L::kKBytes / 2 + lane * box_rows * 128, &kv_map, bar,
                                     0, row, policy);
            } else {
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)L::kKBytes);
                __syncwarp();
                if (lane < nbox) {
#pragma unroll
                    for (int p = 0; p < L::kPanels; ++p)
                        tma_load_2d_hint(dst + p * L::kKvPanel + lane * box_rows * 128, &kv_map,
                                         bar, 64 * p, row, policy);
                }
            }
        };
        for (int kt = 0; kt < n_kt; ++kt) {
            const int cur = nxt;
            if (kt + 1 < n_kt) nxt = box_row(kt + 1);
            const int ks = kt % kKSlots, vs = kt % kVSlots;
            if (kt >= kKSlots &&
                !warp_wait(&k_empty[ks], (uint32_t)(kt / kKSlots - 1) & 1u)) {
                if (lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
                break;
            }
            load(sK + ks * L::kKBytes, KV8 ? &k_staged[ks] : &k_full[ks], cur);
            if (kt >= kVSlots &&
                !warp_wait(&v_empty[vs], (uint32_t)(kt / kVSlots - 1) & 1u)) {
                if (lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
                issued = -(kt + 1);  // K of tile kt is in flight, V is not
                break;
            }
            load(sV + vs * L::kKBytes, KV8 ? &v_staged[vs] : &v_full[vs],
                 cur < -(1 << 29) ? cur : cur + v_off);
            issued = kt + 1;
        }
        // Never leave with copies in flight into this CTA's shared memory.
        {
            const int last = issued < 0 ? -issued : issued;   // tiles whose K was issued
            const int vlast = issued < 0 ? last - 1 : last;    // tiles whose V was issued
            uint64_t *kb = KV8 ? k_staged : k_full, *vb = KV8 ? v_staged : v_full;
            for (int kt = std::max(0, last - kKSlots); kt < last; ++kt)
                mbar_wait_bounded(&kb[kt % kKSlots], (uint32_t)(kt / kKSlots) & 1u);
            for (int kt = std::max(0, vlast - kVSlots); kt < vlast; ++kt)
                mbar_wait_bounded(&vb[kt % kVSlots], (uint32_t)(kt / kVSlots) & 1u);
        }
    } else if (warp == 1 || (warp == kTcWarps - 1 && has1)) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues for query tile 0, the last warp for tile 1: each waits only
        // on its own tile, so one tile's products never queue behind the other's
        // hand-over, and while one issuer waits for its P.V to finish the other's
        // products keep the tensor cores busy.
        const int t = warp == 1 ? 0 : 1;
        const uint32_t idesc_s =
            KV8 ? tc_idesc_f16(kTcRows, kTcKeys, 0) : tc_idesc_bf16(kTcRows, kTcKeys, 0);
        const uint32_t idesc_pv = KV8 ? tc_idesc_f16(kTcRows, D, 1) : tc_idesc_bf16(kTcRows, D, 1);
        // Operand descriptors are built once: an offset within an operand is added
        // to the start-address field (bits 0-13, address / 16), which cannot carry
        // out since shared-memory addresses stay below 2^18.  The issuing thread's
        // per-product work is then one add, not a descriptor rebuilt from scratch,
        // and the products reach the tensor pipe as fast as it takes them.
        const uint64_t q_desc = tc_desc_sw128(smem_u32(sQ) + t * L::kQTile, 16, 1024);
        const uint64_t k_desc = tc_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t v_desc = tc_desc_sw128(smem_u32(sV), L::kKvPanel, 1024);
        // S_t = Q_t . K_j^T into tensor-memory columns [128 t, 128 t + 128).
        auto issue_s = [&](int j) {
            if (lane == 0) {
                const uint64_t kd = k_desc + (uint64_t)(((j % kKSlots) * L::kKBytes) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t qo = ((k >> 2) * L::kQPanel + (k & 3) * 32) >> 4;
                    const uint32_t ko = ((k >> 2) * L::kKvPanel + (k & 3) * 32) >> 4;
                    tc_mma_ss(tmem + t * kTcRows, q_desc + qo, kd + ko, idesc_s, k > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[t]);
                tc_commit(&k_empty[j % kKSlots]);
            }
            __syncwarp();
        };
        // O_t += P_t . V_j for keys [64 h, 64 h + 64) of the tile; P_t is packed two
        // per column in the first 64 columns of its scores (16 keys per 8 columns).
        auto issue_pv = [&](int j, int h) {
            if (lane == 0) {
                const uint64_t vd = v_desc + (uint64_t)(((j % kVSlots) * L::kKBytes) >> 4);
#pragma unroll
                for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                    tc_mma_ts(tmem + kColO + t * kTcRows, tmem + t * kTcRows + kk * 8,
                              vd + (uint64_t)((kk * 16 * 128) >> 4), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
                if (h == 1) {
                    tc_commit(&pv_done[t]);
                    tc_commit(&v_empty[j % kVSlots]);
                }
            }
            __syncwarp();
        };
        bool ok = warp_wait(&q_full[t], 0) && warp_wait(&k_full[0], 0);
        if (ok) {
            tc_fence_after();
            issue_s(0);
        }
        // O_t += P_t.V_j in two 64-key parts, each as soon as its P is written;
        // once that product is done (P_t sits where S_t is written), S_t for the
        // next K tile.  V_j is waited for before P (it normally arrives far
        // ahead, so the hand-over is not delayed by the check); the next K tile
        // after the P.V is issued (from an FP8 pool it arrives later, through the
        // conversion warp).  The other tile's products run meanwhile.
        for (int j = 0; ok && j < n_kt; ++j) {
            if (!(ok = warp_wait(&v_full[j % kVSlots], (uint32_t)(j / kVSlots) & 1u))) break;
            if (!(ok = warp_wait(&p_full[t], (uint32_t)j & 1u))) break;
            tc_fence_after();
            issue_pv(j, 0);
            if (!(ok = warp_wait(&p_hi[t], (uint32_t)j & 1u))) break;
            tc_fence_after();
            issue_pv(j, 1);
            if (j + 1 < n_kt) {
                if (!(ok = warp_wait(&k_full[(j + 1) % kKSlots],
                                     (uint32_t)((j + 1) / kKSlots) & 1u)))
                    break;
                if (!(ok = warp_wait(&pv_done[t], (uint32_t)j & 1u))) break;
                tc_fence_after();
                issue_s(j + 1);
            }
        }
        if (!ok && lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
        // Wait for every product this thread issued before tensor memory is freed.
        if (lane == 0) tc_commit(&drain[t]);
        __syncwarp();
        mbar_wait_bounded(&drain[t], 0);
    } else if (KV8 && warp == kTcWarps) {
        // ------------------------------------------------------------ e4m3 -> f16
        // A lane converts whole rows (keys) of the tile: reads the row's 128 codes
        // (8 chunks, 128B-swizzled as TMA left them in the upper half), then writes
        // its 128 f16 values into the two 64-dim panels.  Panel 1 is the upper
        // half, and row r of it is exactly the bytes of code row r, which this lane
        // has already read.
        auto convert = [&](uint8_t *slot) {
            const uint8_t *codes = slot + L::kKBytes / 2;
#pragma unroll 1
            for (int r = lane; r < kTcKeys; r += 32) {
                uint4 in[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    in[c] = *reinterpret_cast<const uint4 *>(codes + r * 128 + ((c ^ (r & 7)) << 4));
                asm volatile("" ::: "memory");
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t f[8];
                    e4m3x4_to_f16x4(in[c].x, f[0], f[1]);
                    e4m3x4_to_f16x4(in[c].y, f[2], f[3]);
                    e4m3x4_to_f16x4(in[c].z, f[4], f[5]);
                    e4m3x4_to_f16x4(in[c].w, f[6], f[7]);
                    uint8_t *dst = slot + (c >> 2) * L::kKvPanel + r * 128;
                    const int ch = 2 * (c & 3);
                    *reinterpret_cast<uint4 *>(dst + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<uint4 *>(dst + (((ch + 1) ^ (r & 7)) << 4)) =
                        make_uint4(f[4], f[5], f[6], f[7]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        bool ok = true;
        for (int kt = 0; ok && kt < n_kt; ++kt) {
            const int ks = kt % kKSlots, vs = kt % kVSlots;
            if (!(ok = warp_wait(&k_staged[ks], (uint32_t)(kt / kKSlots) & 1u))) break;
            convert(sK + ks * L::kKBytes);
            if (lane == 0) mbar_arrive(&k_full[ks]);
            if (!(ok = warp_wait(&v_staged[vs], (uint32_t)(kt / kVSlots) & 1u))) break;
            convert(sV + vs * L::kKBytes);
            if (lane == 0) mbar_arrive(&v_full[vs]);
        }
        if (!ok && lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
    } else if (warp >= 2 && warp < 2 + 4 * kTcTiles && ((warp - 2) / 4 == 0 || has1)) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 2) / 4;             // query tile of this warpgroup
        const int row = 32 * (warp & 3) + lane;   // this thread's TMEM lane = query row
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t cs = trow + t * kTcRows;   // this tile's score / P columns
        const uint32_t co = trow + kColO + t * kTcRows;
        const int tok = t * QT + row / G, gq = row % G;
        const bool real = row < QT * G && t0 + tok < q_len;
        // Query row -> shared memory in the 128B-swizzled K-major layout.  Loads
        // are bounds-checked: the host does not know the total number of rows.
        float sl2 = a.scale_log2;  // > 0: a negative scale was moved into Q
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                a.q + ((size_t)(q0 + t0 + tok) * a.num_heads + (size_t)h * G + gq) * D);
            const uint32_t flip = a.negate_q ? 0x80008000u : 0u;  // exact bf16 negation
            uint8_t *qt_smem = sQ + t * L::kQTile;
            if constexpr (!KV8) {
                // Every load is issued before the first store: the stores go through
                // generic pointers the compiler cannot tell apart from the loads', so
                // interleaved they would wait for one global round trip each.
                uint4 v[D / 8];
#pragma unroll
                for (int c = 0; c < D / 8; ++c) v[c] = real ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int p = 0; p < L::kPanels; ++p)
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 w = v[p * 8 + c];
                        w.x ^= flip;
                        w.y ^= flip;
                        w.z ^= flip;
                        w.w ^= flip;
                        *reinterpret_cast<uint4 *>(qt_smem + p * L::kQPanel + row * 128 +
                                                   ((c ^ (row & 7)) << 4)) = w;
                    }
            } else {
                // f16 query: the row times the power of two that puts its largest
                // element in [1, 2) (exact: f16 keeps every bf16 significand); the
                // scores are scaled back, together with k_scale, through sl2.
                uint4 v[D / 8];
                float mx = 0.f;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    v[c] = real ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    v[c].x ^= flip;
                    v[c].y ^= flip;
                    v[c].z ^= flip;
                    v[c].w ^= flip;
                    mx = fmax3(mx, fabsf(bf16_lo(v[c].x)), fabsf(bf16_hi(v[c].x)));
                    mx = fmax3(mx, fabsf(bf16_lo(v[c].y)), fabsf(bf16_hi(v[c].y)));
                    mx = fmax3(mx, fabsf(bf16_lo(v[c].z)), fabsf(bf16_hi(v[c].z)));
                    mx = fmax3(mx, fabsf(bf16_lo(v[c].w)), fabsf(bf16_hi(v[c].w)));
                }
                int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127 : 0;
                ex = max(-126, min(126, ex));
                const float down = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex
                sl2 *= a.k_scale * __uint_as_float((uint32_t)(127 + ex) << 23);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 h4 = make_uint4(
                        pack_f16(bf16_lo(v[c].x) * down, bf16_hi(v[c].x) * down),
                        pack_f16(bf16_lo(v[c].y) * down, bf16_hi(v[c].y) * down),
                        pack_f16(bf16_lo(v[c].z) * down, bf16_hi(v[c].z) * down),
                        pack_f16(bf16_lo(v[c].w) * down, bf16_hi(v[c].w) * down));
                    const int p = c / 8, ch = c % 8;
                    *reinterpret_cast<uint4 *>(qt_smem + p * L::kQPanel + row * 128 +
                                               ((ch ^ (row & 7)) << 4)) = h4;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full[t]);
        }
        const int lim = real && !prefix ? std::min(ctx + t0 + tok, len - 1) : len - 1;
        const int other = has1 ? 1 - t : -1;  // the warpgroup this one takes turns with
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < n_kt; ++j) {
            // Tile 0 goes first: tile 0's softmax of K tile j follows tile 1's of
            // j - 1, and tile 1's follows tile 0's of j.
            if (other >= 0 && (t == 1 || j > 0) &&
                !(ok = warp_wait(&sm_turn[other], (uint32_t)(t == 1 ? j : j - 1) & 1u)))
                break;
            if (!(ok = warp_wait(&s_full[t], (uint32_t)j & 1u))) break;
            tc_fence_after();
            const int k0 = j * kTcKeys;
            float x[kTcKeys];
#pragma unroll
            for (int c = 0; c < kTcKeys / 32; ++c)
                tmem_ld32(cs + 32 * c, *reinterpret_cast<float(*)[32]>(&x[32 * c]));
            tc_wait_ld();
            if (k0 + kTcKeys - 1 > lim) {
                // Diagonal / last keys: those past this row's limit get -inf.
#pragma unroll
                for (int c = 0; c < kTcKeys; ++c)
                    if (k0 + c > lim) x[c] = -INFINITY;
            }
            // The scale is folded into the exponent below, so the max is taken
            // over raw scores (three-input max, four independent chains).
            float r0m = -INFINITY, r1m = -INFINITY, r2m = -INFINITY, r3m = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTcKeys; c += 8) {
                r0m = fmax3(r0m, x[c], x[c + 1]);
                r1m = fmax3(r1m, x[c + 2], x[c + 3]);
                r2m = fmax3(r2m, x[c + 4], x[c + 5]);
                r3m = fmax3(r3m, x[c + 6], x[c + 7]);
            }
            const float mx = fmaxf(fmaxf(r0m, r1m), fmaxf(r2m, r3m)) * sl2;
            const bool grow = mx > m + kTcRescaleSlack;
            const bool rescale = __any_sync(0xffffffffu, grow);
            float cr = 1.f;
            if (rescale) {
                const float mn = grow ? fmaxf(m, mx) : m;
                cr = fast_exp2(m - mn);
                l *= cr;
                m = mn;
            }
            // P = 2^(x*scale - m) <= 2^8, packed two per column into the first 64
            // columns (already read), keys 0-63 first: their P.V starts while keys
            // 64-127 are worked.  Packed fp32 pairs: one FFMA for (x*scale - m) and
            // one add for the row sums per two scores.  The row sum adds the fp32
            // P before its rounding to 16 bits (the rule of every kernel here:
            // summing the rounded values instead costs two more instructions per
            // pair, 3.6 % of this kernel's time on the mixed workload).
            const float nm = -m;
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            auto p_part = [&](int h) {
#pragma unroll
                for (int qr = 2 * h; qr < 2 * h + 2; ++qr) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        float t0, t1, t2, t3;
                        fma2(t0, t1, x[32 * qr + 2 * c], x[32 * qr + 2 * c + 1], sl2, sl2, nm, nm);
                        fma2(t2, t3, x[32 * qr + 2 * c + 2], x[32 * qr + 2 * c + 3], sl2, sl2, nm,
                             nm);
                        const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        const float p2 = fast_exp2(t2), p3 = fast_exp2(t3);
                        add2(s0, s1, p0, p1);
                        add2(s2, s3, p2, p3);
                        pk[c] = KV8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
                        pk[c + 1] = KV8 ? pack_f16(p2, p3) : pack_bf16(p2, p3);
                    }
                    tmem_st16(cs + 16 * qr, pk);
                }
            };
            p_part(0);
            if (rescale && j > 0) {
                // The scores being ready means every earlier P.V of this tile is
                // done (the scores are issued after it), and the next one waits for
                // this warpgroup: O is idle and is rescaled in place.
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(co + 32 * c, o);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= cr;
                    tmem_st32(co + 32 * c, *reinterpret_cast<const uint32_t(*)[32]>(o));
                }
            }
            tc_wait_st();
            if (j * kTcKeys + kTcKeys > len) {
                // Keys at or past the sequence end: zero their V rows so P=0 adds
                // exactly nothing whatever the stale data is.  Each tile's
                // warpgroup zeroes them before its hand-over of the tile (the two
                // write the same zeros), since the two tiles' products are issued
                // independently.
                if (!(ok = warp_wait(&v_full[j % kVSlots], (uint32_t)(j / kVSlots) & 1u)))
                    break;
                const int r0 = len - j * kTcKeys, nr = kTcKeys - r0;
                uint8_t *vs = sV + (size_t)(j % kVSlots) * L::kKBytes;
                for (int e = row; e < nr * 8 * L::kPanels; e += 128) {
                    const int p = e / (nr * 8), rr = (e >> 3) % nr, ch = e & 7;
                    *reinterpret_cast<uint4 *>(vs + p * L::kKvPanel + (r0 + rr) * 128 +
                                               ch * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[t]);
            p_part(1);
            l += (s0 + s1) + (s2 + s3);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&p_hi[t]);
                mbar_arrive(&sm_turn[t]);
            }
        }
        // The last P.V completes after every earlier product of the tile.
        if (ok) ok = warp_wait(&pv_done[t], (uint32_t)(n_kt - 1) & 1u);
        if (!ok) {
            if (lane == 0) atomicOr(&g_err_prefill, kErrTimeout);
        } else {
            tc_fence_after();
            if (prefix) {
                // Unnormalised partial of this (split, sequence, query head); an
                // FP8 pool's v_scale is applied here, as the decode applies it to
                // the pieces it merges with.
                const float vsc = KV8 ? a.v_scale : 1.f;
                const size_t rec =
                    ((size_t)bid.z * q_len + (t0 + tok)) * a.num_heads + (size_t)h * G + gq;
                float4 *pacc = reinterpret_cast<float4 *>(a.part_acc + rec * D);
                const uint64_t keep = policy_evict_last();  // read back by the merge
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(co + 32 * c, o);
                    tc_wait_ld();
                    if (real) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            st_hint(pacc + c * 8 + e,
                                    make_float4(o[4 * e] * vsc, o[4 * e + 1] * vsc,
                                                o[4 * e + 2] * vsc, o[4 * e + 3] * vsc),
                                    keep);
                    }
                }
                if (real)
                    st_hint(reinterpret_cast<float2 *>(a.part_ml) + rec, make_float2(m, l), keep);
            } else {
            const float inv = (KV8 ? a.v_scale : 1.f) / l;
            uint4 *dst = reinterpret_cast<uint4 *>(
                a.out + ((size_t)(q0 + t0 + tok) * a.num_heads + (size_t)h * G + gq) * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(co + 32 * c, o);
                tc_wait_ld();
                if (real) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[c * 4 + e] = make_uint4(
                            pack_bf16(o[8 * e + 0] * inv, o[8 * e + 1] * inv),
                            pack_bf16(o[8 * e + 2] * inv, o[8 * e + 3] * inv),
                            pack_bf16(o[8 * e + 4] * inv, o[8 * e + 5] * inv),
                            pack_bf16(o[8 * e + 6] * inv, o[8 * e + 7] * inv));
                }
            }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool KV8 = false>
__global__ void __launch_bounds__((kTcWarps + (KV8 ? 1 : 0)) * 32, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const PrefillArgs a) {
    prefill_body<D, KV8>(kv_map, a, blockIdx, gridDim);
}

template <int D, bool KV8 = false>
cudaError_t launch_prefill_tc(const PrefillArgs &a, const CUtensorMap &map, dim3 grid,
                              cudaStream_t stream) {
    const size_t smem = TcLay<D>::kSmem;
    auto kern = prefill_tc_kernel<D, KV8>;
    cudaError_t e = ensure_smem<prefill_tc_kernel<D, KV8>>(smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, (kTcWarps + (KV8 ? 1 : 0)) * 32, smem, stream>>>(map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t take_error_prefill(unsigned *bits) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_err_prefill, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_prefill, &zero, sizeof(unsigned));
    return e;
}

namespace {

// Arguments and grid of a chunked-prefill launch.
PrefillArgs make_prefill_args(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                              int max_q_len, const KvGeom &g, int num_heads,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, float scale, dim3 *grid) {
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
    // The kernel folds a positive scale into the exponent; a negative scale is
    // applied by negating Q (exact in bf16), and a zero scale is replaced by a
    // positive value far too small to change any finite score.
    a.negate_q = scale < 0.f ? 1 : 0;
    a.scale_log2 = std::max(std::fabs(scale) * 1.4426950408889634f, 1e-30f);
    a.q_tile = kTcRows / a.group;
    a.part_ml = nullptr;
    a.part_acc = nullptr;
    a.shared_len = a.split_tiles = a.prefix_rows = 0;
    a.k_scale = a.v_scale = 1.f;
    const int per_cta = kTcTiles * a.q_tile;
    *grid = dim3((unsigned)((max_q_len + per_cta - 1) / per_cta), (unsigned)g.num_kv_heads,
                 (unsigned)num_chunks);
    return a;
}

}  // namespace

cudaError_t launch_prefill(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                           int max_q_len, const void *kv_cache, const KvGeom &g, int num_heads,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, float scale, cudaStream_t stream) {
    CUtensorMap map;
    if (!encode_kv_map(&map, kv_cache, g, g.block_size >= 16 ? 16 : g.block_size))
        return cudaErrorInvalidValue;
    dim3 grid;
    const PrefillArgs a = make_prefill_args(out, q, cu_q_lens, num_chunks, max_q_len, g,
                                            num_heads, block_tables, max_blocks_per_seq,
                                            seq_lens, scale, &grid);
    if (g.head_size == 128) return launch_prefill_tc<128>(a, map, grid, stream);
    return launch_prefill_tc<64>(a, map, grid, stream);
}

cudaError_t launch_prefill_fp8(void *out, const void *q, const int32_t *cu_q_lens,
                               int num_chunks, int max_q_len, const void *kv_cache,
                               const KvGeom &g, int num_heads, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, float scale,
                               float k_scale, float v_scale, cudaStream_t stream) {
    CUtensorMap map;
    if (g.head_size != 128 ||
        !encode_kv_map_fp8(&map, kv_cache, g, g.block_size >= 16 ? 16 : g.block_size))
        return cudaErrorInvalidValue;
    dim3 grid;
    PrefillArgs a = make_prefill_args(out, q, cu_q_lens, num_chunks, max_q_len, g, num_heads,
                                      block_tables, max_blocks_per_seq, seq_lens, scale, &grid);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return launch_prefill_tc<128, true>(a, map, grid, stream);
}

int prefix_splits(int num_seqs, int num_heads, int num_kv_heads, int shared_len, int sm_count) {
    if (shared_len <= 0 || num_seqs <= 0) return 0;
    const int group = num_heads / num_kv_heads;
    const int per_cta = kTcTiles * (kTcRows / group);
    const long long ctas = (long long)((num_seqs + per_cta - 1) / per_cta) * num_kv_heads;
    const int tiles = (shared_len + kTcKeys - 1) / kTcKeys;
    // About one wave of CTAs, at least two K/V tiles per CTA.
    long long want = (sm_count + ctas - 1) / ctas;
    want = std::min<long long>(want, std::max(1, tiles / 2));
    const int per = (int)((tiles + want - 1) / want);
    return (tiles + per - 1) / per;
}

cudaError_t launch_prefix_partials(const void *q, const void *kv_cache, const KvGeom &g,
                                   int num_heads, const int32_t *block_tables,
                                   int max_blocks_per_seq, int num_seqs, int shared_len,
                                   float scale, int splits, float *part_ml, float *part_acc,
                                   bool kv8, float k_scale, float v_scale, cudaStream_t stream) {
    CUtensorMap map;
    const int box_rows = g.block_size >= 16 ? 16 : g.block_size;
    if (kv8 ? (g.head_size != 128 || !encode_kv_map_fp8(&map, kv_cache, g, box_rows))
            : !encode_kv_map(&map, kv_cache, g, box_rows))
        return cudaErrorInvalidValue;
    PrefillArgs a;
    a.out = nullptr;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.cu_q_lens = nullptr;
    a.block_tables = block_tables;
    a.seq_lens = nullptr;
    a.num_heads = num_heads;
    a.num_kv_heads = g.num_kv_heads;
    a.group = num_heads / g.num_kv_heads;
    a.block_size = g.block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = g.num_blocks;
    a.negate_q = scale < 0.f ? 1 : 0;
    a.scale_log2 = std::max(std::fabs(scale) * 1.4426950408889634f, 1e-30f);
    a.q_tile = kTcRows / a.group;
    a.part_ml = part_ml;
    a.part_acc = part_acc;
    a.shared_len = shared_len;
    const int tiles = (shared_len + kTcKeys - 1) / kTcKeys;
    a.split_tiles = (tiles + splits - 1) / splits;
    a.prefix_rows = num_seqs;
    a.k_scale = kv8 ? k_scale : 1.f;
    a.v_scale = kv8 ? v_scale : 1.f;
    const int per_cta = kTcTiles * a.q_tile;
    dim3 grid((unsigned)((num_seqs + per_cta - 1) / per_cta), (unsigned)g.num_kv_heads,
              (unsigned)splits);
    if (kv8) return launch_prefill_tc<128, true>(a, map, grid, stream);
    if (g.head_size == 128) return launch_prefill_tc<128>(a, map, grid, stream);
    return launch_prefill_tc<64>(a, map, grid, stream);
}

}  // namespace pa
