// pa_decode.cuh - paged decode attention: one query token per sequence.
//
// The method: "Inside vLLM: Anatomy of a High-Throughput LLM Inference System"
// (§Engine core: a sequence's tokens are found through the blocks its block table
// names; §Block size: one block holds K and V of block_size tokens for every KV
// head).  Each sequence's query attends to all its cached tokens.
//
// GB300 design
//   * Work = the flattened list of 16-token tiles over (sequence, KV head).  The
//     list is cut into equal contiguous ranges, one per warp of a persistent grid
//     (152 SMs x W warps), so skewed lengths cost nothing in balance.  A
//     (sequence, head) segment that falls across ranges is finished in pieces whose
//     (max, sum, acc) states are merged by log-sum-exp in a second small kernel;
//     for a shared-prefix batch that kernel merges every segment with the prefix
//     pass's partials, one warp per segment (pa_merge.cuh).
//   * Every warp runs its own pipeline: lane 0 issues 128B-swizzled 2-D TMA
//     copies of the K and V tiles named by the block table into an S-stage ring in
//     shared memory (plus the segment's G query rows with a bulk copy); the warp
//     waits on the stage's mbarrier, computes, and refills the stage.  No
//     CTA-wide synchronisation inside the loop.
//   * Per tile the warp computes S^T = K.Q^T (16 tokens x 8 query heads of the GQA
//     group) with one m16n8k16 bf16 MMA per 16 dims, runs the online softmax in
//     fp32 (log2 domain), transposes P in registers (movmatrix) and accumulates
//     O^T += V^T.P^T with ldmatrix.trans.  The math is a few hundred instructions
//     per 8 KB tile, far below what HBM delivers per SM, so the kernel is
//     HBM-bound.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_merge.cuh"

namespace pa {
namespace {

__device__ unsigned g_err_decode;

// Warps per CTA and ring depth per warp (one CTA per SM).  Measured on GB300:
// 12 warps with one stage each keeps the most bytes in flight for the smallest
// issue cost; more warps help only when the context is served from L2.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 12
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 1
#endif

constexpr int kTile = 16;                        // tokens per tile (the MMA's M)
constexpr int kHeadsPad = 8;                     // query heads per KV head, padded to the MMA's N
constexpr int kDecodeWarps = PA_DECODE_WARPS;
constexpr int kDecodeStages = PA_DECODE_STAGES;
// An FP8 tile is half the bytes, so an FP8 pool gets twice the stages to keep the
// same bytes in flight per warp.
constexpr int kDecodeStagesFp8 = 2 * PA_DECODE_STAGES;
// The running max used as the exponent reference is only raised when a score
// exceeds it by more than this (log2 units), so P stays <= 2^8 and the
// accumulator is rescaled rarely.
constexpr float kRescaleSlack = 8.0f;

// KV8: an FP8 pool (one e4m3 byte per element) instead of bf16.
template <int D, bool KV8 = false>
struct Lay {
    static constexpr int kElemBytes = KV8 ? 1 : 2;
    static constexpr int kElemsPerPanel = 128 / kElemBytes;  // elements in a 128-byte row
    static constexpr int kPanels = D * kElemBytes / 128;     // 128-byte-wide column panels
    static constexpr int kPanelBytes = kTile * 128;    // 16 rows of one panel
    static constexpr int kKvBytes = kPanels * kPanelBytes;
};

// A stage: K panels, V panels, then the segment's G query rows (also used to
// stage a finished segment's output), rounded up to keep stages 1024-aligned.
__host__ __device__ constexpr int q_slot_bytes(int group, int head_size) {
    return (group * head_size * 2 + 1023) / 1024 * 1024;
}

struct DecodeArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *part_acc;   // [2*total_warps][8][D]
    float *part_ml;    // [2*total_warps][8][2]  (max in log2 units, sum)
    int32_t *prefix;   // [num_seqs+1] tile prefix over sequences
    int num_seqs, num_heads, num_kv_heads, group;
    int block_size, max_blocks, num_blocks;
    int total_warps;
    int stage_bytes;   // 2 * K/V tile bytes + query slot
    float scale_log2;  // scale * log2(e)
    float k_scale, v_scale;  // FP8 pool: real K/V = e4m3 value * scale (1 for bf16)
    // Cascade (cs.pre_splits > 0): each sequence's tokens [0, shared_len) are
    // attended by the prefix pass; this kernel covers tokens [shared_len,
    // seq_len).  Every piece of a segment (a segment one warp finishes whole
    // included) leaves its (m, l, acc) record for the cascade merge kernel.
    int shared_len;
    CascadeState cs;
    // Mixed-batch launch: the number of decode CTAs and their total warps were
    // chosen on the device; plan = {ctas, total_warps} (nullptr otherwise).
    const int *plan;
    // Tiles a warp keeps in flight, at most the ring's stages (0: all of them).
    // Fewer than the ring holds when enough SMs stream that HBM is saturated
    // anyway: the bytes in flight then only lengthen every request's queueing,
    // the loads of the kernel's other role included.
    int depth;
    // Segment-per-CTA mode (1): CTA c covers segment c (sequence c / num_kv_heads,
    // KV head c % num_kv_heads), its warps taking equal shares of the segment's
    // tiles; the CTA's last warp to finish merges the pieces and writes the rows
    // (zeros for a sequence of no tokens), so no merge kernel follows.  For
    // batches of at most one segment per SM, each a few tiles long: the split
    // partition would leave a merge launch on the step's critical path.
    int seg_ctas;
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int D, bool KV8 = false, int S = kDecodeStages, int W = kDecodeWarps>
__host__ __device__ constexpr size_t decode_smem_bytes(int num_seqs, int group) {
    return 1024 /* alignment slack */ +
           (size_t)W * S * (2 * Lay<D, KV8>::kKvBytes + q_slot_bytes(group, D)) +
           (size_t)W * S * 8 + (size_t)(2 * num_seqs + 1) * 4;
}

// TMA row of (block, K, head, offset) in the pool viewed as rows of head_size.
__device__ __forceinline__ int kv_row(int blk, int h, int off, const DecodeArgs &a) {
    if (blk < 0 || blk >= a.num_blocks) {
        atomicOr(&g_err_decode, kErrOob);
        return -(1 << 30);  // wholly outside the map: TMA fills zeros, nothing is read
    }
    return ((blk * 2) * a.num_kv_heads + h) * a.block_size + off;
}

// Decode pieces of segment (sequence s, KV head h) under the split kernel's
// partition (the first min(NW, T) warps, equal shares of the T tiles): warps
// g0..g1, and the record of warp g0's piece (its first record unless it began in
// an earlier segment).  n_dec = 0 for a segment with no own tokens.
__device__ __forceinline__ void segment_pieces(const int *prefix, int num_seqs, int Hkv,
                                               long long NW, int s, int h, int &n_dec,
                                               int &rec0) {
    const int pre = prefix[s];
    const int nt = prefix[s + 1] - pre;
    n_dec = 0;
    rec0 = -1;
    if (nt == 0) return;
    const long long T = (long long)prefix[num_seqs] * Hkv;
    const long long NWe = NW < T ? NW : T;
    const long long S0 = (long long)Hkv * pre + (long long)h * nt;
    const long long g0 = div_floor_small((S0 + 1) * NWe - 1, T);
    const long long g1 = div_floor_small((S0 + nt) * NWe - 1, T);
    n_dec = (int)(g1 - g0 + 1);
    rec0 = (int)(g0 * 2 + (g0 * T < S0 * NWe ? 1 : 0));  // floor(g0 T / NWe) < S0
}

// The split-context decode of one CTA (index cta of a grid whose warps number
// total_warps), W warps with an S-stage ring each; called by decode_kernel and by
// the mixed-batch kernel, whose CTAs may have more warps than W: those take part
// in the set-up and its two CTA-wide barriers, then leave.
template <int D, int W, int S, bool KV8>
__device__ __forceinline__ void decode_body(const CUtensorMap &kv_map, const DecodeArgs &a,
                                            int cta, int total_warps) {
    using L = Lay<D, KV8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(align_up(reinterpret_cast<size_t>(smem_raw), 1024));
    const int stage_bytes = a.stage_bytes;
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)W * S * stage_bytes);
    int *s_len = reinterpret_cast<int *>(bars + W * S);
    int *s_pre = s_len + a.num_seqs;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.num_seqs, Hkv = a.num_kv_heads, G = a.group, bs = a.block_size;

    if (tid == 0) prefetch_tensormap(&kv_map);
    // Lengths (clamped to what the table can hold) and the tile prefix over sequences.
    const int max_len = a.max_blocks * bs;
    // s_len holds the tokens this kernel covers: those past the shared prefix.
    const int sh = a.shared_len;
    for (int s = tid; s < B; s += blockDim.x) {
        int len = a.seq_lens[s];
        if (len < sh || len > max_len) {
            atomicOr(&g_err_decode, kErrOob);
            len = len < sh ? sh : max_len;
        }
        s_len[s] = len - sh;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int s = base + lane;
            const int nt = s < B ? (s_len[s] + kTile - 1) / kTile : 0;
            int v = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (s < B) s_pre[s] = carry + v - nt;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_pre[B] = carry;
    }
    if (lane == 0 && warp < W) {
        for (int st = 0; st < S; ++st) mbar_init(&bars[warp * S + st], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (cta == 0)
        for (int s = tid; s <= B; s += blockDim.x) a.prefix[s] = s_pre[s];
    // The merge kernel may be scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (warp >= W) return;
    // This warp's equal share of the flattened tile list.  With fewer tiles than
    // warps only the first T warps take one each, so no warp's range is empty
    // and a segment's pieces are the consecutive warps g0..g1.
    const long long T = (long long)s_pre[B] * Hkv;
    const long long NW = total_warps;
    const long long NWe = NW < T ? NW : (T > 0 ? T : 1);
    const long long g = (long long)cta * W + warp;
    int t_begin = g < NWe ? (int)((g * T) / NWe) : 0;
    int t_end = g < NWe ? (int)(((g + 1) * T) / NWe) : 0;
    if (a.seg_ctas) {
        const int s = cta / Hkv, h = cta - (cta / Hkv) * Hkv;
        const int nt = s_pre[s + 1] - s_pre[s];
        const int ne = nt < W ? nt : W;
        t_begin = t_end = 0;
        if (warp < ne) {
            t_begin = Hkv * s_pre[s] + h * nt + warp * nt / ne;
            t_end = Hkv * s_pre[s] + h * nt + (warp + 1) * nt / ne;
        }
    }
    const int n = t_end - t_begin;
    // Cascade: the prefix pass reads the shared blocks through sequence 0's table,
    // so every other sequence's first shared_len / block_size entries must equal
    // sequence 0's.  The decode warps compare them, a strided share each, and flag
    // a mismatch (the result is then not that of the caller's tables).
    auto check_shared_tables = [&]() {
        if (sh == 0) return;
        const int nsh = sh / bs;
        const long long total = (long long)(B - 1) * nsh;
        for (long long x = g * 32 + lane; x < total; x += NW * 32) {
            const int s = 1 + (int)(x / nsh), i = (int)(x - (long long)(s - 1) * nsh);
            if (a.block_tables[(size_t)s * a.max_blocks + i] != a.block_tables[i])
                atomicOr(&g_err_decode, kErrPrecondition);
        }
    };
    if (n <= 0) {
        check_shared_tables();
        return;
    }

    uint8_t *wring = ring + (size_t)warp * S * stage_bytes;
    uint64_t *wbar = bars + warp * S;

    // Tile descriptors, one tile per lane, for two batches of 32 tiles.
    //   rk0 / rk1: TMA row of the K rows of the tile's first / second box (-1: none)
    //   seg: (sequence << 8) | kv head;   jt: tile index inside the segment
    auto make_desc = [&](int batch, int &rk0, int &rk1, int &seg, int &jt) {
        const int x = t_begin + batch * 32 + lane;
        rk0 = -1;
        rk1 = -1;
        seg = -1;
        jt = 0;
        if (batch * 32 + lane >= n) return;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (Hkv * s_pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        const int s = lo;
        const int nt = s_pre[s + 1] - s_pre[s];
        const int r = x - Hkv * s_pre[s];
        const int h = r / nt;
        const int j = r - h * nt;
        seg = (s << 8) | h;
        jt = j;
        const int32_t *bt = a.block_tables + (size_t)s * a.max_blocks;
        const int tok0 = sh + j * kTile;  // absolute position of the tile's first token
        if (bs >= kTile) {
            rk0 = kv_row(bt[tok0 / bs], h, tok0 % bs, a);
        } else {  // block_size 8: two blocks per tile, the second only if it holds tokens
            rk0 = kv_row(bt[tok0 / bs], h, 0, a);
            if (j * kTile + bs < s_len[s]) rk1 = kv_row(bt[tok0 / bs + 1], h, 0, a);
        }
    };

    int dA0, dA1, dA2, dA3, dB0, dB1, dB2, dB3;
    make_desc(0, dA0, dA1, dA2, dA3);
    make_desc(1, dB0, dB1, dB2, dB3);
    int cur_batch = 0;

    const int box_rows = bs >= kTile ? kTile : bs;
    const uint32_t box_bytes = (uint32_t)box_rows * 128u;
    const uint32_t q_bytes = (uint32_t)G * D * 2u;
    const int v_row_off = Hkv * bs;
    const uint64_t policy = policy_evict_first();
    // Records the merge reads back: kept in L2 ahead of the streamed K/V.
    const uint64_t keep = policy_evict_last();

    auto issue = [&](int i) {
        const bool in_a = (i >> 5) == cur_batch;
        const int src = i & 31;
        const int rk0 = __shfl_sync(0xffffffffu, in_a ? dA0 : dB0, src);
        const int rk1 = __shfl_sync(0xffffffffu, in_a ? dA1 : dB1, src);
        const int seg = __shfl_sync(0xffffffffu, in_a ? dA2 : dB2, src);
        int prev = -1;
        if (i > 0) {
            const bool pa_ = ((i - 1) >> 5) == cur_batch;
            prev = __shfl_sync(0xffffffffu, pa_ ? dA2 : dB2, (i - 1) & 31);
        }
        if (lane == 0) {
            uint8_t *stg = wring + (size_t)(i % S) * stage_bytes;
            uint64_t *bar = wbar + (i % S);
            const bool new_seg = seg != prev;
            const int nbox = rk1 >= 0 ? 2 : 1;
            const uint32_t bytes =
                (uint32_t)(2 * L::kPanels * nbox) * box_bytes + (new_seg ? q_bytes : 0u);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int p = 0; p < L::kPanels; ++p) {
                const int x = L::kElemsPerPanel * p;
                tma_load_2d_hint(stg + p * L::kPanelBytes, &kv_map, bar, x, rk0, policy);
                tma_load_2d_hint(stg + L::kKvBytes + p * L::kPanelBytes, &kv_map, bar, x,
                                 rk0 + v_row_off, policy);
                if (rk1 >= 0) {
                    tma_load_2d_hint(stg + p * L::kPanelBytes + bs * 128, &kv_map, bar, x, rk1,
                                     policy);
                    tma_load_2d_hint(stg + L::kKvBytes + p * L::kPanelBytes + bs * 128, &kv_map,
                                     bar, x, rk1 + v_row_off, policy);
                }
            }
            if (new_seg) {
                const int s = seg >> 8, h = seg & 255;
                bulk_load(stg + 2 * L::kKvBytes,
                          a.q + ((size_t)s * a.num_heads + (size_t)h * G) * D, q_bytes, bar);
            }
        }
    };

    const int ahead = a.depth > 0 && a.depth < S ? a.depth : S;
    const int first_issue = n < ahead ? n : ahead;
    // Launched as a programmatic dependent of the cache write that fills the
    // pool, the set-up above overlaps that write; the pool is read only after it
    // has completed (a no-op in any other launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = 0; i < first_issue; ++i) issue(i);
    int issued = first_issue;
    // While the first tiles are in flight.
    check_shared_tables();

    float acc[D / 16][4];
    uint32_t qf[D / 16][2];
    // Score multipliers (log2 units) of this lane's two score columns (query
    // heads 2t, 2t+1): scale*log2(e), times, for an FP8 pool, k_scale and the
    // power of two that brought the head's query into f16 range.
    float cs0 = a.scale_log2, cs1 = a.scale_log2;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int prev_seg = -1, first_j = 0;
    bool first_piece = true;
    const int hq_row = lane >> 2;          // query head (MMA column) this lane feeds
    const int hh0 = 2 * (lane & 3);        // query heads whose results this lane holds
    const int tr0 = lane >> 2;             // tokens whose scores this lane holds: tr0, tr0+8
    // Output dim of accumulator row tr0 (+8 if hi) of MMA tile mt.
    auto dim_of = [&](int mt, int hi) {
        if constexpr (KV8) return 16 * mt + 2 * tr0 + hi;
        return mt * 16 + tr0 + 8 * hi;
    };

    for (int c = 0; c < n; ++c) {
        const int st = c % S;
        uint8_t *stg = wring + (size_t)st * stage_bytes;
        if (!mbar_wait_bounded(wbar + st, (uint32_t)(c / S) & 1u)) {
            if (lane == 0) atomicOr(&g_err_decode, kErrTimeout);
            // Give the copies still in flight a bounded chance to land, then leave.
            for (int k = c + 1; k < issued; ++k)
                mbar_wait_bounded(wbar + (k % S), (uint32_t)(k / S) & 1u);
            return;
        }
        const int src = c & 31;
        const int seg = __shfl_sync(0xffffffffu, dA2, src);
        const int j = __shfl_sync(0xffffffffu, dA3, src);
        int next_seg = -2;
        if (c + 1 < n) {
            const bool in_a = ((c + 1) >> 5) == cur_batch;
            next_seg = __shfl_sync(0xffffffffu, in_a ? dA2 : dB2, (c + 1) & 31);
        }
        const int s = seg >> 8, h = seg & 255;
        const __nv_bfloat16 *qslot = reinterpret_cast<const __nv_bfloat16 *>(stg + 2 * L::kKvBytes);
        if (seg != prev_seg) {
            if constexpr (!KV8) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    if (hq_row < G) {
                        const __nv_bfloat16 *qr = qslot + hq_row * D + 16 * k + 2 * (lane & 3);
                        qf[k][0] = *reinterpret_cast<const uint32_t *>(qr);
                        qf[k][1] = *reinterpret_cast<const uint32_t *>(qr + 8);
                    } else {
                        qf[k][0] = 0u;
                        qf[k][1] = 0u;
                    }
                }
            } else {
                // f16 operands.  The K fragment of MMA k-slots (2t, 2t+1, 2t+8, 2t+9)
                // holds dims 4t..4t+3 of each 16-dim chunk (one 32-bit word of e4m3
                // codes), so the query fragment takes the same dims.  Each head's
                // query is scaled by a power of two into [1, 2) at its largest
                // element (exact; f16 keeps every bf16 significand), and the
                // scores are scaled back.
                float qv[D / 16][4];
                float mx = 0.f;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    uint2 w = make_uint2(0u, 0u);
                    if (hq_row < G)
                        w = *reinterpret_cast<const uint2 *>(qslot + hq_row * D + 16 * k +
                                                             4 * (lane & 3));
                    qv[k][0] = bf16_lo(w.x);
                    qv[k][1] = bf16_hi(w.x);
                    qv[k][2] = bf16_lo(w.y);
                    qv[k][3] = bf16_hi(w.y);
                    mx = fmax3(mx, fabsf(qv[k][0]), fabsf(qv[k][1]));
                    mx = fmax3(mx, fabsf(qv[k][2]), fabsf(qv[k][3]));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127 : 0;
                ex = max(-126, min(126, ex));
                const float down = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    qf[k][0] = pack_f16(qv[k][0] * down, qv[k][1] * down);
                    qf[k][1] = pack_f16(qv[k][2] * down, qv[k][3] * down);
                }
                const int e0 = __shfl_sync(0xffffffffu, ex, 4 * hh0);
                const int e1 = __shfl_sync(0xffffffffu, ex, 4 * (hh0 + 1));
                const float base = a.scale_log2 * a.k_scale;
                cs0 = base * __uint_as_float((uint32_t)(127 + e0) << 23);
                cs1 = base * __uint_as_float((uint32_t)(127 + e1) << 23);
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            first_j = j;
        }
        const int len = s_len[s];
        const int valid = min(kTile, len - j * kTile);
        bool wrote_smem = false;
        if (valid < kTile) {
            // Stale rows past the sequence end may hold anything (NaN included):
            // zero their V so P=0 contributes exactly nothing.
            const int rows = kTile - valid;
            for (int e = lane; e < rows * 8 * L::kPanels; e += 32) {
                const int p = e / (rows * 8);
                const int rr = (e / 8) % rows;
                const int ch = e & 7;
                *reinterpret_cast<uint4 *>(stg + L::kKvBytes + p * L::kPanelBytes +
                                           (valid + rr) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
            wrote_smem = true;
            __syncwarp();
        }

        // S^T[token][head] = K . Q^T, as two independent accumulation chains
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t kbase = smem_u32(stg);
        if constexpr (!KV8) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t panel = kbase + (k >> 2) * L::kPanelBytes;
                const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int chunk = 2 * (k & 3) + (lane >> 4);
                uint32_t af[4];
                ldsm_x4(af, swz128(panel, row, chunk));
                if (k & 1)
                    mma_bf16(sd, af, qf[k][0], qf[k][1]);
                else
                    mma_bf16(sc, af, qf[k][0], qf[k][1]);
            }
        } else {
            // One ldmatrix.x4 reads 16 tokens x 32 dims of e4m3 codes: per lane a
            // word of 4 codes (dims 4t..4t+3 of a 16-dim chunk) for tokens g, g+8
            // and two chunks; each word becomes the f16 pairs of MMA k-slots
            // (2t, 2t+1) and (2t+8, 2t+9).
            const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2) {
                uint32_t w[4];
                ldsm_x4(w, swz128(kbase, row, 2 * k2 + (lane >> 4)));
                uint32_t af[4], ag[4];
                e4m3x4_to_f16x4(w[0], af[0], af[2]);
                e4m3x4_to_f16x4(w[1], af[1], af[3]);
                e4m3x4_to_f16x4(w[2], ag[0], ag[2]);
                e4m3x4_to_f16x4(w[3], ag[1], ag[3]);
                mma_f16(sc, af, qf[2 * k2][0], qf[2 * k2][1]);
                mma_f16(sd, ag, qf[2 * k2 + 1][0], qf[2 * k2 + 1][1]);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] += sd[e];
        // Scores in log2 units; tokens past the sequence end get -inf.
        float x0 = sc[0] * cs0, x1 = sc[1] * cs1;
        float x2 = sc[2] * cs0, x3 = sc[3] * cs1;
        if (valid < kTile) {
            if (tr0 >= valid) x0 = x1 = -INFINITY;
            if (tr0 + 8 >= valid) x2 = x3 = -INFINITY;
        }
        // The exponent reference m only moves when some score exceeds it by the
        // slack (first tile, sharp rises): one warp vote decides, and only then is
        // the tile max reduced across lanes and the accumulator rescaled.
        const bool grow = fmaxf(x0, x2) > m0 + kRescaleSlack || fmaxf(x1, x3) > m1 + kRescaleSlack;
        float cr0 = 1.f, cr1 = 1.f;
        const bool rescale = __any_sync(0xffffffffu, grow);
        if (rescale) {
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            cr0 = fast_exp2(m0 - mn0);
            cr1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
        }
        // Per-lane partial sums of P in fp32, before its rounding to 16 bits for
        // the P.V product (the rule of every kernel here); the head's 8 lanes are
        // summed once, at the end of the segment.
        const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
        const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
        l0 = l0 * cr0 + (p0 + p2);
        l1 = l1 * cr1 + (p1 + p3);
        const uint32_t plo = KV8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
        const uint32_t phi = KV8 ? pack_f16(p2, p3) : pack_bf16(p2, p3);
        const uint32_t b0 = movmatrix_t(plo), b1 = movmatrix_t(phi);

        // O^T[dim][head] += V^T . P^T
        const uint32_t vbase = kbase + L::kKvBytes;
        if (rescale) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                acc[mt][0] *= cr0;
                acc[mt][1] *= cr1;
                acc[mt][2] *= cr0;
                acc[mt][3] *= cr1;
            }
        }
        if constexpr (!KV8) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const uint32_t panel = vbase + (mt >> 2) * L::kPanelBytes;
                const int mi = lane >> 3;
                const int row = (lane & 7) + (mi >> 1) * 8;
                const int chunk = 2 * (mt & 3) + (mi & 1);
                uint32_t af[4];
                ldsm_x4_t(af, swz128(panel, row, chunk));
                mma_bf16(acc[mt], af, b0, b1);
            }
        } else {
            // V^T fragments from e4m3 codes.  ldmatrix.trans on 16-bit units gives a
            // lane, for tokens 2t, 2t+1 (or 2t+8, 2t+9) and dims 2g, 2g+1 of a 16-dim
            // chunk, the four codes (t0,d0) (t0,d1) (t1,d0) (t1,d1); one byte permute
            // makes them the token pairs of dim 2g and of dim 2g+1, and each pair is
            // one f16x2.  MMA row g of tile mt stands for dim 16 mt + 2g, row g+8 for
            // dim 16 mt + 2g + 1.
            const int mi = lane >> 3;
            const int row = (lane & 7) + (mi & 1) * 8;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t w[4];
                ldsm_x4_t(w, swz128(vbase, row, 2 * q + (mi >> 1)));
                uint32_t af[4], ag[4];
                e4m3x4_to_f16x4(prmt(w[0], 0u, 0x3120u), af[0], af[1]);  // tokens 2t, 2t+1
                e4m3x4_to_f16x4(prmt(w[1], 0u, 0x3120u), af[2], af[3]);  // tokens 2t+8, 2t+9
                e4m3x4_to_f16x4(prmt(w[2], 0u, 0x3120u), ag[0], ag[1]);
                e4m3x4_to_f16x4(prmt(w[3], 0u, 0x3120u), ag[2], ag[3]);
                mma_f16(acc[2 * q], af, b0, b1);
                mma_f16(acc[2 * q + 1], ag, b0, b1);
            }
        }

        if (next_seg != seg) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            if constexpr (KV8) {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][e] *= a.v_scale;
            }
            const int nt = s_pre[s + 1] - s_pre[s];
            const bool whole = first_j == 0 && j == nt - 1;
            if (whole && a.cs.pre_splits == 0) {
                // Whole segment in this warp: normalise and write bf16 rows, staged in
                // the stage's query slot (G rows) for 16-byte stores.  Only the G real
                // heads are staged: the slot holds no room for the padding heads.
                __nv_bfloat16 *stage_out =
                    reinterpret_cast<__nv_bfloat16 *>(stg + 2 * L::kKvBytes);
                const float i0 = 1.f / l0, i1 = 1.f / l1;
                const bool w0 = hh0 < G, w1 = hh0 + 1 < G;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d0 = dim_of(mt, 0), d1 = dim_of(mt, 1);
                    if (w0) {
                        stage_out[hh0 * D + d0] = __float2bfloat16_rn(acc[mt][0] * i0);
                        stage_out[hh0 * D + d1] = __float2bfloat16_rn(acc[mt][2] * i0);
                    }
                    if (w1) {
                        stage_out[(hh0 + 1) * D + d0] = __float2bfloat16_rn(acc[mt][1] * i1);
                        stage_out[(hh0 + 1) * D + d1] = __float2bfloat16_rn(acc[mt][3] * i1);
                    }
                }
                __syncwarp();
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.out + ((size_t)s * a.num_heads + (size_t)h * G) * D);
                const uint4 *srcv = reinterpret_cast<const uint4 *>(stage_out);
                for (int v = lane; v < G * D / 8; v += 32) dst[v] = srcv[v];
                wrote_smem = true;
            } else if (a.seg_ctas) {
                // Segment-per-CTA mode: this warp's piece (its one tile is consumed)
                // stays in its stage, [8 heads][D] of acc then [8 heads] of (m, l),
                // for the CTA's merge after its barrier.
                float *sacc = reinterpret_cast<float *>(stg);
                float *sml = sacc + kHeadsPad * D;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d0 = dim_of(mt, 0), d1 = dim_of(mt, 1);
                    sacc[hh0 * D + d0] = acc[mt][0];
                    sacc[(hh0 + 1) * D + d0] = acc[mt][1];
                    sacc[hh0 * D + d1] = acc[mt][2];
                    sacc[(hh0 + 1) * D + d1] = acc[mt][3];
                }
                if (lane < 4) {
                    sml[hh0 * 2] = m0;
                    sml[hh0 * 2 + 1] = l0;
                    sml[(hh0 + 1) * 2] = m1;
                    sml[(hh0 + 1) * 2 + 1] = l1;
                }
                wrote_smem = true;
            } else {
                // A piece of a split segment, or (cascade) a whole one: unnormalised
                // (m, l, acc) for the merge kernel.
                const size_t rec = (size_t)g * 2 + (first_piece ? 0 : 1);
                const size_t wrec = (size_t)s * Hkv + h;
                float *pacc = whole ? a.cs.whole_acc + wrec * kHeadsPad * D
                                    : a.part_acc + rec * kHeadsPad * D;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d0 = dim_of(mt, 0), d1 = dim_of(mt, 1);
                    st_hint(pacc + hh0 * D + d0, acc[mt][0], keep);
                    st_hint(pacc + (hh0 + 1) * D + d0, acc[mt][1], keep);
                    st_hint(pacc + hh0 * D + d1, acc[mt][2], keep);
                    st_hint(pacc + (hh0 + 1) * D + d1, acc[mt][3], keep);
                }
                if (lane < 4) {
                    float *pml = whole ? a.cs.whole_ml + wrec * kHeadsPad * 2
                                       : a.part_ml + rec * kHeadsPad * 2;
                    st_hint(reinterpret_cast<float2 *>(pml + hh0 * 2), make_float2(m0, l0), keep);
                    st_hint(reinterpret_cast<float2 *>(pml + (hh0 + 1) * 2), make_float2(m1, l1),
                            keep);
                }
            }
            first_piece = false;
        }
        prev_seg = seg;
        if (wrote_smem) fence_proxy_async_smem();
        __syncwarp();
        if (c + ahead < n) {
            issue(c + ahead);
            issued = c + ahead + 1;
        }
        if ((c & 31) == 31) {
            dA0 = dB0;
            dA1 = dB1;
            dA2 = dB2;
            dA3 = dB3;
            ++cur_batch;
            make_desc(cur_batch + 1, dB0, dB1, dB2, dB3);
        }
    }
}

// Segment-per-CTA mode, once every warp of CTA cta has left decode_body: warp 0
// merges the segment's pieces, which the warps left in their stages (warps
// 0 .. ne - 1, one tile each), by log-sum-exp and writes its rows; a segment of
// one tile is already written by its warp, and a sequence of no tokens gets
// zero rows.  The tile counts come from the tables decode_body built in shared
// memory.  Kept out of line: inlined, its registers made the streaming loop of
// every decode kernel spill.
template <int D, int W, int S, bool KV8>
__device__ __noinline__ void seg_cta_merge(const DecodeArgs &a, int cta) {
    __syncthreads();  // every piece's record is in its warp's stage
    if (threadIdx.x >= 32) return;
    extern __shared__ uint8_t smem_raw[];
    const uint8_t *ring =
        reinterpret_cast<const uint8_t *>(align_up(reinterpret_cast<size_t>(smem_raw), 1024));
    const int *s_len = reinterpret_cast<const int *>(ring + (size_t)W * S * a.stage_bytes +
                                                     (size_t)W * S * 8);
    const int *s_pre = s_len + a.num_seqs;
    const int lane = threadIdx.x, G = a.group;
    const int Hkv = a.num_kv_heads, s = cta / Hkv, h = cta - s * Hkv;
    const int nt = s_pre[s + 1] - s_pre[s];
    const int ne = nt < W ? nt : W;
    __nv_bfloat16 *orow = a.out + ((size_t)s * a.num_heads + (size_t)h * G) * D;
    if (nt == 0) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow);
        for (int v = lane; v < G * D / 8; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    if (ne <= 1) return;
    const size_t stride = (size_t)S * a.stage_bytes;  // between two warps' first stages
    for (int e = lane; e < G * D / 4; e += 32) {
        const int hh = e / (D / 4), c4 = 4 * (e - hh * (D / 4));
        float M = -INFINITY;
        for (int k = 0; k < ne; ++k) {
            const float *ml = reinterpret_cast<const float *>(ring + k * stride) + kHeadsPad * D;
            M = fmaxf(M, ml[hh * 2]);
        }
        float den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < ne; ++k) {
            const float *acc = reinterpret_cast<const float *>(ring + k * stride);
            const float *ml = acc + kHeadsPad * D;
            const float w = fast_exp2(ml[hh * 2] - M);
            den += w * ml[hh * 2 + 1];
            const float4 v = *reinterpret_cast<const float4 *>(acc + hh * D + c4);
            num.x += w * v.x;
            num.y += w * v.y;
            num.z += w * v.z;
            num.w += w * v.w;
        }
        const float inv = 1.f / den;
        *reinterpret_cast<uint2 *>(orow + hh * D + c4) =
            make_uint2(pack_bf16(num.x * inv, num.y * inv), pack_bf16(num.z * inv, num.w * inv));
    }
}

template <int D, int W, int S, bool KV8>
__global__ void __launch_bounds__(W * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
    decode_body<D, W, S, KV8>(kv_map, a, blockIdx.x, a.total_warps);
    if (a.seg_ctas) seg_cta_merge<D, W, S, KV8>(a, blockIdx.x);
}

// Merge the pieces of segments that were split across warps; zero empty
// sequences.  One CTA per (sequence, KV head); one thread per (query head, 4
// dims).  Launched as a programmatic dependent of the split kernel: it may start
// early and waits for that grid's completion before reading anything it wrote.
template <int D>
__global__ void __launch_bounds__(kHeadsPad * D / 4) decode_merge_kernel(const DecodeArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int k = blockIdx.x;
    const int Hkv = a.num_kv_heads, G = a.group;
    const int s = k / Hkv, h = k - s * Hkv;
    const int pre = a.prefix[s];
    const int nt = a.prefix[s + 1] - pre;
    const int i = threadIdx.x;
    if (i >= G * D / 4) return;
    const int hh = i / (D / 4), d4 = i - hh * (D / 4);
    uint2 *orow =
        reinterpret_cast<uint2 *>(a.out + ((size_t)s * a.num_heads + (size_t)h * G + hh) * D);
    if (nt == 0) {
        orow[d4] = make_uint2(0u, 0u);
        return;
    }
    // Pieces g0..g1 of this segment, under the split kernel's partition (the
    // first min(NW, T) warps, equal shares).
    const long long NW = a.plan ? a.plan[1] : a.total_warps;
    const long long T = (long long)a.prefix[a.num_seqs] * Hkv;
    const long long NWe = NW < T ? NW : T;
    const long long S0 = (long long)Hkv * pre + (long long)h * nt;
    const long long S1 = S0 + nt;
    const long long g0 = div_floor_small((S0 + 1) * NWe - 1, T);
    const long long g1 = div_floor_small(S1 * NWe - 1, T);
    if (g0 == g1) return;  // written whole by that warp
    // Warp gw covers tiles [floor(gw*T/NWe), floor((gw+1)*T/NWe)); its record of
    // this segment is its first (slot 0) unless it began in an earlier segment.
    const int slot0 = g0 * T < S0 * NWe ? 1 : 0;  // floor(g0 T / NWe) < S0
    float M = -INFINITY;
    for (long long gw = g0; gw <= g1; ++gw) {
        const size_t rec = (size_t)gw * 2 + (gw == g0 ? slot0 : 0);
        M = fmaxf(M, a.part_ml[(rec * kHeadsPad + hh) * 2]);
    }
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (long long gw = g0; gw <= g1; ++gw) {
        const size_t rec = (size_t)gw * 2 + (gw == g0 ? slot0 : 0);
        const float2 ml = reinterpret_cast<const float2 *>(a.part_ml)[rec * kHeadsPad + hh];
        const float4 v =
            reinterpret_cast<const float4 *>(a.part_acc + (rec * kHeadsPad + hh) * D)[d4];
        const float w = exp2f(ml.x - M);
        num.x += w * v.x;
        num.y += w * v.y;
        num.z += w * v.z;
        num.w += w * v.w;
        den += w * ml.y;
    }
    const float inv = 1.f / den;
    orow[d4] = make_uint2(pack_bf16(num.x * inv, num.y * inv), pack_bf16(num.z * inv, num.w * inv));
}

// Batches of at most this many sequences have their tile prefix rebuilt by each
// merge CTA (16 KB of shared memory) instead of read from the decode's table.
constexpr int kMergeOwnPrefix = 4096;

// The cascade's merge as its own launch, one warp per segment; launched as a
// programmatic dependent of the kernel that wrote the records: it waits for that
// grid's completion before reading any record.  What the segment's pieces are
// depends only on the inputs (the lengths) and the decode grid's shape, so for
// batches up to kMergeOwnPrefix sequences each CTA rebuilds the tile prefix of
// the own tokens, clamped exactly as decode_body clamps them, before the wait,
// while the decode grid's last warps still run: after the wait only the records
// are loaded.
template <int D>
__global__ void __launch_bounds__(256) cascade_merge_kernel(const DecodeArgs a) {
    __shared__ int s_pre[kMergeOwnPrefix + 1];
    __shared__ int s_warp[8];
    const int B = a.num_seqs, Hkv = a.num_kv_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = blockIdx.x * 8 + warp;
    const int s = k / Hkv, h = k - (k / Hkv) * Hkv;
    const bool own_prefix = B <= kMergeOwnPrefix && a.plan == nullptr;
    int n_dec = 0, rec0 = -1;
    if (own_prefix) {
        const int per = (B + 255) / 256;  // consecutive sequences per thread
        const int sh = a.shared_len, max_len = a.max_blocks * a.block_size;
        int t[16];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int q = tid * per + i;
            int nt = 0;
            if (i < per && q < B) {
                int len = a.seq_lens[q];
                if (len < sh || len > max_len) len = len < sh ? sh : max_len;
                nt = (len - sh + kTile - 1) / kTile;
            }
            t[i] = nt;
            sum += nt;
        }
        int v = sum;  // inclusive scan over the warp, then over the warps
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) s_warp[warp] = v;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += s_warp[w];
        int run = base + v - sum;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int q = tid * per + i;
            if (i < per && q < B) s_pre[q] = run;
            run += t[i];
        }
        if (tid == 255) s_pre[B] = run;
        __syncthreads();
        if (k < B * Hkv) segment_pieces(s_pre, B, Hkv, a.total_warps, s, h, n_dec, rec0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (k >= B * Hkv) return;
    if (!own_prefix)
        segment_pieces(a.prefix, B, Hkv, a.plan ? a.plan[1] : a.total_warps, s, h, n_dec, rec0);
    merge_segment<D, 4>(a.cs, s, h, n_dec, rec0);
}

// after_write: the kernel just before on the stream is this library's cache write
// of the pool (it triggers its dependents at its start), so the decode launches
// as its programmatic dependent.  Its inputs other than the pool were written
// before that write began.
template <int D, bool KV8>
cudaError_t launch_decode_d(const DecodeArgs &a0, const CUtensorMap &map, int grid,
                            cudaStream_t stream, bool after_write) {
    constexpr int S = KV8 ? kDecodeStagesFp8 : kDecodeStages;
    const size_t smem = decode_smem_bytes<D, KV8, S>(a0.num_seqs, a0.group);
    auto kern = decode_kernel<D, kDecodeWarps, S, KV8>;
    cudaError_t e = ensure_smem<decode_kernel<D, kDecodeWarps, S, KV8>>(smem);
    if (e != cudaSuccess) return e;
    if (after_write) {
        cudaLaunchConfig_t dcfg = {};
        dcfg.gridDim = dim3((unsigned)grid);
        dcfg.blockDim = dim3(kDecodeWarps * 32);
        dcfg.dynamicSmemBytes = smem;
        dcfg.stream = stream;
        cudaLaunchAttribute dattr[1];
        dattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        dattr[0].val.programmaticStreamSerializationAllowed = 1;
        dcfg.attrs = dattr;
        dcfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&dcfg, kern, map, a0);
    } else {
        kern<<<grid, kDecodeWarps * 32, smem, stream>>>(map, a0);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess || a0.seg_ctas) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a0.num_seqs * a0.num_kv_heads));
    cfg.blockDim = dim3((unsigned)(a0.group * D / 4));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a0.cs.pre_splits > 0) {
        cfg.gridDim = dim3((unsigned)((a0.num_seqs * a0.num_kv_heads + 7) / 8));
        cfg.blockDim = dim3(256);
        return cudaLaunchKernelEx(&cfg, cascade_merge_kernel<D>, a0);
    }
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, a0);
}

}  // namespace

int decode_max_seqs(int head_size, int group, bool kv8) {
    const size_t limit = 227 * 1024;
    const size_t fixed = kv8 ? decode_smem_bytes<128, true, kDecodeStagesFp8>(0, group)
                         : head_size == 128 ? decode_smem_bytes<128>(0, group)
                                            : decode_smem_bytes<64>(0, group);
    return fixed >= limit ? 0 : (int)((limit - fixed) / 8);
}

bool decode_seg_ctas(int num_seqs, int num_kv_heads, int max_seq_len, int sm_count) {
    // At most one segment per SM, each at most a tile per warp: a CTA per segment,
    // merged in place (one launch).
    const long long segs = (long long)num_seqs * num_kv_heads;
    const long long seg_tiles = ((long long)std::max(max_seq_len, 1) + kTile - 1) / kTile;
    return segs >= 1 && segs <= sm_count && seg_tiles <= kDecodeWarps;
}

size_t decode_workspace_bytes(int num_seqs, int head_size, int sm_count) {
    const size_t nw = (size_t)sm_count * kDecodeWarps;
    return align_up((size_t)(num_seqs + 1) * 4, 256) + align_up(nw * 2 * kHeadsPad * 2 * 4, 256) +
           align_up(nw * 2 * kHeadsPad * (size_t)head_size * 4, 256);
}

cudaError_t take_error_decode(unsigned *bits) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_err_decode, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_decode, &zero, sizeof(unsigned));
    return e;
}

namespace {

// Arguments of a decode launch over ctas CTAs (workspace carved as
// decode_workspace_bytes lays it out); no cascade, scales 1.
DecodeArgs make_decode_args(void *out, const void *q, const KvGeom &g, int num_heads,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int num_seqs, float scale, void *workspace,
                            bool kv8, int ctas) {
    const int sms = device_sm_count();
    const int D = g.head_size;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t nw_max = (size_t)sms * kDecodeWarps;
    DecodeArgs a;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.prefix = reinterpret_cast<int32_t *>(ws);
    ws += align_up((size_t)(num_seqs + 1) * 4, 256);
    a.part_ml = reinterpret_cast<float *>(ws);
    ws += align_up(nw_max * 2 * kHeadsPad * 2 * 4, 256);
    a.part_acc = reinterpret_cast<float *>(ws);
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = g.num_kv_heads;
    a.group = num_heads / g.num_kv_heads;
    a.block_size = g.block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = g.num_blocks;
    a.total_warps = ctas * kDecodeWarps;
    a.stage_bytes = 2 * (D * (kv8 ? 1 : 2) / 128) * kTile * 128 + q_slot_bytes(a.group, D);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.k_scale = 1.f;
    a.v_scale = 1.f;
    a.shared_len = 0;
    a.cs = CascadeState{};
    a.cs.out = a.out;
    a.cs.part_ml = a.part_ml;
    a.cs.part_acc = a.part_acc;
    a.cs.num_seqs = num_seqs;
    a.cs.num_heads = num_heads;
    a.cs.num_kv_heads = g.num_kv_heads;
    a.cs.group = a.group;
    a.plan = nullptr;
    a.depth = 0;
    a.seg_ctas = 0;
    return a;
}

// Point a's cascade state at the per-segment records (as cascade_whole_bytes
// lays them out) and at the prefix partials.
void set_cascade(DecodeArgs &a, void *whole, const float *pre_ml, const float *pre_acc,
                 int pre_splits) {
    const size_t segs = (size_t)a.num_seqs * a.num_kv_heads;
    uint8_t *w = static_cast<uint8_t *>(whole);
    a.cs.whole_ml = reinterpret_cast<float *>(w);
    a.cs.whole_acc = reinterpret_cast<float *>(w + align_up(segs * kHeadsPad * 2 * 4, 256));
    a.cs.pre_ml = pre_ml;
    a.cs.pre_acc = pre_acc;
    a.cs.pre_splits = pre_splits;
}

cudaError_t launch_decode_impl(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                               int num_heads, const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, int num_seqs, int max_seq_len,
                               int shared_len, float scale, void *workspace, const float *pre_ml,
                               const float *pre_acc, int pre_splits, void *whole, bool kv8,
                               float k_scale, float v_scale, cudaStream_t stream,
                               bool after_write = false) {
    const int sms = device_sm_count();
    const int D = g.head_size;
    CUtensorMap map;
    const int box_rows = g.block_size >= kTile ? kTile : g.block_size;
    if (!(kv8 ? encode_kv_map_fp8(&map, kv_cache, g, box_rows)
              : encode_kv_map(&map, kv_cache, g, box_rows)))
        return cudaErrorInvalidValue;
    // As many warps as there can be tiles, at most one CTA per SM.  A warp has a
    // single stage, so a small batch finishes soonest with one tile per warp; a
    // large one fills every SM and each warp streams its share.
    const long long seg_tiles = (std::max(max_seq_len - shared_len, 1) + kTile - 1) / kTile;
    const long long segs = (long long)num_seqs * g.num_kv_heads;
    const long long tmax = segs * seg_tiles;
    long long ctas = (tmax + kDecodeWarps - 1) / kDecodeWarps;
    ctas = std::max(1LL, std::min<long long>(ctas, sms));
    const bool seg_ctas = !whole && shared_len == 0 && decode_seg_ctas(num_seqs, g.num_kv_heads,
                                                                        max_seq_len, sms);
    if (seg_ctas) ctas = segs;
    DecodeArgs a = make_decode_args(out, q, g, num_heads, block_tables, max_blocks_per_seq,
                                    seq_lens, num_seqs, scale, workspace, kv8, (int)ctas);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.shared_len = shared_len;
    a.seg_ctas = seg_ctas ? 1 : 0;
    if (whole) set_cascade(a, whole, pre_ml, pre_acc, pre_splits);
    if (kv8) return launch_decode_d<128, true>(a, map, (int)ctas, stream, after_write);
    if (D == 128) return launch_decode_d<128, false>(a, map, (int)ctas, stream, after_write);
    return launch_decode_d<64, false>(a, map, (int)ctas, stream, after_write);
}



}  // namespace

cudaError_t launch_decode(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                          int num_heads, const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                          void *workspace, cudaStream_t stream, bool after_write) {
    return launch_decode_impl(out, q, kv_cache, g, num_heads, block_tables, max_blocks_per_seq,
                              seq_lens, num_seqs, max_seq_len, 0, scale, workspace, nullptr,
                              nullptr, 0, nullptr, false, 1.f, 1.f, stream, after_write);
}

cudaError_t launch_decode_fp8(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                              int num_heads, const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                              float k_scale, float v_scale, void *workspace, cudaStream_t stream,
                              bool after_write) {
    return launch_decode_impl(out, q, kv_cache, g, num_heads, block_tables, max_blocks_per_seq,
                              seq_lens, num_seqs, max_seq_len, 0, scale, workspace, nullptr,
                              nullptr, 0, nullptr, true, k_scale, v_scale, stream, after_write);
}

cudaError_t launch_decode_suffix(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                                 int num_heads, const int32_t *block_tables,
                                 int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                                 int max_seq_len, int shared_len, float scale, void *workspace,
                                 const float *pre_ml, const float *pre_acc, int pre_splits,
                                 void *whole, bool kv8, float k_scale, float v_scale,
                                 cudaStream_t stream) {
    return launch_decode_impl(out, q, kv_cache, g, num_heads, block_tables, max_blocks_per_seq,
                              seq_lens, num_seqs, max_seq_len, shared_len, scale, workspace,
                              pre_ml, pre_acc, pre_splits, pre_splits > 0 ? whole : nullptr, kv8,
                              kv8 ? k_scale : 1.f, kv8 ? v_scale : 1.f, stream);
}

size_t prefix_partial_bytes(int splits, int num_seqs, int num_heads, int head_size) {
    const size_t rows = (size_t)splits * num_seqs * num_heads;
    return align_up(rows * 2 * 4, 256) + align_up(rows * (size_t)head_size * 4, 256);
}

size_t cascade_whole_bytes(int num_seqs, int num_kv_heads, int head_size) {
    const size_t segs = (size_t)num_seqs * num_kv_heads;
    return align_up(segs * kHeadsPad * 2 * 4, 256) +
           align_up(segs * kHeadsPad * (size_t)head_size * 4, 256);
}

}  // namespace pa
