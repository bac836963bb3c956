// pa_merge.cuh - the merge of a shared-prefix (cascade) decode.
//
// Prefix caching ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
// System", advanced features) lets a batch's sequences share their first
// shared_len tokens' blocks.  The cascade attends those tokens once per KV head
// for the whole batch (the prefix pass) and each sequence's own tokens apart
// (the decode pieces); softmax states of disjoint key sets combine exactly by
// log-sum-exp.  Every contributor to a segment (one sequence, one KV head)
// leaves its unnormalised (m, l, acc) record; a warp per segment then merges
// them, in one fixed order (decode pieces in warp order, then the prefix
// splits), and writes the segment's output rows.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct CascadeState {
    __nv_bfloat16 *out;  // [num_seqs][num_heads][D]
    // Decode pieces of split segments: two records per warp of the decode grid
    // (its first and its last segment), [2 * warps][8][2] (m in log2 units, l)
    // and [2 * warps][8][D] (acc).
    const float *part_ml;
    const float *part_acc;
    // Segments one decode warp holds whole: one record per segment.
    float *whole_ml;   // [num_seqs * num_kv_heads][8][2]
    float *whole_acc;  // [num_seqs * num_kv_heads][8][D]
    // Prefix pass: pre_splits partials per (sequence, query head).
    const float *pre_ml;   // [pre_splits][num_seqs][num_heads][2]
    const float *pre_acc;  // [pre_splits][num_seqs][num_heads][D]
    int num_seqs, num_heads, num_kv_heads, group;
    int pre_splits;        // prefix partials per row (0: no cascade)
};

// Global loads that bypass L1 (records written by other SMs), with an L2
// eviction hint: a record is dead once merged, so its lines go first.
__device__ __forceinline__ float2 ld_cg2(const float *p, uint64_t policy) {
    float2 v;
    asm volatile("ld.global.cg.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
                 : "=f"(v.x), "=f"(v.y)
                 : "l"(p), "l"(policy));
    return v;
}
__device__ __forceinline__ float4 ld_cg4(const float *p, uint64_t policy) {
    float4 v;
    asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// floor(a / b) for 0 <= a < 2^62, 0 < b, when the quotient is below 2^20 (a warp
// index): a single-precision estimate, off by less than one, corrected with
// exact integer products.  A few instructions instead of a 64-bit integer
// division routine (and no FP64, which this GPU runs at a small fraction of its
// FP32 rate).
__device__ __forceinline__ long long div_floor_small(long long a, long long b) {
    long long q = (long long)((float)a / (float)b);
    if (q < 0) q = 0;
#pragma unroll 1
    while (q * b > a) --q;
#pragma unroll 1
    while ((q + 1) * b <= a) ++q;
    return q;
}

// Merge segment (s, h) from its n_dec decode records (the whole-segment record if
// n_dec == 1; else the piece at record rec0, then slot 0 of each following warp)
// and the pre_splits prefix partials, by log-sum-exp; write its G output rows in
// bf16.  Called by a whole warp.
//
// Records come RG (at most four) at a time: lane 8k + hh holds the (m, l) of
// record k for query head hh, and each lane loads, for every one of its (head, 4
// dims) slots of the G x D outputs, the RG records' accumulators at once.  So a
// segment of up to RG records costs one round trip: every load is issued before
// any is used (RG = 2 where registers are scarce).  The reference max M, the weights 2^(m - M) and the denominator are
// computed once per (record, head) in the lane that holds its (m, l), and each
// slot takes its weight by one shuffle.  More than four records (long segments,
// several prefix splits) take a first pass over their (m, l) for M.  Every
// record keeps head hh's (m, l) at base_ml + 2 hh and its acc at base_acc + D hh.
template <int D, int RG = 4>
__device__ __forceinline__ void merge_segment(const CascadeState &c, int s, int h, int n_dec,
                                              int rec0) {
    const int lane = threadIdx.x & 31;
    const int G = c.group;
    const size_t seg = (size_t)s * c.num_kv_heads + h;
    const int R = n_dec + c.pre_splits;
    const size_t prow = (size_t)s * c.num_heads + (size_t)h * G;  // first query row
    const size_t pstride = (size_t)c.num_seqs * c.num_heads;     // between prefix splits
    auto rec_off = [&](int k) -> size_t {  // record index within its array
        if (k < n_dec) return n_dec == 1 ? seg : (k == 0 ? (size_t)rec0 : (size_t)(rec0 / 2 + k) * 2);
        return (size_t)(k - n_dec) * pstride + prow;
    };
    auto base_ml = [&](int k) -> const float * {
        if (k < n_dec) return (n_dec == 1 ? c.whole_ml : c.part_ml) + rec_off(k) * 16;
        return c.pre_ml + rec_off(k) * 2;
    };
    auto base_acc = [&](int k) -> const float * {
        if (k < n_dec) return (n_dec == 1 ? c.whole_acc : c.part_acc) + rec_off(k) * 8 * D;
        return c.pre_acc + rec_off(k) * D;
    };
    constexpr int kQuads = D / 4;
    const int nslot = (G * kQuads + 31) / 32;
    const int kk = lane >> 3, hh = lane & 7;  // the (m, l) this lane holds: record kk, head hh
    const uint64_t drop = policy_evict_first();
    int hi[8], off[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane;
        hi[i] = idx / kQuads < G ? idx / kQuads : 0;  // slots past G heads read head 0
        off[i] = hi[i] * D + 4 * (idx % kQuads);
    }
    // The first four records' accumulators and (m, l) are all requested before
    // any is used.
    float4 v[RG][8];
    auto load_group = [&](int k0, int nk) {
#pragma unroll
        for (int j = 0; j < RG; ++j) {
            const float *a = base_acc(k0 + (j < nk ? j : 0));
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < nslot && j < nk) v[j][i] = ld_cg4(a + off[i], drop);
        }
    };
    auto load_ml = [&](int k0, int nk) {
        return kk < nk && hh < G ? ld_cg2(base_ml(k0 + kk) + 2 * hh, drop)
                                 : make_float2(-INFINITY, 0.f);
    };
    const int nk0 = R < RG ? R : RG;
    load_group(0, nk0);
    const float2 ml0 = load_ml(0, nk0);
    // Reference max per head over all records: lane (kk, hh) covers records
    // kk, kk + 4, ... (the first of them already in ml0 when kk < nk0).
    float M = -INFINITY;
    for (int k = kk; k < R; k += 4)
        M = fmaxf(M, k < nk0 ? ml0.x
                             : (hh < G ? ld_cg2(base_ml(k) + 2 * hh, drop).x : -INFINITY));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
    float4 num[8];
    float den = 0.f;  // this lane's share of its head's denominator
#pragma unroll
    for (int i = 0; i < 8; ++i) num[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fold_group = [&](int nk, const float2 ml) {
        const float w = kk < nk && hh < G ? fast_exp2(ml.x - M) : 0.f;
        den += w * ml.y;
#pragma unroll
        for (int j = 0; j < RG; ++j) {
            if (j >= nk) break;  // warp-uniform
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float wj = __shfl_sync(0xffffffffu, w, 8 * j + hi[i]);
                if (i < nslot) {
                    num[i].x += wj * v[j][i].x;
                    num[i].y += wj * v[j][i].y;
                    num[i].z += wj * v[j][i].z;
                    num[i].w += wj * v[j][i].w;
                }
            }
        }
    };
    fold_group(nk0, ml0);
    for (int k0 = RG; k0 < R; k0 += RG) {
        const int nk = R - k0 < RG ? R - k0 : RG;
        load_group(k0, nk);
        fold_group(nk, load_ml(k0, nk));
    }
    den += __shfl_xor_sync(0xffffffffu, den, 8);
    den += __shfl_xor_sync(0xffffffffu, den, 16);
    const float inv_h = 1.f / den;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float inv = __shfl_sync(0xffffffffu, inv_h, hi[i]);
        const int idx = i * 32 + lane;
        if (i < nslot && idx / kQuads < G) {
            uint2 *orow = reinterpret_cast<uint2 *>(c.out + (prow + idx / kQuads) * D);
            orow[idx % kQuads] = make_uint2(pack_bf16(num[i].x * inv, num[i].y * inv),
                                            pack_bf16(num[i].z * inv, num[i].w * inv));
        }
    }
}

}  // namespace pa
