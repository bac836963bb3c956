// pa_merge.cuh - the last-arriver merge of a shared-prefix (cascade) decode.
//
// Prefix caching ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
// System", advanced features) lets a batch's sequences share their first
// shared_len tokens' blocks.  The cascade attends those tokens once per KV head
// for the whole batch (the prefix pass) and each sequence's own tokens apart
// (the decode pieces); softmax states of disjoint key sets combine exactly by
// log-sum-exp.  Here no separate merge launch combines them: every contributor
// to a segment (one sequence, one KV head) leaves its unnormalised (m, l, acc)
// record and then counts its arrival in the segment's counter; the one whose
// arrival completes the count merges all the segment's records and writes its
// output rows.  Nobody waits for anybody.
//
// Counting without knowing how many will arrive: the decode warp holding the
// segment's first tile knows how many decode pieces the segment has (n) and
// whether the prefix pass counts as an arrival (p, 1 when it runs in the same
// launch, 0 when its partials were complete before the launch).  It adds
// kArrivalsDone - n - p + 1, every other contributor adds 1; the sum reaches
// kArrivalsDone exactly when everyone has arrived, and no partial sum does
// (without the first piece the sum is at most n + p - 1, with it at most
// kArrivalsDone - 1 until the last arrival).  So the prefix pass needs no
// knowledge of the decode's split.  Counters start at zero (cleared before the
// launch).
//
// Records are read back in one fixed order (decode pieces in warp order, then
// the prefix splits), whoever merges, so the result does not depend on which
// contributor arrived last.
#pragma once

#include "pa_common.cuh"

namespace pa {

constexpr unsigned kArrivalsDone = 1u << 30;

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
    // Per segment: (record index of the first decode piece, or -1 for a whole
    // segment's record; number of decode pieces), written by the warp holding
    // the segment's first tile before it arrives.
    int2 *seg_info;
    unsigned *seg_cnt;     // per segment: arrivals (zero before the launch)
    int num_seqs, num_heads, num_kv_heads, group;
    int pre_splits;        // prefix partials per row (0: no cascade)
    int prefix_arrives;    // 1: the prefix pass runs in the same launch and counts
};

// Global loads that bypass L1: records written by other SMs during this launch.
__device__ __forceinline__ float2 ld_cg2(const float *p) {
    return __ldcg(reinterpret_cast<const float2 *>(p));
}
__device__ __forceinline__ float4 ld_cg4(const float *p) {
    return __ldcg(reinterpret_cast<const float4 *>(p));
}

// Count one arrival at segment seg (one thread).  True for the arrival that
// completes the count; its caller then merges.  Everything this contributor
// wrote before must be ordered before the call (stores, then a warp or named
// barrier among the writers).  The launch may be a programmatic dependent of the
// kernel that clears the counters: wait for that grid first.
__device__ __forceinline__ bool arrive(unsigned *cnt, unsigned add) {
    __threadfence();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const unsigned old = atomicAdd(cnt, add);
    const bool last = old + add == kArrivalsDone;
    if (last) __threadfence();
    return last;
}

// Merge segment (s, h) from its n_dec decode records (the whole-segment record if
// n_dec == 1; else the piece at record rec0, then slot 0 of each following warp)
// and the pre_splits prefix partials, by log-sum-exp; write its G output rows in
// bf16.  Called by a whole warp.
//
// The merge is latency-bound (a few KB from L2 per record), so it is organised
// around round trips: the (m, l) of up to four records come in one load per
// lane (lane 8k + hh: record k, head hh), and the accumulators of two records
// are in flight at a time, each lane holding up to 8 (head, 4 dims) slots of the
// G x D outputs.  One pass, in record order, with a running reference max per
// slot (the accumulators rescaled when it rises): up to two records cost one
// round trip, up to four two.  Every record keeps head hh's (m, l) at
// base_ml + 2 hh and its acc at base_acc + D hh.  Not inlined: it runs once per
// segment, and its live registers would otherwise be allocated against the
// callers' streaming loops.
template <int D>
__device__ __forceinline__ void merge_segment(const CascadeState &c, int s, int h, int n_dec,
                                           int rec0) {
    const int lane = threadIdx.x & 31;
    const int G = c.group;
    const size_t seg = (size_t)s * c.num_kv_heads + h;
    const int R = n_dec + c.pre_splits;
    const size_t prow = (size_t)s * c.num_heads + (size_t)h * G;  // first query row
    const size_t pstride = (size_t)c.num_seqs * c.num_heads;     // between prefix splits
    // Base of record k: (m, l) of head 0, acc of head 0.
    auto base_ml = [&](int k) -> const float * {
        if (k < n_dec) {
            if (n_dec == 1) return c.whole_ml + seg * 16;
            return c.part_ml + (k == 0 ? (size_t)rec0 : (size_t)(rec0 / 2 + k) * 2) * 16;
        }
        return c.pre_ml + ((size_t)(k - n_dec) * pstride + prow) * 2;
    };
    auto base_acc = [&](int k) -> const float * {
        if (k < n_dec) {
            if (n_dec == 1) return c.whole_acc + seg * 8 * D;
            return c.part_acc + (k == 0 ? (size_t)rec0 : (size_t)(rec0 / 2 + k) * 2) * 8 * D;
        }
        return c.pre_acc + ((size_t)(k - n_dec) * pstride + prow) * D;
    };
    constexpr int kQuads = D / 4;
    const int nslot = (G * kQuads + 31) / 32;
    float4 num[8];
    float den[8], Mr[8];
    int hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane;
        hi[i] = idx / kQuads < G ? idx / kQuads : 0;  // slots past G heads read head 0
        num[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        den[i] = 0.f;
        Mr[i] = -INFINITY;
    }
    // Fold record k (its (m, l) in lane 8 j + head of ml_lane, its acc in v).
    auto fold = [&](int j, const float2 ml_lane, const float4 (&v)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float m = __shfl_sync(0xffffffffu, ml_lane.x, 8 * j + hi[i]);
            const float l = __shfl_sync(0xffffffffu, ml_lane.y, 8 * j + hi[i]);
            if (i < nslot) {
                const float mn = fmaxf(Mr[i], m);
                const float f = Mr[i] == -INFINITY ? 0.f : exp2f(Mr[i] - mn);
                const float w = exp2f(m - mn);
                num[i].x = num[i].x * f + w * v[i].x;
                num[i].y = num[i].y * f + w * v[i].y;
                num[i].z = num[i].z * f + w * v[i].z;
                num[i].w = num[i].w * f + w * v[i].w;
                den[i] = den[i] * f + w * l;
                Mr[i] = mn;
            }
        }
    };
    for (int k0 = 0; k0 < R; k0 += 4) {
        const int nk = R - k0 < 4 ? R - k0 : 4;
        float2 ml = make_float2(-INFINITY, 0.f);
        if ((lane >> 3) < nk && (lane & 7) < G) ml = ld_cg2(base_ml(k0 + (lane >> 3)) + 2 * (lane & 7));
        for (int j = 0; j < nk; j += 2) {
            float4 v0[8], v1[8];
            const float *a0 = base_acc(k0 + j);
            const float *a1 = j + 1 < nk ? base_acc(k0 + j + 1) : a0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < nslot) {
                    const int off = hi[i] * D + 4 * ((i * 32 + lane) % kQuads);
                    v0[i] = ld_cg4(a0 + off);
                    v1[i] = ld_cg4(a1 + off);
                }
            fold(j, ml, v0);
            if (j + 1 < nk) fold(j + 1, ml, v1);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane;
        if (i < nslot && idx / kQuads < G) {
            const float inv = 1.f / den[i];
            uint2 *orow = reinterpret_cast<uint2 *>(c.out + (prow + idx / kQuads) * D);
            orow[idx % kQuads] = make_uint2(pack_bf16(num[i].x * inv, num[i].y * inv),
                                            pack_bf16(num[i].z * inv, num[i].w * inv));
        }
    }
}

// Zero the arrival counters of n segments; launched just before a launch that
// counts (which may start early as its programmatic dependent).
__global__ void __launch_bounds__(256) cascade_clear_kernel(unsigned *cnt, int n) {
    asm volatile("griddepcontrol.launch_dependents;" :::);
    for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256) cnt[i] = 0u;
}

}  // namespace pa
