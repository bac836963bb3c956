// pa_plan.cuh - the device-side split of a mixed launch's SMs between its decode
// and chunked-prefill roles ("Inside vLLM: Anatomy of a High-Throughput LLM
// Inference System", §Generate function: decode and prefill tokens of one step
// are flattened into one forward pass).  One block computes it: either its own
// one-block launch or one extra block of the cache-write launch that precedes the
// attention launch, so the split costs no launch of its own.
#pragma once

#include "pa_internal.h"

namespace pa {

// Decode bytes and prefill flops of the batch, then the number of decode SMs k
// that makes both parts finish together: min over k of
// max(bytes / min(k * decode rate, HBM), flops / ((sms - k) * prefill rate)).
// fp32 throughout (the choice needs no more; this GPU's fp64 rate is low), the
// search spread over one warp.  Any block of whole warps (32 to 1024 threads).
static __device__ __forceinline__ void mix_plan_block(const MixPlanArgs &a) {
    __shared__ float s_dec[32], s_pre[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;
    float dec = 0.f, pre = 0.f;
    for (int s = tid; s < a.num_seqs; s += nthreads) {
        const long long len = max(0, min(a.seq_lens[s], a.max_len));
        if (s < a.num_prefills) {
            const long long ql = a.cu_q_lens[s + 1] - a.cu_q_lens[s];
            const long long ctx = max(0LL, len - ql);
            pre += (float)(ql * ctx + ql * (ql + 1) / 2);
        } else {
            dec += (float)len;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        dec += __shfl_xor_sync(0xffffffffu, dec, o);
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    if (lane == 0) {
        s_dec[warp] = dec;
        s_pre[warp] = pre;
    }
    __syncthreads();
    if (warp != 0) return;
    dec = lane < (nthreads >> 5) ? s_dec[lane] : 0.f;
    pre = lane < (nthreads >> 5) ? s_pre[lane] : 0.f;
    for (int o = 16; o > 0; o >>= 1) {
        dec += __shfl_xor_sync(0xffffffffu, dec, o);
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    // times in microseconds: bytes / (GB/s * 1e3), flops / (TFLOP/s * 1e6)
    const float bytes = dec * a.dec_bytes_per_token;
    const float flops = pre * a.pre_flops_per_pair;
    int best = 1;
    float best_t = 3.0e38f;
    for (int k = 1 + lane; k < a.sms; k += 32) {
        const float td = bytes / (fminf(k * a.dec_sm_gbs, a.hbm_gbs) * 1e3f);
        const float tp = flops / ((a.sms - k) * a.pre_sm_tflops * 1e6f);
        const float t = fmaxf(td, tp);
        if (t < best_t) {
            best_t = t;
            best = k;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
        const int ok = __shfl_xor_sync(0xffffffffu, best, o);
        if (ot < best_t || (ot == best_t && ok < best)) {
            best_t = ot;
            best = ok;
        }
    }
    if (lane == 0) {
        a.plan[0] = best;
        a.plan[1] = best * a.dec_warps;
    }
}

}  // namespace pa
