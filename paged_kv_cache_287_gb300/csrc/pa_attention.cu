// pa_attention.cu - the attention kernels of libpagedattn in one translation unit:
// decode (pa_decode.cuh), chunked prefill (pa_prefill.cuh), and the single-launch
// kernel for a flattened mixed batch that runs both side by side.
#include <type_traits>

#include "pa_decode.cuh"
#include "pa_plan.cuh"
#include "pa_prefill.cuh"

// ----------------------------------------------------------------------------
// One launch for a flattened mixed batch ("Inside vLLM: Anatomy of a
// High-Throughput LLM Inference System", §Generate function: the forward pass
// flattens the batch into a single sequence).  Decode is bound by HBM and the
// chunked prefill by the tensor-core hand-over chain, so the two run side by
// side on disjoint SMs: the grid's first `sms` CTAs are decode slots, of which
// the first k stream the decode tiles (k chosen on the device, below) and the
// rest exit at once; the remaining CTAs are the prefill's, dispatched onto every
// SM the decode does not hold.  The decode's pieces are merged by the usual
// merge kernel, launched after (not as a programmatic dependent: waiting merge
// CTAs would occupy the SMs the prefill needs).
namespace pa {
namespace {

// Decode CTAs of the mixed launch keep two stages per warp: on part of the GPU
// each SM has to hold twice the bytes in flight.
constexpr int kMixStages = 2;
// An FP8 tile is half the bytes: three stages per warp.
constexpr int kMixStagesFp8 = 3;
// Rates measured on GB300 for the split (bf16 pool): decode with 12 warps x 2
// stages streams about 88 GB/s per SM beside the prefill (whose CTAs start while
// the step's cache write runs), 7.0 TB/s at most in all; chunked prefill does
// about 7.5 TFLOP/s per SM.  On the mixed workload the step is fastest with 56
// decode SMs (433-436 us against 461-466 with 52 and 445 with 60), which these
// rates choose.  FP8 pool: see launch_mixed.
constexpr float kMixDecodeSmGBs = 88.0f, kMixHbmGBs = 7000.0f, kMixPrefillSmTflops = 7.5f;
// FP8 pool: the decode issues about 2.6 times the instructions per byte and
// streams about 46 GB/s per SM on part of the GPU (measured: the mixed step is
// within 1 % of its best for 52 to 70 decode SMs on the mixed workload).
constexpr float kMixDecodeSmGBsFp8 = 46.0f;

// The split as a launch of its own, where no cache write precedes the mixed
// launch.
__global__ void __launch_bounds__(256) mix_plan_kernel(const MixPlanArgs a) {
    mix_plan_block(a);
}

// KV8: an FP8 pool for both roles (the prefill role's converter is warp 11).
// DW: warps of the decode role (12, or 11 where 12 rings of the decode's stages
// would not fit the prefill role's shared memory; the 12th then idles).
template <int D, bool KV8, int DW>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
    mixed_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs da,
                 const PrefillArgs pa, int dec_slots, uint3 pre_grid) {
    if ((int)blockIdx.x < dec_slots) {
        // The plan may come from the cache write this launch depends on.
        if (da.plan) asm volatile("griddepcontrol.wait;" ::: "memory");
        // Without a device plan every decode slot streams (da.total_warps warps).
        const int dec_ctas = da.plan ? da.plan[0] : dec_slots;
        if ((int)blockIdx.x < dec_ctas)
            decode_body<D, DW, KV8 ? kMixStagesFp8 : kMixStages, KV8>(
                kv_map, da, blockIdx.x, da.plan ? da.plan[1] : da.total_warps);
    } else {
        const unsigned v = blockIdx.x - (unsigned)dec_slots;
        const uint3 bid = make_uint3(v % pre_grid.x, (v / pre_grid.x) % pre_grid.y,
                                     v / (pre_grid.x * pre_grid.y));
        prefill_body<D, KV8>(kv_map, pa, bid, pre_grid);
    }
}

// dec_slots: the grid's leading decode CTAs (with a device plan, the first
// plan[0] of them stream and the rest exit).  cascade: a shared-prefix decode,
// whose merge kernel (a warp per segment) follows as a programmatic dependent:
// the grid (one CTA per SM) is resident at once, and the merge CTAs take SMs as
// this grid's CTAs leave them.  Otherwise the plain merge kernel follows as a
// plain launch (the prefill CTAs come in waves, and early merge CTAs would hold
// SMs they need).  after_write: the launch just before on the stream is the
// step's cache write (which triggers its dependents at its start); this launch
// is then its programmatic dependent, and every read of the pool or of the
// plan waits for the write to complete.
template <int D, bool KV8, int DW = kDecodeWarps>
cudaError_t launch_mixed_d(const CUtensorMap &map, const DecodeArgs &da, const PrefillArgs &pa,
                           dim3 pgrid, int dec_slots, size_t smem, cudaStream_t stream,
                           bool cascade = false, bool after_write = false) {
    auto kern = mixed_kernel<D, KV8, DW>;
    cudaError_t e = ensure_smem<mixed_kernel<D, KV8, DW>>(smem);
    if (e != cudaSuccess) return e;
    const unsigned n_pre = pgrid.x * pgrid.y * pgrid.z;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)dec_slots + n_pre);
    cfg.blockDim = dim3(kDecodeWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = after_write ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, map, da, pa, dec_slots,
                           make_uint3(pgrid.x, pgrid.y, pgrid.z));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t mcfg = {};
    mcfg.stream = stream;
    mcfg.attrs = attr;
    if (cascade) {
        mcfg.gridDim = dim3((unsigned)((da.num_seqs * da.num_kv_heads + 7) / 8));
        mcfg.blockDim = dim3(256);
        mcfg.numAttrs = 1;
        return cudaLaunchKernelEx(&mcfg, cascade_merge_kernel<D>, da);
    }
    mcfg.gridDim = dim3((unsigned)(da.num_seqs * da.num_kv_heads));
    mcfg.blockDim = dim3((unsigned)(da.group * D / 4));
    return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<D>, da);
}

}  // namespace

size_t mixed_workspace_bytes(int num_decodes, int head_size, int sm_count) {
    return decode_workspace_bytes(num_decodes, head_size, sm_count) + 256;
}

namespace {

// Warps of the mixed launch's decode role: 12 when their rings fit the prefill
// role's shared memory (which is the launch's), else 11 for a bf16 pool of head
// size 128 (the launch instantiated for that), else 0 (no one launch).
int mixed_decode_warps(int num_decodes, int num_heads, const KvGeom &g, bool kv8) {
    const int G = num_heads / g.num_kv_heads;
    if (kv8 && g.head_size != 128) return 0;
    const size_t pre = g.head_size == 128 ? TcLay<128>::kSmem : TcLay<64>::kSmem;
    auto fits = [&](auto w) {
        constexpr int W = decltype(w)::value;
        const size_t dec =
            kv8 ? decode_smem_bytes<128, true, kMixStagesFp8, W>(num_decodes, G)
            : g.head_size == 128 ? decode_smem_bytes<128, false, kMixStages, W>(num_decodes, G)
                                 : decode_smem_bytes<64, false, kMixStages, W>(num_decodes, G);
        return dec <= pre;
    };
    if (fits(std::integral_constant<int, kDecodeWarps>{})) return kDecodeWarps;
    if (!kv8 && g.head_size == 128 && fits(std::integral_constant<int, kDecodeWarps - 1>{}))
        return kDecodeWarps - 1;
    return 0;
}

}  // namespace

bool mixed_supported(int num_decodes, int num_heads, const KvGeom &g, bool kv8) {
    return mixed_decode_warps(num_decodes, num_heads, g, kv8) > 0;
}

bool mixed_plan_args(MixPlanArgs *pl, const int32_t *cu_q_lens, int num_prefills,
                     const KvGeom &g, int num_heads, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_seqs, void *workspace, bool kv8) {
    const int sms = device_sm_count();
    const int D = g.head_size, num_decodes = num_seqs - num_prefills;
    // The decode's rate per SM scales with its warps (each holds the same bytes
    // in flight).
    const int dw = mixed_decode_warps(num_decodes, num_heads, g, kv8);
    if (dw == 0) return false;
    pl->seq_lens = seq_lens;
    pl->cu_q_lens = cu_q_lens;
    pl->num_prefills = num_prefills;
    pl->num_seqs = num_seqs;
    pl->sms = sms;
    pl->max_len = max_blocks_per_seq * g.block_size;
    pl->dec_bytes_per_token = 2.0f * g.num_kv_heads * D * (kv8 ? 1 : 2);
    pl->pre_flops_per_pair = 4.0f * num_heads * D;
    // FP8 pool (measured on GB300): decode about kMixDecodeSmGBsFp8 per SM with 12
    // warps x 3 stages, 6.3 TB/s at most; the prefill, with its conversion, about
    // 7.1 TFLOP/s per SM.
    pl->dec_warps = dw;
    pl->dec_sm_gbs = (kv8 ? kMixDecodeSmGBsFp8 : kMixDecodeSmGBs) * dw / kDecodeWarps;
    pl->hbm_gbs = kv8 ? 6300.f : kMixHbmGBs;
    pl->pre_sm_tflops = kv8 ? 7.1f : kMixPrefillSmTflops;
    pl->plan = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) +
                                       decode_workspace_bytes(num_decodes, D, sms));
    return true;
}

cudaError_t launch_mixed(void *out, const void *q, const int32_t *cu_q_lens, int num_prefills,
                         int num_prefill_tokens, int max_prefill_q_len, const void *kv_cache,
                         const KvGeom &g, int num_heads, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                         float scale, void *workspace, bool kv8, float k_scale, float v_scale,
                         cudaStream_t stream, bool plan_done, bool after_write) {
    const int sms = device_sm_count();
    const int D = g.head_size, num_decodes = num_seqs - num_prefills;
    CUtensorMap map;
    const int box_rows = g.block_size >= kTile ? kTile : g.block_size;
    if (!(kv8 ? encode_kv_map_fp8(&map, kv_cache, g, box_rows)
              : encode_kv_map(&map, kv_cache, g, box_rows)))
        return cudaErrorInvalidValue;
    MixPlanArgs pl;
    if (!mixed_plan_args(&pl, cu_q_lens, num_prefills, g, num_heads, max_blocks_per_seq,
                         seq_lens, num_seqs, workspace, kv8))
        return cudaErrorInvalidValue;
    const int dw = pl.dec_warps;
    int *plan = pl.plan;
    if (!plan_done) {
        mix_plan_kernel<<<1, 256, 0, stream>>>(pl);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t off = (size_t)num_prefill_tokens * num_heads * D * 2;
    DecodeArgs da = make_decode_args(static_cast<uint8_t *>(out) + off,
                                     static_cast<const uint8_t *>(q) + off, g, num_heads,
                                     block_tables + (size_t)num_prefills * max_blocks_per_seq,
                                     max_blocks_per_seq, seq_lens + num_prefills, num_decodes,
                                     scale, workspace, kv8, sms);
    da.plan = plan;
    da.k_scale = k_scale;
    da.v_scale = v_scale;
    dim3 pgrid;
    PrefillArgs pa =
        make_prefill_args(out, q, cu_q_lens, num_prefills, max_prefill_q_len, g, num_heads,
                          block_tables, max_blocks_per_seq, seq_lens, scale, &pgrid);
    pa.k_scale = k_scale;
    pa.v_scale = v_scale;
    const bool aw = after_write;
    if (kv8)
        return launch_mixed_d<128, true>(map, da, pa, pgrid, sms, TcLay<128>::kSmem, stream,
                                         false, aw);
    if (D == 128 && dw < kDecodeWarps)
        return launch_mixed_d<128, false, kDecodeWarps - 1>(map, da, pa, pgrid, sms,
                                                            TcLay<128>::kSmem, stream, false, aw);
    if (D == 128)
        return launch_mixed_d<128, false>(map, da, pa, pgrid, sms, TcLay<128>::kSmem, stream,
                                          false, aw);
    return launch_mixed_d<64, false>(map, da, pa, pgrid, sms, TcLay<64>::kSmem, stream, false,
                                     aw);
}

// ----------------------------------------------------------------------------
// Shared-prefix decode in one launch of the same kernel.  Once the prefix
// partials are merged by the merge kernel, the prefix pass and the own tokens'
// decode are independent, so they run side by side: the prefix pass on P SMs
// (its CTAs the grid's tail: row groups x KV heads x key splits), the decode on
// the other sms - P as the leading CTAs; then the merge.  The key splits (1 to
// 4) balance the two by the rates below; the one launch is taken when the
// prefix CTAs fit in half the SMs and the prefix pass, so split, does not
// outlast the decode by more than a sixth.  Otherwise the separate launches
// (the prefix pass first, split over the whole GPU) are faster.
namespace {
// Rates for the choice (measured on GB300, prefix-sharing workload, one launch
// with the decode role keeping one tile in flight per warp): a prefix CTA takes
// about 2.5 us per 128-key tile plus 4 us to start and finish, beside a decode
// that keeps HBM busy; the own tokens' decode streams about 50 GB/s per SM.
constexpr float kCascadeTileUs = 2.5f, kCascadeStartUs = 4.0f, kCascadeDecSmGBs = 50.0f;
// FP8 pool: the prefix pass converts each tile (about 2.5 us with it), the
// decode streams about 44 GB/s per SM.
constexpr float kCascadeTileUsFp8 = 2.5f, kCascadeDecSmGBsFp8 = 44.0f;
#ifndef PA_CASCADE_DEPTH
#define PA_CASCADE_DEPTH 1
#endif
constexpr int kCascadeDepth = PA_CASCADE_DEPTH;
}  // namespace

int cascade_one_launch_ctas(int num_seqs, int num_heads, const KvGeom &g, int max_seq_len,
                            int shared_len, bool kv8, int sms, int *splits) {
    if (shared_len <= 0 || num_seqs <= 0) return 0;
    const int G = num_heads / g.num_kv_heads;
    const int per_cta = kTcTiles * (kTcRows / G);
    const long long groups = (long long)((num_seqs + per_cta - 1) / per_cta) * g.num_kv_heads;
    if (mixed_decode_warps(num_seqs, num_heads, g, kv8) == 0) return 0;
    const int tiles = (shared_len + kTcKeys - 1) / kTcKeys;
    // At most as many splits as the workspace holds prefix partials for.
    const int room = prefix_splits(num_seqs, num_heads, g.num_kv_heads, shared_len, sms);
    // Own tokens: about half the longest suffix per sequence on average.
    const double own_bytes = (double)num_seqs * g.num_kv_heads *
                             (0.5 * std::max(max_seq_len - shared_len, 0)) * 2.0 *
                             g.head_size * (kv8 ? 1 : 2);
    const double tile_us = kv8 ? kCascadeTileUsFp8 : kCascadeTileUs;
    const double sm_gbs = kv8 ? kCascadeDecSmGBsFp8 : kCascadeDecSmGBs;
    int best_p = 0;
    double best_t = 0.0, best_pre = 0.0, best_dec = 0.0;
    for (int p = 1; p <= std::min(4, std::min(room, tiles)); ++p) {
        // Every split must hold keys (the merge reads one partial per split).
        if ((tiles + (tiles + p - 1) / p - 1) / ((tiles + p - 1) / p) != p) continue;
        const long long n_pre = groups * p;
        if (n_pre > sms / 2) break;
        const double pre_us = (double)((tiles + p - 1) / p) * tile_us + kCascadeStartUs;
        const double dec_us = own_bytes / ((double)(sms - n_pre) * sm_gbs * 1e3);
        const double t = std::max(pre_us, dec_us);
        if (best_p == 0 || t < best_t) {
            best_p = p;
            best_t = t;
            best_pre = pre_us;
            best_dec = dec_us;
        }
    }
    if (best_p == 0 || best_pre > best_dec * 7.0 / 6.0) return 0;
    if (splits) *splits = best_p;
    return sms - (int)(groups * best_p);
}

cudaError_t launch_cascade_one(void *out, const void *q, const void *kv_cache, const KvGeom &g,
                               int num_heads, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                               int max_seq_len, int shared_len, float scale, void *workspace,
                               float *pre_ml, float *pre_acc, void *whole, bool kv8,
                               float k_scale, float v_scale, cudaStream_t stream) {
    const int sms = device_sm_count();
    const int D = g.head_size, G = num_heads / g.num_kv_heads;
    int splits = 1;
    const int dec_ctas = cascade_one_launch_ctas(num_seqs, num_heads, g, max_seq_len, shared_len,
                                                 kv8, sms, &splits);
    if (dec_ctas == 0) return cudaErrorNotSupported;
    const int dw = mixed_decode_warps(num_seqs, num_heads, g, kv8);
    const int q_tile = kTcRows / G, per_cta = kTcTiles * q_tile;
    const int tiles = (shared_len + kTcKeys - 1) / kTcKeys;

    CUtensorMap map;
    const int box_rows = g.block_size >= kTile ? kTile : g.block_size;
    if (!(kv8 ? encode_kv_map_fp8(&map, kv_cache, g, box_rows)
              : encode_kv_map(&map, kv_cache, g, box_rows)))
        return cudaErrorInvalidValue;
    DecodeArgs da = make_decode_args(out, q, g, num_heads, block_tables, max_blocks_per_seq,
                                     seq_lens, num_seqs, scale, workspace, kv8, dec_ctas);
    da.total_warps = dec_ctas * dw;
    da.k_scale = kv8 ? k_scale : 1.f;
    da.v_scale = kv8 ? v_scale : 1.f;
    da.shared_len = shared_len;
    set_cascade(da, whole, pre_ml, pre_acc, splits);
    // Most SMs stream the own tokens, so one tile in flight per warp (two from an
    // FP8 pool, half the bytes) saturates HBM; more only lengthens the queueing
    // of the prefix pass's loads beside them.
    da.depth = kCascadeDepth + (kv8 ? 1 : 0);
    // The prefix pass: every sequence's query rows against keys [0, shared_len)
    // of sequence 0's blocks, one split.
    PrefillArgs pa;
    pa.out = nullptr;
    pa.q = static_cast<const __nv_bfloat16 *>(q);
    pa.cu_q_lens = nullptr;
    pa.block_tables = block_tables;
    pa.seq_lens = nullptr;
    pa.num_heads = num_heads;
    pa.num_kv_heads = g.num_kv_heads;
    pa.group = G;
    pa.block_size = g.block_size;
    pa.max_blocks = max_blocks_per_seq;
    pa.num_blocks = g.num_blocks;
    pa.negate_q = scale < 0.f ? 1 : 0;
    pa.scale_log2 = std::max(std::fabs(scale) * 1.4426950408889634f, 1e-30f);
    pa.q_tile = q_tile;
    pa.part_ml = pre_ml;
    pa.part_acc = pre_acc;
    pa.shared_len = shared_len;
    pa.split_tiles = (tiles + splits - 1) / splits;
    pa.prefix_rows = num_seqs;
    pa.k_scale = da.k_scale;
    pa.v_scale = da.v_scale;
    const dim3 pgrid((unsigned)((num_seqs + per_cta - 1) / per_cta), (unsigned)g.num_kv_heads,
                     (unsigned)splits);
    if (kv8)
        return launch_mixed_d<128, true>(map, da, pa, pgrid, dec_ctas, TcLay<128>::kSmem, stream,
                                         true);
    if (D == 128 && dw < kDecodeWarps)
        return launch_mixed_d<128, false, kDecodeWarps - 1>(map, da, pa, pgrid, dec_ctas,
                                                            TcLay<128>::kSmem, stream, true);
    if (D == 128)
        return launch_mixed_d<128, false>(map, da, pa, pgrid, dec_ctas, TcLay<128>::kSmem, stream,
                                          true);
    return launch_mixed_d<64, false>(map, da, pa, pgrid, dec_ctas, TcLay<64>::kSmem, stream,
                                     true);
}

}  // namespace pa
