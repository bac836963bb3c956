/*
 * CPU fp64 oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library; the product path never does, and this
 * file shares no code, header or constant with the CUDA library.
 *
 * What it restates ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
 * System"):
 *   - §Block size: a KV block of a standard (non-MLA) layer holds K and V for
 *     block_size tokens of every KV head, 2*block_size*num_kv_heads*head_size*
 *     dtype_bytes bytes, bf16 being 2 bytes;
 *   - §Engine core: blocks drawn from a free-block pool are the index that maps
 *     a sequence's tokens to where their K/V live;
 *   - §Generate function: the batch is one flattened token sequence, each
 *     sequence contributing its new (query) tokens.
 * Paging, splitting the context and online softmax are exact reorganisations
 * of ordinary attention, so the oracle is the plain definition: gather each
 * sequence's K/V into logical order, then softmax(q.K^T * scale) V with a
 * causal limit, everything in double precision, sums in token order.
 *
 * Layout (a convention both sides share; the pages do not fix one):
 *   kv_cache  bf16 bits [num_blocks][2][num_kv_heads][block_size][head_size],
 *             index 0 = K, 1 = V;
 *   slot      = physical_block * block_size + offset inside the block;
 *   query head h reads KV head h / (num_heads / num_kv_heads).
 * FP8 pools (the pages name FP8 among the supported quantisation formats and
 * give the block size per dtype byte count): one byte per element in the same
 * layout, each an OCP FP8 E4M3 ("e4m3fn") code; the real value is the code's
 * value times a per-tensor scale (k_scale for K, v_scale for V).  A new row is
 * stored as the e4m3 code nearest to (float)x / scale, ties to the even code,
 * magnitudes beyond the largest finite code (448) saturating to it.
 * Every function here is pinned by the CPU tests (closed forms, brute force
 * on contiguous data, library attention, placement invariance).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * OCP FP8 E4M3 (e4m3fn): sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; exponent 15 with mantissa 7 is NaN; exponent 0 is subnormal,
 * m * 2^-9.  Otherwise (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10).
 */
double oracle_e4m3_to_double(uint8_t code)
{
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/*
 * Nearest e4m3 code to x, ties to the code with an even mantissa (its low bit
 * clear), |x| >= 448 saturating to 448; the sign is kept (so a negative value
 * that rounds to zero gives the negative-zero code); NaN gives the NaN code.
 * Plain search over the 127 non-negative finite codes, whose values increase
 * with the code.
 */
uint8_t oracle_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0;
    for (int c = 0; c <= 0x7E; ++c)
        if (oracle_e4m3_to_double((uint8_t)c) <= a)
            lo = c;
    const double vlo = oracle_e4m3_to_double((uint8_t)lo);
    const double vhi = oracle_e4m3_to_double((uint8_t)(lo + 1));
    const double mid = 0.5 * (vlo + vhi); /* exact: both have few significant bits */
    int c;
    if (a < mid)
        c = lo;
    else if (a > mid)
        c = lo + 1;
    else
        c = (lo & 1) == 0 ? lo : lo + 1;
    return sign | (uint8_t)c;
}

/* §Block size: 2 (key and value) * block_size * num_kv_heads * head_size * dtype bytes. */
size_t oracle_kv_block_bytes(int block_size, int num_kv_heads, int head_size, int dtype_bytes)
{
    return (size_t)2 * (size_t)block_size * (size_t)num_kv_heads * (size_t)head_size *
           (size_t)dtype_bytes;
}

/* Element index of (block, K|V, kv head, offset, dim) in the pool. */
static size_t pool_index(int64_t block, int kv, int head, int offset, int dim,
                         int num_kv_heads, int block_size, int head_size)
{
    return ((((size_t)block * 2 + (size_t)kv) * (size_t)num_kv_heads + (size_t)head) *
                (size_t)block_size + (size_t)offset) * (size_t)head_size + (size_t)dim;
}

/*
 * Cache write: new token i's K and V rows go to slot_mapping[i] (§Engine core:
 * tokens map to the block that holds their KV).  A negative slot is padding
 * and is skipped.  Pure bit copy.  Returns 0, or -1 if a slot lies outside the
 * pool (nothing is written for that row).
 */
int oracle_cache_write(uint16_t *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                       int head_size, const uint16_t *k_new, const uint16_t *v_new,
                       const int32_t *slot_mapping, int num_tokens)
{
    int status = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = -1;
            continue;
        }
        int64_t block = slot / block_size;
        int offset = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_size; ++d) {
                size_t src = ((size_t)i * num_kv_heads + h) * head_size + d;
                kv_cache[pool_index(block, 0, h, offset, d, num_kv_heads, block_size, head_size)] =
                    k_new[src];
                kv_cache[pool_index(block, 1, h, offset, d, num_kv_heads, block_size, head_size)] =
                    v_new[src];
            }
        }
    }
    return status;
}

/*
 * FP8 cache write: as oracle_cache_write, but element x of new token i is
 * stored as oracle_e4m3_from_float((float)x / scale), the division in binary32
 * (k_scale for K, v_scale for V).
 */
int oracle_cache_write_fp8(uint8_t *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                           int head_size, const uint16_t *k_new, const uint16_t *v_new,
                           const int32_t *slot_mapping, int num_tokens, float k_scale,
                           float v_scale)
{
    int status = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = -1;
            continue;
        }
        int64_t block = slot / block_size;
        int offset = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_size; ++d) {
                size_t src = ((size_t)i * num_kv_heads + h) * head_size + d;
                const float k = (float)bf16_bits_to_double(k_new[src]);
                const float v = (float)bf16_bits_to_double(v_new[src]);
                kv_cache[pool_index(block, 0, h, offset, d, num_kv_heads, block_size, head_size)] =
                    oracle_e4m3_from_float(k / k_scale);
                kv_cache[pool_index(block, 1, h, offset, d, num_kv_heads, block_size, head_size)] =
                    oracle_e4m3_from_float(v / v_scale);
            }
        }
    }
    return status;
}

/* Value of pool element idx: bf16 bits, or an e4m3 code times its scale. */
static double pool_value(const void *kv_cache, int fp8, size_t idx, double scale)
{
    if (fp8)
        return oracle_e4m3_to_double(((const uint8_t *)kv_cache)[idx]) * scale;
    return bf16_bits_to_double(((const uint16_t *)kv_cache)[idx]);
}

/*
 * Gather: token t of a sequence lives in block block_table_row[t / block_size]
 * at offset t % block_size (§Engine core).  Writes K and V as contiguous
 * [len][num_kv_heads][head_size] doubles, tokens in logical order.
 * Returns 0, or -1 if a table entry lies outside the pool.
 */
int oracle_gather(double *K, double *V, const uint16_t *kv_cache, int num_blocks,
                  int block_size, int num_kv_heads, int head_size,
                  const int32_t *block_table_row, int len)
{
    for (int t = 0; t < len; ++t) {
        int64_t block = block_table_row[t / block_size];
        if (block < 0 || block >= num_blocks)
            return -1;
        int offset = t % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_size; ++d) {
                size_t dst = ((size_t)t * num_kv_heads + h) * head_size + d;
                K[dst] = bf16_bits_to_double(kv_cache[pool_index(
                    block, 0, h, offset, d, num_kv_heads, block_size, head_size)]);
                V[dst] = bf16_bits_to_double(kv_cache[pool_index(
                    block, 1, h, offset, d, num_kv_heads, block_size, head_size)]);
            }
        }
    }
    return 0;
}

/*
 * One query row against one sequence's gathered K/V.  The row sits at
 * absolute position pos and sees tokens 0..pos (causal); query head h uses KV
 * head g.  x_j = scale * <q, K_j>, m = max_j x_j, w_j = exp(x_j - m),
 * out = sum_j w_j V_j / sum_j w_j, all sums in j order.  No visible token
 * (pos < 0) gives zeros.  x is scratch of at least pos+1 doubles.
 */
static void attend_row(double *out, const uint16_t *q_row, const double *K, const double *V,
                       int pos, int g, int num_kv_heads, int head_size, double scale, double *x)
{
    const int D = head_size;
    if (pos < 0) {
        for (int d = 0; d < D; ++d)
            out[d] = 0.0;
        return;
    }
    double qd[512];
    for (int d = 0; d < D; ++d)
        qd[d] = bf16_bits_to_double(q_row[d]);
    double m = -INFINITY;
    for (int j = 0; j <= pos; ++j) {
        const double *k = K + ((size_t)j * num_kv_heads + g) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qd[d] * k[d];
        x[j] = scale * dot;
        if (x[j] > m)
            m = x[j];
    }
    double denom = 0.0;
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int j = 0; j <= pos; ++j) {
        double w = exp(x[j] - m);
        denom += w;
        const double *v = V + ((size_t)j * num_kv_heads + g) * D;
        for (int d = 0; d < D; ++d)
            out[d] += w * v[d];
    }
    for (int d = 0; d < D; ++d)
        out[d] /= denom;
}

/*
 * Attention for a flattened batch (§Generate function).  Sequence s owns query
 * rows cu_q_lens[s] .. cu_q_lens[s+1]-1 and seq_lens[s] cached tokens, the last
 * q_len of which are its own new tokens, so row i of the sequence sits at
 * position (seq_lens[s] - q_len) + i.  Decode is q_len = 1 (position
 * seq_lens[s]-1); a chunk of a long prompt is q_len > 1 after its cached
 * context (chunked prefill).
 *
 * q:   bf16 bits [total_q][num_heads][head_size]
 * out: doubles [n_out][num_heads][head_size], where the rows computed are
 *      rows[0..num_rows-1] if rows != NULL, else every row in order.
 * Returns 0; -1 on a bad argument or an out-of-pool table entry; -2 on
 * allocation failure.
 */
static int attention_impl(double *out, const uint16_t *q, const int32_t *cu_q_lens,
                          int num_seqs, const void *kv_cache, int kv_fp8, double k_scale,
                          double v_scale, int num_blocks, int block_size, int num_heads,
                          int num_kv_heads, int head_size, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *seq_lens, double scale,
                          const int32_t *rows, int num_rows, int num_threads)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_size <= 0 ||
        head_size > 512 || block_size <= 0)
        return -1;
    const int group = num_heads / num_kv_heads;
    const int total_q = cu_q_lens[num_seqs];
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    /* out_index[r] = where query row r goes in out, or -1 if not requested */
    int *out_index = (int *)malloc(sizeof(int) * (size_t)(total_q > 0 ? total_q : 1));
    if (!out_index)
        return -2;
    for (int r = 0; r < total_q; ++r)
        out_index[r] = rows ? -1 : r;
    if (rows) {
        for (int i = 0; i < num_rows; ++i) {
            if (rows[i] < 0 || rows[i] >= total_q) {
                free(out_index);
                return -1;
            }
            out_index[rows[i]] = i;
        }
    }
    int status = 0;
    for (int s = 0; s < num_seqs && status == 0; ++s) {
        const int r0 = cu_q_lens[s], r1 = cu_q_lens[s + 1];
        int want = 0;
        for (int r = r0; r < r1; ++r)
            want |= out_index[r] >= 0;
        if (!want)
            continue;
        const int len = seq_lens[s];
        const int context = len - (r1 - r0);
        const size_t n_kv = (size_t)(len > 0 ? len : 1) * num_kv_heads * head_size;
        double *K = (double *)malloc(sizeof(double) * n_kv);
        double *V = (double *)malloc(sizeof(double) * n_kv);
        if (!K || !V) {
            free(K);
            free(V);
            status = -2;
            break;
        }
        const int32_t *table = block_tables + (size_t)s * max_blocks_per_seq;
        if (len > 0) {
            /* gather in parallel over blocks of tokens; same result as one pass */
            int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
            for (int t0 = 0; t0 < len; t0 += block_size) {
                int n = len - t0 < block_size ? len - t0 : block_size;
                int64_t block = table[t0 / block_size];
                if (block < 0 || block >= num_blocks) {
                    bad |= 1;
                    continue;
                }
                for (int t = t0; t < t0 + n; ++t)
                    for (int h = 0; h < num_kv_heads; ++h)
                        for (int d = 0; d < head_size; ++d) {
                            size_t dst = ((size_t)t * num_kv_heads + h) * head_size + d;
                            K[dst] = pool_value(kv_cache, kv_fp8,
                                                pool_index(block, 0, h, t - t0, d, num_kv_heads,
                                                           block_size, head_size),
                                                k_scale);
                            V[dst] = pool_value(kv_cache, kv_fp8,
                                                pool_index(block, 1, h, t - t0, d, num_kv_heads,
                                                           block_size, head_size),
                                                v_scale);
                        }
            }
            if (bad) {
                free(K);
                free(V);
                status = -1;
                break;
            }
        }
        const int work = (r1 - r0) * num_heads;
        int no_scratch = 0;
#pragma omp parallel reduction(| : no_scratch)
        {
            double *x = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
            no_scratch |= (x == NULL);
#pragma omp for schedule(dynamic, 1)
            for (int w = 0; w < work; ++w) {
                const int r = r0 + w / num_heads;
                const int h = w % num_heads;
                if (out_index[r] < 0 || !x)
                    continue;
                const int pos = context + (r - r0);
                attend_row(out + ((size_t)out_index[r] * num_heads + h) * head_size,
                           q + ((size_t)r * num_heads + h) * head_size, K, V, pos, h / group,
                           num_kv_heads, head_size, scale, x);
            }
            free(x);
        }
        free(K);
        free(V);
        if (no_scratch)
            status = -2;
    }
    free(out_index);
    return status;
}

int oracle_attention(double *out, const uint16_t *q, const int32_t *cu_q_lens, int num_seqs,
                     const uint16_t *kv_cache, int num_blocks, int block_size, int num_heads,
                     int num_kv_heads, int head_size, const int32_t *block_tables,
                     int max_blocks_per_seq, const int32_t *seq_lens, double scale,
                     const int32_t *rows, int num_rows, int num_threads)
{
    return attention_impl(out, q, cu_q_lens, num_seqs, kv_cache, 0, 1.0, 1.0, num_blocks,
                          block_size, num_heads, num_kv_heads, head_size, block_tables,
                          max_blocks_per_seq, seq_lens, scale, rows, num_rows, num_threads);
}

/*
 * oracle_attention over an FP8 pool: K = e4m3 value * k_scale, V = e4m3 value *
 * v_scale (exact in double), then the same definition.
 */
int oracle_attention_fp8(double *out, const uint16_t *q, const int32_t *cu_q_lens, int num_seqs,
                         const uint8_t *kv_cache, double k_scale, double v_scale, int num_blocks,
                         int block_size, int num_heads, int num_kv_heads, int head_size,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, double scale, const int32_t *rows,
                         int num_rows, int num_threads)
{
    return attention_impl(out, q, cu_q_lens, num_seqs, kv_cache, 1, k_scale, v_scale,
                          num_blocks, block_size, num_heads, num_kv_heads, head_size,
                          block_tables, max_blocks_per_seq, seq_lens, scale, rows, num_rows,
                          num_threads);
}

/* Threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
