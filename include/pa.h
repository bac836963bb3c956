/*
 * pa.h - C ABI of libpagedattn: attention over a paged KV cache on GB300 (sm_103a).
 *
 * The method is the one "Inside vLLM: Anatomy of a High-Throughput LLM Inference
 * System" describes: KV lives in fixed-size physical blocks drawn from a pool of
 * free blocks (§Engine core, "free_block_queue"); each sequence reaches its tokens'
 * K/V through a block table (§Engine core: blocks are the index from tokens to
 * their KV; §Worker procedures: the input batch holds the block tables); a block
 * of a standard layer holds 2*block_size*num_kv_heads*head_size*dtype_bytes bytes
 * (§Block size); the forward pass sees the batch as one flattened sequence
 * (§Generate function) and long prompts arrive in chunks (chunked prefill, listed
 * under the post's advanced features).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory and never synchronises: every call
 *     only enqueues work on `stream` and returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - bf16 tensors are raw IEEE bfloat16 (2 bytes).  Every bf16 pointer must be
 *     16-byte aligned; integer arrays 4-byte aligned.
 *   - KV pool layout: bf16 [num_blocks][2][num_kv_heads][block_size][head_size],
 *     contiguous; index 0 of the second axis is K, 1 is V.  One physical block is
 *     therefore one contiguous run of pa_kv_block_bytes() bytes.
 *   - A slot is physical_block * block_size + offset_in_block.
 *   - Query head h uses KV head h / (num_heads / num_kv_heads) (grouped-query
 *     attention, contiguous groups).
 *   - Supported shapes: head_size 64 or 128; block_size 8, 16 or 32;
 *     num_heads / num_kv_heads from 1 to 8.  Others return PA_ERR_UNSUPPORTED.
 *   - Host-checkable faults return PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and
 *     enqueue nothing.  A failed launch returns PA_ERR_CUDA.  Device-side data
 *     (slots, block ids, lengths) is a precondition: the kernels check block ids
 *     and slots against the pool, skip what lies outside and record it in a
 *     device error word that pa_error_check() reads (PA_ERR_OOB).  Nothing on
 *     the device traps.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad scale ...   */
    PA_ERR_UNSUPPORTED = 2, /* valid but outside the supported shapes listed above    */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed            */
    PA_ERR_OOB = 4,         /* a kernel met a block id or slot outside the pool       */
    PA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait on its own copies gave up      */
    PA_ERR_WORKSPACE = 6,   /* workspace pointer null/misaligned or smaller than asked */
    PA_ERR_PRECONDITION = 7 /* a kernel found a stated device-side precondition broken
                               (pa_decode_cascade: a sequence's shared blocks differ) */
} pa_status;

/* Human-readable name of a status; never NULL. */
const char *pa_status_string(pa_status status);

/*
 * Bytes of one KV block, 2 * block_size * num_kv_heads * head_size * 2 (bf16),
 * the formula of §Block size.  Returns 0 for non-positive arguments.
 */
size_t pa_kv_block_bytes(int block_size, int num_kv_heads, int head_size);

/*
 * pa_cache_write - scatter new tokens' K and V rows into their slots.
 *
 * Follows §Engine core (a token's KV lives in the block its sequence was given).
 *   kv_cache      [num_blocks][2][num_kv_heads][block_size][head_size] bf16, in/out
 *   k_new, v_new  [num_tokens][num_kv_heads][head_size] bf16 rows; row i starts
 *                 at element i * new_row_stride (new_row_stride >= num_kv_heads *
 *                 head_size, a multiple of 8), heads contiguous inside a row
 *   slot_mapping  [num_tokens] int32; slot < 0 skips the row (padding); a slot
 *                 >= num_blocks*block_size is skipped and flagged PA_ERR_OOB
 * Bit-exact copy.  Two rows with the same slot in one call are a precondition
 * violation (which one lands is unspecified).  num_tokens == 0 is a no-op.
 */
pa_status pa_cache_write(void *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                         int head_size, const void *k_new, const void *v_new,
                         int64_t new_row_stride, const int32_t *slot_mapping, int num_tokens,
                         pa_stream_t stream);

/*
 * pa_kv_block_bytes_dtype - the same formula for any element size:
 * 2 * block_size * num_kv_heads * head_size * dtype_num_bytes (§Block size);
 * 1 for an FP8 pool.  Returns 0 for non-positive arguments.
 */
size_t pa_kv_block_bytes_dtype(int block_size, int num_kv_heads, int head_size,
                               int dtype_num_bytes);

/*
 * FP8 KV cache.  The pages list FP8 among the quantisation formats the engine
 * supports and size a block by its element bytes (§Block size); here an FP8
 * pool has the bf16 pool's layout, [num_blocks][2][num_kv_heads][block_size]
 * [head_size], one byte per element holding an OCP FP8 E4M3 ("e4m3fn") code,
 * and real values are code values times a per-tensor scale: k_scale for every
 * K element, v_scale for every V element (finite, > 0; else
 * PA_ERR_INVALID_ARG).
 *
 * pa_cache_write_fp8 - pa_cache_write into an FP8 pool: element x of a new
 * bf16 row is stored as the e4m3 code nearest to x / scale (binary32
 * division; ties to the even code; magnitudes beyond 448 saturate to +-448).
 * Arguments as pa_cache_write, plus k_scale / v_scale; kv_cache is the FP8
 * pool (16-byte aligned).
 */
pa_status pa_cache_write_fp8(void *kv_cache, int num_blocks, int block_size, int num_kv_heads,
                             int head_size, const void *k_new, const void *v_new,
                             int64_t new_row_stride, const int32_t *slot_mapping, int num_tokens,
                             float k_scale, float v_scale, pa_stream_t stream);

/*
 * pa_decode_fp8 - pa_decode over an FP8 pool: K = code value * k_scale,
 * V = code value * v_scale.  head_size must be 128 (else PA_ERR_UNSUPPORTED).
 * Codes convert to f16 exactly and the products run on f16 MMAs with fp32
 * accumulation; each query head is scaled by a power of two into f16 range
 * first (exact), P is rounded to f16.  Workspace: pa_decode_workspace_bytes.
 * Other arguments, results and errors as pa_decode.
 */
pa_status pa_decode_fp8(void *out, const void *q, const void *kv_cache, int num_blocks,
                        int block_size, int num_heads, int num_kv_heads, int head_size,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                        float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                        pa_stream_t stream);

/*
 * pa_prefill_chunk_fp8 - pa_prefill_chunk over an FP8 pool: K = code value *
 * k_scale, V = code value * v_scale.  head_size must be 128 (else
 * PA_ERR_UNSUPPORTED).  Each K/V tile is converted to f16 in shared memory
 * (exactly) and the products run as f16 tcgen05 MMAs with fp32 accumulation;
 * each query row is scaled by a power of two into f16 range first (exact), P
 * is rounded to f16.  Other arguments, results and errors as pa_prefill_chunk.
 */
pa_status pa_prefill_chunk_fp8(void *out, const void *q, const int32_t *cu_q_lens,
                               int num_chunks, int max_q_len, const void *kv_cache,
                               int num_blocks, int block_size, int num_heads, int num_kv_heads,
                               int head_size, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, float scale,
                               float k_scale, float v_scale, pa_stream_t stream);

/*
 * Workspace pa_decode needs on the current device for this shape, in bytes
 * (partial softmax states of split contexts plus a small table).  Depends on
 * the device's SM count and the batch size, not on sequence lengths: every
 * context is split over the whole GPU, so the partial states are per warp of
 * the persistent grid.  Returns 0 for invalid arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_size);

/*
 * pa_decode - one query token per sequence against its paged context.
 *
 * Follows §Engine core (a sequence's tokens are found through the blocks its
 * block table names: the blocks are the index from tokens to their KV) and
 * §Generate function (the batch's decode tokens are rows of one flattened
 * forward pass, each attending to its own sequence's cached KV).
 * Sequence s attends to its tokens 0 .. seq_lens[s]-1, found through
 * block_tables[s][t / block_size] at offset t % block_size; the new token's own
 * K/V must already be written (pa_cache_write), so seq_lens[s] counts it.
 *   out           [num_seqs][num_heads][head_size] bf16, written
 *   q             [num_seqs][num_heads][head_size] bf16
 *   block_tables  [num_seqs][max_blocks_per_seq] int32 physical block ids
 *   seq_lens      [num_seqs] int32, 0 <= seq_lens[s] <= max_blocks_per_seq*block_size;
 *                 0 yields a zero output row
 *   max_seq_len   host-side upper bound of seq_lens (sizes the launch only)
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(head_size)), finite
 *   workspace     device scratch of >= pa_decode_workspace_bytes(...) bytes,
 *                 256-byte aligned, owned by the caller, contents need no
 *                 initialisation; two calls that overlap on the GPU must not
 *                 share one workspace
 * out[s][h] = sum_t softmax_t(scale * q[s][h].K[t][h/G]) V[t][h/G], computed
 * with an online softmax in fp32 over bf16 products; contexts are split evenly
 * over the whole GPU and the pieces merged by log-sum-exp (a second, dependent
 * kernel).  A batch of at most one (sequence, KV head) pair per SM whose
 * max_seq_len is at most 12 tiles of 16 tokens runs as one kernel instead: a CTA
 * per pair, its warps splitting the pair's tiles, merged in the CTA
 * (pa_decode_cascade_kernels with shared_len 0 says which).  num_seqs == 0 is a
 * no-op.
 */
pa_status pa_decode(void *out, const void *q, const void *kv_cache, int num_blocks,
                    int block_size, int num_heads, int num_kv_heads, int head_size,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                    void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_noalloc - pa_decode without a caller-provided workspace.
 *
 * The pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory on this path: an engine that has already reserved
 * nearly all of HBM for its KV-cache pool, a host program that only receives
 * device pointers and owns no allocator, or a decode loop that cannot afford
 * cudaMalloc/cudaFree (they may synchronise the device).
 *   Arguments and results are those of pa_decode, minus workspace.
 *   Scratch comes from a 16 MiB array in this library's device image, held by
 *   every GPU that loads the library until the process exits.  A shape whose
 *   pa_decode_workspace_bytes() exceeds 16 MiB returns PA_ERR_UNSUPPORTED.
 *   The call allocates nothing.  Its first call in a CUDA context (the device's
 *   primary context, or another one made current) looks up the array's device
 *   address in that context and keeps it for that context's later calls; make
 *   that first call before any stream capture.  The 16 MiB hold every shape
 *   pa_decode accepts on a 152-SM GB300 (the largest, 15 091 sequences of head
 *   size 128, needs 15.1 MB).
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other threads) race and must be serialised by the caller.  No
 *   byte of the array needs to start at zero: each call writes before it reads.
 */
pa_status pa_decode_noalloc(void *out, const void *q, const void *kv_cache, int num_blocks,
                            int block_size, int num_heads, int num_kv_heads, int head_size,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int num_seqs, int max_seq_len, float scale,
                            pa_stream_t stream);

/*
 * Workspace pa_decode_cascade needs on the current device, in bytes: that of
 * pa_decode plus the shared prefix's partial softmax states and one partial
 * state per (sequence, KV head) for the sequences' own tokens.  Depends on the
 * device's SM count.  Returns 0 for invalid arguments.
 */
size_t pa_decode_cascade_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                         int head_size, int shared_len);

/*
 * Kernels one pa_decode_cascade call (pa_decode_cascade_fp8 when kv8 != 0) with
 * these shapes launches on the current device: 2 when the shared prefix and the
 * sequences' own tokens are attended side by side in one launch on disjoint
 * SMs, then merged (chosen from the shapes and the pool's type); 3 when the
 * prefix is attended by its own launch before the own tokens and the merge;
 * when shared_len is 0, pa_decode's count: 1 (a CTA per segment, merged in
 * place) or 2 (split kernel and merge kernel); 0 when num_seqs is 0; -1 for
 * invalid shapes.  For planning only (e.g. counting a CUDA graph's nodes): the results
 * are the same either way, up to floating-point summation order.
 */
int pa_decode_cascade_kernels(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                              int block_size, int max_seq_len, int shared_len, int kv8);

/*
 * pa_decode_cascade - pa_decode for a batch whose sequences share a prefix.
 *
 * Prefix caching ("Inside vLLM: Anatomy of a High-Throughput LLM Inference
 * System", advanced features: prefix caching) lets sequences with a common
 * prompt start hold the same physical KV blocks.  Here the first shared_len
 * tokens of every sequence are those blocks: block_tables[s][i] equals
 * block_tables[0][i] for i < shared_len / block_size (a precondition; the
 * prefix is read through sequence 0's table; the kernels compare the entries,
 * and a mismatch makes pa_error_check() return PA_ERR_PRECONDITION).  The prefix is attended once per
 * KV head for all queries of the batch on the tensor cores, each sequence's own
 * tokens [shared_len, seq_lens[s]) as in pa_decode, and the softmax states
 * are merged by log-sum-exp, one warp per (sequence, KV head).  The result is
 * pa_decode's up to floating-point summation order, and the same bits on every
 * call.
 *   Arguments are those of pa_decode, plus:
 *   shared_len    tokens shared by every sequence, 0 <= shared_len <= max_seq_len,
 *                 a multiple of 16 and of block_size (else PA_ERR_UNSUPPORTED);
 *                 every seq_lens[s] >= shared_len (else PA_ERR_OOB is flagged);
 *                 0 makes the call pa_decode
 *   workspace     >= pa_decode_cascade_workspace_bytes(...) bytes, 256-byte
 *                 aligned, caller-owned, no initialisation needed
 */
pa_status pa_decode_cascade(void *out, const void *q, const void *kv_cache, int num_blocks,
                            int block_size, int num_heads, int num_kv_heads, int head_size,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int num_seqs, int max_seq_len,
                            int shared_len, float scale, void *workspace,
                            size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_cascade_fp8 - pa_decode_cascade over an FP8 pool: K = code value *
 * k_scale, V = code value * v_scale (the pool pa_cache_write_fp8 fills).
 * head_size must be 128 (else PA_ERR_UNSUPPORTED); k_scale and v_scale must be
 * finite and > 0 (else PA_ERR_INVALID_ARG).  The prefix pass converts K/V to
 * f16 as pa_prefill_chunk_fp8 does, the own tokens are read as in
 * pa_decode_fp8.  Workspace: pa_decode_cascade_workspace_bytes.  Other
 * arguments, results and errors as pa_decode_cascade.
 */
pa_status pa_decode_cascade_fp8(void *out, const void *q, const void *kv_cache, int num_blocks,
                                int block_size, int num_heads, int num_kv_heads, int head_size,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *seq_lens, int num_seqs, int max_seq_len,
                                int shared_len, float scale, float k_scale, float v_scale,
                                void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill_chunk - chunked-prefill attention of query chunks against their
 * cached context and themselves, causal.
 *
 * The batch is flattened (§Generate function): chunk s owns query rows
 * cu_q_lens[s] .. cu_q_lens[s+1]-1.  Its q_len = cu_q_lens[s+1]-cu_q_lens[s]
 * new tokens sit at positions seq_lens[s]-q_len .. seq_lens[s]-1 and their K/V
 * must already be written to the pool; row i sees tokens 0 .. seq_lens[s]-q_len+i.
 *   out           [total_q][num_heads][head_size] bf16, written
 *   q             [total_q][num_heads][head_size] bf16
 *   cu_q_lens     [num_chunks+1] int32, cu_q_lens[0] == 0, non-decreasing
 *   max_q_len     host-side upper bound of any chunk's q_len (sizes the launch)
 *   block_tables  [num_chunks][max_blocks_per_seq] int32
 *   seq_lens      [num_chunks] int32 context + chunk, >= that chunk's q_len
 * Tensor cores compute q.K^T and P.V in bf16 with fp32 accumulation.
 * num_chunks == 0 or max_q_len == 0 is a no-op.
 */
pa_status pa_prefill_chunk(void *out, const void *q, const int32_t *cu_q_lens, int num_chunks,
                           int max_q_len, const void *kv_cache, int num_blocks, int block_size,
                           int num_heads, int num_kv_heads, int head_size,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, float scale, pa_stream_t stream);

/*
 * Workspace pa_attention_varlen needs: pa_decode's for the batch's
 * num_seqs - num_prefills decode sequences.  Returns 0 for invalid arguments.
 */
size_t pa_attention_varlen_workspace_bytes(int num_seqs, int num_prefills, int num_heads,
                                           int num_kv_heads, int head_size);

/*
 * pa_attention_varlen - one step of attention over a flattened mixed batch.
 *
 * The forward pass "flattens the batch into a single sequence"
 * (§Generate function) mixing prompt chunks (chunked prefill) with decode
 * tokens.  The batch lists its num_prefills chunk sequences first (query rows
 * [0, num_prefill_tokens), cu_q_lens[0..num_prefills] their row offsets, so
 * cu_q_lens[num_prefills] == num_prefill_tokens) and then its decode
 * sequences, one query row each, in order.  The call
 *   1. writes the step's new K/V rows into their slots (pa_cache_write), one
 *      per query row, unless slot_mapping is NULL;
 *   2. attends every chunk row causally to its sequence (pa_prefill_chunk);
 *   3. attends every decode row to its whole sequence (pa_decode).
 *   out, q        [num_prefill_tokens + num_decodes][num_heads][head_size] bf16
 *   k_new, v_new  [same rows][num_kv_heads][head_size] bf16 (read only if
 *                 slot_mapping != NULL)
 *   slot_mapping  [same rows] int32 slots, or NULL
 *   cu_q_lens     [num_prefills + 1] int32 (read only if num_prefills > 0)
 *   max_prefill_q_len  host bound of the chunks' query lengths
 *   block_tables, seq_lens  for all num_seqs sequences, chunks first
 *   max_seq_len   host bound of the decode sequences' lengths
 *   workspace     >= pa_attention_varlen_workspace_bytes(...) bytes, 256-byte
 *                 aligned
 * Launches on `stream` in that order.  Every argument is checked (as by the
 * three calls, and the workspace) before anything is enqueued: a host-checkable
 * fault returns its status with the pool untouched.
 */
pa_status pa_attention_varlen(void *out, const void *q, const void *k_new, const void *v_new,
                              const int32_t *slot_mapping, const int32_t *cu_q_lens,
                              int num_seqs, int num_prefills, int num_prefill_tokens,
                              int max_prefill_q_len, void *kv_cache, int num_blocks,
                              int block_size, int num_heads, int num_kv_heads, int head_size,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int max_seq_len, float scale,
                              void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_varlen_fp8 - pa_attention_varlen over an FP8 pool: the writes
 * quantise as pa_cache_write_fp8, the chunks and decode tokens read as
 * pa_prefill_chunk_fp8 and pa_decode_fp8 (head_size 128), in one launch when
 * both are present.  Workspace: pa_attention_varlen_workspace_bytes.
 */
pa_status pa_attention_varlen_fp8(void *out, const void *q, const void *k_new,
                                  const void *v_new, const int32_t *slot_mapping,
                                  const int32_t *cu_q_lens, int num_seqs, int num_prefills,
                                  int num_prefill_tokens, int max_prefill_q_len, void *kv_cache,
                                  int num_blocks, int block_size, int num_heads,
                                  int num_kv_heads, int head_size, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *seq_lens,
                                  int max_seq_len, float scale, float k_scale, float v_scale,
                                  void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_varlen_args - every argument of pa_attention_varlen(_fp8) in one struct,
 * for callers whose per-argument marshalling costs more than the call itself
 * (an interpreter's foreign-function layer).  Each field means what the
 * parameter of the same name means; kv8 != 0 selects the FP8 pool form
 * (k_scale and v_scale are read only then).  Natural C layout, as declared: on
 * a 64-bit target 12 eight-byte fields, 12 int32, 3 float (pa_varlen_args_bytes
 * reports its size).
 */
typedef struct pa_varlen_args {
    void *out;
    const void *q;
    const void *k_new;
    const void *v_new;
    const int32_t *slot_mapping;
    const int32_t *cu_q_lens;
    void *kv_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    void *workspace;
    size_t workspace_bytes;
    pa_stream_t stream;
    int32_t num_seqs, num_prefills, num_prefill_tokens, max_prefill_q_len;
    int32_t num_blocks, block_size, num_heads, num_kv_heads, head_size;
    int32_t max_blocks_per_seq, max_seq_len, kv8;
    float scale, k_scale, v_scale;
} pa_varlen_args;

/* sizeof(pa_varlen_args), for callers that lay the struct out themselves. */
size_t pa_varlen_args_bytes(void);

/*
 * pa_attention_varlen_packed - pa_attention_varlen (kv8 == 0) or
 * pa_attention_varlen_fp8 (kv8 != 0) with the arguments read from *args, which
 * the call does not keep.  Same checks and statuses; PA_ERR_INVALID_ARG for a
 * NULL args.
 */
pa_status pa_attention_varlen_packed(const pa_varlen_args *args);

/*
 * Synchronise `stream`, then read and clear the device error word the kernels
 * of this library set on the current device.  Returns PA_OK, PA_ERR_TIMEOUT,
 * PA_ERR_OOB or PA_ERR_PRECONDITION (the first of these that was set, in this
 * order), or PA_ERR_CUDA if the synchronisation itself failed.
 */
pa_status pa_error_check(pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
