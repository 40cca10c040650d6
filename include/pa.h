/*
 * pa.h -- C interface of the GB300 paged-KV decode library (libpa.so).
 *
 * The library implements the data-parallel hot path of paged KV caching:
 *   pa_reshape_and_cache  write new tokens' K/V into pool slots,
 *   pa_copy_blocks        copy-on-write of shared blocks (one layer, or
 *                         all layers: pa_copy_blocks_layers),
 *   pa_swap_blocks        block copies between a device and a host pool,
 *   pa_decode             one decode step of attention over a paged pool,
 *   pa_attention          several causal query tokens per sequence.
 *
 * Layouts (row-major, innermost last):
 *   k_cache, v_cache   [num_blocks, block_size, num_kv_heads, head_dim]
 *                      one pool per layer, K and V separate
 *                      ("kv-cache-memory-core", section 2.2).
 *   block_tables       int32 [num_seqs, max_blocks_per_seq]; entry j of row i
 *                      is the physical block holding tokens
 *                      [j*block_size, (j+1)*block_size) of sequence i
 *                      ("vLLM intro part 2", section 3.2).  Entries at or past
 *                      cdiv(seq_lens[i], block_size) are never read.
 *   seq_lens           int32 [num_seqs], tokens attended per sequence.
 *   slot_mapping       int64 [num_tokens], absolute pool slot of each new
 *                      token, block*block_size + offset (same section).
 *   q, out             [num_seqs, num_q_heads, head_dim], one decode query
 *                      per sequence; out has the type of q.
 *   key, value         [num_tokens, num_kv_heads, head_dim].
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads)
 *   ("kv-cache-memory-core", section 4.2, grouped-query attention).
 *
 * Ownership and execution: every pointer is a device pointer owned by the
 * caller, including the workspace.  Every call is asynchronous on `stream`,
 * allocates nothing and never synchronises the host.  Host-side argument
 * checks return a status before anything is launched.  Out-of-range indices
 * met on the device (a block id, a slot or a copy pair outside the pool, a
 * sequence longer than its table) skip the affected unit and OR a bit into
 * *err_flag (if err_flag is non-null); kernels never trap.  Identical inputs
 * give bit-identical outputs (no floating-point atomics).
 *
 * Supported shapes: head_dim 64 or 128; block_size 8, 16, 32, 64 or 128;
 * num_q_heads a multiple of num_kv_heads; num_kv_heads <= 256.
 * Element types: f32 caches need f32 q; f16/bf16 caches need q of the same
 * type; fp8 caches (e4m3 or e5m2) take f16 or bf16 q (head_dim 128 only).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shape */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not supported (dtype combo, head_dim, ...) */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4           /* a CUDA runtime/driver call failed; see pa_last_error_detail */
} pa_status;

typedef enum {
    PA_F32 = 0,
    PA_F16 = 1,
    PA_BF16 = 2,
    PA_FP8_E4M3 = 3,          /* OCP E4M3 (finite-only, max 448), one byte */
    PA_FP8_E5M2 = 4           /* OCP E5M2 (IEEE-like inf/NaN, max 57344), one byte */
} pa_dtype;

/* Bits OR-ed into *err_flag by device code. */
#define PA_ERRBIT_BAD_BLOCK     1u   /* block table entry outside [0, num_blocks) */
#define PA_ERRBIT_BAD_SLOT      2u   /* slot_mapping entry >= num_blocks*block_size */
#define PA_ERRBIT_BAD_PAIR      4u   /* copy pair id outside [0, num_blocks) */
#define PA_ERRBIT_SEQ_TOO_LONG  8u   /* seq_lens[i] < 0 or > max_blocks_per_seq*block_size */
#define PA_ERRBIT_WAIT_TIMEOUT 16u   /* an internal pipeline wait exceeded its time limit */
#define PA_ERRBIT_BAD_QUERY    32u   /* pa_attention: q_start entries not increasing within
                                        [0, total_q], or a sequence with more than max_q_len
                                        query tokens; its rows are left unwritten */

/* Human-readable name of a status. */
const char* pa_status_string(pa_status s);

/* Detail of the most recent failure on the calling host thread ("" if none). */
const char* pa_last_error_detail(void);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs on the
 * current device for these bounds.  max_seq_len bounds every seq_lens[i];
 * partition_tokens is the value that will be passed to pa_decode.
 * Returns 0 for invalid arguments.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int max_seq_len,
                                int head_dim, int partition_tokens);

/*
 * pa_decode -- single-query decode attention over a paged KV pool
 * ("vLLM intro part 2", section 4 (kernel layer, the softmax and dot-product
 * formulas); PagedAttention note (vagrantpi PKM), kernel steps: look up the
 * block table, load block by block, merge across blocks with online softmax).
 *
 * For every sequence i and query head h, with g = h / (num_q_heads /
 * num_kv_heads) and L = seq_lens[i]:
 *   s_t   = scale * <q[i,h,:], K_t>            t in [0, L)
 *   out   = sum_t softmax(s)_t * V_t
 * where K_t, V_t are row (t % block_size, g) of physical block
 * block_tables[i][t / block_size].  fp8 caches are read as
 * K_t = e4m3(k) * k_scale, V_t = e4m3(v) * v_scale (scales ignored otherwise);
 * the scales are applied to the scores and the output, never per element.
 * L == 0 writes zeros.
 *
 * The work is split into chunks of 16 tokens (32 for fp8 caches with
 * head_dim 128 and at most 8 query heads per KV head), balanced over
 * persistent CTAs; sequences spanning several CTAs (or longer than
 * partition_tokens) are merged afterwards by a log-sum-exp reduction kernel
 * on the same stream.
 *   partition_tokens  0 lets the library choose split points; otherwise a
 *                     positive multiple of 16: sequences are additionally
 *                     split every partition_tokens tokens.
 * Precision: scores and sums accumulate in fp32.  The probabilities enter
 * P*V rounded to the MMA operand type: bf16 (8 significant bits) for bf16
 * caches, f16 (11 bits) for f16 caches and fp8 caches on 16-token chunks.
 * On the fp8 32-token path (e4m3 and e5m2 caches: the key and value bytes
 * are MMA operands as stored) the query and the probabilities are each carried
 * as two e4m3 terms, 8 significant bits (exact for bf16 queries, except
 * elements below 2^-9 of the largest in their GQA group); an infinite query
 * element saturates to +-448 there instead of propagating.  pa_decode_simt
 * keeps everything in fp32.  f32 caches (with f32 q) run on CUDA-core
 * FMAs in fp32 throughout: fp32 is no tensor-core operand type here, so that
 * kernel is the only one for them.
 *   workspace         device buffer of at least pa_decode_workspace_size(...)
 *                     bytes, 256-byte aligned; contents need no initialisation
 *                     and are scratch between calls.  Calls sharing one
 *                     workspace must not overlap on the GPU.
 *   err_flag          optional device int32 receiving PA_ERRBIT_* bits.
 * Alignment: q, out, k_cache, v_cache must be 16-byte aligned.
 */
pa_status pa_decode(void* out, const void* q, pa_dtype q_dtype,
                    const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* seq_lens, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks,
                    float scale, float k_scale, float v_scale,
                    int partition_tokens, void* workspace, size_t workspace_bytes,
                    int32_t* err_flag, cudaStream_t stream);

/*
 * pa_decode_simt -- the same operation, arguments and results as pa_decode,
 * computed with CUDA-core FMAs instead of tensor-core MMAs, for every cache
 * type.  pa_decode runs this kernel for f32 caches; for the other types it
 * is a measured comparison point.
 */
pa_status pa_decode_simt(void* out, const void* q, pa_dtype q_dtype,
                         const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, float k_scale, float v_scale,
                         int partition_tokens, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, cudaStream_t stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot supply a workspace.
 * The pages have no counterpart: this exists for callers that must not
 * allocate device memory on the call path, such as a serving loop whose
 * memory is fully pre-partitioned by its own allocator, or a plugin inside a
 * host framework that owns all device memory.  Arguments and results are
 * those of pa_decode without the workspace; the split-KV partials go to a
 * scratch array of PA_NOALLOC_SCRATCH_BYTES that the library keeps in device
 * memory on every GPU it is loaded on, until the process exits.
 *   - The first call on a device looks up the array's address on that device
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - A batch needing more scratch than PA_NOALLOC_SCRATCH_BYTES (see
 *     pa_decode_workspace_size) returns PA_ERR_WORKSPACE and launches nothing.
 *   - All calls on a device share the array and it keeps the previous call's
 *     contents; calls whose GPU work overlaps race on it.  No contents need
 *     to start at zero.
 *   - Nothing is allocated or freed.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
pa_status pa_decode_noalloc(void* out, const void* q, pa_dtype q_dtype,
                            const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* seq_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale, float k_scale, float v_scale,
                            int partition_tokens, int32_t* err_flag, cudaStream_t stream);

/*
 * pa_reshape_and_cache -- write token t's K and V rows ([num_kv_heads,
 * head_dim] each) into pool slot slot_mapping[t] ("vLLM intro part 2",
 * section 3.2, slot_mapping; "kv-cache-memory-core", section 3, decode
 * appends one slot per step).
 *   slot < 0                          padding: skipped, no error.
 *   slot >= num_blocks*block_size     skipped, PA_ERRBIT_BAD_SLOT.
 * Same-type writes copy bits.  An fp8 cache quantises on write
 * ("kv-cache-memory-core", section 4.4): byte = e4m3_satfinite_rne(x / scale)
 * with x the source value widened to float, IEEE float division, round to
 * nearest even, saturation to +-448; NaN becomes the NaN code.  Sources for
 * an fp8 cache may be f32, f16 or bf16; other caches need src == kv dtype.
 * Duplicate slots within one call leave one of the writes (unspecified which).
 */
pa_status pa_reshape_and_cache(void* k_cache, void* v_cache, pa_dtype kv_dtype,
                               const void* key, const void* value, pa_dtype src_dtype,
                               const int64_t* slot_mapping, int num_tokens,
                               int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, float k_scale, float v_scale,
                               int32_t* err_flag, cudaStream_t stream);

/*
 * pa_copy_blocks -- copy-on-write block copies ("vLLM intro part 2",
 * section 5; aibook "显存与 KV 缓存", the copy-on-write steps: copy first,
 * repoint the table, then write).  For each pair p, the whole K block and V
 * block block_mapping[2p] are copied onto block block_mapping[2p+1].
 * num_pairs == 0 is a no-op.  A pair with an id outside [0, num_blocks) is
 * skipped with PA_ERRBIT_BAD_PAIR.  Destinations must be distinct and must
 * not be the source of another pair in the same call.
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_dtype kv_dtype,
                         const int64_t* block_mapping, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int32_t* err_flag, cudaStream_t stream);

/*
 * pa_attention -- causal attention of several new query tokens per sequence
 * over the paged pool, their K/V already written (speculative lookahead
 * tokens, or a chunk of a prompt: the "new" and "lookahead" spans one request
 * computes in one iteration, "分页省的不是 KV 字节", section 2, the
 * allocate_slots layout).  Sequence i owns query rows q_start[i] ..
 * q_start[i+1]-1 of q and out ([total_q, num_q_heads, head_dim]); they are the
 * last n_i = q_start[i+1] - q_start[i] of its L_i = seq_lens[i] tokens, and
 * query token j, at position p = L_i - n_i + j, attends keys 0..p:
 *   out[q_start[i] + j, h] = sum_{t<=p} softmax_t(scale * <q, K_t>) V_t.
 * A token with p < 0 (n_i > L_i) gets zeros.  One pass reads each K/V byte
 * once for all of a sequence's query tokens: the (token, head) rows of a GQA
 * group share the MMA tile.  q_start is a device int32 array of num_seqs + 1
 * entries, non-decreasing, q_start[0] = 0, q_start[num_seqs] = total_q; every
 * n_i <= max_q_len, and max_q_len * (num_q_heads / num_kv_heads) <= 128.
 * Tensor cores only (f16, bf16 and fp8 caches); other arguments as for
 * pa_decode.  With every n_i = 1 the result equals pa_decode's.
 * Kernels: with at least 48 rows per KV head (max_q_len * G), a 16-bit cache
 * and partition_tokens a multiple of 32, the rows of up to four KV heads
 * (each padded to a multiple of 32) fill one 128-row tcgen05 tile whose S and
 * O accumulators live in tensor memory (32-token chunks, P rounded to the
 * cache's 16-bit type); otherwise 16-row mma.sync tiles as in pa_decode.
 */
size_t pa_attention_workspace_size(int num_seqs, int max_q_len, int num_q_heads, int max_seq_len,
                                   int head_dim, int partition_tokens);
pa_status pa_attention(void* out, const void* q, pa_dtype q_dtype,
                       const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* q_start, int num_seqs,
                       int total_q, int max_q_len, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, float scale,
                       float k_scale, float v_scale, int partition_tokens, void* workspace,
                       size_t workspace_bytes, int32_t* err_flag, cudaStream_t stream);

/*
 * pa_copy_blocks_layers -- pa_copy_blocks for every layer of a model in one
 * launch: the same pairs are copied in each of the num_layers K and V pools.
 * k_caches and v_caches are HOST arrays of num_layers device pointers (pools
 * of identical shape, 16-byte aligned); num_layers <= 256.
 */
pa_status pa_copy_blocks_layers(void* const* k_caches, void* const* v_caches, int num_layers,
                                pa_dtype kv_dtype, const int64_t* block_mapping, int num_pairs,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                int32_t* err_flag, cudaStream_t stream);

/*
 * pa_swap_blocks -- block-granular swap between two pools of the same block
 * shape, typically a device pool and a host pool (preemption by swapping a
 * request's KV out to CPU memory and back in, "kv-cache-memory-core", the
 * preemption section: swap keeps the progress at the cost of CPU memory and
 * interconnect bandwidth).  For each pair p the K and V block
 * block_mapping[2p] of the source pool are copied to block
 * block_mapping[2p+1] of the destination pool.  Either pool may be host
 * memory the device can address (pinned with cudaHostAlloc / cudaMallocHost,
 * or cudaHostRegister-ed); block_mapping must be device-accessible.  Ids
 * outside their pool are skipped with PA_ERRBIT_BAD_PAIR.  The two pools must
 * not overlap.  A kernel performs the copy, so swaps of many scattered blocks
 * cost one launch, not one transfer per block.
 */
pa_status pa_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks, const void* src_k,
                         const void* src_v, int src_num_blocks, pa_dtype kv_dtype,
                         const int64_t* block_mapping, int num_pairs, int num_kv_heads,
                         int head_dim, int block_size, int32_t* err_flag, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
