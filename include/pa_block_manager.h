/*
 * pa_block_manager.h -- C interface of the host-side block manager
 * (libpa_host.so): the allocator that produces the block tables, slot
 * mappings and copy-on-write pairs consumed by pa_decode,
 * pa_reshape_and_cache and pa_copy_blocks.
 *
 * What it implements (the pages' allocator):
 *   - A pool of num_blocks physical blocks with reference counts and one
 *     free queue holding every block with ref_cnt == 0, head = next to be
 *     handed out ("分页省的不是 KV 字节", section 3: BlockPool and the
 *     six-block walk T0-T4).
 *   - Taking blocks pops them from the head; a block that still carries a
 *     prefix-cache hash loses it then (eviction as a side effect of reuse).
 *   - Releasing a request drops one reference per block, last block first;
 *     a block reaching zero goes to the head if it has no hash and to the
 *     tail, hash kept, if it has one (same section, T2).  The other page
 *     ("vLLM intro part 2", section 6.3) sends every freed block to the
 *     tail; the worked trace is followed.
 *   - Prefix cache: a new request's full blocks come with their chained
 *     hashes; the lookup walks them from block 0 and stops at the first miss
 *     ("vLLM intro part 2", section 6.1 and 6.3).  A hit held by nobody
 *     leaves the free queue (touch).  The hashes themselves are computed by
 *     the caller (the Python binding uses sha256 from its standard library);
 *     this library treats them as opaque 32-byte keys.
 *   - Copy-on-write: the next token of a request whose last block is partly
 *     filled and shared takes a new block, emits the pair (old, new) for
 *     pa_copy_blocks, repoints the table and drops one reference from the
 *     old block ("vLLM intro part 2", section 5, steps 1-4).
 *
 * Requests are named by caller-chosen 64-bit ids.  A manager is not thread
 * safe: one host thread at a time.  All output buffers are caller-owned host
 * memory.  Nothing here touches a GPU.
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_bm pa_bm;

typedef enum {
    PA_BM_OK = 0,
    PA_BM_WAIT = 1,          /* allocation incomplete: the request holds its prefix hits and waits */
    PA_BM_NO_SPACE = 2,      /* not enough free blocks; nothing changed for the failing request */
    PA_BM_BAD_REQUEST = 3,   /* unknown request id, existing id on create, or a waiting request */
    PA_BM_INVALID_ARG = 4    /* null pointer, bad size, capacity too small */
} pa_bm_status;

#define PA_BM_HASH_BYTES 32

/* A manager over blocks 0..num_blocks-1 of block_size tokens.  `order`
 * (nullable) is the initial free queue from head to tail, a permutation of
 * the block ids; null means 0, 1, 2, ...  Returns null on invalid arguments. */
pa_bm* pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* order);
void pa_bm_destroy(pa_bm* m);

int32_t pa_bm_num_free(const pa_bm* m);
/* ref_cnt of a block, -1 for an id outside the pool. */
int32_t pa_bm_ref_cnt(const pa_bm* m, int32_t block);
/* The free queue from head to tail: writes min(cap, length) ids (and, if
 * has_hash is non-null, 1 for blocks carrying a hash); returns the length. */
int32_t pa_bm_free_queue(const pa_bm* m, int32_t* ids, uint8_t* has_hash, int32_t cap);

/* A new request of num_tokens tokens.  hashes: num_hashes chained hashes of
 * its first full blocks, PA_BM_HASH_BYTES each (may be 0 / null).  Prefix
 * hits are taken first; the remaining blocks come from the free queue and
 * its new full blocks are registered under their hashes.
 * *num_cached_tokens = hits * block_size.  Returns PA_BM_OK, or PA_BM_WAIT
 * when the free queue is too short: the request then exists, holds its hits
 * and completes with pa_bm_resume. */
pa_bm_status pa_bm_allocate(pa_bm* m, int64_t req, int32_t num_tokens, const uint8_t* hashes,
                            int32_t num_hashes, int32_t* num_cached_tokens);
pa_bm_status pa_bm_resume(pa_bm* m, int64_t req);

/* A new request `child` sharing every block of the (complete) `parent`. */
pa_bm_status pa_bm_fork(pa_bm* m, int64_t parent, int64_t child);

/* One decode step: reserve the slot of the next token of each of the n
 * requests, in order.  slot_mapping[k] = block * block_size + offset for
 * request k; copy-on-write pairs go to pairs[2*p], pairs[2*p+1] (int64
 * src, dst; room for pair_cap pairs, n suffices).  Stops at the first
 * request that cannot get a block and returns PA_BM_NO_SPACE; *num_done is
 * the number of requests served (their slots and pairs are valid). */
pa_bm_status pa_bm_append_slots(pa_bm* m, int32_t n, const int64_t* reqs, int64_t* slot_mapping,
                                int64_t* pairs, int32_t pair_cap, int32_t* num_pairs, int32_t* num_done);

/* Register the hash of logical block j of a request once it is full (a
 * block filled by decode appends).  A block that already has a hash keeps
 * it. */
pa_bm_status pa_bm_cache_block(pa_bm* m, int64_t req, int32_t j, const uint8_t* hash);

/* Release a request (complete or waiting). */
pa_bm_status pa_bm_free(pa_bm* m, int64_t req);

/* Number of tokens of a request, -1 if unknown. */
int64_t pa_bm_num_tokens(const pa_bm* m, int64_t req);
/* A request's block table: writes min(cap, n) ids (none when out is NULL),
 * returns n, or -1 for an unknown or swapped-out request. */
int32_t pa_bm_block_table(const pa_bm* m, int64_t req, int32_t* out, int32_t cap);
/* Block tables of n requests as int32 rows of max_blocks entries, the
 * unused tail of each row set to `pad`: the layout pa_decode reads.
 * PA_BM_INVALID_ARG if a table is longer than max_blocks. */
pa_bm_status pa_bm_block_tables(const pa_bm* m, int32_t n, const int64_t* reqs, int32_t* out,
                                int32_t max_blocks, int32_t pad);

/* What row k of a persistent block-table buffer holds, for
 * pa_bm_block_tables_update.  Fill with 0xff bytes (len = -1: unknown)
 * before the first call and whenever the buffer is rewritten elsewhere. */
typedef struct {
    int64_t req;
    uint32_t epoch;
    int32_t len;
} pa_bm_row;

/* pa_bm_block_tables for a buffer kept across decode steps: row k is
 * rewritten in full only if it held another request, or the same request
 * before a copy-on-write changed one of its entries; otherwise only the
 * entries appended since the last call are written.  rows[k] is updated. */
pa_bm_status pa_bm_block_tables_update(const pa_bm* m, int32_t n, const int64_t* reqs, int32_t* out,
                                       int32_t max_blocks, int32_t pad, pa_bm_row* rows);

/*
 * Preemption by swapping: a preempted request's KV is copied to CPU memory
 * and its progress kept ("显存与 KV 缓存", section on preemption, 抢占;
 * "vLLM intro part 2", section 9 weighs it against recomputation).  A
 * second pool of host blocks 0..num_host_blocks-1 receives the blocks; the
 * pairs returned are the copies to make with pa_swap_blocks, on the stream,
 * before anything else writes the blocks named as destinations.
 *
 * pa_bm_set_host_pool: (re)creates the host pool, free queue in `order`
 * (nullable: 0, 1, 2, ...).  PA_BM_BAD_REQUEST while a request is swapped
 * out.
 */
pa_bm_status pa_bm_set_host_pool(pa_bm* m, int32_t num_host_blocks, const int32_t* order);
int32_t pa_bm_num_host_free(const pa_bm* m);

/* Swap a complete request out: every block it holds alone (ref_cnt 1) gets
 * a host block from the head of the host queue, in table order, and the
 * pairs (gpu block, host block) go to pairs[2*p], pairs[2*p+1]; those GPU
 * blocks are then released last block first, as by pa_bm_free.  Blocks it
 * shares with other requests stay on the GPU with its reference (moving one
 * holder would free no memory).  The request keeps its token count; until
 * pa_bm_swap_in it has no block table and cannot append or fork.
 * PA_BM_NO_SPACE (nothing changed) if the host queue is short. */
pa_bm_status pa_bm_swap_out(pa_bm* m, int64_t req, int64_t* pairs, int32_t pair_cap, int32_t* num_pairs);

/* Swap it back in: each host-resident entry, in table order, takes a GPU
 * block from the free queue; pairs (host block, gpu block); the host blocks
 * return to the tail of the host queue; the request's prompt blocks are
 * registered under their prefix hashes again.  PA_BM_NO_SPACE (nothing
 * changed) if the GPU free queue is short. */
pa_bm_status pa_bm_swap_in(pa_bm* m, int64_t req, int64_t* pairs, int32_t pair_cap, int32_t* num_pairs);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
