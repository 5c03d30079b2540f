/*
 * pkv.h -- C ABI of the paged-KV-cache decode-attention library (libpkv.so).
 *
 * One decode step of a transformer layer over a paged KV cache, for one GPU
 * (NVIDIA GB300, sm_103a):
 *
 *   1. the new token's K and V are written in place into their cache slots
 *      (pkv_append) -- no reallocation, old entries are never recomputed
 *      ("为什么“推理优化”不是锦上添花", sec. 3.1; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 *      sec. 4.3);
 *   2. every query head attends over all cached positions of its request,
 *      out = softmax(scale * q . K^T) . V, with K/V gathered block by block
 *      through the request's block table (pkv_decode_attention, or the
 *      explicit split pair pkv_decode_partition + pkv_merge)
 *      ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2 and 4.2).
 *
 * The cache is cut into fixed-size blocks that requests reference through
 * per-request block tables; blocks can be shared between requests (a common
 * prompt prefix) ("推理优化这件事，为什么值得反复复盘", sec. 4.2 and 4.3;
 * "为什么“推理优化”不是锦上添花", sec. 3.2, scheme 1).  The host block pool
 * (pkv_pool_*) hands out block ids, counts references and frees blocks.
 *
 * Conventions shared by every call
 * --------------------------------
 *   * Cache layout: k_cache and v_cache are fp16 arrays
 *     [num_blocks][num_kv_heads][block_size][head_dim], contiguous.  Slot s
 *     is (block s / block_size, offset s % block_size).
 *   * GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   * block_tables: int32 [num_seqs][max_blocks_per_seq]; entry i of row b
 *     is the physical block holding logical tokens [i*bs, (i+1)*bs) of
 *     request b.  Entries at or past ceil(context_lens[b] / block_size) are
 *     never read.
 *   * context_lens: int32 [num_seqs], the number of cached tokens of each
 *     request INCLUDING the token appended in this step.  0 is allowed and
 *     yields a zero output row.
 *   * Pointers named *_cache, q, out, k_new, v_new, o_part, m_part, l_part,
 *     block_tables, context_lens, slot_mapping and workspace are DEVICE
 *     pointers owned by the caller.  The library never allocates, frees or
 *     retains device memory (its only device memory is the static scratch
 *     array of pkv_decode_attention_noalloc, part of the loaded module) and
 *     keeps no pointer after a call returns.
 *   * Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream): they validate arguments on the host, enqueue
 *     kernels and return without synchronising.  A call that returns an
 *     error has enqueued nothing.
 *   * Inside the kernels, indices that would leave a buffer (a block id
 *     outside [0, num_blocks), a context longer than its table, a slot
 *     outside the pool) are clamped or skipped and recorded in a per-device
 *     error word; pkv_get_device_error reports and clears it.  No kernel
 *     traps, asserts or spins without bound.
 *   * Thread safety: calls may be issued from several host threads; the
 *     pool object is not internally locked (one owner thread per pool).
 *   * Cache formats: fp16 K and V (the calls without a suffix); int8 keys with
 *     fp16 values (*_int8k); int8 keys and values (*_int8kv); fp8 (E4M3) keys
 *     and values (*_fp8kv).  The 8-bit forms keep one float32 scale per
 *     (token, kv head) row beside the codes; their sections below give the
 *     layouts and the quantisation rule.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

/* ---------------------------------------------------------------- status */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG -1   /* null pointer, bad shape, misaligned pointer */
#define PKV_ERR_UNSUPPORTED -2   /* valid but not implemented (head_dim, group size, ...) */
#define PKV_ERR_CUDA -3          /* a CUDA runtime call or kernel launch failed */
#define PKV_ERR_OUT_OF_BLOCKS -4 /* the pool has fewer free blocks than requested */
#define PKV_ERR_WORKSPACE -5     /* workspace missing or smaller than required */
#define PKV_ERR_DEVICE_CHECK -6  /* a kernel recorded an out-of-range index */

/* Codes recorded in the device error word (see pkv_get_device_error). */
#define PKV_DEV_OK 0
#define PKV_DEV_BAD_BLOCK_ID 1   /* block table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT 2    /* context_lens[b] > max_blocks_per_seq * block_size */
#define PKV_DEV_BAD_SLOT 3       /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEV_WAIT_TIMEOUT 4   /* an asynchronous copy did not complete in time */
#define PKV_DEV_PREFIX_MISMATCH 5 /* a block table does not start with the shared prefix's blocks */
#define PKV_DEV_SMEM_MISALIGNED 6 /* dynamic shared memory not 1024-byte aligned (the CTA skipped its tokens) */

/* Defaults and limits of the decode kernels. */
#define PKV_HEAD_DIM 128             /* the only head_dim the decode kernels take */
#define PKV_DEFAULT_PARTITION 1024   /* split-context partition used by pkv_decode_attention */
#define PKV_MAX_PARTITION 4096       /* largest partition_size accepted */
#define PKV_MIN_BLOCK_SIZE 16        /* block_size must be a multiple of 16 ... */
#define PKV_MAX_BLOCK_SIZE 256       /* ... and at most 256 */

/* Flags of the pkv_decode_step* calls.
 * PKV_STEP_OVERLAP: the call's kernels may start reading this call's block
 * tables, context lengths and cached K/V rows (every position before each
 * request's new token; with prefix_len > 0 the shared prefix) while the kernel
 * issued just before them on `stream` is still running; q, k_new, v_new, the
 * workspace and out are touched only after that kernel has completed, and the
 * call's own kernels let the next kernel on the stream start the same way.  Set
 * it only when that preceding kernel writes neither this call's caches nor its
 * tables or context lengths: e.g. the previous layer's step (another cache) or
 * the projection that produced q, k_new and v_new.  Not for two steps in a row
 * on the same cache, where the second reads the row the first appended.
 * Source: the library's scheduling (programmatic dependent launch), not the
 * pages; results are identical with and without it.  Without the flag every
 * kernel still launches as a programmatic dependent but reads nothing before
 * the preceding kernel completes. */
#define PKV_STEP_OVERLAP 1u

typedef struct CUstream_st *pkv_stream_t; /* == cudaStream_t */
typedef struct pkv_pool pkv_pool;         /* opaque host object */

/* Human-readable name of a PKV_* status code (static storage, never NULL).
 * Library plumbing; the pages describe no counterpart. */
PKV_API const char *pkv_status_string(int status);

/* Library version as 10000*major + 100*minor + patch.  Library plumbing; the
 * pages describe no counterpart. */
PKV_API int pkv_version(void);

/* ================================================================ host pool
 * Paged allocation of KV-cache blocks, freed on every exit path of a request,
 * with reference counts for blocks shared as a common prefix
 * ("推理优化这件事，为什么值得反复复盘", sec. 4.2: paged management, allocate on
 * demand and free at request end including on failure, shared-prefix cache).
 * All pool calls are host-only and synchronous.
 */

/* Create a pool of num_blocks (1 .. 2^31-1) free blocks (the preallocated
 * block pool of the pages' paged cache, sec. 4.2 of the page above).  The free
 * list is a permutation of 0..num_blocks-1 drawn from `seed` (splitmix64 +
 * Fisher-Yates), so consecutive allocations scatter over the pool, as the pages
 * say history K/V ends up ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2:
 * random addresses).  *out receives the pool;
 * release it with pkv_pool_destroy.  Errors: INVALID_ARG. */
PKV_API int pkv_pool_create(int64_t num_blocks, uint64_t seed, pkv_pool **out);

/* Release a pool (NULL is ignored).  Outstanding block ids become invalid. */
PKV_API void pkv_pool_destroy(pkv_pool *pool);

/* Allocate n blocks (all or nothing), each with reference count 1, writing
 * their ids to ids[0..n-1].  Errors: INVALID_ARG, OUT_OF_BLOCKS (nothing is
 * allocated and ids is untouched). */
PKV_API int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *ids);

/* Add one reference to each of n allocated blocks (prefix sharing, sec. 4.2 of
 * the page above).  All ids
 * are checked before any count changes.  Errors: INVALID_ARG (an id that is
 * out of range or not allocated). */
PKV_API int pkv_pool_share(pkv_pool *pool, int n, const int32_t *ids);

/* Drop one reference from each of n blocks; a block whose count reaches 0
 * returns to the free list.  All ids are checked first (and an id listed
 * more times than its count is an error), so a failed call changes nothing.
 * Errors: INVALID_ARG. */
PKV_API int pkv_pool_free(pkv_pool *pool, int n, const int32_t *ids);

/* Number of free blocks, or -1 for a NULL pool. */
PKV_API int64_t pkv_pool_num_free(const pkv_pool *pool);

/* Reference count of block id (0 = free), or -1 if id is out of range. */
PKV_API int pkv_pool_refcount(const pkv_pool *pool, int32_t id);

/* Grow one request's block table so that it covers new_tokens tokens:
 * table_row[0 .. ceil(cur_tokens/bs)) are the blocks the request holds; the
 * blocks needed for tokens [cur_tokens, new_tokens) are allocated (all or
 * nothing) and written after them.  Errors: INVALID_ARG (new_tokens would
 * exceed max_blocks * block_size, or new_tokens < cur_tokens), OUT_OF_BLOCKS. */
PKV_API int pkv_pool_reserve(pkv_pool *pool, int32_t *table_row, int max_blocks,
                             int cur_tokens, int new_tokens, int block_size);

/* Fork: a new request starts as a copy of the first num_tokens tokens of another
 * (a shared prefix, sec. 4.2 of the page above).
 * dst_row[0 .. ceil(num_tokens/bs)) receives the same block ids as src_row and
 * every one of those blocks gains a reference (shared, not copied).  Errors:
 * INVALID_ARG (an id not allocated, or more blocks than max_blocks). */
PKV_API int pkv_pool_fork(pkv_pool *pool, const int32_t *src_row, int32_t *dst_row, int max_blocks,
                          int num_tokens, int block_size);

/* Make position `cur_tokens` of a request writable before its token is
 * appended (copy-on-write: this library's reading of how a block shared as a
 * prefix, sec. 4.2 of the page above, stays unchanged for its other readers).  If the position starts a new block, one block is allocated and
 * written to table_row.  If it falls inside a block that other requests also
 * reference (reference count > 1), that block is copied on write: a fresh
 * block replaces it in table_row, the old block loses this request's
 * reference, and *copy_src / *copy_dst receive the pair the caller must copy
 * on the device (pkv_copy_blocks) before appending; *n_copies is 1 then, else
 * 0.  Errors: INVALID_ARG, OUT_OF_BLOCKS (nothing changed). */
PKV_API int pkv_pool_prepare_append(pkv_pool *pool, int32_t *table_row, int max_blocks,
                                    int cur_tokens, int block_size, int32_t *copy_src,
                                    int32_t *copy_dst, int *n_copies);

/* Drop the request's reference to each of its ceil(num_tokens/bs) blocks (the
 * end of a request, whether it finished or failed); all-or-nothing as
 * pkv_pool_free.  Errors: INVALID_ARG. */
PKV_API int pkv_pool_free_table(pkv_pool *pool, const int32_t *table_row, int num_tokens,
                                int block_size);

/* Swap a request's blocks between two pools (device cache <-> host swap space,
 * either direction; the pages name page-level swap in/out as a benefit of
 * paging: "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2).  For the
 * n = ceil(num_tokens / bs) blocks of table_row (ids in `from`): n blocks are
 * allocated in `to`, src_ids[i] / dst_ids[i] receive the pair (old id, new id)
 * to copy (pkv_copy_blocks_between), the old blocks are released in `from`,
 * and table_row[i] becomes the new id.  Every block must be held by this
 * request alone (reference count 1): a block other requests still read cannot
 * leave.  All-or-nothing: on error nothing changes.  The copy must be enqueued
 * before any later kernel reuses the released blocks (same stream order).
 * Errors: INVALID_ARG (shared or unallocated block, row too short),
 * OUT_OF_BLOCKS (`to` has fewer than n free blocks). */
PKV_API int pkv_pool_swap(pkv_pool *from, pkv_pool *to, int32_t *table_row, int max_blocks, int num_tokens,
                          int block_size, int32_t *src_ids, int32_t *dst_ids);

/* Host slot mapping for one new token per request: the page-table lookup from a
 * logical position to its physical slot ("为什么“推理优化”不是锦上添花", sec. 3.2,
 * scheme 1: fixed-size pages found through a page table):
 *   slots[b] = block_tables[b][positions[b] / bs] * bs + positions[b] % bs,
 * and slots[b] = -1 when positions[b] < 0 (no token for that request).
 * block_tables, positions and slots are HOST pointers.  Errors: INVALID_ARG
 * (a position past the table or a negative block id in a read entry). */
PKV_API int pkv_slot_mapping(int64_t *slots, const int32_t *block_tables, const int32_t *positions,
                             int num_seqs, int max_blocks_per_seq, int block_size);

/* ================================================================ device calls */

/* In-place append of one decode step's new K/V into the cache: the new token's
 * entries are written into the preallocated cache at their slots, no tensor is
 * rebuilt or reallocated ("为什么“推理优化”不是锦上添花", sec. 3.1: write the new
 * K/V into a preallocated cache; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 4.3: in-place append instead of torch.cat).
 *   k_cache, v_cache : fp16 [num_blocks][num_kv_heads][block_size][head_dim], 16-byte aligned
 *   slot_mapping     : int64 [num_tokens]; token t goes to slot slot_mapping[t];
 *                      a negative slot skips the token (padding)
 *   k_new, v_new     : fp16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 * Each (token, kv head) row is copied bit for bit with 16-byte stores.  Two
 * tokens naming the same slot race (the caller must not do that).
 * head_dim must be a multiple of 8; block_size >= 1.  A slot >= num_blocks *
 * block_size is skipped and recorded as PKV_DEV_BAD_SLOT.
 * Errors: INVALID_ARG, CUDA. */
PKV_API int pkv_append(void *k_cache, void *v_cache, const int64_t *slot_mapping,
                       const void *k_new, const void *v_new, int num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, pkv_stream_t stream);

/* Copy whole blocks (every kv head, every slot) of both caches -- the device
 * half of copy-on-write for blocks shared between requests
 * ("推理优化这件事，为什么值得反复复盘", sec. 4.2 shares prefix blocks; the copy of
 * a shared block before a write into it is this library's reading of that
 * sharing):
 *   k_cache[dst[i]] <- k_cache[src[i]], v_cache[dst[i]] <- v_cache[src[i]], i < n,
 * bit for bit (copy-on-write of a shared block).  src and dst are DEVICE int32
 * arrays; a destination must not appear twice nor also be a source.  Ids
 * outside [0, num_blocks) skip the pair and are recorded as
 * PKV_DEV_BAD_BLOCK_ID.  head_dim must be a multiple of 8.
 * Errors: INVALID_ARG, CUDA. */
PKV_API int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst, int n,
                            int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                            pkv_stream_t stream);

/* Copy whole blocks from one pool to another of the same geometry -- the
 * device half of swapping a request's pages out of and back into the cache
 * ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2: page-level swap):
 *   dst_k[dst_ids[i]] <- src_k[src_ids[i]], dst_v[dst_ids[i]] <- src_v[src_ids[i]],
 * bit for bit (swap out / swap in).  Either pool may be host memory the GPU can
 * address (page-locked, e.g. cudaHostAlloc or a pinned torch tensor): the copy
 * kernel reads and writes it directly.  src_ids / dst_ids must be readable by
 * the GPU.  Pair i is skipped, and PKV_DEV_BAD_BLOCK_ID recorded, when an id
 * is outside its pool.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
PKV_API int pkv_copy_blocks_between(void *dst_k, void *dst_v, int64_t dst_num_blocks, const void *src_k,
                                    const void *src_v, int64_t src_num_blocks, const int32_t *src_ids,
                                    const int32_t *dst_ids, int n, int num_kv_heads, int head_dim,
                                    int block_size, pkv_stream_t stream);

/* Bytes of workspace pkv_decode_attention needs for contexts up to
 * max_context tokens (0 when one partition covers max_context): fp32 partials
 * for every (request, q head, partition) followed by one int completion
 * counter per (request, q head).  Source: the pages attend over a request's
 * whole context in one pass and do not split it; the split into partitions
 * and their log-sum-exp merge (see pkv_decode_partition) is this library's
 * design for long contexts, exact because softmax over a union of token
 * ranges is the l-weighted merge of the softmaxes over the ranges. */
PKV_API size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                         int max_context, int partition_size);

/* One decode step of attention for every request and query head: read every
 * cached K of the request, score it against q, normalise with softmax and take
 * the weighted sum of V ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.2),
 * with K/V gathered through the request's page table (same page, sec. 3.2):
 *   out[b][h][:] = softmax(scale * q[b][h] . K_b^T) . V_b
 * over the context_lens[b] cached tokens of request b, K_b/V_b gathered
 * through block_tables (kv head h / (num_q_heads / num_kv_heads)).
 *   out : fp16 [num_seqs][num_q_heads][head_dim], 8-byte aligned
 *   q   : fp16 [num_seqs][num_q_heads][head_dim], 16-byte aligned
 * Requirements: head_dim == 128; num_q_heads / num_kv_heads in {1, 2, 4, 8};
 * block_size a multiple of 16 in [16, 256]; caches 16-byte aligned.
 * When max_blocks_per_seq * block_size <= PKV_DEFAULT_PARTITION every request
 * is done by one pass and the workspace is not used (may be NULL).  Otherwise
 * contexts are split into partitions of PKV_DEFAULT_PARTITION tokens that run
 * in parallel and are merged by log-sum-exp inside the same kernel (the last
 * partition of a request to finish merges them); requests that fit one
 * partition still finish in one pass.  When a request can span at least 8
 * partitions and the grid fills at least three waves of resident CTAs, odd
 * partitions start a quarter partition early, so that partition lengths
 * alternate (P - P/4, P + P/4; the count per request is unchanged) and the
 * CTAs of one wave do not all end together; the result is the same up to
 * rounding order.  The split needs
 * pkv_decode_workspace_size(num_seqs, num_q_heads, 128, max_blocks_per_seq *
 * block_size, PKV_DEFAULT_PARTITION) bytes of 256-byte-aligned workspace whose
 * counter region is zero when the workspace is first used (zero-fill a new
 * workspace once, e.g. cudaMemsetAsync); every call leaves the counters zero.
 * Calls that share a workspace must be ordered (one stream).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
PKV_API int pkv_decode_attention(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, int num_seqs,
                                 int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size, int64_t num_blocks, float scale,
                                 void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Bytes of workspace pkv_decode_attention_shared_prefix needs: fp32 partials for
 * ceil(prefix_len / 128) prefix chunks plus up to ceil((max_context - prefix_len) / 64)
 * suffix partitions per (request, q head) (the call picks the suffix partition,
 * 64..512 tokens, from the grid it gives), then one int counter per
 * (request, q head).  0 for invalid arguments. */
PKV_API size_t pkv_shared_prefix_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                                int max_context, int prefix_len);

/* Decode attention for a batch whose block tables all begin with the same
 * prefix_len / block_size blocks (a shared prompt prefix: "推理优化这件事，为什么值得
 * 反复复盘", sec. 4.2; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2).  The
 * result equals pkv_decode_attention on the same arguments, but the prefix's
 * K/V is read once per kv head for the whole batch instead of once per
 * request: a first kernel scores every request's query rows against the
 * prefix in 128-token chunks (tensor-core MMA over the B x G rows of each kv
 * head), a second runs the split decode over each request's suffix (tokens
 * from prefix_len on) and a third merges each request's prefix chunks and
 * suffix partitions by log-sum-exp (the three launched back to back on
 * `stream`, the later two as programmatic dependents).
 * Requirements (besides those of pkv_decode_attention): prefix_len > 0 and a
 * multiple of block_size; context_lens[b] >= prefix_len; row b of
 * block_tables starts with the same prefix_len / block_size ids as row 0
 * (checked on the device: PKV_DEV_PREFIX_MISMATCH); workspace of
 * pkv_shared_prefix_workspace_size(num_seqs, num_q_heads, 128,
 * max_blocks_per_seq * block_size, prefix_len) bytes, 256-byte aligned, whose
 * counter region is zero before first use (calls leave it zero).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
PKV_API int pkv_decode_attention_shared_prefix(void *out, const void *q, const void *k_cache,
                                               const void *v_cache, const int32_t *block_tables,
                                               const int32_t *context_lens, int num_seqs,
                                               int max_blocks_per_seq, int num_q_heads,
                                               int num_kv_heads, int head_dim, int block_size,
                                               int64_t num_blocks, float scale, int prefix_len,
                                               void *workspace, size_t workspace_bytes,
                                               pkv_stream_t stream);

/* Workspace for pkv_decode_step: pkv_decode_workspace_size(..., max_context,
 * PKV_DEFAULT_PARTITION) when prefix_len is 0, else
 * pkv_shared_prefix_workspace_size(..., prefix_len).  Source: the split and its
 * merge are this library's (see pkv_decode_workspace_size), not the pages'. */
PKV_API size_t pkv_decode_step_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                              int max_context, int prefix_len);

/* One whole decode step in one call: append each request's new token in
 * place, then attend over every cached token including it
 * ("为什么“推理优化”不是锦上添花", sec. 3.1; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 4.2 and 4.3).
 *   k_new, v_new : fp16 [num_seqs][num_kv_heads][head_dim], 16-byte aligned; the
 *                  token of request b goes to logical position context_lens[b] - 1,
 *                  i.e. slot block_tables[b][(ctx-1)/bs] * bs + (ctx-1) % bs, which
 *                  must lie in an allocated block (a request with context 0
 *                  appends nothing; an invalid block id skips the write and is
 *                  recorded as PKV_DEV_BAD_BLOCK_ID)
 *   k_cache, v_cache : written (the new rows) and read.
 * prefix_len 0: same result as pkv_slot_mapping(positions = ctx - 1) +
 * pkv_append + pkv_decode_attention.  prefix_len > 0: same as pkv_append +
 * pkv_decode_attention_shared_prefix (the new token must lie past the prefix).
 * The append is fused into the decode kernel: the CTA that owns a request's
 * last position writes the row to the cache and uses it directly, so a step
 * is one kernel launch (three with a shared prefix).  Workspace rules as for the
 * matching attention call.  flags: 0 or PKV_STEP_OVERLAP (other bits are
 * INVALID_ARG).  Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
PKV_API int pkv_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                            void *k_cache, void *v_cache, const int32_t *block_tables,
                            const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, float scale, int prefix_len, void *workspace,
                            size_t workspace_bytes, unsigned flags, pkv_stream_t stream);

/* ---- int8 key cache ------------------------------------------------------
 * Keys stored as int8 codes with one float32 scale per (block, kv head, slot);
 * values stay fp16.  The pages report that int8 halves cache memory but that
 * quality suffers on long sequences, and advise quantising only the keys
 * ("推理优化这件事，为什么值得反复复盘", sec. 4.4; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 4.2).  Scheme (the pages give none): per key row of 128 dims,
 *   scale = max_d |k_d| / 127           (float32, IEEE division)
 *   code_d = round-half-even(k_d / scale), in [-127, 127]   (float32 quotient)
 * and an all-zero row stores scale 0 and zero codes.  Attention uses
 * k_d = code_d * scale.  Layouts:
 *   k_codes : int8 [num_blocks][num_kv_heads][block_size][128], 16-byte aligned
 *   k_scale : float32 [num_blocks][num_kv_heads][block_size], 16-byte aligned
 *   v_cache : fp16 [num_blocks][num_kv_heads][block_size][128] as for pkv_append.
 * Per cached token and kv head this reads 128 + 4 + 256 bytes instead of 512. */

/* Append into the int8-key cache: for each token t with slot_mapping[t] >= 0,
 * quantise k_new[t][j] into k_codes/k_scale at that slot and copy v_new[t][j]
 * into v_cache.  Argument rules, skips and errors as pkv_append (k_new/v_new
 * 8-byte aligned).  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
PKV_API int pkv_append_int8k(void *k_codes, float *k_scale, void *v_cache, const int64_t *slot_mapping,
                             const void *k_new, const void *v_new, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, pkv_stream_t stream);

/* pkv_decode_attention over the int8-key cache: the same result definition with
 * every key dequantised, the same shapes, workspace (pkv_decode_workspace_size)
 * and error rules.  Any group size 1, 2, 4 or 8 runs on the tensor cores. */
PKV_API int pkv_decode_attention_int8k(void *out, const void *q, const void *k_codes, const float *k_scale,
                                       const void *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                       pkv_stream_t stream);

/* pkv_decode_step over the int8-key cache: the new token's key is quantised and
 * written (codes and scale) with its value by the decode kernel itself, then
 * attended.  Same as pkv_append_int8k at positions ctx - 1 followed by
 * pkv_decode_attention_int8k.  No shared-prefix form.  Workspace as
 * pkv_decode_attention_int8k.  flags as pkv_decode_step.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
PKV_API int pkv_decode_step_int8k(void *out, const void *q, const void *k_new, const void *v_new, void *k_codes,
                                  float *k_scale, void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                  unsigned flags, pkv_stream_t stream);

/* ---- int8 keys and values (optional) --------------------------------------
 * Values quantised by the same per-row scheme as the keys: int8 codes
 * v_codes [num_blocks][num_kv_heads][block_size][128] and float32 v_scale
 * [num_blocks][num_kv_heads][block_size]; attention uses v_d = code_d * scale.
 * 128 + 4 + 128 + 4 bytes per cached token and kv head instead of 512.  The
 * pages advise keeping values in high precision (quality on long generations,
 * "推理优化这件事，为什么值得反复复盘", sec. 4.4): this is the option for callers
 * that accept that trade; the int8-key cache above is the default form. */

/* Append into the int8 K + V cache: both rows quantised at each slot.  Rules and
 * errors as pkv_append_int8k. */
PKV_API int pkv_append_int8kv(void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                              const int64_t *slot_mapping, const void *k_new, const void *v_new, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                              pkv_stream_t stream);

/* pkv_decode_attention over the int8 K + V cache (keys and values dequantised).
 * Scales 16-byte aligned.  Workspace and errors as pkv_decode_attention_int8k. */
PKV_API int pkv_decode_attention_int8kv(void *out, const void *q, const void *k_codes, const float *k_scale,
                                        const void *v_codes, const float *v_scale, const int32_t *block_tables,
                                        const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                        pkv_stream_t stream);

/* pkv_decode_step over the int8 K + V cache: the new token's key and value rows
 * are quantised and written by the decode kernel, then attended.  Same as
 * pkv_append_int8kv at positions ctx - 1 followed by pkv_decode_attention_int8kv.
 * flags as pkv_decode_step. */
PKV_API int pkv_decode_step_int8kv(void *out, const void *q, const void *k_new, const void *v_new, void *k_codes,
                                   float *k_scale, void *v_codes, float *v_scale, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                   int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                   unsigned flags, pkv_stream_t stream);

/* ---- fp8 (E4M3) keys and values (optional) ---------------------------------
 * The pages compress the cache to 8 bits per element ("推理优化这件事，为什么值得反复复盘",
 * sec. 4.4; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.2) and name FP8 as the
 * 8-bit number format the hardware handles natively (the latter page, sec. 2).
 * This cache stores 8-bit floating-point codes in the layout of the int8 K + V
 * cache: k_codes and v_codes uint8 [num_blocks][num_kv_heads][block_size][128],
 * 16-byte aligned; k_scale and v_scale float32 [num_blocks][num_kv_heads]
 * [block_size], 16-byte aligned for the decode calls.  Each code is E4M3 (sign,
 * 4 exponent bits with bias 7, 3 fraction bits; exponent field 0 holds
 * subnormals; 0x7F and 0xFF are NaN; largest finite 448).  Per row (token, kv
 * head): scale = max_d |x_d| / 448 and code_d = the E4M3 value nearest to
 * x_d / scale (ties to the even code; a negative quotient that rounds to zero
 * gives -0, 0x80), both in float32, magnitudes clamped to 448; an all-zero row
 * has scale 0 and codes 0.  Attention uses x_d = value(code_d) * scale.  Same
 * bytes as int8 K + V (264 per cached token and kv head); a relative step of
 * 2^-3 instead of int8's uniform max/127, so coarser for large elements and
 * finer for small ones.  Rows the caller writes itself must hold no NaN code
 * at positions below the context length. */

/* Append into the fp8 K + V cache: both rows quantised at each slot.  Rules and
 * errors as pkv_append_int8k. */
PKV_API int pkv_append_fp8kv(void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                             const int64_t *slot_mapping, const void *k_new, const void *v_new, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                             pkv_stream_t stream);

/* pkv_decode_attention over the fp8 K + V cache (keys and values dequantised).
 * Workspace and errors as pkv_decode_attention_int8kv. */
PKV_API int pkv_decode_attention_fp8kv(void *out, const void *q, const void *k_codes, const float *k_scale,
                                       const void *v_codes, const float *v_scale, const int32_t *block_tables,
                                       const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                       pkv_stream_t stream);

/* pkv_decode_step over the fp8 K + V cache: the new token's key and value rows
 * are quantised and written by the decode kernel, then attended.  Same as
 * pkv_append_fp8kv at positions ctx - 1 followed by pkv_decode_attention_fp8kv.
 * flags as pkv_decode_step. */
PKV_API int pkv_decode_step_fp8kv(void *out, const void *q, const void *k_new, const void *v_new, void *k_codes,
                                  float *k_scale, void *v_codes, float *v_scale, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                                  unsigned flags, pkv_stream_t stream);

/* ---- several new tokens per request ----------------------------------------
 * A verified draft (speculative decoding) or a prefill chunk: request b brings
 * n_b = query_start[b + 1] - query_start[b] new tokens whose K/V are already in
 * the cache (pkv_append with their slots), so context_lens[b] counts them.
 * Query row i of the request sits at logical position ctx_b - n_b + i and
 * attends causally to positions 0 .. ctx_b - n_b + i:
 *   out[t][h] = softmax(scale * q[t][h] . K[0..pos]^T) V[0..pos],
 *   t = query_start[b] + i, pos = ctx_b - n_b + i
 * (the pages list chunked prefill and speculative decoding among the ways to
 * run decode over the same cache: "LLM推理优化：从硬件瓶颈到KV Cache的工程实践",
 * sec. 3.2).  n_b = 1 for every request is pkv_decode_attention. */
#define PKV_MAX_QUERY_LEN 1024

/* Workspace bytes for pkv_decode_attention_multi (0 when no request can need
 * a split: every table fits one PKV_DEFAULT_PARTITION-token partition). */
PKV_API size_t pkv_decode_multi_workspace_size(int num_seqs, int total_q, int max_query_len, int num_q_heads,
                                               int num_kv_heads, int head_dim, int max_context);

/* Causal attention of every request's new tokens over its paged cache.
 *   q, out      : fp16 [total_q][num_q_heads][head_dim] (q 16-byte, out 8-byte aligned)
 *   query_start : device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0,
 *                 query_start[num_seqs] = total_q; every n_b <= max_query_len
 *                 (<= PKV_MAX_QUERY_LEN) and n_b <= ctx_b.  A request with n_b = 0
 *                 is skipped; inconsistent rows are skipped and recorded as
 *                 PKV_DEV_BAD_CONTEXT.
 * Other arguments as pkv_decode_attention.  One CTA serves C (token, head) rows
 * of one kv head and one PKV_DEFAULT_PARTITION-token partition, C = 8 when
 * max_query_len * G <= 8 and 16 otherwise, so K/V is read by ceil(n_b * G / C)
 * CTAs that run back to back (L2 serves the repeats); the split's merge is
 * fused as in pkv_decode_attention.  Workspace: zero-filled
 * before first use, left zeroed, at least pkv_decode_multi_workspace_size bytes,
 * 256-byte aligned.  Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
PKV_API int pkv_decode_attention_multi(void *out, const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       const int32_t *query_start, int num_seqs, int total_q, int max_query_len,
                                       int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int64_t num_blocks, float scale, void *workspace,
                                       size_t workspace_bytes, pkv_stream_t stream);

/* Largest max_query_len of pkv_decode_step_multi (the new rows a CTA patches are
 * staged in its shared memory). */
#define PKV_MAX_STEP_QUERY_LEN 16

/* One several-token step in one launch: append each request's new tokens in
 * place, then attend causally over its cache (the append of pkv_decode_step,
 * "为什么“推理优化”不是锦上添花", sec. 3.1, applied to a verified draft or a
 * prefill chunk, "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2).
 *   k_new, v_new : fp16 [total_q][num_kv_heads][head_dim], 16-byte aligned; row
 *                  query_start[b] + i goes to logical position ctx_b - n_b + i of
 *                  request b (its slot in block_tables[b]; an invalid block id skips
 *                  the write and is recorded as PKV_DEV_BAD_BLOCK_ID)
 *   k_cache, v_cache : written (the new rows) and read.
 * Same result as pkv_append at those positions followed by
 * pkv_decode_attention_multi; max_query_len <= PKV_MAX_STEP_QUERY_LEN (else
 * UNSUPPORTED).  Every CTA whose token range holds new positions patches their
 * rows into its shared-memory tiles; the CTA of the request's last row group
 * also writes them to the cache.  flags: 0 or PKV_STEP_OVERLAP (as
 * pkv_decode_step; the query starts count among what the preceding kernel must
 * not write).  Other arguments, workspace and errors as pkv_decode_attention_multi. */
PKV_API int pkv_decode_step_multi(void *out, const void *q, const void *k_new, const void *v_new, void *k_cache,
                                  void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                                  const int32_t *query_start, int num_seqs, int total_q, int max_query_len,
                                  int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int64_t num_blocks, float scale, void *workspace,
                                  size_t workspace_bytes, unsigned flags, pkv_stream_t stream);

/* pkv_decode_step (prefix_len 0) with the split-context partition chosen by the
 * caller instead of PKV_DEFAULT_PARTITION (the split and its log-sum-exp merge
 * are this library's design, exact by the softmax identity noted at
 * pkv_decode_workspace_size; the pages do not split a context): a multiple of 16 in
 * [16, PKV_MAX_PARTITION]; 0 selects the default.  Smaller partitions give more
 * CTAs per request (short batches, very long contexts), larger ones amortise
 * each CTA's start-up.  Workspace: pkv_decode_workspace_size(..., max_context,
 * partition_size).  Other arguments, results and errors as pkv_decode_step. */
PKV_API int pkv_decode_step_partition(void *out, const void *q, const void *k_new, const void *v_new,
                                      void *k_cache, void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, float scale, int partition_size, void *workspace,
                                      size_t workspace_bytes, unsigned flags, pkv_stream_t stream);

/* Split-context partial attention.  Source: not the pages, which attend over a
 * whole context in one pass; this is one half of the library's split for long
 * contexts, defined so that pkv_merge of these partials equals the one-pass
 * softmax exactly in real arithmetic (softmax over a union of token ranges is
 * the merge below of per-range statistics).  Partition p of request b covers logical
 * tokens [p * partition_size, min(ctx_b, (p + 1) * partition_size)); for each
 * such partition and query head h it writes
 *   m_part[b][h][p]      = max score (natural-log units, scale applied)
 *   l_part[b][h][p]      = sum over the partition of exp(score - m)
 *   o_part[b][h][p][:]   = sum exp(score - m) v / l   (normalised, fp32)
 * o_part: fp32 [num_seqs][num_q_heads][max_partitions][head_dim];
 * m_part, l_part: fp32 [num_seqs][num_q_heads][max_partitions].
 * Partitions at or past ceil(ctx_b / partition_size) are not written, except
 * that an empty request (ctx_b == 0) gets m = -inf, l = 0, o = 0 in partition 0.
 * max_partitions must be >= ceil(max_blocks_per_seq * block_size / partition_size);
 * partition_size a multiple of 16 in [16, PKV_MAX_PARTITION].  Other
 * requirements as pkv_decode_attention.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
PKV_API int pkv_decode_partition(float *o_part, float *m_part, float *l_part, const void *q,
                                 const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 int num_seqs, int max_blocks_per_seq, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int64_t num_blocks, float scale, int partition_size,
                                 int max_partitions, pkv_stream_t stream);

/* Log-sum-exp merge of the partials of pkv_decode_partition (the other half of
 * the library's split; the pages do not define it: it is the softmax identity
 * that rebuilds the one-pass result from per-range max, sum and average):
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
 * over the ceil(ctx_b / partition_size) partitions of each request, rounded
 * to fp16 (round to nearest even); an empty request gets a zero row.
 * out: fp16 [num_seqs][num_q_heads][head_dim].  Errors: INVALID_ARG, CUDA. */
PKV_API int pkv_merge(void *out, const float *o_part, const float *m_part, const float *l_part,
                      const int32_t *context_lens, int num_seqs, int num_q_heads, int head_dim,
                      int partition_size, int max_partitions, pkv_stream_t stream);

/* Size of the library's built-in scratch array used by pkv_decode_attention_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */

/* Allocation-free form of pkv_decode_attention.  The pages describe no
 * counterpart: this call exists for callers that cannot allocate device memory.
 *
 * Who needs it: plugins hosted by another runtime that owns all device memory
 * and hands them only input and output pointers; latency-bound serving loops
 * that ban allocator calls (and the device-wide synchronisation cudaMalloc
 * implies) once they are running.  Neither can supply the split workspace
 * pkv_decode_attention asks for.
 *
 * Same arguments, semantics and results as pkv_decode_attention, minus the
 * workspace: the split partials live in a file-scope static __device__ array
 * of PKV_NOALLOC_SCRATCH_BYTES bytes inside libpkv.so.  Every GPU on which the
 * library's kernels are loaded holds that array until the process exits.  The
 * first call on a device looks up the array's device address (with that
 * device current) and caches it for the life of the process; make that first
 * call before any stream capture begins.  A cudaDeviceReset of the device
 * invalidates the cached address: do not call this entry on a device after
 * resetting it.  Nothing here calls cudaMalloc, cudaFree or any allocating
 * routine.  Every argument is checked before any CUDA call.
 *
 * Limit and sharing: a call whose split needs more than
 * PKV_NOALLOC_SCRATCH_BYTES (pkv_decode_workspace_size with max_context =
 * max_blocks_per_seq * block_size and partition PKV_DEFAULT_PARTITION) is
 * refused with PKV_ERR_WORKSPACE before anything is enqueued.  All calls share
 * the one array, and it keeps the previous call's contents; the only part
 * that must start at zero (the split's completion counters) is cleared by
 * each call on `stream` before its kernel runs, and every partial a call
 * reads it has written itself.  Calls whose kernels overlap on the GPU
 * (unordered streams, or several host threads) race on the array: order them
 * on one stream.
 * Errors: as pkv_decode_attention, plus WORKSPACE for oversize requests and
 * CUDA if the address look-up fails. */
PKV_API int pkv_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, int num_seqs,
                                         int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int64_t num_blocks,
                                         float scale, pkv_stream_t stream);

/* Synchronise `stream`, then report (in *code) and clear the device error
 * word of the current device (library plumbing for failure detection; the pages
 * describe no counterpart): PKV_DEV_OK when no kernel recorded an index
 * problem since the last call.  Returns PKV_OK, or CUDA when a runtime call
 * fails.  This is the only library call that synchronises. */
PKV_API int pkv_get_device_error(pkv_stream_t stream, int *code);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
