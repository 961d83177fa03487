/*
 * pagedkv.h — C ABI of the paged KV-cache decode library (libpagedkv.so).
 *
 * The library implements the hot path of PagedAttention-style serving on one
 * GPU: single-query decode attention that walks a per-sequence block table
 * (pkv_paged_attn_decode), the scatter of each step's new K/V into its slot
 * (pkv_kv_append), block-granular copy-on-write (pkv_block_copy), and a
 * host-side refcounted block allocator that decides slots and copies
 * (pkv_alloc_*).
 *
 * Sources, cited by page title and section:
 *   [P1] "800 kilobytes per token" (shashforge.dev)
 *   [P2] "Only 20.4% of your KV cache held actual tokens: how PagedAttention
 *        put a page table inside the attention kernel" (blog.teqners.com)
 *   [P3] "The KV cache is a systems problem" (rsw.lol)
 *
 * Conventions shared by every call
 *   - Pointers named *_cache, q, out, k, v, block_tables, context_lens,
 *     slot_mapping, src_dst_pairs and workspace are DEVICE pointers owned by
 *     the caller; the library never allocates, frees or retains them.
 *     Tensors are dense row-major with the shapes given per call; q, out, k,
 *     v and both caches must be 16-byte aligned.
 *   - The KV cache is two arrays (K and V) of shape
 *     [num_blocks, num_kv_heads, block_size, head_dim]: token position t of a
 *     sequence lives in logical block t / block_size at offset
 *     t % block_size, and logical block i lives in physical block
 *     block_tables[s][i].  ([P2] "The page table, relocated into attention".)
 *   - Every device call enqueues its kernels on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream) and returns without synchronising.
 *     Argument checks happen on the host before anything is enqueued; a call
 *     that returns an error has enqueued nothing.
 *   - Stream order is kept as for any kernel.  The decode, append and copy
 *     kernels are launched with programmatic stream serialization: their
 *     blocks may be placed on the GPU while the previous kernel on the stream
 *     is still running, but each waits for that kernel to finish (and for its
 *     writes to be visible) before it reads or writes memory.  A kernel the
 *     caller launches after them without that attribute starts after they
 *     finish, as usual.
 *   - Problems only visible on the device (a block id outside the pool, a
 *     context length beyond the table, a slot beyond the pool) never fault:
 *     the offending access is skipped or redirected to block 0, the result is
 *     undefined, and a PKV_DEV_* flag is raised in a per-device status word
 *     read by pkv_device_status().
 *   - The kernels never spin on another block or another launch.  Apart from
 *     the wait for the previous kernel on the stream described above, the
 *     only waits are on their own copies into shared memory, each bounded in
 *     time (PKV_DEV_WAIT_TIMEOUT).
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,          /* null pointer, bad size, misaligned pointer, ... */
  PKV_ERR_UNSUPPORTED = 2,          /* valid but not built: head_dim, block_size, grid limits */
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,  /* split decode needs more workspace than given */
  PKV_ERR_OUT_OF_BLOCKS = 4,        /* allocator: pool exhausted, state unchanged */
  PKV_ERR_CUDA = 5,                 /* a CUDA runtime call failed, see pkv_last_cuda_error() */
  PKV_ERR_UNKNOWN_SEQ = 6,          /* allocator: sequence id not live */
  PKV_ERR_SEQ_EXISTS = 7,           /* allocator: sequence id already live */
  PKV_ERR_TABLE_TOO_SMALL = 8       /* allocator: caller's table row shorter than the sequence */
} pkv_status_t;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype_t;

/* Flags of the per-device status word (bitwise OR of everything seen since
 * the last clear). */
#define PKV_DEV_BAD_BLOCK_ID 1u     /* a table entry or copy pair outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT_LEN 2u  /* context_lens[s] < 0 or > max_context_len or > table row */
#define PKV_DEV_BAD_SLOT 4u         /* slot_mapping[t] >= num_blocks * block_size */
#define PKV_DEV_WAIT_TIMEOUT 8u     /* a bounded wait inside a kernel gave up (never expected) */

/* Human-readable name of a status code (static string). */
const char* pkv_status_string(pkv_status_t status);

/* cudaError_t of the last PKV_ERR_CUDA returned on this host thread. */
int pkv_last_cuda_error(void);

/* ABI version, bumped on any incompatible change. */
int pkv_version(void);

/* ------------------------------------------------------------------------
 * Paged single-query decode attention.
 *
 * [P2] "The page table, relocated into attention": the kernel follows each
 * sequence's block table and gathers K and V from non-contiguous physical
 * blocks; [P2] "Why the KV cache is the thing that limits your batch": each
 * decode step is a memory-bound matrix-vector product per request.
 *
 * For every sequence s < num_seqs and query head h < num_q_heads:
 *   out[s][h][:] = softmax_t( scale * q[s][h] . K_s[t][h / G] ) @ V_s[t][h / G]
 * over t < context_lens[s], where G = num_q_heads / num_kv_heads (query head
 * h reads KV head h / G) and K_s[t] = k_cache[block_tables[s][t / B]][.][t % B].
 * Logits, softmax and the weighted sum are fp32; out is rounded to dtype
 * (round to nearest even).  On the tensor-core path (groups G of 2 to 32
 * query heads by default, see pkv_set_decode_path) the softmax
 * weights are rounded to dtype before the weighted sum, which the tensor
 * core accumulates in fp32 ([P3] "Calculate bytes per token before choosing
 * a batch": groups of query heads share one KV head, and a group of G heads
 * does 2 G flops per cache byte).  A sequence with context_lens[s] == 0 gets
 * zeros.
 * Positions at or beyond context_lens[s] are never read, and neither are
 * table entries past ceil(context_lens[s] / B).
 *
 *   out           [num_seqs, num_q_heads, head_dim]            dtype, written
 *   q             [num_seqs, num_q_heads, head_dim]            dtype
 *   k_cache/v_cache [num_blocks, num_kv_heads, block_size, head_dim] dtype
 *   block_tables  int32 [num_seqs, max_blocks_per_seq] (row stride
 *                 max_blocks_per_seq); entries must lie in [0, num_blocks)
 *   context_lens  int32 [num_seqs], each in [0, max_context_len] and
 *                 <= max_blocks_per_seq * block_size
 *   max_context_len  host-side upper bound on context_lens (sizes the grid)
 *   head_dim      64 or 128;  block_size 8, 16, 32, 64 or 128
 *   partition_size   tokens per split-context partition: 0 lets the library
 *                 choose (pkv_decode_partition_size); otherwise a positive
 *                 multiple of 32.  When ceil(max_context_len / partition_size)
 *                 > 1 the call writes per-partition partial results into
 *                 `workspace` and launches a second, reduction kernel.
 *   workspace     device scratch of at least pkv_decode_workspace_size(...)
 *                 bytes (may be NULL when that size is 0); its contents on
 *                 entry do not matter and it is not read after the call.
 *
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED,
 * PKV_ERR_WORKSPACE_TOO_SMALL, PKV_ERR_CUDA (launch failure).
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_paged_attn_decode(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused decode step: append the step's new token, then attend.
 *
 * One decode step appends one token per sequence and attends over the whole
 * context including it ([P2] "Why the KV cache is the thing that limits your
 * batch": the cache grows token by token; [P2] "The page table, relocated
 * into attention").  This call does both in one launch: for every sequence
 * with context_lens[s] > 0 the new token is position ctx - 1 =
 * context_lens[s] - 1, its slot is
 *   block_tables[s][(ctx - 1) / B] * B + (ctx - 1) % B,
 * and the call writes k_new[s][h][:] / v_new[s][h][:] there (bit-exact, as
 * pkv_kv_append would) while the attention uses those rows directly.  The
 * result equals pkv_kv_append followed by pkv_paged_attn_decode.
 *
 *   k_new, v_new  [num_seqs, num_kv_heads, head_dim] dtype, 16-byte aligned
 *   k_cache/v_cache are written (one row per sequence and KV head)
 * The slot's block must not be shared with another sequence (do the
 * copy-on-write pkv_block_copy first, on the same stream).  Sequences with
 * context_lens[s] == 0 append nothing.  Other arguments, results, workspace
 * and errors as pkv_paged_attn_decode.
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_paged_attn_decode_append(
    void* out, const void* q, const void* k_new, const void* v_new,
    void* k_cache, void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Allocation-free decode.  (The source pages have no counterpart: this is an
 * interface for callers, not part of the method.)
 *
 * For callers that cannot provide a workspace: engines that reserve all
 * device memory for their own pool and forbid allocation while serving, and
 * latency-critical loops where cudaMalloc, which may synchronise the device,
 * is not allowed.  Same arguments and result as pkv_paged_attn_decode minus
 * the workspace: the split-context partials go to a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.
 *
 *   - Allocates nothing (no cudaMalloc/cudaFree, no allocating library call).
 *   - Sizes whose pkv_decode_workspace_size(...) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES are rejected with PKV_ERR_WORKSPACE_TOO_SMALL
 *     before anything is enqueued; use a larger partition_size or the
 *     workspace entry point for them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - All calls on a device share the one array, which keeps whatever the
 *     last call left in it.  Nothing in it needs to start at zero (each
 *     partial is written before it is read), but calls that overlap on the
 *     GPU (different streams without ordering between them) race on it:
 *     order them on one stream or with events.
 * ---------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */

pkv_status_t pkv_paged_attn_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, pkv_stream_t stream);

/* Partition size the library picks for partition_size == 0 on the current
 * device (depends on its SM count and on the decode kernel the call will
 * use).  Returns a positive multiple of 32, or -1 for invalid arguments. */
int pkv_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int max_context_len);

/* Which decode kernel the decode calls use, process-wide (a tuning and test
 * control; the default suits every shape measured):
 *   0  chosen per call (default): the tensor-core kernel for grouped heads
 *      (groups of 2 to 32 query heads, head_dim 64 or 128, partition_size 0
 *      or a multiple of 128) and for single-head groups (MHA) with fewer
 *      than 8 (sequence, KV head) pairs per SM; the CUDA-core kernel
 *      otherwise (MHA with more pairs, or a partition the tensor-core
 *      kernel cannot take);
 *   1  always the CUDA-core kernel;
 *   2  the tensor-core kernel wherever it can run (groups of 1 to 32, head_dim
 *      64 or 128, partition_size 0 or a multiple of 128), else the CUDA-core
 *      one.
 * Both compute the same attention within the stated tolerance.  It changes
 * the partition pkv_decode_partition_size and pkv_decode_workspace_size
 * report, so set it before sizing a workspace, and not while another host
 * thread issues decode calls.  Returns PKV_ERR_INVALID_ARG for other
 * values. */
pkv_status_t pkv_set_decode_path(int path);
int pkv_get_decode_path(void);

/* 1 if a decode call with these sizes (partition_size as in
 * pkv_paged_attn_decode) runs the tensor-core kernel under the current
 * setting, 0 if the CUDA-core kernel, -1 for invalid arguments. */
int pkv_decode_uses_tensor_cores(int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_context_len, int partition_size);

/* Workspace bytes pkv_paged_attn_decode needs for these sizes (0 when the
 * call will not split).  partition_size as in pkv_paged_attn_decode.
 * Layout: fp32 partial outputs [num_seqs, num_q_heads, parts, head_dim],
 * then fp32 running maxima and fp32 denominators [num_seqs, num_q_heads,
 * parts] each, parts = ceil(max_context_len / partition).  Returns
 * (size_t)-1 for invalid arguments. */
size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_context_len, int partition_size);

/* ------------------------------------------------------------------------
 * Contiguous-cache decode: the baseline without a block table.
 *
 * [P3] "When the extra machinery is not worth it": keep a simple contiguous
 * cache as a baseline and compare both under identical token distributions;
 * [P2] "What the indirection costs": the paged kernel's price is the table
 * reads, extra branches and variable lengths.  This call runs the same
 * kernels over the pre-paging layout ([P2] opening section: one contiguous
 * tensor per request, reserved at its maximum length), so the difference to
 * pkv_paged_attn_decode on the same tokens is the cost of the indirection.
 *
 *   k_cache/v_cache [num_seqs, num_kv_heads, capacity, head_dim] dtype:
 *                 sequence s holds its positions t < context_lens[s] at
 *                 [s][h][t][:]; capacity is the reservation per sequence
 *   context_lens  int32 [num_seqs], each in [0, capacity]
 * It runs the CUDA-core decode kernel (and its partition choice) whatever
 * pkv_set_decode_path says, so it is the contiguous twin of
 * pkv_paged_attn_decode under setting 1; the workspace it needs is
 * pkv_contiguous_workspace_size.  Other arguments, results and errors as
 * pkv_paged_attn_decode (with max_context_len = capacity).
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_contiguous_attn_decode(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* context_lens, int capacity,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    float scale, pkv_dtype_t dtype, int partition_size,
    void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Workspace bytes pkv_contiguous_attn_decode needs (0 when it will not
 * split); (size_t)-1 for invalid arguments. */
size_t pkv_contiguous_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int capacity, int partition_size);

/* ------------------------------------------------------------------------
 * Multi-query (chunked prompt) attention over the paged cache.
 *
 * Prompts are processed in chunks that share the step budget with decoding
 * ([P3] "Memory savings change the scheduling question"); each chunk attends
 * causally to the sequence's cached prefix and to itself, through the block
 * table ([P2] "The page table, relocated into attention").
 *
 * Sequence s brings L_s = query_start[s+1] - query_start[s] query rows
 * q[query_start[s] .. query_start[s+1]), the last L_s positions of its
 * context: query j is position p = context_lens[s] - L_s + j, and its K/V
 * (like every position < context_lens[s]) must already be in the cache
 * (pkv_kv_append).  For every query head h:
 *   out[query_start[s] + j][h] = softmax_{t <= p}(scale * q . K_s[t][h/G]) @ V_s[t][h/G]
 * Q.K and P.V run on the tensor cores (fp32 accumulation); the softmax
 * weights P are rounded to dtype before P.V, as the operand type requires.
 *
 *   q, out        [total_queries, num_q_heads, head_dim] dtype, with
 *                 total_queries >= query_start[num_seqs] (rows of either past
 *                 total_queries are neither read nor written)
 *   query_start   int32 [num_seqs + 1], non-decreasing, starting at 0
 *   max_query_len host-side bound on L_s (sizes the grid)
 *   context_lens  int32 [num_seqs] with L_s <= context_lens[s] <= max_context_len
 *   num_q_heads / num_kv_heads <= 128
 * Other arguments as pkv_paged_attn_decode.  Errors: PKV_ERR_INVALID_ARG,
 * PKV_ERR_UNSUPPORTED (also when the caches cannot be described to the
 * tensor-memory-access unit, or when num_seqs * num_kv_heads * query tiles
 * exceeds 2^31 - 1), PKV_ERR_CUDA.
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_paged_attn_prefill(
    void* out, const void* q, int total_queries, const int32_t* query_start, int max_query_len,
    const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, pkv_dtype_t dtype,
    pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Append new tokens' K and V into their cache slots.
 *
 * The cache grows token by token ([P2] "Why the KV cache is the thing that
 * limits your batch"); logical blocks fill left to right ([P2] "The page
 * table, relocated into attention").
 *
 * For each token t < num_tokens with slot = slot_mapping[t] >= 0 and every
 * KV head h:  k_cache[slot / B][h][slot % B][:] = k[t][h][:]  (same for V).
 * Tokens with a negative slot are skipped (padding).  A byte copy: bit-exact.
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim] dtype
 *   k_cache/v_cache [num_blocks, num_kv_heads, block_size, head_dim] dtype
 *   slot_mapping  int64 [num_tokens]; flat slot = physical_block * B + offset
 * Slots must be distinct (two tokens writing one slot race).  A slot at or
 * beyond num_blocks * block_size is skipped and flags PKV_DEV_BAD_SLOT.
 * Errors: PKV_ERR_INVALID_ARG (null or misaligned pointer, negative sizes,
 * bad dtype), PKV_ERR_UNSUPPORTED (head_dim or block_size not built, or more
 * than 2^31 16-byte chunks of K in one call: 32 GiB), PKV_ERR_CUDA.
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_kv_append(
    const void* k, const void* v, void* k_cache, void* v_cache,
    const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, pkv_dtype_t dtype, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Block-granular copy-on-write.
 *
 * [P2] "The part everyone forgets: pages enable sharing, not just packing":
 * when a sample writes into a shared, partially filled block, a fresh block
 * is allocated and one block's worth of data is copied ([P1] "The old
 * answer, imported honestly": copy on write when a shared block diverges).
 *
 * For each pair i < num_pairs: copies block_bytes bytes of physical block
 * src = src_dst_pairs[2i] onto block dst = src_dst_pairs[2i+1], in k_cache
 * and in v_cache (block_bytes = num_kv_heads * block_size * head_dim *
 * element size, a multiple of 16).  Destinations must be distinct and no
 * destination may also be a source in the same call (pairs run in parallel).
 * Ids outside [0, num_blocks) skip the pair and flag PKV_DEV_BAD_BLOCK_ID.
 *
 *   src_dst_pairs int64 [num_pairs, 2], device memory
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_block_copy(
    void* k_cache, void* v_cache, const int64_t* src_dst_pairs, int num_pairs,
    int num_blocks, size_t block_bytes, pkv_stream_t stream);

/* Read (and optionally clear) the status word of the current device.
 * Synchronises `stream` first so that flags from work already enqueued on it
 * are visible.  flags may be NULL when only clearing. */
pkv_status_t pkv_device_status(uint32_t* flags, int clear, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostic for the kernels' bounded waits.
 *
 * Every wait inside the decode and prefill kernels (on the CTA's own copies,
 * MMA completions and warps) gives up after a limit (2 s), raises
 * PKV_DEV_WAIT_TIMEOUT in the device status word and lets the kernel end,
 * so that a wait that cannot complete never hangs the GPU.  This call
 * enqueues one such wait on a barrier that nothing completes: it returns
 * PKV_OK at once, the kernel ends after the limit, and pkv_device_status()
 * then reports PKV_DEV_WAIT_TIMEOUT.  The context stays usable.  Not part of
 * the hot path.
 * ---------------------------------------------------------------------- */
pkv_status_t pkv_debug_wait_timeout(pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Host-side refcounted block allocator (not on the device path).
 *
 * Fixed-size blocks, a block table per sequence, blocks taken only when all
 * earlier ones are full ([P2] "The page table, relocated into attention");
 * forked samples share blocks by reference count, a write into a shared,
 * partially filled block triggers copy-on-write, and blocks whose count
 * reaches zero return to the pool ([P2] "The part everyone forgets: pages
 * enable sharing, not just packing"; [P3] "Shared prefixes need ownership
 * rules").
 *
 * Policy: LIFO free list handing out 0, 1, 2, ... first; a sequence's blocks
 * are released from its last logical block to its first; copy-on-write iff
 * the write position is inside the last block and that block's count is
 * above one.  Every call that fails leaves the allocator unchanged.  The
 * allocator owns only ids and counts; the caller owns every tensor and must
 * order the device work it derives from these answers on its streams
 * ([P3] "Shared prefixes need ownership rules": a delayed device write must
 * not land in a block that has already been handed to another sequence).
 * Not thread-safe: one handle per host thread, or external locking.
 * ---------------------------------------------------------------------- */
typedef struct pkv_allocator pkv_allocator;

typedef struct {
  int64_t num_blocks;      /* pool size */
  int64_t free_blocks;     /* on the free list */
  int64_t used_blocks;     /* refcount > 0 */
  int64_t shared_blocks;   /* refcount > 1 */
  int64_t num_seqs;        /* live sequences */
  int64_t logical_tokens;  /* sum of live sequence lengths */
  int64_t filled_slots;    /* distinct physical slots holding a token */
  int64_t cow_copies;      /* copy-on-write events since creation */
} pkv_alloc_stats_t;

pkv_status_t pkv_alloc_create(int num_blocks, int block_size, pkv_allocator** out);
void pkv_alloc_destroy(pkv_allocator* a);
/* New sequence holding num_tokens >= 0 positions (ceil(n / B) blocks). */
pkv_status_t pkv_alloc_add_seq(pkv_allocator* a, int64_t seq_id, int num_tokens);
/* child shares every block of parent; both keep parent's length. */
pkv_status_t pkv_alloc_fork(pkv_allocator* a, int64_t parent, int64_t child);
/* Reserve the slot of the sequence's next token.  *cow_src / *cow_dst are
 * the block pair to copy before writing (both -1 when no copy is needed). */
pkv_status_t pkv_alloc_append_slot(pkv_allocator* a, int64_t seq_id, int64_t* slot,
                                   int64_t* cow_src, int64_t* cow_dst);
/* append_slot for n sequences in order.  slots[i] receives the slot of
 * seq_ids[i]; every copy needed is written to cow_pairs (int64 [n, 2]) and
 * *num_pairs receives their count.  All or nothing: if any sequence fails
 * (unknown id, pool exhausted) the appends already made in the batch are
 * undone, the allocator is left as before the call and *num_pairs is 0.
 * A sequence id may appear at most once per batch. */
pkv_status_t pkv_alloc_append_slots(pkv_allocator* a, const int64_t* seq_ids, int n,
                                    int64_t* slots, int64_t* cow_pairs, int* num_pairs);
/* Drop a sequence (finish or cancel); blocks reaching count 0 are freed. */
pkv_status_t pkv_alloc_free_seq(pkv_allocator* a, int64_t seq_id);
/* Host int32 rows [n, max_blocks] of physical ids, padded with -1. */
pkv_status_t pkv_alloc_block_table(pkv_allocator* a, const int64_t* seq_ids, int n,
                                   int32_t* out, int max_blocks);
/* Slots of positions [start, start + count) of a sequence (host int64). */
pkv_status_t pkv_alloc_seq_slots(pkv_allocator* a, int64_t seq_id, int start, int count,
                                 int64_t* out);
pkv_status_t pkv_alloc_seq_info(pkv_allocator* a, int64_t seq_id, int* num_tokens,
                                int* num_blocks);
pkv_status_t pkv_alloc_refcount(pkv_allocator* a, int block, int* refcount);
pkv_status_t pkv_alloc_stats(pkv_allocator* a, pkv_alloc_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
