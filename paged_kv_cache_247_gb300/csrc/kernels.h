// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Everything one paged decode launch needs.  Filled and checked by the API
// layer; the kernels trust it.
struct DecodeParams {
  void* out;                  // [S, Hq, D] element type
  const void* q;              // [S, Hq, D]
  const void* k_cache;        // [NB, Hkv, B, D]
  const void* v_cache;        // [NB, Hkv, B, D]
  const void* k_new;          // fused append only: [S, Hkv, D] rows of position ctx - 1
  const void* v_new;          // (nullptr: plain decode)
  const int32_t* block_tables;  // [S, max_blocks_per_seq]
  const int32_t* context_lens;  // [S]
  float* ws_o;                // split only: [S, Hq, num_parts, D]
  float* ws_m;                // split only: [S, Hq, num_parts] (log2 domain)
  float* ws_l;                // split only: [S, Hq, num_parts]
  unsigned int* status;       // device status word
  int max_blocks_per_seq;
  int max_context_len;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;        // Hq / Hkv
  int head_chunks;  // CTAs per KV head (ceil(group / heads per CTA))
  int block_size;
  int log2_block;
  int num_blocks;
  int partition_size;  // tokens per CTA (multiple of 32)
  int num_parts;       // ceil(max_context_len / partition_size), >= 1
  float qscale;        // scale * log2(e): logits are kept in base-2 units
};

// Query heads one CTA processes for a group size (1, 2 or 4).
int decode_heads_per_cta(int group);

// Decode CTAs resident per SM on the current device (0 if unknown).
int decode_ctas_per_sm(int head_dim, int heads_per_cta);

// Shared memory one decode CTA uses.
size_t decode_smem_bytes(int head_dim, int heads_per_cta);

// Launch the decode kernel and, when num_parts > 1, the reduction kernel.
cudaError_t launch_paged_decode(const DecodeParams& p, int dtype, int head_dim,
                                int heads_per_cta, cudaStream_t stream);

// Only the split reduction (merging num_parts partials per (sequence, query
// head)); used after the tensor-core decode kernel.
cudaError_t launch_decode_reduce(const DecodeParams& p, int dtype, int head_dim,
                                 cudaStream_t stream);

// Decode on the tensor cores: head size 64 or 128, groups of
// kMinTcGroup..kMaxTcGroup query heads (grouped heads by default, single
// heads when forced), partitions of whole 128-key tiles.
constexpr int kMinTcGroup = 1;
constexpr int kMaxTcGroup = 32;
constexpr int kTcPartitionQuantum = 128;
bool decode_tc_supported(int head_dim, int group, int partition_size);

// Persistent: min(work items, sms) CTAs, one per SM.  unsupported is set when
// the tensor maps of the caches or of q cannot be encoded.
cudaError_t launch_paged_decode_tc(const DecodeParams& p, int dtype, int head_dim, int sms,
                                   cudaStream_t stream, bool* unsupported);

// Same kernels over a contiguous cache [S, Hkv, capacity, D]: block_size is
// the capacity, block_tables is unused and sequence s reads rows of s.
cudaError_t launch_contiguous_decode(const DecodeParams& p, int dtype, int head_dim,
                                     int heads_per_cta, cudaStream_t stream);

// Multi-query (chunked prompt) attention over the paged cache.
struct PrefillArgs {
  void* out;
  const void* q;
  int total_queries;  // rows of q and out
  const int32_t* query_start;
  int max_query_len;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int max_context_len;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  float scale;
  int dtype;
  unsigned int* status;
  int sm_count;  // SMs of the device (sizes the launch order's groups)
};

// unsupported is set when the tensor maps of q or of the caches cannot be
// encoded, or the work needs more CTAs than a 1-D grid holds.
cudaError_t launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream, bool* unsupported);

// kv_append indexes (token, 16-byte chunk) pairs with 32 bits: a call may move
// at most this many chunks of K (and as many of V), 32 GiB each.
constexpr long long kMaxAppendChunks = 1LL << 31;

cudaError_t launch_kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks,
                             unsigned int* status, cudaStream_t stream);

cudaError_t launch_block_copy(void* k_cache, void* v_cache, const int64_t* pairs,
                              int num_pairs, int num_blocks, size_t block_bytes,
                              unsigned int* status, cudaStream_t stream);

// Diagnostic: one bounded wait on an mbarrier that nothing completes; it
// gives up after the wait limit and raises PKV_DEV_WAIT_TIMEOUT.
cudaError_t launch_wait_probe(unsigned int* status, cudaStream_t stream);

}  // namespace pkv
