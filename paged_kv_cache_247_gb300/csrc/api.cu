// The C ABI: argument checks, launch planning, and the device status word.
// Nothing here allocates device memory.

#include <cuda_runtime.h>

#include <algorithm>
#include <math.h>
#include <mutex>

#include "kernels.h"
#include "pagedkv.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kPartitionQuantum = 32;    // partitions are whole pipeline stages
constexpr int kMaxAutoPartition = 2048;  // longest partition the library picks
constexpr int kAssumedSms = 152;         // used only when no device can be queried
constexpr int kAssumedCtasPerSm = 3;

// Sticky per-device record of problems the kernels saw (PKV_DEV_* bits).
__device__ unsigned int g_device_status;

thread_local int g_last_cuda_error = 0;

std::mutex g_mutex;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

pkv_status_t cuda_fail(cudaError_t err) {
  g_last_cuda_error = static_cast<int>(err);
  return PKV_ERR_CUDA;
}

// Device address of the status word on the current device (host code may not
// take the symbol's address directly: that is a host-side shadow).
cudaError_t status_word(unsigned int** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_device_status);
    if (err != cudaSuccess) return err;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_block_size(int b) { return b == 8 || b == 16 || b == 32 || b == 64 || b == 128; }

int log2_int(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

bool decode_shape_ok(int num_seqs, int num_q_heads, int num_kv_heads, int max_context_len) {
  return num_seqs >= 0 && num_q_heads > 0 && num_kv_heads > 0 &&
         num_q_heads % num_kv_heads == 0 && max_context_len >= 0;
}

// Tokens per partition when the caller leaves the choice to the library.
//
// Every partition costs a CTA start-up (barrier set-up, table window,
// pipeline fill), a drain and a round trip of its partial result through the
// workspace, so partitions are kept long (up to 2048 tokens; measured best on
// GB300 for 1k-32k contexts).  Contexts are split into whole waves of CTAs
// where a split allows it, otherwise only as far as needed to give about four
// waves.  Batches with very few (sequence, KV head) units split finer (down to
// 256 tokens) because idle SMs cost more than partition overhead there.
//
// units: CTAs per partition index ((sequence, KV head[, head chunk]) triples);
// slots: CTAs resident on the device at once; quantum: partitions are a
// multiple of it.
int partition_for(long long units, long long slots, int max_context_len, int quantum) {
  if (max_context_len <= quantum) return quantum;
  const long long target = 4 * slots;
  const int floor_tokens = units * 4 >= slots ? 1024 : 256;
  if (units < target) {
    // Prefer a split whose CTAs fill whole waves: units * p within 5 % below
    // k waves of resident CTAs, for the fewest waves k that allows a
    // partition of [floor_tokens, kMaxAutoPartition] tokens (a multiple of
    // the quantum).  On GB300 a full single wave beat the four-wave split by
    // 11 % (8 sequences x 8k tokens) and two full waves by 6 % (16 x 8k).
    for (long long k = 1; k <= 4; ++k) {
      const long long p = k * slots / units;
      if (p < 2) continue;
      long long part = (max_context_len + p - 1) / p;
      part = ((part + quantum - 1) / quantum) * quantum;
      const long long ctas = units * ((max_context_len + part - 1) / part);
      if (part < floor_tokens || part > kMaxAutoPartition || ctas > k * slots ||
          ctas * 20 < k * slots * 19)
        continue;
      return (int)part;
    }
  }
  // Otherwise split until about four waves of CTAs: on GB300 four waves beat
  // two by up to 6 % and lost nowhere on 8-64 sequences x 1k-32k tokens, the
  // last partial wave being a smaller share of the call.
  const long long parts = units >= target ? 1 : (target + units - 1) / units;
  long long part = (max_context_len + parts - 1) / parts;
  part = ((part + 255) / 256) * 256;
  if (part < floor_tokens) part = floor_tokens;
  if (part > kMaxAutoPartition) part = kMaxAutoPartition;
  if (part >= max_context_len)
    return (int)(((long long)max_context_len + quantum - 1) / quantum * quantum);
  return (int)part;
}

int device_sms() {
  const int sms = sm_count();
  return sms > 0 ? sms : kAssumedSms;  // no device: assume a GB300
}

// Partition of the CUDA-core decode kernel.
int auto_partition(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                   int max_context_len) {
  const int group = num_q_heads / num_kv_heads;
  const int gt = pkv::decode_heads_per_cta(group);
  const long long units = (long long)num_seqs * num_kv_heads * ((group + gt - 1) / gt);
  int per_sm = sm_count() > 0 ? pkv::decode_ctas_per_sm(head_dim, gt) : 0;
  if (per_sm <= 0) per_sm = kAssumedCtasPerSm;
  return partition_for(units, (long long)device_sms() * per_sm, max_context_len,
                       kPartitionQuantum);
}

// Partition of the tensor-core decode kernel.  Its CTAs are persistent and
// take the work items (sequence, KV head, partition) in turn; the launch
// uses ceil(items / rounds) CTAs for rounds = ceil(items / SMs), so every CTA
// walks the same number of items.  The choice minimises a model of the
// call's time in units of one 128-key tile streamed at an SM's share of HBM:
//   * each round takes its items' tiles times the fraction of the SMs it
//     occupies (HBM is shared), but no less than half a tile per tile, since
//     one SM streams at most about twice its share (the bytes its copy rings
//     keep in flight);
//   * each item costs about half a tile more (its output and the switch to
//     the next item), and a split about two tiles (the partials' round trip
//     and the merge).
// On GB300 this picks the fastest of the partitions measured on 8 and 64
// sequences x 1k to 8k tokens (query-head group 4) and on 32 sequences x 4k
// tokens with groups of 4 and 32: two partitions for 8 x 8k and 8 x 32k
// (64 sequence-heads, fewer than the SMs), none from 512 sequence-heads on
// (64 x 8k: 1.04 of the copy peak unsplit against 1.00 in two), none for 4k
// tokens over 256 of them, where splitting at 2k cost 4-10 %.
int tc_partition(int num_seqs, int num_kv_heads, int max_context_len) {
  const double units = (double)num_seqs * num_kv_heads;
  const double sms = (double)device_sms();
  const long long tiles = ((long long)max_context_len + pkv::kTcPartitionQuantum - 1) /
                          pkv::kTcPartitionQuantum;
  if (tiles <= 1) return pkv::kTcPartitionQuantum;
  constexpr double kMaxRate = 2.0;    // an SM alone streams about twice its share
  constexpr double kItemCost = 0.5;   // tiles per work item
  constexpr double kSplitCost = 2.0;  // tiles for a split call
  double best_cost = 0.0;
  long long best = tiles;
  // more than about eight rounds of items never pays: the search stops there
  const double most = ceil(8.0 * sms / units);
  for (long long parts = 1; parts <= tiles && (double)parts <= most; ++parts) {
    const long long pt = (tiles + parts - 1) / parts;  // tiles per partition
    if ((tiles + pt - 1) / pt != parts) continue;      // the same partition as fewer parts
    const double items = units * (double)parts;
    const double avg = (double)tiles / (double)parts;  // tiles per item
    const double rounds = ceil(items / sms);
    const double ctas = ceil(items / rounds);          // CTAs of the launch
    const double cost = rounds * avg * fmax(ctas / sms, 1.0 / kMaxRate) + rounds * kItemCost +
                        (parts > 1 ? kSplitCost : 0.0);
    if (parts == 1 || cost < best_cost) {  // ties: fewer partitions
      best_cost = cost;
      best = pt;
    }
  }
  return (int)(best * pkv::kTcPartitionQuantum);
}

// Which decode kernel runs: 0 = chosen per call, 1 = CUDA cores, 2 = tensor
// cores (where supported).  Process-wide; see pkv_set_decode_path.
int g_decode_path = 0;

// The decode kernel and partition size of one call.  The CUDA-core kernel
// streams K/V through its FMA pipes; from a group of 8 query heads on, the
// group's 2 G flops per byte exceed what those deliver at the HBM rate.  The
// tensor-core kernel (persistent, one CTA per SM, every head of the group
// per work item) leaves the threads a few instructions per key and measured
// faster than the CUDA-core one on every grouped shape of GB300 (groups of 2
// to 32, head sizes 64 and 128, 8 to 256 sequences, 1k to 32k tokens, blocks
// of 8 to 128), so it takes every grouped call it supports.  Single-head
// groups (MHA) take the CUDA-core kernel once there are enough (sequence,
// head) pairs to fill the GPU without splitting: on the OPT-13B layer (64
// sequences of lognormal lengths, 2,560 pairs) it reaches the HBM roofline,
// 0.1172 ms, where the tensor-core kernel's static walk of unequal items
// takes 0.128-0.131.  With fewer pairs the CUDA-core kernel splits the
// contexts and pays the reduction, and the tensor-core kernel measured
// faster: 2 to 16 sequences of that layer 10-50 %, 4 and 16 sequences of 4k
// tokens over 40 heads 12 and 3 %, 8 to 64 sequences of 4k tokens over 8
// heads 4-16 % (at head size 64 as well: 8-26 %); the two
// tie at 32 sequences of the layer (1,280 pairs) and at 128 of 4k tokens over
// 8 heads (1,024).
constexpr int kMhaTcPairsPerSm = 8;  // below this many pairs per SM: tensor cores

struct DecodePlan {
  bool tc;
  int partition;
};

DecodePlan decode_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_context_len, int partition_size) {
  const int group = num_q_heads / num_kv_heads;
  const int path = __atomic_load_n(&g_decode_path, __ATOMIC_RELAXED);
  const bool few_pairs =
      (long long)num_seqs * num_kv_heads < (long long)kMhaTcPairsPerSm * device_sms();
  bool tc = path == 2 || (path == 0 && (group >= 2 || few_pairs));
  if (tc && !pkv::decode_tc_supported(head_dim, group,
                                      partition_size ? partition_size
                                                     : pkv::kTcPartitionQuantum))
    tc = false;
  if (partition_size) return {tc, partition_size};
  if (!tc)
    return {false, auto_partition(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  max_context_len)};
  return {true, tc_partition(num_seqs, num_kv_heads, max_context_len)};
}

long long num_parts_for(int max_context_len, int partition) {
  if (max_context_len <= 0) return 1;
  return (max_context_len + (long long)partition - 1) / partition;
}

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status_t status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKV_ERR_OUT_OF_BLOCKS: return "out of blocks";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_UNKNOWN_SEQ: return "unknown sequence";
    case PKV_ERR_SEQ_EXISTS: return "sequence exists";
    case PKV_ERR_TABLE_TOO_SMALL: return "block table row too small";
  }
  return "unknown status";
}

int pkv_last_cuda_error(void) { return g_last_cuda_error; }

int pkv_version(void) { return 1; }

int pkv_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int max_context_len) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, max_context_len)) return -1;
  if (head_dim != 64 && head_dim != 128) return -1;
  return decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, 0).partition;
}

size_t pkv_contiguous_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int capacity, int partition_size) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, capacity)) return (size_t)-1;
  if (head_dim != 64 && head_dim != 128) return (size_t)-1;
  if (partition_size < 0 || partition_size % kPartitionQuantum) return (size_t)-1;
  const int part = partition_size ? partition_size
                                  : auto_partition(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                   capacity);
  const long long parts = num_parts_for(capacity, part);
  if (parts <= 1) return 0;
  return (size_t)num_seqs * num_q_heads * parts * (head_dim + 2) * sizeof(float);
}

int pkv_decode_uses_tensor_cores(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_context_len, int partition_size) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, max_context_len)) return -1;
  if (head_dim != 64 && head_dim != 128) return -1;
  if (partition_size < 0 || partition_size % kPartitionQuantum) return -1;
  return decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                     partition_size).tc ? 1 : 0;
}

pkv_status_t pkv_set_decode_path(int path) {
  if (path < 0 || path > 2) return PKV_ERR_INVALID_ARG;
  __atomic_store_n(&g_decode_path, path, __ATOMIC_RELAXED);
  return PKV_OK;
}

int pkv_get_decode_path(void) { return __atomic_load_n(&g_decode_path, __ATOMIC_RELAXED); }

size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_context_len, int partition_size) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, max_context_len)) return (size_t)-1;
  if (head_dim != 64 && head_dim != 128) return (size_t)-1;
  if (partition_size < 0 || partition_size % kPartitionQuantum) return (size_t)-1;
  const int part = decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                               partition_size).partition;
  const long long parts = num_parts_for(max_context_len, part);
  if (parts <= 1) return 0;
  return (size_t)num_seqs * num_q_heads * parts * (head_dim + 2) * sizeof(float);
}

namespace {

// Shared body of the paged decode calls.  k_new/v_new (both or neither) are
// the step's new-token rows [num_seqs, num_kv_heads, head_dim] for the fused
// append.
pkv_status_t paged_decode_impl(void* out, const void* q, const void* k_new, const void* v_new,
                               void* k_cache, void* v_cache, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens,
                               int max_context_len, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               float scale, pkv_dtype_t dtype, int partition_size,
                               void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, max_context_len))
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (partition_size < 0 || partition_size % kPartitionQuantum) return PKV_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!supported_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(context_lens)) & 3u)
    return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size < max_context_len) return PKV_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;

  const int group = num_q_heads / num_kv_heads;
  const int gt = pkv::decode_heads_per_cta(group);
  const DecodePlan plan = decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_context_len, partition_size);
  const int head_chunks = plan.tc ? 1 : (group + gt - 1) / gt;
  const int part = plan.partition;
  const long long parts = num_parts_for(max_context_len, part);
  if (num_seqs > 65535 || (long long)num_kv_heads * head_chunks > 65535 || parts > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  if ((long long)num_seqs * num_q_heads > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (plan.tc && (long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;

  pkv::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_new = k_new;
  p.v_new = v_new;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_context_len = max_context_len;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.head_chunks = head_chunks;
  p.block_size = block_size;
  p.log2_block = log2_int(block_size);
  p.num_blocks = num_blocks;
  p.partition_size = part;
  p.num_parts = (int)parts;
  p.qscale = scale * 1.4426950408889634f;  // log2(e): softmax is evaluated with exp2
  if (parts > 1) {
    const size_t need = (size_t)num_seqs * num_q_heads * parts * (head_dim + 2) * sizeof(float);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    float* ws = static_cast<float*>(workspace);
    const size_t rows = (size_t)num_seqs * num_q_heads * parts;
    p.ws_o = ws;
    p.ws_m = ws + rows * head_dim;
    p.ws_l = p.ws_m + rows;
  }
  cudaError_t err = status_word(&p.status);
  if (err != cudaSuccess) return cuda_fail(err);
  if (plan.tc) {
    bool unsupported = false;
    // CTAs for the persistent walk: as many as the SMs, or fewer so that
    // every CTA walks the same number of items.  512 items on 152 SMs, say,
    // run as 4 rounds of 128 CTAs instead of 3 rounds of 152 and a fourth of
    // 56; each round still keeps HBM busy (one CTA streams about twice its
    // share), and no CTA waits out a short last round.
    const long long items = parts * num_kv_heads * (long long)num_seqs;
    const long long sms = device_sms();
    const long long rounds = (items + sms - 1) / sms;
    const int ctas = (int)std::max(1LL, (items + rounds - 1) / rounds);
    err = pkv::launch_paged_decode_tc(p, dtype, head_dim, ctas,
                                      reinterpret_cast<cudaStream_t>(stream), &unsupported);
    if (unsupported) return PKV_ERR_UNSUPPORTED;
  } else {
    err = pkv::launch_paged_decode(p, dtype, head_dim, gt,
                                   reinterpret_cast<cudaStream_t>(stream));
  }
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

}  // namespace

pkv_status_t pkv_paged_attn_decode(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int max_context_len, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int num_blocks, float scale, pkv_dtype_t dtype,
                                   int partition_size, void* workspace, size_t workspace_bytes,
                                   pkv_stream_t stream) {
  // The caches are only read on this path.
  return paged_decode_impl(out, q, nullptr, nullptr, const_cast<void*>(k_cache),
                           const_cast<void*>(v_cache), block_tables, max_blocks_per_seq,
                           context_lens, max_context_len, num_seqs, num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, scale, dtype, partition_size,
                           workspace, workspace_bytes, stream);
}

pkv_status_t pkv_paged_attn_decode_append(void* out, const void* q, const void* k_new,
                                          const void* v_new, void* k_cache, void* v_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int max_context_len,
                                          int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, int num_blocks,
                                          float scale, pkv_dtype_t dtype, int partition_size,
                                          void* workspace, size_t workspace_bytes,
                                          pkv_stream_t stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
  return paged_decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                           max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                           dtype, partition_size, workspace, workspace_bytes, stream);
}

pkv_status_t pkv_contiguous_attn_decode(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* context_lens,
                                        int capacity, int num_seqs, int num_q_heads,
                                        int num_kv_heads, int head_dim, float scale,
                                        pkv_dtype_t dtype, int partition_size, void* workspace,
                                        size_t workspace_bytes, pkv_stream_t stream) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, capacity)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (partition_size < 0 || partition_size % kPartitionQuantum) return PKV_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(context_lens) & 3u) return PKV_ERR_INVALID_ARG;
  if (capacity <= 0) return PKV_ERR_INVALID_ARG;

  const int group = num_q_heads / num_kv_heads;
  const int gt = pkv::decode_heads_per_cta(group);
  const int head_chunks = (group + gt - 1) / gt;
  const int part = partition_size ? partition_size
                                  : auto_partition(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                   capacity);
  const long long parts = num_parts_for(capacity, part);
  if (num_seqs > 65535 || (long long)num_kv_heads * head_chunks > 65535 || parts > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  if ((long long)num_seqs * num_q_heads > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;

  pkv::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = nullptr;
  p.context_lens = context_lens;
  p.max_blocks_per_seq = 1;   // one "block" per sequence: its whole reservation
  p.max_context_len = capacity;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.head_chunks = head_chunks;
  p.block_size = capacity;
  p.log2_block = 0;
  p.num_blocks = num_seqs;
  p.partition_size = part;
  p.num_parts = (int)parts;
  p.qscale = scale * 1.4426950408889634f;
  if (parts > 1) {
    const size_t need = (size_t)num_seqs * num_q_heads * parts * (head_dim + 2) * sizeof(float);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    float* ws = static_cast<float*>(workspace);
    const size_t rows = (size_t)num_seqs * num_q_heads * parts;
    p.ws_o = ws;
    p.ws_m = ws + rows * head_dim;
    p.ws_l = p.ws_m + rows;
  }
  cudaError_t err = status_word(&p.status);
  if (err != cudaSuccess) return cuda_fail(err);
  err = pkv::launch_contiguous_decode(p, dtype, head_dim, gt,
                                      reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

pkv_status_t pkv_paged_attn_prefill(void* out, const void* q, int total_queries,
                                    const int32_t* query_start, int max_query_len,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context_len,
                                    int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int num_blocks, float scale,
                                    pkv_dtype_t dtype, pkv_stream_t stream) {
  if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, max_context_len))
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (!isfinite(scale) || max_query_len < 0 || total_queries < 0) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!supported_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > 128) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0 || max_query_len == 0 || total_queries == 0) return PKV_OK;
  if (!out || !q || !query_start || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(context_lens) |
       reinterpret_cast<uintptr_t>(query_start)) & 3u)
    return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size < max_context_len) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if ((long long)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;

  pkv::PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.total_queries = total_queries;
  a.query_start = query_start;
  a.max_query_len = max_query_len;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  cudaError_t err = status_word(&a.status);
  if (err != cudaSuccess) return cuda_fail(err);
  a.sm_count = sm_count() > 0 ? sm_count() : kAssumedSms;
  bool unsupported = false;
  err = pkv::launch_paged_prefill(a, reinterpret_cast<cudaStream_t>(stream), &unsupported);
  if (unsupported) return PKV_ERR_UNSUPPORTED;
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

pkv_status_t pkv_kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                           const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, pkv_dtype_t dtype,
                           pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!supported_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return PKV_ERR_INVALID_ARG;
  if ((long long)num_tokens * num_kv_heads * head_dim * 2 / 16 > pkv::kMaxAppendChunks)
    return PKV_ERR_UNSUPPORTED;
  unsigned int* status = nullptr;
  cudaError_t err = status_word(&status);
  if (err != cudaSuccess) return cuda_fail(err);
  err = pkv::launch_kv_append(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                              head_dim, block_size, num_blocks, status,
                              reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

pkv_status_t pkv_block_copy(void* k_cache, void* v_cache, const int64_t* src_dst_pairs,
                            int num_pairs, int num_blocks, size_t block_bytes,
                            pkv_stream_t stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16)
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) return PKV_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  cudaError_t err = status_word(&status);
  if (err != cudaSuccess) return cuda_fail(err);
  err = pkv::launch_block_copy(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks,
                               block_bytes, status, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

pkv_status_t pkv_device_status(uint32_t* flags, int clear, pkv_stream_t stream) {
  unsigned int* status = nullptr;
  cudaError_t err = status_word(&status);
  if (err != cudaSuccess) return cuda_fail(err);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return cuda_fail(err);
  if (flags) {
    unsigned int host = 0;
    err = cudaMemcpyAsync(&host, status, sizeof(host), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return cuda_fail(err);
    *flags = host;
  }
  if (clear) {
    err = cudaMemsetAsync(status, 0, sizeof(unsigned int), st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return cuda_fail(err);
  }
  return PKV_OK;
}

pkv_status_t pkv_debug_wait_timeout(pkv_stream_t stream) {
  unsigned int* status = nullptr;
  cudaError_t err = status_word(&status);
  if (err != cudaSuccess) return cuda_fail(err);
  err = pkv::launch_wait_probe(status, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err);
  return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot hand this library a workspace: serving engines that
// reserve all device memory for their own pool up front and do not let a
// library allocate while it runs, and latency-critical loops where a
// cudaMalloc (which may synchronise the device) is not allowed.  For them,
// pkv_paged_attn_decode_noalloc runs the same decode with its split-context
// partials kept in a fixed array that lives in this library's device image.
// Every GPU that loads the library holds this array until the process exits.

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  Host code only sees a
// host-side stand-in under the array's name, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pkv_status_t pkv_paged_attn_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, pkv_dtype_t dtype, int partition_size,
    pkv_stream_t stream) {
  const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                max_context_len, partition_size);
  if (need == (size_t)-1) {
    // Invalid sizes: the regular entry point reports the precise error
    // before it touches any memory.
    return pkv_paged_attn_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                 context_lens, max_context_len, num_seqs, num_q_heads,
                                 num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                                 partition_size, nullptr, 0, stream);
  }
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (need > 0) {
    const cudaError_t err = noalloc_scratch(&scratch);
    if (err != cudaSuccess) return cuda_fail(err);
  }
  // The partials need no clearing: every partition writes its slot before
  // the reduction reads it, so what an earlier call left behind is ignored.
  return pkv_paged_attn_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, max_context_len, num_seqs, num_q_heads, num_kv_heads,
                               head_dim, block_size, num_blocks, scale, dtype, partition_size,
                               scratch, need > 0 ? (size_t)PKV_NOALLOC_SCRATCH_BYTES : 0, stream);
}
