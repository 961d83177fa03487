// Cache maintenance kernels: kv_append (slot scatter) and block_copy
// (copy-on-write), both plain 16-byte vector copies.
//
// kv_append: each decode step writes one token of K and V per sequence into
// its slot ("Only 20.4% of your KV cache held actual tokens", sections "Why
// the KV cache is the thing that limits your batch" and "The page table,
// relocated into attention").  The source row of a token is contiguous
// ([Hkv, D]); in the cache each head's D elements are contiguous at
// ((block * Hkv + h) * B + offset) * D.
//
// block_copy: copy-on-write of a shared, partially filled block copies one
// block's worth of data ("Only 20.4% ...", section "The part everyone
// forgets: pages enable sharing, not just packing"); one block of one cache
// is Hkv * B * D contiguous elements.
//
// Both are HBM-bound byte copies: every thread moves 16-byte chunks and
// keeps several loads in flight before it stores.

#include "common.cuh"
#include "overlap.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 2;      // kv_append: 2 chunks of K and 2 of V per thread
constexpr int kCopyUnroll = 8;  // block_copy: 16 chunks (K and V) in flight per thread

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// The (token, 16-byte chunk) pairs of the whole call form one index space,
// chunk i being chunk i % row_chunks of token i / row_chunks (the source rows
// are contiguous, so i also indexes k and v).  Every thread moves kUnroll
// chunks of K and of V whatever the width of a token's row: 128 chunks for 8
// heads of 128, 640 for 40.  Chunk c of a token belongs to head
// c >> log2_cpr.  The data loads are issued first, since their addresses do
// not depend on the slot; the slot reads then overlap them.
__global__ void __launch_bounds__(kCopyThreads)
    kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     const int64_t* __restrict__ slot_mapping, unsigned total_chunks,
                     unsigned row_chunks, int log2_cpr, int num_kv_heads, int block_size,
                     long long num_slots, unsigned int* status) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  const unsigned cpr_mask = (1u << log2_cpr) - 1u;
  const unsigned i0 = blockIdx.x * (unsigned)(kCopyThreads * kUnroll) + threadIdx.x;
  uint4 rk[kUnroll], rv[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const unsigned i = i0 + u * kCopyThreads;
    if (i < total_chunks) {
      rk[u] = load_stream(k + i);
      rv[u] = load_stream(v + i);
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const unsigned i = i0 + u * kCopyThreads;
    if (i >= total_chunks) continue;
    const unsigned t = i / row_chunks;
    const unsigned c = i - t * row_chunks;
    const long long slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (c == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const long long blk = slot / block_size;
    const long long off = slot - blk * block_size;
    const size_t dst =
        ((((size_t)blk * num_kv_heads + (c >> log2_cpr)) * block_size + off) << log2_cpr) +
        (c & cpr_mask);
    k_cache[dst] = rk[u];
    v_cache[dst] = rv[u];
  }
}

// grid.x covers one block's chunks, grid.y walks the pairs.
__global__ void __launch_bounds__(kCopyThreads)
    block_copy_kernel(uint4* k_cache, uint4* v_cache, const int64_t* __restrict__ pairs,
                      int num_pairs, long long chunks_per_block, int num_blocks,
                      unsigned int* status) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  for (int i = blockIdx.y; i < num_pairs; i += gridDim.y) {
    const long long src = pairs[2 * i];
    const long long dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK_ID);
      continue;
    }
    const uint4* ks = k_cache + src * chunks_per_block;
    const uint4* vs = v_cache + src * chunks_per_block;
    uint4* kd = k_cache + dst * chunks_per_block;
    uint4* vd = v_cache + dst * chunks_per_block;
    for (long long c0 = (long long)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
         c0 < chunks_per_block; c0 += (long long)gridDim.x * kCopyThreads * kCopyUnroll) {
      uint4 rk[kCopyUnroll], rv[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const long long c = c0 + u * kCopyThreads;
        if (c < chunks_per_block) {
          // Sources are read-only for the whole launch (no destination may
          // be a source in the same call), so the non-coherent path is safe.
          rk[u] = load_stream(ks + c);
          rv[u] = load_stream(vs + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const long long c = c0 + u * kCopyThreads;
        if (c < chunks_per_block) {
          kd[c] = rk[u];
          vd[c] = rv[u];
        }
      }
    }
  }
}

// Diagnostic: thread 0 waits on an mbarrier that nothing arrives on, with
// the same bounded wait the decode and prefill pipelines use.  The wait
// gives up after the limit, raises PKV_DEV_WAIT_TIMEOUT and returns, so the
// kernel ends and the context stays usable.
__global__ void wait_probe_kernel(unsigned int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status);
}

}  // namespace

cudaError_t launch_wait_probe(unsigned int* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks,
                             unsigned int* status, cudaStream_t stream) {
  const int cpr = head_dim * 2 / 16;  // 16-byte chunks per head row
  const int log2_cpr = cpr == 8 ? 3 : 4;
  const long long row_chunks = (long long)num_kv_heads * cpr;
  const long long total = (long long)num_tokens * row_chunks;
  if (total > kMaxAppendChunks) return cudaErrorInvalidValue;  // rejected by the caller first
  const long long span = kCopyThreads * kUnroll;
  const unsigned gx = (unsigned)((total + span - 1) / span);
  return launch_overlapped(
      kv_append_kernel, dim3(gx), dim3(kCopyThreads), 0, stream,
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, (unsigned)total, (unsigned)row_chunks,
      log2_cpr, num_kv_heads, block_size, (long long)num_blocks * block_size, status);
}

cudaError_t launch_block_copy(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                              int num_blocks, size_t block_bytes, unsigned int* status,
                              cudaStream_t stream) {
  const long long cpb = (long long)(block_bytes / 16);
  long long gx = (cpb + kCopyThreads * kCopyUnroll - 1) / (kCopyThreads * kCopyUnroll);
  if (gx > 65535) gx = 65535;
  const int gy = num_pairs < 65535 ? num_pairs : 65535;
  return launch_overlapped(block_copy_kernel, dim3((unsigned)gx, gy), dim3(kCopyThreads), 0,
                           stream, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                           pairs, num_pairs, cpb, num_blocks, status);
}

}  // namespace pkv
