// 5th-generation tensor-core (tcgen05) and TMA tensor-copy helpers shared by
// the tensor-core kernels: chunked-prompt attention and grouped-head decode.
// sm_103a only.
//
// Shared-memory operand tiles all use one layout: groups of 8 rows, the
// groups (cols / 64) KiB apart; within a group, one 1024-byte atom per 64
// columns of 16-bit elements with the 128-byte swizzle (16-byte chunk c of
// row r sits at chunk position c ^ (r & 7) of its 128-byte row).  For a
// K-major operand (K along the columns) this is the canonical layout with
// SBO = group stride; for an MN-major one (M or N along the columns) LBO is
// the 1024-byte atom stride and SBO the group stride.  One 4-D TMA copy
// (make_cache_map) fills whole groups of a cache tile with all their atoms.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pagedkv.h"

namespace pkv {
namespace tc {

// Keys per K/V tile of the tensor-core kernels (also the longest TMA run).
constexpr int kTileKeys = 128;

// Shared-memory matrix descriptor: start, leading/stride byte offsets,
// descriptor version 1 (bits 46-47), 128-byte swizzle (bits 61-63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bit 4), A and B
// type (bits 7 and 10: fp16 or bf16, always the same for both), A and B
// major (bits 15 and 16: K-major or MN-major), N / 8 (bits 17-22), M / 16
// (bits 24-28).
__device__ __forceinline__ uint32_t instr_desc(bool bf16, bool a_mn_major, bool b_mn_major, int n,
                                               int m) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// The MMA and commit helpers are warp-collective: every lane of a converged
// warp calls them with the same arguments and one lane, chosen by
// elect.sync, issues the instruction.  Issuing from a converged warp keeps
// the descriptors in the warp's uniform registers: on GB300 one warp then
// issues an MMA about every 40 cycles, against about 64 when a branch taken
// by a single lane issues it.

// D (+)= A.B with both operands described by shared-memory descriptors.
__device__ __forceinline__ void mma_f16_ss_warp(uint32_t d_tmem, uint64_t a, uint64_t b,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// D (+)= A.B with the A operand read from tensor memory (row r in lane r,
// element pairs packed low-first, 8 columns per 16 elements of K) and B
// described by a shared-memory descriptor.
__device__ __forceinline__ void mma_f16_ta_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// The barrier completes once every MMA issued before by the elected lane
// (elect.sync picks the same lane of a converged warp every time) has.
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}


// 32 consecutive 32-bit columns of this thread's TMEM lane, loaded straight
// into float registers, and a wait that names them, so that no use of the
// loaded values can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]),
        "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]),
        "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr));
}

// The same load, which also returns the maximum of the 32 loaded values of
// this thread's lane (tcgen05.ld.red with .max; on GB300 the loaded values
// are returned unchanged and the maximum matches fmaxf over them).
__device__ __forceinline__ void tmem_ld32f_max(uint32_t taddr, float* v, float* mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
      "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, "
      "[%33];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]),
        "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]),
        "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31]), "=f"(*mx)
      : "r"(taddr));
}

// Wait for this thread's outstanding tensor-memory loads, naming the loaded
// registers (and, below, a reduction result) so that no use is scheduled
// before the wait.
__device__ __forceinline__ void tmem_wait_ld_bind(float* v) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
        "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]),
        "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]),
        "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]),
        "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]), "+f"(v[31])
      :
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld_bind_max(float* v, float* mx) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
        "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]),
        "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]),
        "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]),
        "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]), "+f"(v[31]), "+f"(*mx)
      :
      : "memory");
}

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 16 consecutive 32-bit columns of this thread's lane, the wait that binds
// them, and the store back.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld_bind16(float* v) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
        "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]),
        "+f"(v[14]), "+f"(v[15])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Copy the box at coordinates (0, 0, 0, g) of a 4-D tensor map.
__device__ __forceinline__ void tma_load_group(void* dst, const CUtensorMap* map, int g,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %2, %2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(g), "r"(smem_addr(bar))
      : "memory");
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Copy the box at coordinates (0, row, 0) of a 3-D tensor map (make_rows_map).
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, int row,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %2}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_addr(bar))
      : "memory");
}

// Copy the box at coordinates (0, head, token, 0) of a 4-D map
// (make_token_head_map).
__device__ __forceinline__ void tma_load_token_heads(void* dst, const CUtensorMap* map, int head,
                                                     int token, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %2}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(head), "r"(token), "r"(smem_addr(bar))
      : "memory");
}

// 4, 8 or 16 consecutive 32-bit columns of this thread's lane, loaded and
// waited for.
template <int C>
__device__ __forceinline__ void tmem_load_small(uint32_t taddr, float* v) {
  static_assert(C == 4 || C == 8 || C == 16, "4, 8 or 16 columns");
  if constexpr (C == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3])
                 :
                 : "memory");
  } else if constexpr (C == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                   "=f"(v[6]), "=f"(v[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7])
                 :
                 : "memory");
  } else {
    tmem_ld16f(taddr, v);
    tmem_wait_ld_bind16(v);
  }
}

// 4, 8 or 16 consecutive 32-bit columns of this thread's lane stored, and
// waited for.
template <int C>
__device__ __forceinline__ void tmem_store_small(uint32_t taddr, const float* v) {
  static_assert(C == 4 || C == 8 || C == 16, "4, 8 or 16 columns");
  if constexpr (C == 4) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
                 : "memory");
  } else if constexpr (C == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
  } else {
    tmem_st16f(taddr, v);
  }
  tmem_wait_st();
}

// 32 consecutive 32-bit columns of packed pairs into this thread's lane.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]),
      "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]),
      "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]),
      "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}

// Byte offset of 16-byte chunk c of row r in a tile with COLS 16-bit columns
// in the layout above.
template <int COLS>
__device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
  return (uint32_t)((r >> 3) * (COLS / 64) * 1024 + (c >> 3) * 1024 + (r & 7) * 128 +
                    (((c & 7) ^ (r & 7)) << 4));
}

// ---- host side ------------------------------------------------------------

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    tried = true;
  }
  return fn;
}

// 4-D view of a cache for TMA: see below; boxes of min(block_size, 128)
// rows, 128-byte swizzle.
inline bool make_cache_map(CUtensorMap* map, const void* base, int dtype, long long rows, int head_dim,
                    int block_size) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  // The cache rows [rows, head_dim] seen as (64 columns, 8 rows, head_dim / 64
  // atoms, rows / 8 groups): a box of whole groups lands as the tile layout
  // above, every atom of every group in one copy.
  const int atoms = head_dim / 64;
  const int run = block_size < kTileKeys ? block_size : kTileKeys;
  const cuuint64_t dims[4] = {64, 8, (cuuint64_t)atoms, (cuuint64_t)(rows / 8)};
  const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, 128, (cuuint64_t)head_dim * 2 * 8};
  const cuuint32_t box[4] = {64, 8, (cuuint32_t)atoms, (cuuint32_t)(run / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map,
                        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of a row-major [rows, head_dim] array for TMA: (64 columns, rows,
// head_dim / 64 atoms), 128-byte swizzle.  A box of box_rows rows starting at
// any row lands as head_dim / 64 atoms of box_rows x 128 bytes each (a
// K-major operand with 8-row groups 1024 bytes apart and atoms box_rows x 128
// bytes apart); rows past the end read as zero.
inline bool make_rows_map(CUtensorMap* map, const void* base, int dtype, long long rows,
                          int head_dim, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const int atoms = head_dim / 64;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)atoms};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)atoms};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map,
                        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D view of query (or output) rows [tokens, heads, head_dim] for TMA:
// (64 columns, heads, tokens, head_dim / 64 atoms), 128-byte swizzle.  A box
// of box_heads x box_tokens = 8 rows lands as one 8-row group of the tile
// layout above, token-major, every atom of the group in one copy; rows past
// the end read as zero.
inline bool make_token_head_map(CUtensorMap* map, const void* base, int dtype, long long tokens,
                                int heads, int head_dim, int box_heads, int box_tokens) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const int atoms = head_dim / 64;
  const cuuint64_t dims[4] = {64, (cuuint64_t)heads, (cuuint64_t)tokens, (cuuint64_t)atoms};
  const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2, 128};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_tokens, (cuuint32_t)atoms};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map,
                        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace pkv
