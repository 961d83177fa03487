// Paged multi-query (chunked prompt) attention on the 5th-generation tensor
// cores of sm_103a (tcgen05.mma, accumulators in tensor memory).
//
// What it computes: sequence s brings L_s query rows, the last L_s positions
// of its context (their K/V already appended); query j at position
// p = ctx_s - L_s + j attends causally to positions 0..p, reading K/V through
// the block table ("Only 20.4% of your KV cache held actual tokens", section
// "The page table, relocated into attention"; prompt chunks: "The KV cache is
// a systems problem", section "Memory savings change the scheduling
// question").  Unlike decode this is a dense contraction: a tile of 128
// (query, head) rows against 128 keys is a 128x128xD product, twice.
//
// One CTA owns (sequence, KV head, tile of query rows).  Rows are
// (query, head-of-group) pairs, so every head of a KV group shares each K/V
// tile (grouped-query attention packs into the MMA's M dimension).
//
//   warp 4   producer: per key tile, reads the tile's block ids and loads
//            every (block, head) run of K and V with 2-D TMA
//            (cp.async.bulk.tensor, 128-byte swizzle) into a 2-stage ring.
//   warp 5   MMA issuer (one thread): S = Q K^T into tensor memory, then,
//            once the softmax warps have written P, O += P V (V as an
//            MN-major operand); completion via tcgen05.commit on mbarriers.
//            The warp also allocates and frees the tensor memory.
//   warps 0-3  softmax: thread r owns row r of S (tcgen05.ld), applies the
//            causal mask, keeps the row's running max and sum in base 2,
//            rescales its O row in tensor memory when the max grows, and
//            writes its row of P (same 16-bit type as V) into shared memory
//            in the swizzled K-major layout the next MMA reads.  At the end
//            it divides O by the sum and stores the row.
//
// Tensor memory: S in columns [0, 128), O in [128, 128 + D).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kBM = 128;  // rows of a tile: MMA M
constexpr int kBN = 128;  // keys per tile: N of Q K^T, K of P V
constexpr int kPrefillThreads = 192;
constexpr int kKvStages = 2;
constexpr int kTmemCols = 256;
constexpr int kAtomBytes = kBM * 128;  // one 64-column (128-byte) swizzle region of 128 rows

template <int D>
struct PrefillSmem {
  static constexpr int kAtoms = D / 64;                 // 64-column atoms per row
  static constexpr int kTileBytes = kAtoms * kAtomBytes;  // a Q, K or V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kKvStages * kTileBytes;
  static constexpr int kP = kV + kKvStages * kTileBytes;  // [128 rows x 128 keys]
  static constexpr int kBar = kP + 2 * kAtomBytes;
  static constexpr int kTmemSlot = kBar + 16 * 8;
  static constexpr int kBytes = kTmemSlot + 16 + 1024;    // + 1024-byte alignment slack
};

struct PrefillParams {
  void* out;                    // [total_q, Hq, D]
  const void* q;                // [total_q, Hq, D]
  const int32_t* query_start;   // [S + 1]
  const int32_t* context_lens;  // [S]
  const int32_t* block_tables;  // [S, max_blocks_per_seq]
  unsigned int* status;
  int max_blocks_per_seq;
  int max_context_len;
  int num_q_heads;
  int num_kv_heads;
  int group;        // Hq / Hkv
  int group_pow2;   // rows per query in a tile (group rounded up to a power of two)
  int block_size;
  int num_blocks;
  float qscale;     // scale * log2(e)
};

// ---- tcgen05 helpers ------------------------------------------------------

// Shared-memory matrix descriptor: start, leading/stride byte offsets,
// descriptor version 1 (bits 46-47), 128-byte swizzle (bits 61-63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A/B type, majors,
// N and M.
__device__ __forceinline__ uint32_t instr_desc(bool bf16, bool b_mn_major, int n, int m) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Same load straight into float registers, and a wait that names them, so
// that no use of the loaded values can be scheduled before the wait.
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

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte-row
// region with the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_chunk(int row, int chunk) {
  return (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4);
}

// ---- the kernel -----------------------------------------------------------

template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    paged_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap) {
  using L = PrefillSmem<D>;
  constexpr int kAtoms = L::kAtoms;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + L::kQ;
  unsigned char* sK = smem + L::kK;
  unsigned char* sV = smem + L::kV;
  unsigned char* sP = smem + L::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars;         // [2]
  uint64_t* kv_empty = bars + 2;    // [2]
  uint64_t* q_full = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* s_free = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* o_done = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int G = p.group;
  const int Gp = p.group_pow2;
  const int qpt = kBM / Gp;  // queries per tile

  const int q0 = p.query_start[s];
  const int nq = p.query_start[s + 1] - q0;
  int ctx = p.context_lens[s];
  const long long cap_ll = min((long long)p.max_context_len,
                               (long long)p.max_blocks_per_seq * p.block_size);
  if (ctx < nq || ctx > cap_ll) {
    if (threadIdx.x == 0 && qt == 0) atomicOr(p.status, PKV_DEV_BAD_CONTEXT_LEN);
    if (ctx < nq || nq <= 0) return;  // nothing sensible to attend to
    ctx = (int)cap_ll;
  }
  const int j_first = qt * qpt;
  if (j_first >= nq) return;  // this tile has no queries
  const int j_last = min(nq, j_first + qpt) - 1;
  const int pos_max = ctx - nq + j_last;
  const int n_tiles = pos_max / kBN + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(q_full, kBM);
    mbar_init(s_full, 1);
    mbar_init(s_free, kBM);
    mbar_init(p_full, kBM);
    mbar_init(o_done, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + kBN;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int B = p.block_size;
    const int32_t* trow = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % kKvStages;
      if (i >= kKvStages && !mbar_wait_warp(&kv_empty[st], ((i / kKvStages) - 1) & 1, p.status))
        break;
      const int key0 = i * kBN;
      const int key_end = min(ctx, key0 + kBN);
      const int lb0 = key0 / B;
      const int nblk = (key_end - 1) / B - lb0 + 1;
      int phys = 0;
      if (lane < nblk) {
        phys = __ldg(trow + lb0 + lane);
        if ((unsigned)phys >= (unsigned)p.num_blocks) {
          atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
          phys = 0;
        }
      }
      if (lane == 0)
        mbar_arrive_expect_tx(&kv_full[st], (uint32_t)nblk * B * D * (uint32_t)sizeof(T) * 2);
      __syncwarp();
      if (lane < nblk) {
        const int y = (phys * p.num_kv_heads + kvh) * B;
        const int row = lane * B;  // key row inside the tile
#pragma unroll
        for (int a = 0; a < kAtoms; ++a) {
          tma_load_2d(sK + st * L::kTileBytes + a * kAtomBytes + row * 128, &kmap, 64 * a, y,
                      &kv_full[st]);
          tma_load_2d(sV + st * L::kTileBytes + a * kAtomBytes + row * 128, &vmap, 64 * a, y,
                      &kv_full[st]);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
      const uint32_t idesc_s = instr_desc(bf16, false, kBN, kBM);
      const uint32_t idesc_o = instr_desc(bf16, true, D, kBM);
      const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV),
                     aP = smem_addr(sP);
      bool ok = mbar_wait(q_full, 0, p.status);
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % kKvStages;
        if (!mbar_wait(&kv_full[st], (i / kKvStages) & 1, p.status)) break;
        if (i > 0 && !mbar_wait(s_free, (i - 1) & 1, p.status)) break;
        tc_fence_after();
        // S = Q K^T over D in steps of 16 (4 steps per 64-column atom)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * kAtomBytes + (ks % 4) * 32;
          mma_f16(tmem_s, smem_desc(aQ + off, 16, 1024),
                  smem_desc(aK + st * L::kTileBytes + off, 16, 1024), idesc_s, ks > 0);
        }
        mma_commit(s_full);
        if (!mbar_wait(p_full, i & 1, p.status)) break;
        tc_fence_after();
        // O += P V over the tile's 128 keys in steps of 16; V is read as an
        // MN-major operand: 8-key groups 1024 B apart, 64-column atoms
        // kAtomBytes apart.
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint32_t offp = (ks / 4) * kAtomBytes + (ks % 4) * 32;
          mma_f16(tmem_o, smem_desc(aP + offp, 16, 1024),
                  smem_desc(aV + st * L::kTileBytes + ks * 16 * 128, kAtomBytes, 1024), idesc_o,
                  (i > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&kv_empty[st]);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- softmax / epilogue (rows)
    const int r = threadIdx.x;  // row of the tile == TMEM lane
    const int jq = j_first + r / Gp;
    const int g = r % Gp;
    const bool row_valid = (r / Gp) < qpt && jq < nq && g < G;
    const int pos = row_valid ? ctx - nq + jq : -1;
    const size_t row_elem =
        ((size_t)(q0 + (row_valid ? jq : 0)) * p.num_q_heads + kvh * G + (row_valid ? g : 0)) * D;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    // Q row into the swizzled K-major tile (zeros for padding rows).
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + row_elem);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 w = row_valid ? src[c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sQ + (c / 8) * kAtomBytes + sw128_chunk(r, c % 8)) = w;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(q_full);
    }

    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      if (!mbar_wait_warp(s_full, i & 1, p.status)) { ok = false; break; }
      tc_fence_after();
      float sv[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32f(tmem_s + lane_base + c * 32, &sv[c * 32]);
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_wait_ld_bind(&sv[c * 32]);
      tc_fence_before();
      mbar_arrive(s_free);

      // Causal mask, only on tiles where some row of the warp sees keys past
      // its position (the diagonal); elsewhere every key is visible.
      const int key0 = i * kBN;
      if (__any_sync(0xffffffffu, key0 + kBN - 1 > pos)) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c > pos) sv[c] = -CUDART_INF_F;
      }
      // Row max with 8 independent chains (scaling by qscale > 0 commutes).
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = sv[k];
#pragma unroll
      for (int c = 8; c < kBN; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
#pragma unroll
      for (int k = 4; k >= 1; k >>= 1)
#pragma unroll
        for (int j = 0; j < k; ++j) mx[j] = fmaxf(mx[j], mx[j + k]);
      const float mt = mx[0] * p.qscale;
      // Lazy rescaling: the running max moves only when this tile exceeds it
      // by more than 8 (base 2), so P stays <= 2^8 and O is rescaled rarely.
      // Numerator and denominator share the same max, so the result is exact.
      const float m_new = (mt > m_run + 8.f) ? mt : m_run;
      const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
      const float negm = (m_new == -CUDART_INF_F) ? 0.f : -m_new;
      const float2 qs2 = make_float2(p.qscale, p.qscale);
      const float2 nm2 = make_float2(negm, negm);
      float sm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sm[k] = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), qs2, nm2);
        sv[c] = ex2(x.x);
        sv[c + 1] = ex2(x.y);
        sm[(c >> 1) & 7] += sv[c] + sv[c + 1];
      }
#pragma unroll
      for (int k = 4; k >= 1; k >>= 1)
#pragma unroll
        for (int j = 0; j < k; ++j) sm[j] += sm[j + k];
      l_run = l_run * alpha + sm[0];
      m_run = m_new;

      // P V of the previous tile must be done before P and O are touched.
      if (i > 0) {
        if (!mbar_wait_warp(o_done, (i - 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float t[32];
            tmem_ld32f(tmem_o + lane_base + c * 32, t);
            tmem_wait_ld_bind(t);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float2 y = __fmul2_rn(make_float2(t[k], t[k + 1]), a2);
              t[k] = y.x;
              t[k + 1] = y.y;
            }
            tmem_st32(tmem_o + lane_base + c * 32, t);
          }
          tmem_wait_st();
        }
      }
      // P row, rounded to the operand type, in the swizzled K-major layout.
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        uint4 w;
        w.x = Cvt<T>::from_float2(sv[c * 8 + 0], sv[c * 8 + 1]);
        w.y = Cvt<T>::from_float2(sv[c * 8 + 2], sv[c * 8 + 3]);
        w.z = Cvt<T>::from_float2(sv[c * 8 + 4], sv[c * 8 + 5]);
        w.w = Cvt<T>::from_float2(sv[c * 8 + 6], sv[c * 8 + 7]);
        *reinterpret_cast<uint4*>(sP + (c / 8) * kAtomBytes + sw128_chunk(r, c % 8)) = w;
      }
      // Key rows past the context (the tail of the last block, or rows no
      // block was loaded into) must not feed NaN or stale values into P V.
      if (key0 + r >= ctx) {
        const int st = i % kKvStages;
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sV + st * L::kTileBytes + a * kAtomBytes + r * 128 + c * 16) =
                make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(p_full);
    }

    if (ok && mbar_wait_warp(o_done, (n_tiles - 1) & 1, p.status)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      T* orow = static_cast<T*>(p.out) + row_elem;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float t[32];
        tmem_ld32(tmem_o + lane_base + c * 32, t);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 w;
            w.x = Cvt<T>::from_float2(t[k] * inv, t[k + 1] * inv);
            w.y = Cvt<T>::from_float2(t[k + 2] * inv, t[k + 3] * inv);
            w.z = Cvt<T>::from_float2(t[k + 4] * inv, t[k + 5] * inv);
            w.w = Cvt<T>::from_float2(t[k + 6] * inv, t[k + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + k) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

// ---- host side ------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D view of a cache: rows (block, head, slot), columns head_dim; boxes of
// 64 columns x block_size rows, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, int dtype, long long rows, int head_dim,
                    int block_size) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)block_size};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map,
                        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_prefill_typed(const PrefillParams& p, const CUtensorMap& km,
                                 const CUtensorMap& vm, int q_tiles, int num_seqs,
                                 cudaStream_t stream) {
  using L = PrefillSmem<D>;
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    err = cudaFuncSetAttribute(paged_prefill_kernel<T, D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  const dim3 grid(q_tiles, p.num_kv_heads, num_seqs);
  paged_prefill_kernel<T, D><<<grid, kPrefillThreads, L::kBytes, stream>>>(p, km, vm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream, bool* map_failed) {
  *map_failed = false;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.num_kv_heads * a.block_size;
  if (!make_cache_map(&km, a.k_cache, a.dtype, rows, a.head_dim, a.block_size) ||
      !make_cache_map(&vm, a.v_cache, a.dtype, rows, a.head_dim, a.block_size)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  int gp = 1;
  while (gp < a.num_q_heads / a.num_kv_heads) gp <<= 1;
  PrefillParams p{};
  p.out = a.out;
  p.q = a.q;
  p.query_start = a.query_start;
  p.context_lens = a.context_lens;
  p.block_tables = a.block_tables;
  p.status = a.status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.max_context_len = a.max_context_len;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.group_pow2 = gp;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.qscale = a.scale * 1.4426950408889634f;
  const int qpt = kBM / gp;
  const int q_tiles = (a.max_query_len + qpt - 1) / qpt;
  if (a.dtype == PKV_F16) {
    return a.head_dim == 64
               ? launch_prefill_typed<__half, 64>(p, km, vm, q_tiles, a.num_seqs, stream)
               : launch_prefill_typed<__half, 128>(p, km, vm, q_tiles, a.num_seqs, stream);
  }
  return a.head_dim == 64
             ? launch_prefill_typed<__nv_bfloat16, 64>(p, km, vm, q_tiles, a.num_seqs, stream)
             : launch_prefill_typed<__nv_bfloat16, 128>(p, km, vm, q_tiles, a.num_seqs, stream);
}

}  // namespace pkv
