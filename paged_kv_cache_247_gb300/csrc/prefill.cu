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
//   warps 8, 10  producers: per key tile, read the tile's block ids and
//            load every (block, head) run of K (warp 8, 4-stage ring) and of
//            V (warp 10, 3-stage ring) with 2-D TMA (cp.async.bulk.tensor,
//            128-byte swizzle).
//   warp 9   MMA issuer (one thread): S = Q K^T into tensor memory and,
//            once the softmax warps have written P, O += P V (V as an
//            MN-major operand), each issued as soon as ready; completion via
//            tcgen05.commit on mbarriers.
//            The warp also allocates and frees the tensor memory.
//   warps 0-7  softmax, two warpgroups: thread (wg, r) owns half of row r
//            of S (tcgen05.ld), applies the causal mask, exchanges the
//            half-row max through shared memory, keeps the running max and
//            its half of the sum in base 2, rescales its half of the O row
//            in tensor memory when the max grows, and writes its half of the
//            P row (same 16-bit type as V) into shared memory in the
//            swizzled K-major layout the next MMA reads.  At the end the two
//            halves' sums are combined and each stores its half of O.
//
// Tensor memory: two S buffers in columns [0, 128), O in [128, 128 + D).
// Key tiles are 64 wide; S and P are double-buffered and K and V have rings
// of their own, so the tensor core runs S_(i+1) and P_i V_i while the softmax
// warps work on tiles i and i+1.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kBM = 128;  // rows of a tile: MMA M
constexpr int kBN = 64;   // keys per tile: N of Q K^T, K of P V
constexpr int kSoftmaxWarps = 8;  // two warpgroups share each row (half the columns each)
// Warps 8..13: K producers (8, 12) and V producers (10, 13), each pair
// taking alternate tiles, and the two MMA issuers (9, 11).
constexpr int kKProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;  // issues Q K^T; owns the tensor memory
constexpr int kVProducerWarp = kSoftmaxWarps + 2;
constexpr int kPvWarp = kSoftmaxWarps + 3;   // issues P V
constexpr int kKProducerWarp2 = kSoftmaxWarps + 4;
constexpr int kVProducerWarp2 = kSoftmaxWarps + 5;
constexpr int kPrefillThreads = (kSoftmaxWarps + 6) * 32;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kKStages = 5;  // K is released as soon as its Q K^T is done,
constexpr int kVStages = 4;  // V only after its P V: separate rings
constexpr int kBufs = 2;   // S (tensor memory) and P (shared memory) are double-buffered
constexpr int kTmemCols = 512;
constexpr int kBarSlots = 32;  // mbarriers reserved in shared memory
constexpr int kKvAtom = kBN * 128;  // 64 columns (128 bytes) of the 64 key rows of a tile

// A K or V tile in shared memory: groups of 8 key rows, kGroup bytes apart;
// within a group, one 1024-byte 128-byte-swizzled atom per 64 columns.  A
// single TMA copy fills any number of whole groups with both atoms.
template <int D>
struct PrefillSmem {
  static constexpr int kAtoms = D / 64;  // 64-column atoms per row
  static constexpr int kGroup = kAtoms * 1024;
  static constexpr int kKvTile = kAtoms * kKvAtom;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKStages * kKvTile;
  // row-max exchange [2 tiles][2 halves][128] and row-sum exchange [2][128] floats
  static constexpr int kRed = kV + kVStages * kKvTile;
  static constexpr int kBar = kRed + 3 * 2 * kBM * 4;
  static constexpr int kTmemSlot = kBar + kBarSlots * 8;
  // + 1024-byte alignment slack; at least 116 KiB so that one CTA (which
  // takes all of tensor memory) is resident per SM
  static constexpr int kBytes =
      kTmemSlot + 16 + 1024 > 116 * 1024 ? kTmemSlot + 16 + 1024 : 116 * 1024;
  // tensor-memory columns: S buffers, O, Q (bf16/fp16 pairs), P buffers
  static constexpr int kColO = kBufs * kBN;
  static constexpr int kColQ = kColO + D;
  static constexpr int kColP = kColQ + D / 2;
  static_assert(kColP + kBufs * kBN / 2 <= kTmemCols, "tensor memory overflow");
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

// D (+)= A.B with the A operand read from tensor memory (row r in lane r,
// element pairs packed low-first, 8 columns per 16 elements of K) and B
// described by a shared-memory descriptor.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
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

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
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
  unsigned char* sK = smem + L::kK;
  unsigned char* sV = smem + L::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* k_full = bars;                   // K stage landed (TMA transaction bytes)
  uint64_t* k_empty = k_full + kKStages;     // K stage consumed by Q K^T (MMA commit)
  uint64_t* v_full = k_empty + kKStages;     // V stage landed
  uint64_t* v_empty = v_full + kVStages;     // V stage consumed by P V
  uint64_t* q_full = v_empty + kVStages;     // Q written to tensor memory (softmax threads)
  uint64_t* s_full = q_full + 1;             // S buffer computed (MMA commit)
  uint64_t* s_free = s_full + kBufs;         // S buffer read (softmax threads)
  uint64_t* p_full = s_free + kBufs;         // P buffer written (softmax threads)
  uint64_t* pv_done = p_full + kBufs;        // P V of that buffer finished (MMA commit)
  static_assert(2 * kKStages + 2 * kVStages + 1 + 4 * kBufs <= kBarSlots,
                "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  float* red = reinterpret_cast<float*>(smem + L::kRed);

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
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_full, kSoftmaxThreads);
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kSoftmaxThreads);
      mbar_init(&p_full[b], kSoftmaxThreads);
      mbar_init(&pv_done[b], 1);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + L::kColO;  // S buffers at columns [0, 128)
  const uint32_t tmem_q = tmem + L::kColQ;
  const uint32_t tmem_p = tmem + L::kColP;

  if (warp == kKProducerWarp || warp == kVProducerWarp || warp == kKProducerWarp2 ||
      warp == kVProducerWarp2) {
    // ----------------------------------------------------- K and V producers
    // Two warps stream K tiles and two V tiles, each operand into its own
    // ring, each warp of a pair taking every other tile: a TMA copy costs
    // its issuing warp tens of cycles, and the two warps issue in parallel.
    // Each tile's keys are loaded as runs of R rows; a run never crosses a
    // block boundary (R divides both the block size and the tile).
    const bool is_k = warp == kKProducerWarp || warp == kKProducerWarp2;
    const int first = (warp == kKProducerWarp2 || warp == kVProducerWarp2) ? 1 : 0;
    const int nstages = is_k ? kKStages : kVStages;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    unsigned char* ring = is_k ? sK : sV;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const int B = p.block_size;
    const int R = B < kBN ? B : kBN;
    const int32_t* trow = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    // Lane l copies run l (all of its columns) with one TMA copy.  The
    // block-table entry of this warp's next tile is read before this tile's copies
    // are issued, so its latency is spent while the warp waits for the next
    // free slot.
    const int seg = lane;
    auto table_entry = [&](int t) -> int {
      const int key = t * kBN + seg * R;
      return (seg < kBN / R && t < n_tiles && key < ctx) ? __ldg(trow + key / B) : 0;
    };
    int phys_next = table_entry(first);
    for (int i = first; i < n_tiles; i += 2) {
      const int st = i % nstages;
      if (i >= nstages && !mbar_wait_warp(&empty[st], ((i / nstages) - 1) & 1, p.status)) break;
      const int key0 = i * kBN;
      const int nvalid = min(ctx, key0 + kBN) - key0;
      const int nseg = (nvalid + R - 1) / R;
      int phys = phys_next;
      phys_next = table_entry(i + 2);
      if (lane == 0)
        mbar_arrive_expect_tx(&full[st], (uint32_t)nseg * R * D * (uint32_t)sizeof(T));
      __syncwarp();
      if (seg < nseg) {
        if ((unsigned)phys >= (unsigned)p.num_blocks) {
          atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
          phys = 0;
        }
        const int key = key0 + seg * R;
        const int y = (phys * p.num_kv_heads + kvh) * B + key % B;  // a multiple of 8
        tma_load_group(ring + st * L::kKvTile + seg * (R / 8) * L::kGroup, map, y / 8, &full[st]);
      }
    }
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ------------------------------------------------------- MMA issuers
    // One thread issues the chain S_i = Q K_i^T, another P_j V_j.  A single
    // thread issues a tcgen05.mma (or commit) only every ~50 cycles whatever
    // its size, while S_i with N = 64 keeps the tensor core busy for 32
    // cycles per k-step: two issuers keep it fed, and neither chain waits
    // behind the other.  Each commit tracks only its own thread's MMAs.
    if (lane == 0) {
      constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
      if (warp == kMmaWarp) {
        const uint32_t idesc_s = instr_desc(bf16, false, kBN, kBM);
        const uint32_t aK = smem_addr(sK);
        bool ok = mbar_wait(q_full, 0, p.status);
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int st = i % kKStages, b = i % kBufs;
          if (!mbar_wait(&k_full[st], (i / kKStages) & 1, p.status)) break;
          if (i >= kBufs && !mbar_wait(&s_free[b], ((i / kBufs) - 1) & 1, p.status)) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_f16_ta(tmem + b * kBN, tmem_q + ks * 8,
                       smem_desc(aK + st * L::kKvTile + (ks / 4) * 1024 + (ks % 4) * 32, 16,
                                 L::kGroup),
                       idesc_s, ks > 0);
          mma_commit(&s_full[b]);
          mma_commit(&k_empty[st]);
        }
      } else {
        const uint32_t idesc_o = instr_desc(bf16, true, D, kBM);
        const uint32_t aV = smem_addr(sV);
        for (int j = 0; j < n_tiles; ++j) {
          const int bj = j % kBufs, stj = j % kVStages;
          if (!mbar_wait(&p_full[bj], (j / kBufs) & 1, p.status)) break;
          if (!mbar_wait(&v_full[stj], (j / kVStages) & 1, p.status)) break;
          tc_fence_after();
          // V as an MN-major operand: 8-key groups kGroup bytes apart,
          // 64-column atoms 1024 bytes apart.
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            mma_f16_ta(tmem_o, tmem_p + bj * (kBN / 2) + ks * 8,
                       smem_desc(aV + stj * L::kKvTile + ks * 2 * L::kGroup, 1024, L::kGroup),
                       idesc_o,
                       (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&pv_done[bj]);
          mma_commit(&v_empty[stj]);
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- softmax / epilogue (rows)
    // Thread (wg, r): row r of the tile, columns [wg * half, (wg + 1) * half)
    // of S, P and O, with half = 32 keys of S/P and D / 2 columns of O.
    constexpr int kHalfS = kBN / 2;
    constexpr int kHalfO = D / 2;
    const int wg = warp >> 2;
    const int r = threadIdx.x & (kBM - 1);  // row of the tile == TMEM lane
    const int jq = j_first + r / Gp;
    const int g = r % Gp;
    const bool row_valid = (r / Gp) < qpt && jq < nq && g < G;
    const int pos = row_valid ? ctx - nq + jq : -1;
    const size_t row_elem =
        ((size_t)(q0 + (row_valid ? jq : 0)) * p.num_q_heads + kvh * G + (row_valid ? g : 0)) * D;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // This thread's half of the Q row into tensor memory (the A operand of
    // Q K^T): D/2 elements as D/4 columns of packed pairs.
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + row_elem) +
                         wg * (D / 16);
      uint32_t w[16];
#pragma unroll
      for (int part = 0; part < D / 64; ++part) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = row_valid ? src[part * 4 + c] : make_uint4(0, 0, 0, 0);
          w[c * 4 + 0] = v.x;
          w[c * 4 + 1] = v.y;
          w[c * 4 + 2] = v.z;
          w[c * 4 + 3] = v.w;
        }
        tmem_st16u(tmem_q + wg * (D / 4) + part * 16 + lane_base, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
    }

    float m_run = -CUDART_INF_F, l_run = 0.f;  // l_run: this half's share of the row sum
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int b = i % kBufs;
      // A wait that gives up (never expected) leaves ok false and the loop
      // running without further waits, so that both halves still meet at
      // every named barrier below.
      if (ok && !mbar_wait_warp(&s_full[b], (i / kBufs) & 1, p.status)) ok = false;
      tc_fence_after();
      float sv[kHalfS];
      tmem_ld32f(tmem + b * kBN + wg * kHalfS + lane_base, sv);
      tmem_wait_ld_bind(sv);
      tc_fence_before();
      mbar_arrive(&s_free[b]);

      // Causal mask, only on tiles where some row of the warp sees keys past
      // its position (the diagonal); elsewhere every key is visible.
      const int key0 = i * kBN + wg * kHalfS;
      if (__any_sync(0xffffffffu, key0 + kHalfS - 1 > pos)) {
#pragma unroll
        for (int c = 0; c < kHalfS; ++c)
          if (key0 + c > pos) sv[c] = -CUDART_INF_F;
      }
      // Half-row max with 8 independent chains, then the other half's via
      // shared memory (scaling by qscale > 0 commutes with the max).
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = sv[k];
#pragma unroll
      for (int c = 8; c < kHalfS; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
#pragma unroll
      for (int k = 4; k >= 1; k >>= 1)
#pragma unroll
        for (int j = 0; j < k; ++j) mx[j] = fmaxf(mx[j], mx[j + k]);
      float* red_i = red + (i & 1) * 2 * kBM;
      red_i[wg * kBM + r] = mx[0];
      named_barrier_sync(1, kSoftmaxThreads);
      const float mt = fmaxf(mx[0], red_i[(wg ^ 1) * kBM + r]) * p.qscale;
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
      for (int c = 0; c < kHalfS; c += 2) {
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

      // P buffer b is free once the P V of tile i-2 is done.
      if (ok && i >= kBufs && !mbar_wait_warp(&pv_done[b], ((i / kBufs) - 1) & 1, p.status))
        ok = false;
      // Rescaling O needs every earlier P V finished (the last is tile i-1).
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const int bp = (i - 1) % kBufs;
        if (ok && !mbar_wait_warp(&pv_done[bp], ((i - 1) / kBufs) & 1, p.status)) ok = false;
        tc_fence_after();
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < kHalfO / 32; ++c) {
          float t[32];
          const uint32_t ta = tmem_o + wg * kHalfO + lane_base + c * 32;
          tmem_ld32f(ta, t);
          tmem_wait_ld_bind(t);
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 y = __fmul2_rn(make_float2(t[k], t[k + 1]), a2);
            t[k] = y.x;
            t[k + 1] = y.y;
          }
          tmem_st32(ta, t);
        }
        tmem_wait_st();
      }
      // This half of the P row, rounded to the operand type, into tensor
      // memory (the A operand of P V).
      {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < kHalfS / 2; ++c) w[c] = Cvt<T>::from_float2(sv[2 * c], sv[2 * c + 1]);
        tmem_st16u(tmem_p + b * (kBN / 2) + wg * (kHalfS / 2) + lane_base, w);
        tmem_wait_st();
      }
      // Key rows past the context (the tail of the last block, or rows no
      // block was loaded into) must not feed NaN or stale values into P V.
      if (i * kBN + kBN > ctx) {
        // V of this tile must have landed before its tail rows are cleared.
        if (ok && !mbar_wait_warp(&v_full[i % kVStages], (i / kVStages) & 1, p.status)) ok = false;
      }
      if (wg == 0 && r < kBN && i * kBN + r >= ctx) {
        const int st = i % kVStages;
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sV + st * L::kKvTile + (r / 8) * L::kGroup + a * 1024 +
                                      (r % 8) * 128 + c * 16) =
                make_uint4(0, 0, 0, 0);
      }
      if (i * kBN + kBN > ctx)  // make the cleared V rows visible to the tensor core
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }

    // The row sum is split between the two halves.
    float* red_l = red + 2 * 2 * kBM;
    red_l[wg * kBM + r] = l_run;
    named_barrier_sync(1, kSoftmaxThreads);
    const float l_row = l_run + red_l[(wg ^ 1) * kBM + r];
    const int bl = (n_tiles - 1) % kBufs;
    if (ok && mbar_wait_warp(&pv_done[bl], ((n_tiles - 1) / kBufs) & 1, p.status)) {
      tc_fence_after();
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
      T* orow = static_cast<T*>(p.out) + row_elem + wg * kHalfO;
#pragma unroll
      for (int c = 0; c < kHalfO / 32; ++c) {
        float t[32];
        tmem_ld32f(tmem_o + wg * kHalfO + lane_base + c * 32, t);
        tmem_wait_ld_bind(t);
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
  if (warp == kMmaWarp) {
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
// 64 columns x min(block_size, 64) rows, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, int dtype, long long rows, int head_dim,
                    int block_size) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  // The cache rows [rows, head_dim] seen as (64 columns, 8 rows, head_dim / 64
  // atoms, rows / 8 groups): a box of whole groups lands as the tile layout
  // above, every atom of every group in one copy.
  const int atoms = head_dim / 64;
  const int run = block_size < kBN ? block_size : kBN;
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
