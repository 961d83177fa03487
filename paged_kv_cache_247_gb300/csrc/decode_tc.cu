// Grouped-head paged decode on the 5th-generation tensor cores (tcgen05),
// head sizes 64 and 128.
//
// What it computes is what paged_decode_kernel computes ("Only 20.4% of your
// KV cache held actual tokens", section "The page table, relocated into
// attention"): for each sequence and query head, softmax(scale * q . K) V over
// the sequence's context, K and V gathered through the block table.  It is
// the path for query-head groups ("The KV cache is a systems problem",
// section "Calculate bytes per token before choosing a batch": groups of
// query heads share one KV head).  A group of G heads does 2 G flops per
// cache byte; from G = 8 on, that is more than the CUDA cores deliver at the
// HBM rate, so the contraction goes to the tensor core, and at any G the
// per-key work left to the threads is a few instructions.
//
// Orientation: the keys of a 128-key tile are the MMA's M dimension (one
// tensor-memory lane per key), the group's heads its N dimension:
//
//   S^T [128 keys x N]  = K_tile [128 x D] . Q^T      A = K tile (K-major),
//                                                     B = Q rows (K-major)
//   O^T [D x N]        += V_tile^T . P^T              A = V tile (MN-major),
//                                                     B = P^T (K-major)
//
// for head size 128.  For head size 64 (an M of 64 would need another
// accumulator layout) the second product is O [128 x D] += P . V with the
// heads on M: P^T [heads x keys] is the K-major A operand, V the MN-major B
// operand, rows past the group unused.
//
// N is the group rounded up to 16 or 32.  A work item is (sequence, KV head,
// partition of the context) with every head of the group, so each K/V tile is
// read from HBM once per group.  The kernel is persistent: one CTA per SM
// walks the items c, c + grid, c + 2 grid, ...; its rings, barriers and
// tensor memory flow from item to item, so an SM pays its start-up once and
// the next item's copies are in flight while this one finishes.  Warps:
//
//   key warpgroups (1, or 2 for groups above 16, each with half the heads):
//              thread t reads S^T lane t (key t of the tile) and computes
//              P^T column t = exp2(x - m) per head, with a running maximum per
//              head that moves only when a tile exceeds it by more than 8
//              (base 2; the warpgroup then agrees on the new maxima and
//              rescales its partial sums and O^T); partial row sums stay per
//              thread.  At the end of an item thread d normalises and writes
//              dimension d of its heads (head size 128), or thread h the D
//              outputs of head h (head size 64).
//   K producer the item's Q rows (one TMA copy), and one 4-D TMA copy per
//              (block, head) run of K into a ring of tiles.
//   V producer the same for V.
//   S issuer   S^T of each tile (8 MMAs); owns the tensor memory.
//   O issuer   the P.V product of each tile (8 MMAs).
//
// Tensor memory: S^T in two buffers of N columns, O in two (items alternate,
// so an item's output is read while the next one accumulates).
// The split-context partials (o, m, l in base 2) have the layout and meaning
// of paged_decode_kernel's, so the same reduction kernel merges them.

#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "overlap.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

using namespace tc;

constexpr int kKeys = kTileKeys;        // keys per tile: M of S^T, K of the P.V product
constexpr int kGroupP = (kKeys / 64) * 1024; // bytes between 8-head groups of P^T
constexpr int kBarSlots = 48;

constexpr int pow2_at_least(int x, int p = 32) { return p >= x ? p : pow2_at_least(x, 2 * p); }

// NH: the group rounded up to a power of two (4 .. 32); D: head size (64 or
// 128).  For D = 128 the P.V product is O^T [D x N] = V^T P^T (M = D); for
// D = 64, where an M of 64 would be needed, it is O [128 x D] = P V with the
// heads on M (rows past the group unused) and P^T read as the K-major A
// operand.
template <int NH, int D>
struct TcShape {
  static constexpr bool kTrans = D == 128;     // O^T (M = D) or O (M = 128 heads)
  static constexpr int kGroupKV = (D / 64) * 1024;  // bytes between 8-row groups of a K/V tile
  static constexpr int kKvTile = (kKeys / 8) * kGroupKV;
  static constexpr int N = NH < 16 ? 16 : NH;  // MMA N of S^T
  static constexpr int KG = NH > 16 ? 2 : 1;   // key warpgroups
  static constexpr int NHW = NH / KG;          // heads per key warpgroup
  static constexpr int kKeyThreads = 128 * KG;
  static constexpr int kKWarp = 4 * KG;        // K producer
  static constexpr int kVWarp = kKWarp + 1;    // V producer
  static constexpr int kSWarp = kKWarp + 2;    // S^T issuer, owns tensor memory
  static constexpr int kOWarp = kKWarp + 3;    // O^T issuer
  static constexpr int kThreads = kKeyThreads + 4 * 32;
  static constexpr int kQBytes = N * D * 2;    // D / 64 atoms of N rows x 128 bytes
  // P^T rows: the padded group for O^T; for O the MMA's 128 rows, except that
  // a group of at most 8 heads keeps only one 8-row group, which the A
  // operand's descriptor repeats down all 128 rows (group stride 0: rows
  // 8..127 of O repeat rows 0..7 and are never read).
  static constexpr int kPRows = kTrans ? N : (NH <= 8 ? 8 : 128);
  static constexpr int kPGroupStride = kPRows == 8 ? 0 : kGroupP;
  static constexpr int kPBuf = (kPRows / 8) * kGroupP;
  // K and V ring depth: the bytes in flight per SM set the bandwidth an SM
  // draws (about 2-3 us of latency under load), so the rings hold about 96
  // KiB per operand: 3 tiles at D = 128, as many as fit beside two P^T
  // buffers (4) at D = 64.
  static constexpr int kFixed = 2 * kQBytes + 4096;
  static constexpr int kStages =
      D == 128 ? 3 : (227 * 1024 - kFixed - 2 * kPBuf) / (2 * kKvTile) < 6
                         ? (227 * 1024 - kFixed - 2 * kPBuf) / (2 * kKvTile)
                         : 6;
  // S^T buffers and P^T buffers: three where shared memory allows, else two
  static constexpr int kSB = 2 * kStages * kKvTile + kFixed + 3 * kPBuf <= 227 * 1024 ? 3 : 2;
  static constexpr int kOCols = kTrans ? N : D;  // tensor-memory columns of one O buffer
  static constexpr int kQ = 2 * kStages * kKvTile;  // after the K and V rings
  static constexpr int kP = kQ + 2 * kQBytes;
  static constexpr int kRed = kP + kSB * kPBuf;     // [KG][4 warps][NHW] floats
  static constexpr int kBar = kRed + KG * 4 * NHW * 4;
  static constexpr int kTmemSlot = kBar + kBarSlots * 8;
  static constexpr int kBytes = kTmemSlot + 16 + 1024;  // + alignment slack
  static_assert(kBytes <= 227 * 1024, "shared memory overflow");
  static constexpr int kColO = kSB * N;                 // S^T buffers first
  static constexpr int kTmemCols = pow2_at_least(kSB * N + 2 * kOCols);
  static_assert(kTmemCols <= 512, "tensor memory overflow");
};

// One work item: sequence s, KV head, partition [t_begin, t_end) of the
// context (empty when n_tiles == 0).
struct Item {
  int s, kvh, part, ctx, t_begin, t_end, n_tiles, nparts_seq;
};

__device__ __forceinline__ int item_seq(const DecodeParams& p, int j) {
  return j / p.num_parts / p.num_kv_heads;
}

// The item's fields from its sequence's raw context length.
__device__ __forceinline__ Item item_from(const DecodeParams& p, int j, int ctx) {
  Item it;
  it.part = j % p.num_parts;
  const int r = j / p.num_parts;
  it.kvh = r % p.num_kv_heads;
  it.s = r / p.num_kv_heads;
  const long long cap = min((long long)p.max_context_len,
                            (long long)p.max_blocks_per_seq * p.block_size);
  if (ctx < 0) ctx = 0;
  if (ctx > cap) ctx = (int)cap;
  it.ctx = ctx;
  it.t_begin = it.part * p.partition_size;
  it.t_end = min(ctx, it.t_begin + p.partition_size);
  it.n_tiles = it.t_begin < it.t_end ? (it.t_end - it.t_begin + kKeys - 1) / kKeys : 0;
  it.nparts_seq = (ctx + p.partition_size - 1) / p.partition_size;
  return it;
}

__device__ __forceinline__ Item item_at(const DecodeParams& p, int j) {
  return item_from(p, j, __ldg(p.context_lens + item_seq(p, j)));
}

// Reduction of a predicate over one key warpgroup (named barrier 1 + kg):
// true if any of its 128 threads passes true.
__device__ __forceinline__ bool group_any(int kg, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %2, 0;\n\t"
      "bar.red.or.pred po, %1, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(1 + kg), "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void group_sync(int kg) { named_barrier_sync(1 + kg, 128); }

template <typename T, int NH, int D>
__global__ void __launch_bounds__(TcShape<NH, D>::kThreads, 1)
    paged_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap qmap, int num_items) {
  using L = TcShape<NH, D>;
  constexpr int N = L::N;
  constexpr int S = L::kStages;
  constexpr int NHW = L::NHW;
  constexpr int kGroupKV = L::kGroupKV;
  constexpr int kKvTile = L::kKvTile;
  grid_dep_wait();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sK = smem;
  unsigned char* sV = smem + S * kKvTile;
  unsigned char* sQ = smem + L::kQ;
  unsigned char* sP = smem + L::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* k_full = bars;             // [S] K tile landed (TMA bytes)
  uint64_t* k_empty = k_full + S;      // [S] S^T MMAs done reading it (commit)
  uint64_t* v_full = k_empty + S;      // [S] V tile landed
  uint64_t* v_empty = v_full + S;      // [S] O^T MMAs done reading it (commit)
  constexpr int SB = L::kSB;
  uint64_t* s_full = v_empty + S;      // [SB] S^T buffer computed (commit)
  uint64_t* s_free = s_full + SB;      // [SB] S^T buffer read by the key warpgroups
  uint64_t* p_full = s_free + SB;      // [SB] P^T buffer written (key warpgroups)
  uint64_t* p_free = p_full + SB;      // [SB] P.V MMAs done with P^T buffer (commit)
  uint64_t* q_full = p_free + SB;      // [2] Q rows of an item landed (TMA bytes)
  uint64_t* q_empty = q_full + 2;      // [2] S^T MMAs of that item done (commit)
  uint64_t* o_free = q_empty + 2;      // [2] O^T buffer read by the key warpgroups
  uint64_t* drain = o_free + 2;        // [2] each issuer's last MMAs finished
  static_assert(4 * S + 4 * SB + 8 <= kBarSlots, "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int b = 0; b < SB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], L::kKeyThreads);
      mbar_init(&p_full[b], L::kKeyThreads);
      mbar_init(&p_free[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
      mbar_init(&o_free[b], L::kKeyThreads);
      mbar_init(&drain[b], 1);
    }
    fence_barrier_init();
  }
  if (warp == L::kSWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(L::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == L::kKWarp || warp == L::kVWarp) {
    // ----------------------------------------------------------- producers
    // Tile i of an item covers keys [t_begin + 128 i, +128): runs of B rows,
    // one block each; lane l copies run l with one TMA copy.  The block id
    // of the lane's run of the next tile is read before this tile's copy is
    // issued, so its latency overlaps the wait for a free slot.
    const bool is_k = warp == L::kKWarp;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    unsigned char* ring = is_k ? sK : sV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const void* new_rows = is_k ? p.k_new : p.v_new;
    T* cache = const_cast<T*>(static_cast<const T*>(is_k ? p.k_cache : p.v_cache));
    const int B = p.block_size;
    prefetch_tensormap(map);
    if (is_k) prefetch_tensormap(&qmap);
    int kt = 0, k_item = 0, issued = 0, q_issued = 0;
    bool ok = true;
    for (int j = blockIdx.x; ok && j < num_items; j += gridDim.x) {
      // The context length and the block ids of the item's first tile are
      // loaded together (the ids speculatively, within the table row), so
      // the item costs one memory latency before its first copy.
      const int sj = item_seq(p, j);
      const int32_t* trow = p.block_tables + (size_t)sj * p.max_blocks_per_seq;
      const int lb0 = ((j % p.num_parts) * p.partition_size) / B + lane;
      const bool in_row = lane * B < kKeys && lb0 < p.max_blocks_per_seq;
      const int ctx_raw = __ldg(p.context_lens + sj);
      const int first_id = in_row ? __ldg(trow + lb0) : 0;
      const Item it = item_from(p, j, ctx_raw);
      if (it.n_tiles == 0) continue;
      auto table_entry = [&](int i) -> int {
        const int key = it.t_begin + i * kKeys + lane * B;
        return (lane * B < kKeys && i < it.n_tiles && key < it.t_end) ? __ldg(trow + key / B)
                                                                      : 0;
      };
      int phys_next = (it.t_begin + lane * B < it.t_end && lane * B < kKeys) ? first_id : 0;
      if (is_k) {
        const int qb = k_item & 1;
        if (k_item >= 2 && !mbar_wait_warp(&q_empty[qb], ((k_item - 2) >> 1) & 1, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[qb], L::kQBytes);
          tma_load_rows(sQ + qb * L::kQBytes, &qmap, it.s * p.num_q_heads + it.kvh * G,
                        &q_full[qb]);
        }
        __syncwarp();
        q_issued = k_item + 1;
      }
      // Fused append: the step's new token is position ctx - 1 of the last
      // partition; its row (D / 8 chunks of 16 bytes, one per lane) is written
      // to its cache slot before the copy of the tile that holds it.
      constexpr int kRowChunks = D / 8;
      const bool fused_here = new_rows != nullptr && it.t_end == it.ctx;
      uint4 new_chunk = make_uint4(0, 0, 0, 0);
      if (fused_here && lane < kRowChunks)
        new_chunk = reinterpret_cast<const uint4*>(
            static_cast<const T*>(new_rows) +
            ((size_t)it.s * p.num_kv_heads + it.kvh) * D)[lane];
      for (int i = 0; i < it.n_tiles; ++i, ++kt) {
        const int st = kt % S;
        const int key0 = it.t_begin + i * kKeys;
        const int nvalid = min(kKeys, it.t_end - key0);
        const int nseg = (nvalid + B - 1) / B;
        int phys = phys_next;
        phys_next = table_entry(i + 1);
        if ((unsigned)phys >= (unsigned)p.num_blocks) {
          if (lane < nseg) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
          phys = 0;
        }
        if (fused_here && key0 + nvalid == it.ctx) {
          const int pos = it.ctx - 1;
          const int phys_new = __shfl_sync(0xffffffffu, phys, (pos - key0) / B);
          if (lane < kRowChunks) {
            const size_t dst =
                (((size_t)phys_new * p.num_kv_heads + it.kvh) * B + (pos % B)) * D;
            reinterpret_cast<uint4*>(cache + dst)[lane] = new_chunk;
          }
          // the row must be visible to the copy engine's read below
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
        }
        if (kt >= S && !mbar_wait_warp(&empty[st], ((kt / S) - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)nseg * B * D * sizeof(T));
        __syncwarp();
        if (lane < nseg)
          tma_load_group(ring + st * kKvTile + lane * (B / 8) * kGroupKV, map,
                         ((phys * p.num_kv_heads + it.kvh) * B) / 8, &full[st]);
        issued = kt + 1;
      }
      ++k_item;
    }
    // After a timeout, copies still in flight land before the CTA leaves.
    if (timed_out(p.status)) {
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)
        mbar_drain(&full[i % S], (i / S) & 1);
      if (is_k && q_issued > 0)
        mbar_drain(&q_full[(q_issued - 1) & 1], ((q_issued - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == L::kSWarp || warp == L::kOWarp) {
    // ------------------------------------------------------------ issuers
    // The whole warp runs the loop and one elected lane issues.
    constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    const bool is_s = warp == L::kSWarp;
    const uint32_t idesc = is_s ? instr_desc(bf16, false, false, N, kKeys)
                                : (L::kTrans ? instr_desc(bf16, true, false, N, D)
                                             : instr_desc(bf16, false, true, D, kKeys));
    const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ),
                   aP = smem_addr(sP);
    int kt = 0, k_item = 0;
    bool ok = true;
    for (int j = blockIdx.x; ok && j < num_items; j += gridDim.x) {
      const Item it = item_at(p, j);
      if (it.n_tiles == 0) continue;
      const int b = k_item & 1;
      if (is_s) {
        if (!mbar_wait_warp(&q_full[b], (k_item >> 1) & 1, p.status)) break;
        for (int i = 0; i < it.n_tiles; ++i, ++kt) {
          const int st = kt % S;
          if (!mbar_wait_warp(&k_full[st], (kt / S) & 1, p.status) ||
              (kt >= SB && !mbar_wait_warp(&s_free[kt % SB], ((kt / SB) - 1) & 1, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S^T = K . Q^T: 16 dimensions per MMA; a 32-byte step inside the
          // 128-byte rows, then the next 64-column atom.
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_f16_ss_warp(tmem + (kt % SB) * N,
                            smem_desc(aK + st * kKvTile + (ks / 4) * 1024 + (ks % 4) * 32, 16,
                                      kGroupKV),
                            smem_desc(aQ + b * L::kQBytes + (ks / 4) * (N * 128) + (ks % 4) * 32,
                                      16, 1024),
                            idesc, ks > 0 ? 1u : 0u);
          mma_commit_warp(&s_full[kt % SB]);
          mma_commit_warp(&k_empty[st]);
        }
        if (ok) mma_commit_warp(&q_empty[b]);
      } else {
        if (k_item >= 2 && !mbar_wait_warp(&o_free[b], ((k_item - 2) >> 1) & 1, p.status)) break;
        for (int i = 0; i < it.n_tiles; ++i, ++kt) {
          const int st = kt % S;
          if (!mbar_wait_warp(&v_full[st], (kt / S) & 1, p.status) ||
              !mbar_wait_warp(&p_full[kt % SB], (kt / SB) & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O^T += V^T P^T (D = 128) or O += P V (D = 64): 16 keys per
          // MMA, two 8-key groups of V and a 32-byte step inside P^T's
          // 128-byte rows.
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks) {
            const uint64_t dv = smem_desc(aV + st * kKvTile + ks * 2 * kGroupKV, 1024, kGroupKV);
            const uint64_t dp =
                smem_desc(aP + (kt % SB) * L::kPBuf + (ks / 4) * 1024 + (ks % 4) * 32, 16,
                          L::kTrans ? kGroupP : L::kPGroupStride);
            if constexpr (L::kTrans)
              mma_f16_ss_warp(tmem + L::kColO + b * L::kOCols, dv, dp, idesc,
                              (i > 0 || ks > 0) ? 1u : 0u);
            else
              mma_f16_ss_warp(tmem + L::kColO + b * L::kOCols, dp, dv, idesc,
                              (i > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit_warp(&p_free[kt % SB]);
          mma_commit_warp(&v_empty[st]);
        }
      }
      ++k_item;
    }
    uint64_t* d = &drain[is_s ? 0 : 1];
    mma_commit_warp(d);
    mbar_drain(d, 0);
    __syncwarp();
  } else {
    // ----------------------------------------------------- key warpgroups
    const int kg = warp >> 2;            // which half of the heads
    const int t = threadIdx.x & 127;     // key of the tile == lane; dimension d at the end
    const int hb = kg * NHW;             // first head of this warpgroup within the group
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + L::kRed) + kg * 4 * NHW;
    const float qs = p.qscale;
    if constexpr (!L::kTrans) {
      // P's rows past the group are read by the P V product but never
      // written: clear them once (the first release's proxy fence orders
      // these stores before the tensor core reads them).
      for (int i = threadIdx.x; i < SB * L::kPBuf / 16; i += L::kKeyThreads)
        reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
    }
    int kt = 0, k_item = 0;
    bool ok = true;
    for (int j = blockIdx.x; j < num_items; j += gridDim.x) {
      const Item it = item_at(p, j);
      const int h0 = it.kvh * G;
      if (kg == 0 && t == 0 && it.part == 0) {
        const int raw = __ldg(p.context_lens + it.s);
        if (raw < 0 || raw > it.ctx) atomicOr(p.status, PKV_DEV_BAD_CONTEXT_LEN);
      }
      if (it.n_tiles == 0) {
        if (it.ctx == 0 && it.part == 0) {  // empty context: the output is zero
          T* o = static_cast<T*>(p.out) + ((size_t)it.s * p.num_q_heads + h0 + hb) * D;
          const int n = min(NHW, G - hb) * D;
          for (int i = t; i < n; i += 128) o[i] = static_cast<T>(0.f);
        }
        continue;
      }
      const int ob = k_item & 1;
      // The running maxima per head are the same in every thread of the
      // warpgroup: all start at -inf and all take each move from the same
      // tile maxima, so they stay in registers.
      float mref[NHW], l_part[NHW];
#pragma unroll
      for (int g = 0; g < NHW; ++g) {
        mref[g] = -CUDART_INF_F;
        l_part[g] = 0.f;
      }
      for (int i = 0; i < it.n_tiles; ++i, ++kt) {
        const int nvalid = min(kKeys, it.t_end - (it.t_begin + i * kKeys));
        const bool valid = t < nvalid;
        // A wait that gives up (never expected) leaves ok false; the loop
        // runs on without waiting, so that every named barrier stays matched,
        // and nothing it computes is stored.
        if (ok && !mbar_wait_warp(&s_full[kt % SB], (kt / SB) & 1, p.status)) ok = false;
        tc_fence_after();
        float x[NHW];
        tmem_load_small<NHW>(tmem + (kt % SB) * N + hb + lane_base, x);
        tc_fence_before();
        mbar_arrive(&s_free[kt % SB]);
        bool exceed = false;
#pragma unroll
        for (int g = 0; g < NHW; ++g) {
          x[g] *= qs;  // base-2 logit
          exceed |= valid && hb + g < G && x[g] > mref[g] + 8.f;
        }
        if (group_any(kg, exceed)) {
          // Some key exceeds its head's running max by more than 8: the tile
          // maxima per head, then the heads whose maximum moves.
#pragma unroll
          for (int g = 0; g < NHW; ++g) {
            float v = (valid && hb + g < G) ? x[g] : -CUDART_INF_F;
#pragma unroll
            for (int mk = 16; mk >= 1; mk >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, mk));
            if (lane == 0) red[(warp & 3) * NHW + g] = v;
          }
          group_sync(kg);
          float alpha[NHW];
          bool moved = false;
#pragma unroll
          for (int g = 0; g < NHW; ++g) {
            const float mt =
                fmaxf(fmaxf(red[g], red[NHW + g]), fmaxf(red[2 * NHW + g], red[3 * NHW + g]));
            const float mn = mt > mref[g] + 8.f ? mt : mref[g];
            alpha[g] = (mn == mref[g]) ? 1.f : ex2(mref[g] - mn);
            moved |= mn != mref[g];
            mref[g] = mn;
            l_part[g] *= alpha[g];
          }
          group_sync(kg);  // every thread has read red[] before it is written again
          if (i > 0 && moved) {
            // O holds this item's tiles so far: once their MMAs are done
            // (P^T buffer of the previous tile released), rescale it.
            if (ok && !mbar_wait_warp(&p_free[(kt - 1) % SB], ((kt - 1) / SB) & 1, p.status))
              ok = false;
            tc_fence_after();
            if constexpr (L::kTrans) {
              // O^T: thread d rescales this warpgroup's columns of its lane
              const uint32_t oaddr = tmem + L::kColO + ob * L::kOCols + hb + lane_base;
              float o[NHW];
              tmem_load_small<NHW>(oaddr, o);
#pragma unroll
              for (int g = 0; g < NHW; ++g) o[g] *= alpha[g];
              tmem_store_small<NHW>(oaddr, o);
            } else {
              // O: lane h is head h; the warpgroup that owns head h scales
              // its D columns (the other lanes store what they read)
              float a = 1.f;
#pragma unroll
              for (int g = 0; g < NHW; ++g)
                if (t == hb + g) a = alpha[g];
              const uint32_t oaddr = tmem + L::kColO + ob * L::kOCols + lane_base;
#pragma unroll
              for (int c = 0; c < D / 16; ++c) {
                float o[16];
                tmem_load_small<16>(oaddr + c * 16, o);
#pragma unroll
                for (int k = 0; k < 16; ++k) o[k] *= a;
                tmem_store_small<16>(oaddr + c * 16, o);
              }
            }
            tc_fence_before();
          }
        }
        // P^T column t: exp2(x - m) per head, rounded to the operand type.
        T pt[NHW];
#pragma unroll
        for (int g = 0; g < NHW; ++g) {
          const float e = (valid && hb + g < G) ? ex2(x[g] - mref[g]) : 0.f;
          l_part[g] += e;
          pt[g] = static_cast<T>(e);
        }
        // The buffer was last read by the MMAs of tile kt - SB.
        if (kt >= SB && ok && !mbar_wait_warp(&p_free[kt % SB], ((kt / SB) - 1) & 1, p.status))
          ok = false;
        unsigned char* pb = sP + (kt % SB) * L::kPBuf;
#pragma unroll
        for (int g = 0; g < NHW; ++g)
          if (hb + g < G)
            *reinterpret_cast<T*>(pb + chunk_offset<kKeys>(hb + g, t >> 3) + (t & 7) * 2) = pt[g];
        if (nvalid < kKeys && kg == 0) {
          // The item's last tile: V rows past the context must not feed stale
          // or NaN values into O^T (their P is 0, but 0 * NaN is NaN).
          const int st = kt % S;
          if (ok && !mbar_wait_warp(&v_full[st], (kt / S) & 1, p.status)) ok = false;
          if (!valid) {
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
              *reinterpret_cast<uint4*>(sV + st * kKvTile + chunk_offset<D>(t, c)) =
                  make_uint4(0, 0, 0, 0);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&p_full[kt % SB]);
      }

      // Row sums per head over the 128 keys' partial sums.
#pragma unroll
      for (int g = 0; g < NHW; ++g) {
        float v = l_part[g];
#pragma unroll
        for (int mk = 16; mk >= 1; mk >>= 1) v += __shfl_xor_sync(0xffffffffu, v, mk);
        if (lane == 0) red[(warp & 3) * NHW + g] = v;
      }
      group_sync(kg);
      const int last = kt - 1;
      if (ok && !mbar_wait_warp(&p_free[last % SB], (last / SB) & 1, p.status)) ok = false;
      tc_fence_after();
      if constexpr (L::kTrans) {
        // O^T: thread d writes dimension d of this warpgroup's heads.
        float o[NHW];
        tmem_load_small<NHW>(tmem + L::kColO + ob * L::kOCols + hb + lane_base, o);
        tc_fence_before();
        mbar_arrive(&o_free[ob]);
        if (ok) {
          const int d = t;
          // Every head's sum is read from shared memory before the first
          // store (a store through a plain pointer would otherwise make each
          // later read wait for it), and each head divides by one
          // reciprocal: IEEE divisions, each with its own slow-path branch,
          // ran one after another and cost more than the item's last tile.
          float l[NHW], inv[NHW];
#pragma unroll
          for (int g = 0; g < NHW; ++g) {
            l[g] = (red[g] + red[NHW + g]) + (red[2 * NHW + g] + red[3 * NHW + g]);
            inv[g] = __fdividef(1.f, l[g]);
          }
          const size_t row0 = (size_t)it.s * p.num_q_heads + h0 + hb;
          if (it.nparts_seq == 1) {
            T* dst = static_cast<T*>(p.out) + row0 * D + d;
#pragma unroll
            for (int g = 0; g < NHW; ++g)
              if (hb + g < G) dst[(size_t)g * D] = static_cast<T>(o[g] * inv[g]);
          } else {
            const size_t r0 = row0 * p.num_parts + it.part;
            float* dst = p.ws_o + r0 * D + d;
#pragma unroll
            for (int g = 0; g < NHW; ++g)
              if (hb + g < G) dst[(size_t)g * p.num_parts * D] = o[g] * inv[g];
            // Thread g writes head g's maximum and sum (one thread writing
            // them all took longer than the whole tile).
            float mg = 0.f, lg = 0.f;
#pragma unroll
            for (int g = 0; g < NHW; ++g)
              if (d == g) {
                mg = mref[g];
                lg = l[g];
              }
            if (d < NHW && hb + d < G) {
              p.ws_m[r0 + (size_t)d * p.num_parts] = mg;
              p.ws_l[r0 + (size_t)d * p.num_parts] = lg;
            }
          }
        }
      } else {
        // O: thread h (lane h) writes the D outputs of head h if this
        // warpgroup owns it.
        const int g = t - hb;
        const bool mine = g >= 0 && g < NHW && t < G;
        float l = 1.f, m = 0.f;
#pragma unroll
        for (int k = 0; k < NHW; ++k)
          if (k == g) {
            l = (red[k] + red[NHW + k]) + (red[2 * NHW + k] + red[3 * NHW + k]);
            m = mref[k];
          }
        const float inv = 1.f / l;
        const size_t row = (size_t)it.s * p.num_q_heads + h0 + (mine ? t : 0);
        const size_t r = row * p.num_parts + it.part;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          float o[16];
          tmem_load_small<16>(tmem + L::kColO + ob * L::kOCols + lane_base + c * 16, o);
          if (ok && mine) {
            if (it.nparts_seq == 1) {
              uint4 v0, v1;
              v0.x = Cvt<T>::from_float2(o[0] * inv, o[1] * inv);
              v0.y = Cvt<T>::from_float2(o[2] * inv, o[3] * inv);
              v0.z = Cvt<T>::from_float2(o[4] * inv, o[5] * inv);
              v0.w = Cvt<T>::from_float2(o[6] * inv, o[7] * inv);
              v1.x = Cvt<T>::from_float2(o[8] * inv, o[9] * inv);
              v1.y = Cvt<T>::from_float2(o[10] * inv, o[11] * inv);
              v1.z = Cvt<T>::from_float2(o[12] * inv, o[13] * inv);
              v1.w = Cvt<T>::from_float2(o[14] * inv, o[15] * inv);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + row * D + c * 16);
              dst[0] = v0;
              dst[1] = v1;
            } else {
              float4* dst = reinterpret_cast<float4*>(p.ws_o + r * D + c * 16);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv,
                                     o[4 * k + 3] * inv);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&o_free[ob]);
        if (ok && mine && it.nparts_seq > 1) {
          p.ws_m[r] = m;
          p.ws_l[r] = l;
        }
      }
      ++k_item;
    }
    grid_dep_launch_dependents();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kSWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::kTmemCols));
  }
}

template <typename T, int NH, int D>
cudaError_t launch_tc_typed(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm,
                            const CUtensorMap& qm, int sms, cudaStream_t stream) {
  using L = TcShape<NH, D>;
  static unsigned long long configured = 0;  // bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    err = cudaFuncSetAttribute(paged_decode_tc_kernel<T, NH, D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  const long long items = (long long)p.num_parts * p.num_kv_heads * p.num_seqs;
  const int grid = (int)(items < sms ? items : sms);
  err = launch_overlapped(paged_decode_tc_kernel<T, NH, D>, dim3(grid), dim3(L::kThreads),
                          L::kBytes, stream, p, km, vm, qm, (int)items);
  if (err != cudaSuccess || p.num_parts <= 1) return err;
  return launch_decode_reduce(p, std::is_same<T, __nv_bfloat16>::value ? PKV_BF16 : PKV_F16, D,
                              stream);
}

template <typename T, int D>
cudaError_t launch_tc_group(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm,
                            const CUtensorMap& qm, int sms, cudaStream_t stream) {
  static_assert(kMaxTcGroup == 32, "instantiations cover groups up to 32");
  if (p.group <= 4) return launch_tc_typed<T, 4, D>(p, km, vm, qm, sms, stream);
  if (p.group <= 8) return launch_tc_typed<T, 8, D>(p, km, vm, qm, sms, stream);
  if (p.group <= 16) return launch_tc_typed<T, 16, D>(p, km, vm, qm, sms, stream);
  return launch_tc_typed<T, 32, D>(p, km, vm, qm, sms, stream);
}

}  // namespace

bool decode_tc_supported(int head_dim, int group, int partition_size) {
  static_assert(kTcPartitionQuantum == kKeys, "partitions are whole tiles");
  return (head_dim == 64 || head_dim == 128) && group >= kMinTcGroup &&
         group <= kMaxTcGroup && partition_size % kKeys == 0;
}

cudaError_t launch_paged_decode_tc(const DecodeParams& p, int dtype, int head_dim, int sms,
                                   cudaStream_t stream, bool* unsupported) {
  *unsupported = false;
  CUtensorMap km, vm, qm;
  const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
  // Q rows of an item: a box of N rows from the item's first head (rows past
  // the group are other heads' or zero, and only feed unused columns).
  const int box_rows = p.group <= 16 ? 16 : 32;
  const int d = head_dim;
  if (!make_cache_map(&km, p.k_cache, dtype, rows, d, p.block_size) ||
      !make_cache_map(&vm, p.v_cache, dtype, rows, d, p.block_size) ||
      !make_rows_map(&qm, p.q, dtype, (long long)p.num_seqs * p.num_q_heads, d, box_rows)) {
    *unsupported = true;
    return cudaErrorInvalidValue;
  }
  if (dtype == PKV_F16)
    return d == 64 ? launch_tc_group<__half, 64>(p, km, vm, qm, sms, stream)
                   : launch_tc_group<__half, 128>(p, km, vm, qm, sms, stream);
  return d == 64 ? launch_tc_group<__nv_bfloat16, 64>(p, km, vm, qm, sms, stream)
                 : launch_tc_group<__nv_bfloat16, 128>(p, km, vm, qm, sms, stream);
}

}  // namespace pkv
