// Paged multi-query (chunked prompt) attention on the 5th-generation tensor
// cores of sm_103a (tcgen05.mma, accumulators in tensor memory).
//
// What it computes: sequence s brings L_s query rows, the last L_s positions
// of its context (their K/V already appended); query j at position
// p = ctx_s - L_s + j attends causally to positions 0..p, reading K/V through
// the block table ("Only 20.4% of your KV cache held actual tokens", section
// "The page table, relocated into attention"; prompt chunks: "The KV cache is
// a systems problem", section "Memory savings change the scheduling
// question").  Unlike decode this is a dense contraction.
//
// One CTA owns (sequence, KV head, two tiles A and B of 128 query rows each)
// and one SM: the tensor memory holds S_A, S_B (P written over them) and
// O_A, O_B, 4 x 128 columns; shared memory holds both Q tiles and two slots
// each of K and V (193 KiB at D = 128).  Rows are (query, head-of-group)
// pairs, so every head of a KV group shares each K/V tile (grouped-query
// attention packs into the MMA's M dimension).  Each tile's chain
// S -> softmax -> P V is serial, and the single MMA issuer interleaves the
// two: P V of A, S of A's next key tile, P V of B, S of B's next.  So while
// one tile's softmax runs, the tensor core computes the other tile's
// products, and the two softmax phases do not overlap (left to themselves,
// two such chains on one tensor core fall into step, each softmax running
// beside the other's instead of beside its MMAs).
//
//   warp 8   producer: the Q rows of each tile (one 4-D TMA copy per tile;
//            tile A's, then the first K tile, then tile B's), then per key
//            tile the tile's block ids and every (block, head) run of K and
//            of V (one 4-D TMA copy each, 128-byte swizzle) into the next free
//            slot.
//   warp 9   issues S = Q K^T (Q and K from shared memory) and O += P V (P
//            from tensor memory, V as an MN-major operand, rows past the
//            context cleared first); allocates and frees the tensor memory.
//            S_t of a key tile overwrites P_t of the previous one, so it
//            waits for that P V; the wait for the next V tile sits behind the
//            last P V of a key tile, off the path from one tile's S to the
//            other's P V.
//   warps 0-3 (tile A), 4-7 (tile B)  softmax, one thread per row: per key
//            tile it reads its S row for the row max (off the diagonal with
//            tcgen05.ld.red, which returns each 32-column chunk's maximum with
//            the values; on the diagonal with a masked pass), keeps the
//            running max and sum in base 2 (lazy rescaling, O rescaled in
//            place when the max moved), then computes the exponentials half a
//            row at a time and writes each half of P over S in tensor memory,
//            releasing it to P V at once; at the end it normalises and stores
//            its O row.
//
// Work items (one per CTA) are (query tile pair, KV head, sequence).  The
// (sequence, KV head) pairs go in groups of about one wave of items (one CTA
// per SM), and within a group the latest query tiles (the longest causal
// spans) start first: CTAs that run together share K/V in L2, and the final
// wave holds short items.

#include <math_constants.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

using namespace tc;

constexpr int kBM = 128;     // rows of the row tile: MMA M
constexpr int kRowTiles = 2; // two row tiles per CTA, their chains alternating
constexpr int kStages = 2;   // K and V ring slots
constexpr int kBN = 128;     // keys per K/V tile: N of Q K^T, K of P V
static_assert(kBN == kTileKeys, "TMA runs are capped at the tile length");
constexpr int kSoftmaxWarps = 4 * kRowTiles;
constexpr int kProducerWarp = kSoftmaxWarps;  // Q, K and V copies
constexpr int kMmaWarp = kSoftmaxWarps + 1;   // Q K^T and P V; owns the tensor memory
constexpr int kPrefillThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kTmemCols = 512;
constexpr int kBarSlots = 24;   // mbarriers reserved in shared memory

// Shared-memory K and V tiles: groups of 8 rows, kGroup bytes apart; within
// a group, one 1024-byte 128-byte-swizzled atom per 64 columns.  This is the
// K-major operand layout with SBO = kGroup, and, for V, the MN-major one with
// LBO = 1024 and SBO = kGroup.  A single TMA copy fills any number of whole
// groups with all their atoms.  A Q tile is written by one copy of all its
// 128 rows: one 16 KiB block per 64 columns, 8-row groups 1024 bytes apart
// in it (the K-major layout with SBO = 1024), so the same kQTile bytes.
template <int D>
struct PrefillSmem {
  static constexpr int kAtoms = D / 64;
  static constexpr int kGroup = kAtoms * 1024;
  static constexpr int kQTile = (kBM / 8) * kGroup;
  static constexpr int kKvTile = (kBN / 8) * kGroup;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kRowTiles * kQTile;
  static constexpr int kV = kK + kStages * kKvTile;
  static constexpr int kBar = kV + kStages * kKvTile;
  static constexpr int kTmemSlot = kBar + kBarSlots * 8;
  static constexpr int kBytes = kTmemSlot + 16 + 1024;  // + alignment slack
  static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr int kColO = kRowTiles * kBN;
  static_assert(kColO + kRowTiles * D <= kTmemCols, "tensor memory overflow");
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
  int num_seqs;
  int q_tiles;          // CTAs per (sequence, KV head)
  int pairs_per_group;  // (sequence, KV head) pairs whose items are launched together
  int total_queries;    // rows of q and out
  int prefetch_stride;  // work items between a CTA and the one likely to follow it on its SM
};

// A Q box (as tma_load_token_heads copies it) fetched into L2 only: no
// shared memory, no barrier.
__device__ __forceinline__ void tma_prefetch_token_heads(const CUtensorMap* map, int head,
                                                         int token) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %1}];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(0), "r"(head), "r"(token)
      : "memory");
}

// Byte offset of 16-byte chunk c of row r in a tile of the layout above.
template <int D>
__device__ __forceinline__ uint32_t tile_chunk_offset(int r, int c) {
  return chunk_offset<D>(r, c);
}

// ---- the kernel -----------------------------------------------------------

template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    paged_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap) {
  using L = PrefillSmem<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = smem + L::kQ;
  unsigned char* sK = smem + L::kK;
  unsigned char* sV = smem + L::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* k_full = bars;        // [kStages] K slot landed (TMA transaction bytes)
  uint64_t* k_empty = bars + 2;   // [kStages] K slot read by S (MMA commit)
  uint64_t* v_full = bars + 4;    // [kStages] V slot landed
  uint64_t* v_empty = bars + 6;   // [kStages] V slot read by P V
  uint64_t* q_full = bars + 8;    // [t] Q rows of tile t landed
  uint64_t* s_full = bars + 10;   // [t] S_t computed (MMA commit)
  uint64_t* p_full = bars + 12;   // [2 t + h] half h of P_t written (after O_t was rescaled)
  uint64_t* pv_done = bars + 16;  // [t] O_t += P_t V finished (MMA commit)
  uint64_t* drain = bars + 18;    // the issuer's last MMAs finished
  static_assert(19 <= kBarSlots, "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work item -> (query tile, KV head, sequence): the (sequence, head) pairs
  // are taken in groups of about one wave of work items, and within a group
  // the hardware starts the latest query tiles (the longest causal spans)
  // first.
  const int pairs = p.num_kv_heads * p.num_seqs;
  const int per_group = p.pairs_per_group * p.q_tiles;
  const int grp = (int)(blockIdx.x / per_group);
  const int gsize = min(p.pairs_per_group, pairs - grp * p.pairs_per_group);
  const int rem = (int)(blockIdx.x - (unsigned)(grp * per_group));
  const int qt = p.q_tiles - 1 - rem / gsize;
  const int pair = grp * p.pairs_per_group + rem % gsize;
  const int kvh = pair % p.num_kv_heads;
  const int s = pair / p.num_kv_heads;
  const int G = p.group;
  const int Gp = p.group_pow2;
  const int qpt = kBM / Gp;

  const int q0 = p.query_start[s];
  const int nq = p.query_start[s + 1] - q0;
  int ctx = p.context_lens[s];
  const long long cap_ll = min((long long)p.max_context_len,
                               (long long)p.max_blocks_per_seq * p.block_size);
  if (ctx < nq || ctx > cap_ll) {
    if (threadIdx.x == 0 && qt == 0) atomicOr(p.status, PKV_DEV_BAD_CONTEXT_LEN);
    if (ctx < nq || nq <= 0) return;
    ctx = (int)cap_ll;
  }
  const int j0 = qt * kRowTiles * qpt;  // first query of the CTA
  if (j0 >= nq) return;                 // no queries here
  // Key tiles up to each row tile's last query's position (none for a tile
  // past the sequence's queries).
  int n_t[kRowTiles];
#pragma unroll
  for (int t = 0; t < kRowTiles; ++t) {
    const int jt = j0 + t * qpt;
    n_t[t] = jt < nq ? (ctx - nq + min(nq, jt + qpt) - 1) / kBN + 1 : 0;
  }
  const int n_tiles = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&k_full[st], 1);
      mbar_init(&k_empty[st], 1);
      mbar_init(&v_full[st], 1);
      mbar_init(&v_empty[st], 1);
    }
    for (int t = 0; t < kRowTiles; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[2 * t], kBM);
      mbar_init(&p_full[2 * t + 1], kBM);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer
    // The Q rows, then K and V of each key tile into their slots.  A tile's
    // keys are runs of R rows that never cross a block boundary (R divides
    // the block size and the tile); lane l copies run l with one TMA copy
    // per operand.  The block-table entry of the next tile is read once this
    // tile's copies are issued, so its latency is spent while the warp waits
    // for a free slot.
    const int B = p.block_size;
    const int R = B < kBN ? B : kBN;
    const int32_t* trow = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    auto table_entry = [&](int i) -> int {
      const int key = i * kBN + lane * R;
      return (lane < kBN / R && i < n_tiles && key < ctx) ? __ldg(trow + key / B) : 0;
    };
    int phys_next = table_entry(0);
    // Q rows of tile t: one copy of G' heads x 128 / G' queries.  Heads past
    // the group and queries past the sequence are copied too (their rows are
    // masked out and never written); rows past the end of q read as zero.
    // Tile A's rows go first, then K of the first key tile, then tile B's.
    auto load_q = [&](int t) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[t], L::kQTile);
        tma_load_token_heads(sQ + t * L::kQTile, &qmap, kvh * G, q0 + j0 + t * qpt, &q_full[t]);
      }
      __syncwarp();
    };
    load_q(0);
    int last_k = -1, last_v = -1;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % kStages;
      const uint32_t ph = ((i / kStages) - 1) & 1;
      if (i >= kStages && !mbar_wait_warp(&k_empty[st], ph, p.status)) break;
      const int key0 = i * kBN;
      const int nvalid = min(ctx, key0 + kBN) - key0;
      const int nseg = (nvalid + R - 1) / R;
      const uint32_t bytes = (uint32_t)nseg * R * D * (uint32_t)sizeof(T);
      int phys = phys_next;
      if ((unsigned)phys >= (unsigned)p.num_blocks) {
        if (lane < nseg) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
        phys = 0;
      }
      const int key = key0 + lane * R;
      const int g8 = ((phys * p.num_kv_heads + kvh) * B + key % B) / 8;  // 8-row group
      const uint32_t dst = (uint32_t)(st * L::kKvTile + lane * (R / 8) * L::kGroup);
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], bytes);
      __syncwarp();
      if (lane < nseg) tma_load_group(sK + dst, &kmap, g8, &k_full[st]);
      last_k = i;
      if (i == 0) {
        load_q(1);
        // The CTA that will most likely start on this SM when this one ends
        // (one wave of CTAs later): its Q rows into L2 now, so that its first
        // S does not wait for them from DRAM.
        const int j2 = (int)blockIdx.x + p.prefetch_stride;
        if (lane == 0 && j2 < (int)gridDim.x) {
          const int grp2 = j2 / per_group;
          const int gsize2 = min(p.pairs_per_group, pairs - grp2 * p.pairs_per_group);
          const int rem2 = j2 - grp2 * per_group;
          const int qt2 = p.q_tiles - 1 - rem2 / gsize2;
          const int pair2 = grp2 * p.pairs_per_group + rem2 % gsize2;
          const int q02 = __ldg(p.query_start + pair2 / p.num_kv_heads);
#pragma unroll
          for (int t = 0; t < kRowTiles; ++t)
            tma_prefetch_token_heads(&qmap, (pair2 % p.num_kv_heads) * G,
                                     q02 + qt2 * kRowTiles * qpt + t * qpt);
        }
        __syncwarp();
      }
      if (i >= kStages && !mbar_wait_warp(&v_empty[st], ph, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], bytes);
      __syncwarp();
      if (lane < nseg) tma_load_group(sV + dst, &vmap, g8, &v_full[st]);
      last_v = i;
      // The next tile's block ids, read after this tile's copies are out (read
      // before them, the load held the copies back).
      phys_next = table_entry(i + 1);
    }
    // Copies still in flight at exit (only after a timeout) land before the
    // CTA leaves: wait, bounded, for the last ones this warp issued.
    if (last_k >= 0) mbar_drain(&k_full[last_k % kStages], (last_k / kStages) & 1);
    if (last_v >= 0) mbar_drain(&v_full[last_v % kStages], (last_v / kStages) & 1);
    mbar_drain(&q_full[0], 0);
    if (last_k >= 0) mbar_drain(&q_full[1], 0);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The two row tiles alternate: P V of tile A, S of A's next key tile, P V
    // of tile B, S of B's next; so while one tile's softmax runs the tensor
    // core works on the other's products.  S_t of key tile i + 1 overwrites
    // P_t of tile i, so it waits for that P V.  The whole warp runs the loop
    // and one elected lane issues.
    constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc_s = instr_desc(bf16, false, false, kBN, kBM);
    const uint32_t idesc_o = instr_desc(bf16, false, true, D, kBM);
    const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
    auto issue_s = [&](int t, int i) {
      const uint32_t kb = aK + (uint32_t)((i % kStages) * L::kKvTile);
      const uint32_t qb = aQ + (uint32_t)(t * L::kQTile);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t koff = (ks / 4) * 1024 + (ks % 4) * 32;
        const uint32_t qoff = (ks / 4) * (kBM * 128) + (ks % 4) * 32;
        mma_f16_ss_warp(tmem + t * kBN, smem_desc(qb + qoff, 16, 1024),
                        smem_desc(kb + koff, 16, L::kGroup), idesc_s, ks > 0);
      }
      mma_commit_warp(&s_full[t]);
    };
    bool ok = mbar_wait_warp(&k_full[0], 0, p.status);
#pragma unroll
    for (int t = 0; t < kRowTiles; ++t) {
      if (!ok || n_t[t] == 0) continue;
      ok = mbar_wait_warp(&q_full[t], 0, p.status);
      tc_fence_after();
      if (ok) issue_s(t, 0);
    }
    if (ok) mma_commit_warp(&k_empty[0]);
    // V of key tile i is waited for while the last P V of tile i - 1 runs,
    // off the path from one tile's S to the other's P V.
    ok = ok && mbar_wait_warp(&v_full[0], 0, p.status);
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int st = i % kStages;
      const int last_t = i < n_t[1] ? 1 : 0;  // the last row tile with key tile i
      unsigned char* sVs = sV + st * L::kKvTile;
      // Key rows past the context (the tail of the last block, or rows no
      // run was loaded into) must not feed NaN or stale values into P V
      // (their P is 0, but 0 * NaN is NaN): they are cleared first.
      if (i * kBN + kBN > ctx) {
        for (int r = max(ctx - i * kBN, 0) + lane; r < kBN; r += 32)
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            *reinterpret_cast<uint4*>(sVs + tile_chunk_offset<D>(r, c)) = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      const uint32_t aVs = aV + (uint32_t)(st * L::kKvTile);
      bool k_next = false;  // K of key tile i + 1 has landed
#pragma unroll
      for (int t = 0; t < kRowTiles; ++t) {
        if (i >= n_t[t]) continue;
        // P arrives in two halves of the keys; the first half's MMAs run
        // while the softmax computes the second.  V as an MN-major operand:
        // 8-key groups kGroup bytes apart, 64-column atoms 1024 bytes apart.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait_warp(&p_full[2 * t + h], i & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = h * kBN / 32; ks < (h + 1) * kBN / 32; ++ks)
            mma_f16_ta_warp(tmem + L::kColO + t * D, tmem + t * kBN + ks * 8,
                            smem_desc(aVs + ks * 2 * L::kGroup, 1024, L::kGroup), idesc_o,
                            (i > 0 || ks > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit_warp(&pv_done[t]);
        if (t == last_t) {
          mma_commit_warp(&v_empty[st]);
          if (i + 1 < n_tiles &&
              !mbar_wait_warp(&v_full[(i + 1) % kStages], ((i + 1) / kStages) & 1, p.status)) {
            ok = false;
            break;
          }
        }
        if (i + 1 < n_t[t]) {
          if (!k_next) {
            if (!mbar_wait_warp(&k_full[(i + 1) % kStages], ((i + 1) / kStages) & 1, p.status)) {
              ok = false;
              break;
            }
            k_next = true;
          }
          if (!mbar_wait_warp(&pv_done[t], i & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(t, i + 1);
        }
      }
      if (!ok) break;
      if (k_next) mma_commit_warp(&k_empty[(i + 1) % kStages]);
    }
    mma_commit_warp(drain);
    mbar_drain(drain, 0);
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------- softmax / epilogue (rows)
    const int t = warp / 4;                 // row tile of this warpgroup
    const int r = threadIdx.x & (kBM - 1);  // row of the tile == TMEM lane
    const int nt = t == 0 ? n_t[0] : n_t[1];  // (a select: no local-memory array)
    const int jq = j0 + t * qpt + r / Gp;
    const int g = r % Gp;
    const bool row_valid = jq < nq && g < G && q0 + jq < p.total_queries;
    const int pos = row_valid ? ctx - nq + jq : -1;
    const size_t row_elem =
        ((size_t)(q0 + (row_valid ? jq : 0)) * p.num_q_heads + kvh * G + (row_valid ? g : 0)) * D;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tmem_s = tmem + t * kBN + lane_base;
    const uint32_t tmem_o = tmem + L::kColO + t * D + lane_base;

    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      // A wait that gives up (never expected) leaves ok false; the loop then
      // runs on without waiting and nothing it computes is stored.
      if (ok && !mbar_wait_warp(&s_full[t], i & 1, p.status)) ok = false;
      tc_fence_after();
      // Causal mask, only on tiles where some row of the warp sees keys past
      // its position (the diagonal); elsewhere every key is visible.
      const int key0 = i * kBN;
      const bool diag = __any_sync(0xffffffffu, key0 + kBN - 1 > pos);
      // The row maximum.  Off the diagonal, tcgen05.ld.red returns each
      // 32-column chunk's maximum with its values: the row is read half at a
      // time for the maxima alone (the values are read again below), and no
      // comparisons are needed.  On the diagonal (masked keys must not
      // count) the whole row is read and masked.
      float mt;
      if (!diag) {
        float c[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float sv[kBN / 2];
          tmem_ld32f_max(tmem_s + h * (kBN / 2), sv, &c[2 * h]);
          tmem_ld32f_max(tmem_s + h * (kBN / 2) + 32, sv + 32, &c[2 * h + 1]);
          tmem_wait_ld_bind_max(sv, &c[2 * h]);
          tmem_wait_ld_bind_max(sv + 32, &c[2 * h + 1]);
        }
        mt = fmaxf(fmax3(c[0], c[1], c[2]), c[3]) * p.qscale;
      } else {
        float sv[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32f(tmem_s + c * 32, sv + c * 32);
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_wait_ld_bind(sv + c * 32);
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c > pos) sv[c] = -CUDART_INF_F;
        // Row max with 8 independent chains (scaling by qscale > 0 commutes
        // with the max).
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = sv[k];
        constexpr int kTriples = (kBN - 8) / 16;  // columns 8 .. 8 + 16 kTriples - 1, in threes
#pragma unroll
        for (int c = 0; c < kTriples; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], sv[8 + 16 * c + k], sv[16 + 16 * c + k]);
#pragma unroll
        for (int c = 8 + 16 * kTriples; c < kBN; c += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], sv[c + k]);
        mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
             p.qscale;
      }
      // Lazy rescaling: the running max moves only when this tile exceeds it
      // by more than 8 (base 2), so P stays <= 2^8 and O is rescaled rarely.
      // Numerator and denominator share the same max, so the result is exact.
      const float m_new = (mt > m_run + 8.f) ? mt : m_run;
      const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
      const float negm = (m_new == -CUDART_INF_F) ? 0.f : -m_new;
      const float2 qs2 = make_float2(p.qscale, p.qscale);
      const float2 nm2 = make_float2(negm, negm);
      // O_t is quiescent here (S_t of this tile was issued only after the
      // previous P V into O_t had finished): rescale it, if the max moved,
      // before any P of this tile is released.
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          float o[16];
          tmem_ld16f(tmem_o + c * 16, o);
          tmem_wait_ld_bind16(o);
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const float2 y = __fmul2_rn(make_float2(o[k], o[k + 1]), a2);
            o[k] = y.x;
            o[k + 1] = y.y;
          }
          tmem_st16f(tmem_o + c * 16, o);
        }
      }
      // P, rounded to the operand type, over the first half of S's columns,
      // computed and released in two halves of the keys.
      float2 sm[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) sm[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // Keys [64 h, 64 h + 64): S columns 64 h .. 64 h + 63, still intact (P
        // of the first half went to columns 0..31).
        float sv[kBN / 2];
        tmem_ld32f(tmem_s + h * (kBN / 2), sv);
        tmem_ld32f(tmem_s + h * (kBN / 2) + 32, sv + 32);
        tmem_wait_ld_bind(sv);
        tmem_wait_ld_bind(sv + 32);
        if (diag) {
#pragma unroll
          for (int c = 0; c < kBN / 2; ++c)
            if (key0 + h * (kBN / 2) + c > pos) sv[c] = -CUDART_INF_F;
        }
        uint32_t w[kBN / 4];
#pragma unroll
        for (int c = 0; c < kBN / 2; c += 2) {
          const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), qs2, nm2);
          float2 e;
          e.x = ex2(x.x);
          e.y = ex2(x.y);
          sm[(c >> 1) & 3] = __fadd2_rn(sm[(c >> 1) & 3], e);
          w[c >> 1] = Cvt<T>::from_float2(e.x, e.y);
        }
        tmem_st32u(tmem_s + h * (kBN / 4), w);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[2 * t + h]);
      }
      sm[0] = __fadd2_rn(__fadd2_rn(sm[0], sm[1]), __fadd2_rn(sm[2], sm[3]));
      l_run = l_run * alpha + (sm[0].x + sm[0].y);
      m_run = m_new;
    }

    if (nt > 0 && ok && mbar_wait_warp(&pv_done[t], (nt - 1) & 1, p.status)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      T* orow = static_cast<T*>(p.out) + row_elem;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32f(tmem_o + c * 32, o);
        tmem_wait_ld_bind(o);
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 v;
            v.x = Cvt<T>::from_float2(o[k] * inv, o[k + 1] * inv);
            v.y = Cvt<T>::from_float2(o[k + 2] * inv, o[k + 3] * inv);
            v.z = Cvt<T>::from_float2(o[k + 4] * inv, o[k + 5] * inv);
            v.w = Cvt<T>::from_float2(o[k + 6] * inv, o[k + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + k) = v;
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

template <typename T, int D>
cudaError_t launch_prefill_typed(const PrefillParams& p, const CUtensorMap& qm,
                                 const CUtensorMap& km, const CUtensorMap& vm, int q_tiles,
                                 int num_seqs, cudaStream_t stream) {
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
  const dim3 grid((unsigned)((long long)q_tiles * p.num_kv_heads * num_seqs));
  paged_prefill_kernel<T, D><<<grid, kPrefillThreads, L::kBytes, stream>>>(p, qm, km, vm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream, bool* unsupported) {
  *unsupported = false;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.num_kv_heads * a.block_size;
  if (!make_cache_map(&km, a.k_cache, a.dtype, rows, a.head_dim, a.block_size) ||
      !make_cache_map(&vm, a.v_cache, a.dtype, rows, a.head_dim, a.block_size)) {
    *unsupported = true;
    return cudaErrorInvalidValue;
  }
  int gp = 1;
  while (gp < a.num_q_heads / a.num_kv_heads) gp <<= 1;
  // Q rows: one copy per row tile, G' heads x 128 / G' queries (G' <= 128).
  CUtensorMap qm;
  if (!make_token_head_map(&qm, a.q, a.dtype, a.total_queries, a.num_q_heads, a.head_dim,
                           gp, kBM / gp)) {
    *unsupported = true;
    return cudaErrorInvalidValue;
  }
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
  const int rows_q = kRowTiles * (kBM / gp);  // queries per CTA
  const int q_tiles = (a.max_query_len + rows_q - 1) / rows_q;
  if ((long long)q_tiles * a.num_kv_heads * a.num_seqs > 0x7fffffffLL) {
    *unsupported = true;  // more work items than a 1-D grid holds: unsupported
    return cudaErrorInvalidValue;
  }
  p.num_seqs = a.num_seqs;
  p.q_tiles = q_tiles;
  p.total_queries = a.total_queries;
  p.prefetch_stride = std::max(1, a.sm_count);
  // About one wave of CTAs (one per SM) per group; the count only shapes
  // the order, not the result.
  const int pairs = a.num_kv_heads * a.num_seqs;
  p.pairs_per_group = std::max(1, std::min(pairs, a.sm_count / std::max(1, q_tiles)));
  if (a.dtype == PKV_F16) {
    return a.head_dim == 64
               ? launch_prefill_typed<__half, 64>(p, qm, km, vm, q_tiles, a.num_seqs, stream)
               : launch_prefill_typed<__half, 128>(p, qm, km, vm, q_tiles, a.num_seqs, stream);
  }
  return a.head_dim == 64
             ? launch_prefill_typed<__nv_bfloat16, 64>(p, qm, km, vm, q_tiles, a.num_seqs, stream)
             : launch_prefill_typed<__nv_bfloat16, 128>(p, qm, km, vm, q_tiles, a.num_seqs, stream);
}

}  // namespace pkv
