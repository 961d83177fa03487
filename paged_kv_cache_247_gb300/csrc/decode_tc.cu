// Grouped-head paged decode on the 5th-generation tensor cores (tcgen05).
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
// N is the group rounded up to 16 or 32.  One CTA owns (sequence s, KV
// head, partition of the context) and every head of the group, so each K/V
// tile is read from HBM once per group.  Six warps:
//
//   warps 0-3  key warpgroup: thread t reads S^T lane t (key t of the tile)
//              and computes P^T column t = exp2(x - m) per head with a running
//              maximum per head that moves only when a tile exceeds it by
//              more than 8 (base 2; then the threads agree on the new maxima,
//              rescale their partial sums and O^T); partial row sums stay per
//              thread.  At the end thread d normalises and writes dimension d
//              of every head.
//   warp 4     producer: block-table entries and one 4-D TMA copy per
//              (block, head) run of K and of V into rings of tiles.
//   warp 5     MMA issuer and owner of the tensor memory: S^T of tile i, then
//              O^T += P^T of tile i - 1, so the tensor core works on the next
//              tile while the threads work on this one.
//
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

constexpr int kD = 128;                 // head size of this path
constexpr int kKeys = kTileKeys;        // keys per tile: M of S^T, K of O^T
constexpr int kKeyWarps = 4;            // the key warpgroup
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kGroupKV = (kD / 64) * 1024;   // bytes between 8-row groups of a K/V tile
constexpr int kKvTile = (kKeys / 8) * kGroupKV;
constexpr int kGroupP = (kKeys / 64) * 1024; // bytes between 8-head groups of P^T
constexpr int kBarSlots = 32;

// NH: heads a thread handles (the group rounded up to a power of two);
// N: the MMA's N (at least 16).
template <int NH>
struct TcShape {
  static constexpr int N = NH < 16 ? 16 : NH;
  static constexpr int kStages = 3;                  // K ring and V ring depth
  static constexpr int kQ = 2 * kStages * kKvTile;   // after the K and V rings
  static constexpr int kQBytes = (N / 8) * kGroupKV;
  static constexpr int kP = kQ + kQBytes;
  static constexpr int kPBuf = (N / 8) * kGroupP;
  static constexpr int kRed = kP + 2 * kPBuf;        // cross-warp reductions: [4][NH] floats
  static constexpr int kMref = kRed + kKeyWarps * NH * 4;
  static constexpr int kBar = kMref + NH * 4;
  static constexpr int kTmemSlot = kBar + kBarSlots * 8;
  static constexpr int kBytes = kTmemSlot + 16 + 1024;  // + alignment slack
  static_assert(kBytes <= 227 * 1024, "shared memory overflow");
  // tensor memory: S^T double buffer, then O^T
  static constexpr int kColO = 2 * N;
  static constexpr int kTmemCols = 3 * N <= 64 ? 64 : 128;
  static_assert(3 * N <= kTmemCols, "tensor memory overflow");
};

// Reduction of a predicate over the key warpgroup (named barrier 1): true if
// any of its 128 threads passes true.
__device__ __forceinline__ bool key_group_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void key_group_sync() { named_barrier_sync(1, kKeyWarps * 32); }

// N consecutive 32-bit columns of this thread's lane into v (N = 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float* v) {
  if constexpr (N == 16) {
    tmem_ld16f(taddr, v);
    tmem_wait_ld_bind16(v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32f(taddr + c * 32, v + c * 32);
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_wait_ld_bind(v + c * 32);
  }
}

template <int N>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const float* v) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) tmem_st16f(taddr + c * 16, v + c * 16);
  tmem_wait_st();
}

template <typename T, int NH>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap) {
  using L = TcShape<NH>;
  constexpr int N = L::N;
  constexpr int S = L::kStages;
  grid_dep_wait();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sK = smem;
  unsigned char* sV = smem + S * kKvTile;
  unsigned char* sQ = smem + L::kQ;
  unsigned char* sP = smem + L::kP;
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  float* mref_s = reinterpret_cast<float*>(smem + L::kMref);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* k_full = bars;             // [S] K tile landed (TMA bytes)
  uint64_t* k_empty = k_full + S;      // [S] S^T MMAs done reading it (commit)
  uint64_t* v_full = k_empty + S;      // [S] V tile landed
  uint64_t* v_empty = v_full + S;      // [S] O^T MMAs done reading it (commit)
  uint64_t* s_full = v_empty + S;      // [2] S^T buffer computed (commit)
  uint64_t* s_free = s_full + 2;       // [2] S^T buffer read by the key warpgroup
  uint64_t* p_full = s_free + 2;       // [2] P^T buffer written (key warpgroup)
  uint64_t* p_free = p_full + 2;       // [2] O^T MMAs done with P^T buffer (commit)
  uint64_t* q_full = p_free + 2;       // Q rows in shared memory
  uint64_t* drain = q_full + 1;        // the issuer's last MMAs finished
  static_assert(4 * S + 10 <= kBarSlots, "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int G = p.group;
  const int h0 = kvh * G;

  int ctx = p.context_lens[s];
  const long long cap_ll = min((long long)p.max_context_len,
                               (long long)p.max_blocks_per_seq * p.block_size);
  const int ctx_cap = (int)cap_ll;
  if (ctx < 0 || ctx > ctx_cap) {
    if (threadIdx.x == 0 && part == 0) atomicOr(p.status, PKV_DEV_BAD_CONTEXT_LEN);
    ctx = ctx < 0 ? 0 : ctx_cap;
  }
  const int t_begin = part * p.partition_size;
  const int t_end = min(ctx, t_begin + p.partition_size);
  const int nparts_seq = (ctx + p.partition_size - 1) / p.partition_size;
  if (t_begin >= t_end) {
    if (ctx == 0 && part == 0) {  // empty context: the output is zero
      uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + ((size_t)s * p.num_q_heads + h0) * kD;
      for (int i = threadIdx.x; i < G * kD; i += kThreads) o[i] = 0;
    }
    return;
  }
  const int n_tiles = (t_end - t_begin + kKeys - 1) / kKeys;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kKeyWarps * 32);
      mbar_init(&p_full[b], kKeyWarps * 32);
      mbar_init(&p_free[b], 1);
    }
    mbar_init(q_full, kKeyWarps * 32);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(L::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Tile i covers keys [t_begin + 128 i, +128).  Its keys are runs of B
    // rows, one block each; lane l copies run l of K and of V with one TMA
    // copy each.  The block id of the lane's run of the next tile is read
    // before this tile's copies are issued, so its latency overlaps the wait
    // for a free slot.
    const int B = p.block_size;
    const int32_t* trow = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    auto table_entry = [&](int i) -> int {
      const int key = t_begin + i * kKeys + lane * B;
      return (lane * B < kKeys && i < n_tiles && key < t_end) ? __ldg(trow + key / B) : 0;
    };
    // Fused append: the step's new token is position ctx - 1 of the last
    // partition.  Lanes 0-15 hold its K row and lanes 16-31 its V row (16
    // bytes each); the row is written to its cache slot before the copy of
    // the tile that holds it, so the copy reads the new row.
    const bool fused_here = p.k_new != nullptr && t_end == ctx;
    const bool new_is_v = lane >= 16;
    const int new_c = lane & 15;
    uint4 new_chunk = make_uint4(0, 0, 0, 0);
    if (fused_here) {
      const size_t row_off = ((size_t)s * p.num_kv_heads + kvh) * kD;
      new_chunk = reinterpret_cast<const uint4*>(
          static_cast<const T*>(new_is_v ? p.v_new : p.k_new) + row_off)[new_c];
    }
    int phys_next = table_entry(0);
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % S;
      const uint32_t ph = ((i / S) - 1) & 1;
      const int key0 = t_begin + i * kKeys;
      const int nvalid = min(kKeys, t_end - key0);
      const int nseg = (nvalid + B - 1) / B;
      const uint32_t bytes = (uint32_t)nseg * B * kD * (uint32_t)sizeof(T);
      int phys = phys_next;
      phys_next = table_entry(i + 1);
      if ((unsigned)phys >= (unsigned)p.num_blocks) {
        if (lane < nseg) atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
        phys = 0;
      }
      if (fused_here && key0 + nvalid == ctx) {
        const int pos = ctx - 1;
        const int seg_new = (pos - key0) / B;
        const int phys_new = __shfl_sync(0xffffffffu, phys, seg_new);
        const size_t dst = (((size_t)phys_new * p.num_kv_heads + kvh) * B + (pos % B)) * kD;
        T* cache = const_cast<T*>(static_cast<const T*>(new_is_v ? p.v_cache : p.k_cache));
        reinterpret_cast<uint4*>(cache + dst)[new_c] = new_chunk;
        // the row must be visible to the copy engine's reads below
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
      }
      const int g = ((phys * p.num_kv_heads + kvh) * B) / 8;  // first 8-row group of the run
      const uint32_t dst = (uint32_t)(st * kKvTile + lane * (B / 8) * kGroupKV);
      if (i >= S && !mbar_wait_warp(&k_empty[st], ph, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], bytes);
      __syncwarp();
      if (lane < nseg) tma_load_group(sK + dst, &kmap, g, &k_full[st]);
      if (i >= S && !mbar_wait_warp(&v_empty[st], ph, p.status)) {
        issued = i + 1;  // K of this tile is in flight
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], bytes);
      __syncwarp();
      if (lane < nseg) tma_load_group(sV + dst, &vmap, g, &v_full[st]);
      issued = i + 1;
    }
    // After a timeout, copies still in flight land before the CTA leaves.
    if (timed_out(p.status)) {
      for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
        mbar_drain(&k_full[i % S], (i / S) & 1);
        mbar_drain(&v_full[i % S], (i / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- issuer
    if (lane == 0) {
      constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
      const uint32_t idesc_s = instr_desc(bf16, false, false, N, kKeys);
      const uint32_t idesc_o = instr_desc(bf16, true, false, N, kD);
      const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ),
                     aP = smem_addr(sP);
      bool ok = mbar_wait(q_full, 0, p.status);
      // O^T += V^T P^T for tile j: 16 keys per MMA, two 8-key groups of V
      // and a 32-byte step inside P^T's 128-byte rows.
      auto pv = [&](int j) -> bool {
        const int st = j % S;
        if (!mbar_wait(&v_full[st], (j / S) & 1, p.status)) return false;
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks)
          mma_f16_ss(tmem + L::kColO,
                     smem_desc(aV + st * kKvTile + ks * 2 * kGroupKV, 1024, kGroupKV),
                     smem_desc(aP + (j & 1) * L::kPBuf + (ks / 4) * 1024 + (ks % 4) * 32, 16,
                               kGroupP),
                     idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&p_free[j & 1]);
        mma_commit(&v_empty[st]);
        return true;
      };
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % S;
        if (!mbar_wait(&k_full[st], (i / S) & 1, p.status)) break;
        if (i >= 2 && !mbar_wait(&s_free[i & 1], ((i - 2) >> 1) & 1, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t koff = (ks / 4) * 1024 + (ks % 4) * 32;
          mma_f16_ss(tmem + (i & 1) * N, smem_desc(aK + st * kKvTile + koff, 16, kGroupKV),
                     smem_desc(aQ + koff, 16, kGroupKV), idesc_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[i & 1]);
        mma_commit(&k_empty[st]);
        if (i >= 1 && !pv(i - 1)) ok = false;
        if (ok && i == n_tiles - 1) ok = pv(i);
      }
      mma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ key warpgroup
    const int t = threadIdx.x;  // key of the tile == tensor-memory lane; later dimension d
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    // Q rows of the group into shared memory (K-major operand), padding
    // rows zero.  All loads are issued before the first store.
    {
      constexpr int kChunks = N * (kD / 8);
      constexpr int kPer = (kChunks + 127) / 128;
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                         ((size_t)s * p.num_q_heads + h0) * kD);
      uint4 v[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = t + 128 * k;
        const int r = i / (kD / 8);
        v[k] = (i < kChunks && r < G) ? __ldg(qsrc + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = t + 128 * k;
        if (i < kChunks)
          *reinterpret_cast<uint4*>(sQ + chunk_offset<kD>(i / (kD / 8), i % (kD / 8))) = v[k];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(q_full);
    }
    if (t < NH) mref_s[t] = -CUDART_INF_F;

    float l_part[NH];
#pragma unroll
    for (int g = 0; g < NH; ++g) l_part[g] = 0.f;
    const float qs = p.qscale;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int key0 = t_begin + i * kKeys;
      const int nvalid = min(kKeys, t_end - key0);
      const bool valid = t < nvalid;
      // A wait that gives up (never expected) leaves ok false; the loop runs
      // on without waiting, so that every named barrier stays matched, and
      // nothing it computes is stored.
      if (ok && !mbar_wait_warp(&s_full[i & 1], (i >> 1) & 1, p.status)) ok = false;
      tc_fence_after();
      float x[N];
      tmem_load_cols<N>(tmem + (i & 1) * N + lane_base, x);
      tc_fence_before();
      mbar_arrive(&s_free[i & 1]);
      key_group_sync();  // mref_s written (first tile) or last moved
      float mref[NH];
#pragma unroll
      for (int g = 0; g < NH; ++g) mref[g] = mref_s[g];
      bool exceed = false;
#pragma unroll
      for (int g = 0; g < NH; ++g) {
        x[g] = x[g] * qs;  // base-2 logit
        exceed |= valid && g < G && x[g] > mref[g] + 8.f;
      }
      if (key_group_any(exceed)) {
        // Some key exceeds its head's running max by more than 8: the tile
        // maxima per head, then the heads whose maximum moves.
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          float v = (valid && g < G) ? x[g] : -CUDART_INF_F;
#pragma unroll
          for (int mk = 16; mk >= 1; mk >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, mk));
          if (lane == 0) red[warp * NH + g] = v;
        }
        key_group_sync();
        float alpha[NH];
        bool moved = false;
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          const float mt = fmaxf(fmaxf(red[g], red[NH + g]), fmaxf(red[2 * NH + g], red[3 * NH + g]));
          const float mn = mt > mref[g] + 8.f ? mt : mref[g];
          alpha[g] = (mn == mref[g]) ? 1.f : ex2(mref[g] - mn);
          moved |= mn != mref[g];
          mref[g] = mn;
          l_part[g] *= alpha[g];
        }
        key_group_sync();  // every thread has read red[] and the old maxima
        if (t == 0) {
#pragma unroll
          for (int g = 0; g < NH; ++g) mref_s[g] = mref[g];
        }
        if (i > 0 && moved) {
          // O^T holds tiles 0..i-1: once their MMAs are done (P^T buffer
          // (i-1) released), thread d rescales column g of its lane.
          if (ok && !mbar_wait_warp(&p_free[(i - 1) & 1], ((i - 1) >> 1) & 1, p.status))
            ok = false;
          tc_fence_after();
          float o[N];
          tmem_load_cols<N>(tmem + L::kColO + lane_base, o);
#pragma unroll
          for (int g = 0; g < NH; ++g) o[g] *= alpha[g];
          tmem_store_cols<N>(tmem + L::kColO + lane_base, o);
          tc_fence_before();
        }
      }
      // P^T column t: exp2(x - m) per head, rounded to the operand type.
      T pt[NH];
#pragma unroll
      for (int g = 0; g < NH; ++g) {
        const float e = (valid && g < G) ? ex2(x[g] - mref[g]) : 0.f;
        l_part[g] += e;
        pt[g] = static_cast<T>(e);
      }
      // The buffer was last read by the MMAs of tile i - 2.
      if (i >= 2 && ok && !mbar_wait_warp(&p_free[i & 1], ((i - 2) >> 1) & 1, p.status)) ok = false;
      unsigned char* pb = sP + (i & 1) * L::kPBuf;
#pragma unroll
      for (int g = 0; g < NH; ++g)
        if (g < G)
          *reinterpret_cast<T*>(pb + chunk_offset<kKeys>(g, t >> 3) + (t & 7) * 2) = pt[g];
      if (nvalid < kKeys) {
        // The last tile: V rows past the context must not feed stale or NaN
        // values into O^T (their P is 0, but 0 * NaN is NaN).
        const int st = i % S;
        if (ok && !mbar_wait_warp(&v_full[st], (i / S) & 1, p.status)) ok = false;
        if (!valid) {
#pragma unroll
          for (int c = 0; c < kD / 8; ++c)
            *reinterpret_cast<uint4*>(sV + st * kKvTile + chunk_offset<kD>(t, c)) =
                make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&p_full[i & 1]);
    }
    grid_dep_launch_dependents();

    // Row sums per head over the 128 keys' partial sums.
#pragma unroll
    for (int g = 0; g < NH; ++g) {
      float v = l_part[g];
#pragma unroll
      for (int mk = 16; mk >= 1; mk >>= 1) v += __shfl_xor_sync(0xffffffffu, v, mk);
      if (lane == 0) red[warp * NH + g] = v;
    }
    key_group_sync();
    const int last = n_tiles - 1;
    if (ok && mbar_wait_warp(&p_free[last & 1], (last >> 1) & 1, p.status)) {
      tc_fence_after();
      float o[N];
      tmem_load_cols<N>(tmem + L::kColO + lane_base, o);
      const int d = t;
#pragma unroll
      for (int g = 0; g < NH; ++g) {
        if (g >= G) continue;
        const float l = (red[g] + red[NH + g]) + (red[2 * NH + g] + red[3 * NH + g]);
        const float val = o[g] / l;
        if (nparts_seq == 1) {
          static_cast<T*>(p.out)[((size_t)s * p.num_q_heads + h0 + g) * kD + d] =
              static_cast<T>(val);
        } else {
          const size_t r = ((size_t)s * p.num_q_heads + h0 + g) * p.num_parts + part;
          p.ws_o[r * kD + d] = val;
          if (d == 0) {
            p.ws_m[r] = mref_s[g];
            p.ws_l[r] = l;
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
                 "r"(L::kTmemCols));
  }
}

template <typename T, int NH>
cudaError_t launch_tc_typed(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm,
                            cudaStream_t stream) {
  using L = TcShape<NH>;
  static unsigned long long configured = 0;  // bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    err = cudaFuncSetAttribute(paged_decode_tc_kernel<T, NH>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  const dim3 grid(p.num_parts, p.num_kv_heads, p.num_seqs);
  err = launch_overlapped(paged_decode_tc_kernel<T, NH>, grid, dim3(kThreads), L::kBytes, stream,
                          p, km, vm);
  if (err != cudaSuccess || p.num_parts <= 1) return err;
  return launch_decode_reduce(p, std::is_same<T, __nv_bfloat16>::value ? PKV_BF16 : PKV_F16, kD,
                              stream);
}

template <typename T>
cudaError_t launch_tc_group(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm,
                            cudaStream_t stream) {
  static_assert(kMaxTcGroup == 32, "instantiations cover groups up to 32");
  if (p.group <= 4) return launch_tc_typed<T, 4>(p, km, vm, stream);
  if (p.group <= 8) return launch_tc_typed<T, 8>(p, km, vm, stream);
  if (p.group <= 16) return launch_tc_typed<T, 16>(p, km, vm, stream);
  return launch_tc_typed<T, 32>(p, km, vm, stream);
}

}  // namespace

bool decode_tc_supported(int head_dim, int group, int partition_size) {
  static_assert(kTcPartitionQuantum == kKeys, "partitions are whole tiles");
  return head_dim == kD && group >= kMinTcGroup && group <= kMaxTcGroup &&
         partition_size % kKeys == 0;
}

cudaError_t launch_paged_decode_tc(const DecodeParams& p, int dtype, cudaStream_t stream,
                                   bool* unsupported) {
  *unsupported = false;
  CUtensorMap km, vm;
  const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
  if (!make_cache_map(&km, p.k_cache, dtype, rows, kD, p.block_size) ||
      !make_cache_map(&vm, p.v_cache, dtype, rows, kD, p.block_size)) {
    *unsupported = true;
    return cudaErrorInvalidValue;
  }
  return dtype == PKV_F16 ? launch_tc_group<__half>(p, km, vm, stream)
                          : launch_tc_group<__nv_bfloat16>(p, km, vm, stream);
}

}  // namespace pkv
