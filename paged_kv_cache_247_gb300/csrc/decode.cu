// Paged single-query decode attention for sm_103a.
//
// What it computes ("Only 20.4% of your KV cache held actual tokens", section
// "The page table, relocated into attention"): for each sequence and query
// head, softmax(scale * q . K) V over the sequence's context, with K and V
// gathered block by block through the sequence's block table.
//
// One CTA owns (sequence s, KV head, partition of the context) and computes
// every query head of the KV head's group, so each K/V block is read from HBM
// once per group.  Five warps:
//
//   warp 4      producer: keeps the partition's physical block ids in shared
//               memory (the table walker) and streams K and V into a ring of
//               NSTAGE stages of 32 tokens with bulk asynchronous copies
//               (cp.async.bulk, the 1-D TMA path), one copy per contiguous
//               (block, head) run, completing on an mbarrier per stage.
//   warps 0-3   consumers: each takes 8 of a stage's 32 rows.  Eight lanes
//               share one row (16 bytes each per 64 columns), so a group of
//               8 lanes reads 128 contiguous bytes per load; logits of the
//               warp's rows are summed with a transposed butterfly over the
//               8 lanes, then an online softmax (running max and sum in base
//               2, fp32) updates the warp's accumulator of p * V.
//
// At the end the four warps' (max, sum, accumulator) triples are merged in
// shared memory.  A partition that is the whole context writes the output
// directly; otherwise it writes a normalised partial output with its max and
// sum, and a second kernel merges the partitions (split context,
// flash-decoding style).
//
// HBM traffic is the K and V bytes of the context plus q, the table and the
// output: the kernel is bandwidth-bound; the copy engine keeps up to NSTAGE x
// 16 KiB in flight per CTA.

#include <math_constants.h>

#include "common.cuh"
#include "overlap.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kTokStage = 32;       // tokens per pipeline stage
constexpr int kTbl = 128;           // block ids held in shared memory at once
constexpr unsigned kFull = 0xffffffffu;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// After a timed-out wait the consumers stop early and the CTA would exit with
// bulk copies still landing in its shared memory.  The producer calls this
// before it returns: if a wait timed out anywhere, it waits (bounded) for the
// stages it filled last, whose copies may still be in flight.  On the normal
// path every stage has been consumed and the check is the only cost.
template <int NSTAGE>
__device__ __forceinline__ void drain_if_timed_out(uint64_t* full, int issued,
                                                   const unsigned int* status) {
  if (!timed_out(status)) return;
  for (int it = issued > NSTAGE ? issued - NSTAGE : 0; it < issued; ++it)
    mbar_drain(&full[it % NSTAGE], (it / NSTAGE) & 1);
  __syncwarp();
}

template <int D>
constexpr int stages_for() { return D >= 128 ? 4 : 8; }

// Thread layout of one decode CTA, chosen per head size and group size.
//   LPR   lanes that share one K/V row (each reads D / LPR columns)
//   NCW   consumer warps (the producer is one more warp)
//   MINB  CTAs per SM the register budget is sized for
// More lanes per row means fewer q/accumulator registers per thread, which
// buys more resident warps to hide the latency of the reductions.
#ifndef PKV_G1_LPR
#define PKV_G1_LPR 8
#define PKV_G1_NCW 4
#define PKV_G1_MINB 3
#endif
#ifndef PKV_G2_LPR
#define PKV_G2_LPR 16
#define PKV_G2_NCW 4
#define PKV_G2_MINB 3
#endif
#ifndef PKV_G4_LPR
#define PKV_G4_LPR 16
#define PKV_G4_NCW 4
#define PKV_G4_MINB 3
#endif

template <int LPR_, int NCW_, int MINB_>
struct Layout {
  static constexpr int LPR = LPR_;
  static constexpr int NCW = NCW_;
  static constexpr int MINB = MINB_;
};

template <int D, int GT>
struct LayoutFor;
template <int GT>
struct LayoutFor<64, GT> : Layout<8, 4, 3> {};  // a 128-byte row: one 16-byte chunk per lane
template <>
struct LayoutFor<128, 1> : Layout<PKV_G1_LPR, PKV_G1_NCW, PKV_G1_MINB> {};
template <>
struct LayoutFor<128, 2> : Layout<PKV_G2_LPR, PKV_G2_NCW, PKV_G2_MINB> {};
template <>
struct LayoutFor<128, 4> : Layout<PKV_G4_LPR, PKV_G4_NCW, PKV_G4_MINB> {};

template <typename T, int D, int GT>
struct SmemLayout {
  static constexpr int NCW = LayoutFor<D, GT>::NCW;
  static constexpr int kStages = stages_for<D>();
  static constexpr size_t kStageElems = (size_t)kTokStage * D;
  static constexpr size_t kRing = kStages * kStageElems * sizeof(T);   // one of K, V
  static constexpr size_t kMergeAcc = (size_t)NCW * GT * D * 4;        // floats
  static constexpr size_t kMergeMl = (size_t)NCW * GT * 4;
  static constexpr size_t kTable = kTbl * 4;
  static constexpr size_t kBars = 2 * kStages * 8;
  static constexpr size_t kBytes = 2 * kRing + kMergeAcc + 2 * kMergeMl + kTable + kBars;
  static constexpr int kThreads = (NCW + 1) * 32;
};

// kPaged = false is the contiguous-cache baseline: sequence s owns the rows
// [s][h][0, capacity) of the caches (block_size = capacity, no table).
template <typename T, int D, int GT, bool kPaged>
__global__ void __launch_bounds__(SmemLayout<T, D, GT>::kThreads, LayoutFor<D, GT>::MINB)
    paged_decode_kernel(const DecodeParams p) {
  using L = SmemLayout<T, D, GT>;
  using LY = LayoutFor<D, GT>;
  constexpr int LPR = LY::LPR;
  constexpr int NCW = LY::NCW;
  constexpr int NSTAGE = L::kStages;
  constexpr int RPP = 32 / LPR;              // rows a warp covers per pass
  constexpr int RPW = kTokStage / NCW;       // rows a warp owns per stage
  constexpr int NP = RPW / RPP;              // passes per stage
  constexpr int CPL = D / (8 * LPR);         // 16-byte chunks per lane per row
  constexpr int NF2 = 4 * CPL;               // float2 per lane per row
  constexpr int NV = GT * NP;                // partial sums per lane before the reduction
  constexpr int LBL = ilog2(LPR);
  constexpr int H = ilog2(NV);               // halving steps of the butterfly
  constexpr int SH = LBL - H;                // lane-bit shift of a reduced value's index
  constexpr int LOG2NP = ilog2(NP);
  static_assert(CPL >= 1 && NP >= 1 && NV <= LPR, "unsupported decode layout");

  // Before anything else: no memory is touched until the previous kernel on
  // the stream has finished.  (Placed after the index arithmetic instead, it
  // changed the register allocation of the four-head instantiations, and the
  // paged kernel ran 1 % slower on GB300.)
  grid_dep_wait();
  extern __shared__ __align__(128) unsigned char smem[];
  T* Ks = reinterpret_cast<T*>(smem);
  T* Vs = Ks + NSTAGE * L::kStageElems;
  float* mg_acc = reinterpret_cast<float*>(Vs + NSTAGE * L::kStageElems);
  float* mg_max = mg_acc + NCW * GT * D;
  float* mg_sum = mg_max + NCW * GT;
  int* tbl = reinterpret_cast<int*>(mg_sum + NCW * GT);
  uint64_t* full = reinterpret_cast<uint64_t*>(tbl + kTbl);
  uint64_t* empty = full + NSTAGE;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int kvh = blockIdx.y / p.head_chunks;
  const int hc = blockIdx.y - kvh * p.head_chunks;
  const int s = blockIdx.z;
  const int h0 = kvh * p.group + hc * GT;
  const int nh = min(GT, p.group - hc * GT);

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
      uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + ((size_t)s * p.num_q_heads + h0) * D;
      for (int i = threadIdx.x; i < nh * D; i += L::kThreads) o[i] = 0;
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int nstages = (t_end - t_begin + kTokStage - 1) / kTokStage;

  // ------------------------------------------------------------ producer --
  if (warp == NCW) {
    const uint64_t policy = policy_evict_first();
    const T* kbase = static_cast<const T*>(p.k_cache);
    const T* vbase = static_cast<const T*>(p.v_cache);
    if constexpr (!kPaged) {
      // Contiguous baseline: one run per stage, no table.
      const size_t seq_base = ((size_t)s * p.num_kv_heads + kvh) * (size_t)p.block_size * D;
      int issued = 0;
      for (int it = 0; it < nstages; ++it) {
        const int stg = it % NSTAGE;
        if (it >= NSTAGE && !mbar_wait_warp(&empty[stg], ((it / NSTAGE) - 1) & 1, p.status)) break;
        const int tok0 = t_begin + it * kTokStage;
        const int ntok = min(kTokStage, t_end - tok0);
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)ntok * D * sizeof(T);
          mbar_arrive_expect_tx(&full[stg], 2 * bytes);
          bulk_load(Ks + stg * L::kStageElems, kbase + seq_base + (size_t)tok0 * D, bytes,
                    &full[stg], policy);
          bulk_load(Vs + stg * L::kStageElems, vbase + seq_base + (size_t)tok0 * D, bytes,
                    &full[stg], policy);
        }
        __syncwarp();
        issued = it + 1;
      }
      drain_if_timed_out<NSTAGE>(full, issued, p.status);
      return;
    }
    const int log2B = p.log2_block;
    const int lb_last = (t_end - 1) >> log2B;
    const int32_t* trow = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const size_t tile = (size_t)p.block_size * D;  // elements of one (block, head) tile
    int chunk_base = -1;
    // Fused append: the step's new token is position ctx - 1, the last row of
    // this partition when t_end == ctx.  Its K (lanes 0..kRowChunks-1) and V
    // (the next kRowChunks lanes) 16-byte chunks are fetched now so that the
    // load overlaps the pipeline.
    constexpr int kRowChunks = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
    const bool fused_here = p.k_new != nullptr && t_end == ctx;
    const bool new_is_v = lane >= kRowChunks;
    const int new_c = new_is_v ? lane - kRowChunks : lane;
    uint4 new_chunk = make_uint4(0, 0, 0, 0);
    if (fused_here && lane < 2 * kRowChunks) {
      const size_t row_off = ((size_t)s * p.num_kv_heads + kvh) * D;
      new_chunk = reinterpret_cast<const uint4*>(
          static_cast<const T*>(new_is_v ? p.v_new : p.k_new) + row_off)[new_c];
    }
    int issued = 0;
    for (int it = 0; it < nstages; ++it) {
      const int stg = it % NSTAGE;
      if (it >= NSTAGE && !mbar_wait_warp(&empty[stg], ((it / NSTAGE) - 1) & 1, p.status)) break;
      const int tok0 = t_begin + it * kTokStage;
      const int ntok = min(kTokStage, t_end - tok0);
      const int lb0 = tok0 >> log2B;
      const int lb1 = (tok0 + ntok - 1) >> log2B;
      if (chunk_base < 0 || lb1 >= chunk_base + kTbl) {
        // Walk the next window of the block table into shared memory.
        __syncwarp();
        chunk_base = lb0;
        for (int i = lane; i < kTbl; i += 32) {
          const int lb = chunk_base + i;
          int id = 0;
          if (lb <= lb_last) {
            id = __ldg(trow + lb);
            if ((unsigned)id >= (unsigned)p.num_blocks) {
              atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
              id = 0;
            }
          }
          tbl[i] = id;
        }
        __syncwarp();
      }
      // Fused append: the last row of the sequence's last stage comes from
      // the prefetched new row instead of the cache (the CTA of the first
      // head chunk also writes it to its slot); the cache copy stops one row
      // short.
      int copy_end = tok0 + ntok;
      const bool new_row_stage = fused_here && copy_end == ctx;
      if (new_row_stage) {
        copy_end -= 1;
        if (lane < 2 * kRowChunks) {
          T* srow = (new_is_v ? Vs : Ks) + stg * L::kStageElems + (ntok - 1) * D;
          reinterpret_cast<uint4*>(srow)[new_c] = new_chunk;
        }
        // Only shared-memory stores are outstanding here, so this fence is
        // cheap; the global store of the row into its slot comes after the
        // arrive, off the consumers' path.
        __threadfence_block();
      }
      __syncwarp();
      if (lane == 0)
        mbar_arrive_expect_tx(&full[stg], (uint32_t)(copy_end - tok0) * D * sizeof(T) * 2);
      __syncwarp();
      if (new_row_stage && hc == 0 && lane < 2 * kRowChunks) {
        const int pos = ctx - 1;
        const int lbn = pos >> log2B;
        const size_t dst = ((size_t)tbl[lbn - chunk_base] * p.num_kv_heads + kvh) * tile +
                           (size_t)(pos - (lbn << log2B)) * D;
        T* cache = const_cast<T*>(new_is_v ? vbase : kbase);
        reinterpret_cast<uint4*>(cache + dst)[new_c] = new_chunk;
      }
      // One copy per block the stage touches; rows past the context are not
      // copied, so positions beyond context_lens are never read.
      const int lbc = copy_end > tok0 ? ((copy_end - 1) >> log2B) : lb0 - 1;
      if (lane <= lbc - lb0) {
        const int lb = lb0 + lane;
        const int seg0 = max(tok0, lb << log2B);
        const int seg1 = min(copy_end, (lb + 1) << log2B);
        const size_t off = ((size_t)tbl[lb - chunk_base] * p.num_kv_heads + kvh) * tile +
                           (size_t)(seg0 - (lb << log2B)) * D;
        const uint32_t bytes = (uint32_t)(seg1 - seg0) * D * sizeof(T);
        const int row = seg0 - tok0;
        bulk_load(Ks + stg * L::kStageElems + row * D, kbase + off, bytes, &full[stg], policy);
        bulk_load(Vs + stg * L::kStageElems + row * D, vbase + off, bytes, &full[stg], policy);
      }
      issued = it + 1;
    }
    drain_if_timed_out<NSTAGE>(full, issued, p.status);
    return;
  }

  // ----------------------------------------------------------- consumers --
  const int rg = lane >> LBL;        // row group: which row of a pass this lane reads
  const int li = lane & (LPR - 1);   // position inside the row group

  // q for this lane's columns {8*(li + LPR*c) .. +7}, pre-scaled to base-2 logits.
  float2 qf[GT][NF2];
  {
    const T* qrow = static_cast<const T*>(p.q) + ((size_t)s * p.num_q_heads + h0) * D;
    const float2 sc = make_float2(p.qscale, p.qscale);
#pragma unroll
    for (int g = 0; g < GT; ++g) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (g < nh) w = *reinterpret_cast<const uint4*>(qrow + g * D + (li + LPR * c) * 8);
        qf[g][4 * c + 0] = __fmul2_rn(Cvt<T>::to_float2(w.x), sc);
        qf[g][4 * c + 1] = __fmul2_rn(Cvt<T>::to_float2(w.y), sc);
        qf[g][4 * c + 2] = __fmul2_rn(Cvt<T>::to_float2(w.z), sc);
        qf[g][4 * c + 3] = __fmul2_rn(Cvt<T>::to_float2(w.w), sc);
      }
    }
  }

  float2 acc[GT][NF2];
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int e = 0; e < NF2; ++e) acc[g][e] = make_float2(0.f, 0.f);
  float m_run = -CUDART_INF_F;  // running max of this lane's head (base 2)
  float l_run = 0.f;            // running sum of exp2(logit - m_run)

  const int idx_l = li >> SH;   // (g * NP + j) of the sum this lane ends up with
  const int g_l = idx_l / NP;
  const int j_l = idx_l % NP;

  for (int it = 0; it < nstages; ++it) {
    const int stg = it % NSTAGE;
    if (!mbar_wait_warp(&full[stg], (it / NSTAGE) & 1, p.status)) break;
    const int ntok = min(kTokStage, t_end - (t_begin + it * kTokStage));
    const T* Kst = Ks + stg * L::kStageElems;
    const T* Vst = Vs + stg * L::kStageElems;

    // Partial dot products over this lane's columns of rows
    // warp*RPW + j*RPP + rg, for every head of the group.
    float v[NV];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const int row = warp * RPW + j * RPP + rg;
      float2 kf[NF2];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(Kst + row * D + (li + LPR * c) * 8);
        kf[4 * c + 0] = Cvt<T>::to_float2(w.x);
        kf[4 * c + 1] = Cvt<T>::to_float2(w.y);
        kf[4 * c + 2] = Cvt<T>::to_float2(w.z);
        kf[4 * c + 3] = Cvt<T>::to_float2(w.w);
      }
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float2 a = __fmul2_rn(qf[g][0], kf[0]);
#pragma unroll
        for (int e = 1; e < NF2; ++e) a = __ffma2_rn(qf[g][e], kf[e], a);
        v[g * NP + j] = a.x + a.y;
      }
    }
    // Transposed butterfly over the row group's lanes: each exchange halves
    // the values a lane holds, so NV sums cost NV - 1 shuffles, not NV * LBL.
#pragma unroll
    for (int step = 0; step < H; ++step) {
      const int mk = (LPR >> 1) >> step;
      const bool upper = (li & mk) != 0;
      const int half = NV >> (step + 1);
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, mk);
      }
    }
    float x = v[0];
#pragma unroll
    for (int mk = (1 << SH) >> 1; mk >= 1; mk >>= 1) x += __shfl_xor_sync(kFull, x, mk);

    // Online softmax over the warp's rows of this stage: reduce over the
    // lanes that hold the same head (pass bits, then row-group bits).
    if (warp * RPW + j_l * RPP + rg >= ntok) x = -CUDART_INF_F;
    float mt = x;
#pragma unroll
    for (int b = 0; b < LOG2NP; ++b) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, (1 << SH) << b));
#pragma unroll
    for (int mk = LPR; mk < 32; mk <<= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, mk));
    const float m_new = fmaxf(m_run, mt);
    const float alpha = (m_new == -CUDART_INF_F) ? 1.f : exp2f(m_run - m_new);
    const float pe = (x == -CUDART_INF_F) ? 0.f : exp2f(x - m_new);
    float ps = pe;
#pragma unroll
    for (int b = 0; b < LOG2NP; ++b) ps += __shfl_xor_sync(kFull, ps, (1 << SH) << b);
#pragma unroll
    for (int mk = LPR; mk < 32; mk <<= 1) ps += __shfl_xor_sync(kFull, ps, mk);
    l_run = l_run * alpha + ps;
    m_run = m_new;
    if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const float a = __shfl_sync(kFull, alpha, (g * NP) << SH);
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int e = 0; e < NF2; ++e) acc[g][e] = __fmul2_rn(acc[g][e], a2);
      }
    }

    // acc += p * V for this lane's row of each pass.
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const int row = warp * RPW + j * RPP + rg;
      float pg[GT];
#pragma unroll
      for (int g = 0; g < GT; ++g)
        pg[g] = __shfl_sync(kFull, pe, (rg << LBL) | ((g * NP + j) << SH));
      if (row < ntok) {
        float2 vf[NF2];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(Vst + row * D + (li + LPR * c) * 8);
          vf[4 * c + 0] = Cvt<T>::to_float2(w.x);
          vf[4 * c + 1] = Cvt<T>::to_float2(w.y);
          vf[4 * c + 2] = Cvt<T>::to_float2(w.z);
          vf[4 * c + 3] = Cvt<T>::to_float2(w.w);
        }
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          const float2 pp = make_float2(pg[g], pg[g]);
#pragma unroll
          for (int e = 0; e < NF2; ++e) acc[g][e] = __ffma2_rn(pp, vf[e], acc[g][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stg]);
  }
  // The next kernel on the stream may be placed now (it waits for this
  // grid to finish); triggered this late, its CTAs are resident only during
  // this grid's last epilogues rather than through its whole last wave.
  grid_dep_launch_dependents();

  // The row groups of a warp share its running max: add their sums.
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int e = 0; e < NF2; ++e) {
      float2 a = acc[g][e];
#pragma unroll
      for (int mk = LPR; mk < 32; mk <<= 1) {
        a.x += __shfl_xor_sync(kFull, a.x, mk);
        a.y += __shfl_xor_sync(kFull, a.y, mk);
      }
      acc[g][e] = a;
    }
  if (rg == 0) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float4* dst = reinterpret_cast<float4*>(mg_acc + (warp * GT + g) * D + (li + LPR * c) * 8);
        dst[0] = make_float4(acc[g][4 * c].x, acc[g][4 * c].y, acc[g][4 * c + 1].x, acc[g][4 * c + 1].y);
        dst[1] = make_float4(acc[g][4 * c + 2].x, acc[g][4 * c + 2].y, acc[g][4 * c + 3].x,
                             acc[g][4 * c + 3].y);
      }
    if (j_l == 0 && (li & ((1 << SH) - 1)) == 0) {
      mg_max[warp * GT + g_l] = m_run;
      mg_sum[warp * GT + g_l] = l_run;
    }
  }
  named_barrier_sync(1, NCW * 32);

  // Merge the warps and write out (or the partition's partial result).
  for (int e0 = threadIdx.x * 4; e0 < nh * D; e0 += NCW * 32 * 4) {
    const int g = e0 / D;
    const int e = e0 - g * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, mg_max[w * GT + g]);
    float Lsum = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float mw = mg_max[w * GT + g];
      const float sc = (mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
      Lsum += mg_sum[w * GT + g] * sc;
      const float4 a = *reinterpret_cast<const float4*>(mg_acc + (w * GT + g) * D + e);
      o.x += a.x * sc;
      o.y += a.y * sc;
      o.z += a.z * sc;
      o.w += a.w * sc;
    }
    const float inv = 1.f / Lsum;
    if (nparts_seq == 1) {
      T* orow = static_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + h0 + g) * D + e;
      uint2 pk;
      pk.x = Cvt<T>::from_float2(o.x * inv, o.y * inv);
      pk.y = Cvt<T>::from_float2(o.z * inv, o.w * inv);
      *reinterpret_cast<uint2*>(orow) = pk;
    } else {
      const size_t r = ((size_t)s * p.num_q_heads + h0 + g) * p.num_parts + part;
      *reinterpret_cast<float4*>(p.ws_o + r * D + e) =
          make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
      if (e == 0) {
        p.ws_m[r] = M;
        p.ws_l[r] = Lsum;
      }
    }
  }
}

// Merge the partitions of sequences whose context spans more than one:
// out = sum_p w_p o_p / sum_p w_p with w_p = l_p * 2^(m_p - max m).
// One warp per (sequence, query head).
template <typename T, int D>
__global__ void __launch_bounds__(128) paged_decode_reduce_kernel(const DecodeParams p) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 4 + warp;
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (pair >= p.num_seqs * p.num_q_heads) return;
  const int s = pair / p.num_q_heads;
  int ctx = p.context_lens[s];
  const long long cap_ll = min((long long)p.max_context_len,
                               (long long)p.max_blocks_per_seq * p.block_size);
  ctx = ctx < 0 ? 0 : (ctx > cap_ll ? (int)cap_ll : ctx);
  const int np = (ctx + p.partition_size - 1) / p.partition_size;
  if (np <= 1) return;  // written directly by the decode kernel
  const float* mrow = p.ws_m + (size_t)pair * p.num_parts;
  const float* lrow = p.ws_l + (size_t)pair * p.num_parts;
  const float* orow = p.ws_o + (size_t)pair * p.num_parts * D + lane * EPL;
  T* out = static_cast<T*>(p.out) + (size_t)pair * D + lane * EPL;
  if (np <= 32) {
    // Up to 32 partitions (every automatic choice up to 32k tokens): lane i
    // holds partition i's (m, l), and every load of the warp (the maxima,
    // the sums and the first partials) is issued before any is used, so the
    // merge costs one memory round trip.  Same arithmetic, in the same
    // order, as the general loop below.
    constexpr int kPre = 4;
    float pre[kPre][EPL];
#pragma unroll
    for (int i = 0; i < kPre; ++i)
      if (i < np) {
        if constexpr (EPL == 4) {
          const float4 a = *reinterpret_cast<const float4*>(orow + (size_t)i * D);
          pre[i][0] = a.x;
          pre[i][1] = a.y;
          pre[i][2] = a.z;
          pre[i][3] = a.w;
        } else {
          const float2 a = *reinterpret_cast<const float2*>(orow + (size_t)i * D);
          pre[i][0] = a.x;
          pre[i][1] = a.y;
        }
      }
    const float mi = lane < np ? mrow[lane] : -CUDART_INF_F;
    const float li = lane < np ? lrow[lane] : 0.f;
    float M = mi;
#pragma unroll
    for (int mk = 16; mk >= 1; mk >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, mk));
    const float wi = lane < np ? li * exp2f(mi - M) : 0.f;
    float Lsum = 0.f + wi;
#pragma unroll
    for (int mk = 16; mk >= 1; mk >>= 1) Lsum += __shfl_xor_sync(kFull, Lsum, mk);
    const float inv = 1.f / Lsum;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < kPre; ++i)
      if (i < np) {
        const float w = __shfl_sync(kFull, wi, i) * inv;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] += w * pre[i][e];
      }
#pragma unroll 4
    for (int i = kPre; i < np; ++i) {
      const float w = __shfl_sync(kFull, wi, i) * inv;
      if constexpr (EPL == 4) {
        const float4 a = *reinterpret_cast<const float4*>(orow + (size_t)i * D);
        acc[0] += w * a.x;
        acc[1] += w * a.y;
        acc[2] += w * a.z;
        acc[3] += w * a.w;
      } else {
        const float2 a = *reinterpret_cast<const float2*>(orow + (size_t)i * D);
        acc[0] += w * a.x;
        acc[1] += w * a.y;
      }
    }
    if constexpr (EPL == 4) {
      uint2 pk;
      pk.x = Cvt<T>::from_float2(acc[0], acc[1]);
      pk.y = Cvt<T>::from_float2(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(out) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(out) = Cvt<T>::from_float2(acc[0], acc[1]);
    }
    return;
  }
  float M = -CUDART_INF_F;
  for (int i = lane; i < np; i += 32) M = fmaxf(M, mrow[i]);
#pragma unroll
  for (int mk = 16; mk >= 1; mk >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, mk));
  float Lsum = 0.f;
  for (int i = lane; i < np; i += 32) Lsum += lrow[i] * exp2f(mrow[i] - M);
#pragma unroll
  for (int mk = 16; mk >= 1; mk >>= 1) Lsum += __shfl_xor_sync(kFull, Lsum, mk);
  const float inv = 1.f / Lsum;
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int i = 0; i < np; ++i) {
    const float w = lrow[i] * exp2f(mrow[i] - M) * inv;
    if constexpr (EPL == 4) {
      const float4 a = *reinterpret_cast<const float4*>(orow + (size_t)i * D);
      acc[0] += w * a.x;
      acc[1] += w * a.y;
      acc[2] += w * a.z;
      acc[3] += w * a.w;
    } else {
      const float2 a = *reinterpret_cast<const float2*>(orow + (size_t)i * D);
      acc[0] += w * a.x;
      acc[1] += w * a.y;
    }
  }
  if constexpr (EPL == 4) {
    uint2 pk;
    pk.x = Cvt<T>::from_float2(acc[0], acc[1]);
    pk.y = Cvt<T>::from_float2(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(out) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(out) = Cvt<T>::from_float2(acc[0], acc[1]);
  }
}

// Opt the kernel in to more than 48 KiB of dynamic shared memory, once per
// device.
template <typename T, int D, int GT, bool kPaged>
cudaError_t configure() {
  using L = SmemLayout<T, D, GT>;
  static unsigned long long configured = 0;  // bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    err = cudaFuncSetAttribute(paged_decode_kernel<T, D, GT, kPaged>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  return cudaSuccess;
}

template <typename T, int D, int GT>
int ctas_per_sm_typed() {
  using L = SmemLayout<T, D, GT>;
  int n = 0;
  if (configure<T, D, GT, true>() != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_kernel<T, D, GT, true>,
                                                    L::kThreads, L::kBytes) != cudaSuccess)
    return 0;
  return n;
}

template <typename T, int D, int GT, bool kPaged>
cudaError_t launch_typed(const DecodeParams& p, cudaStream_t stream) {
  using L = SmemLayout<T, D, GT>;
  cudaError_t err = configure<T, D, GT, kPaged>();
  if (err != cudaSuccess) return err;
  const dim3 grid(p.num_parts, p.num_kv_heads * p.head_chunks, p.num_seqs);
  err = launch_overlapped(paged_decode_kernel<T, D, GT, kPaged>, grid, dim3(L::kThreads),
                          L::kBytes, stream, p);
  if (err != cudaSuccess || p.num_parts <= 1) return err;
  const int pairs = p.num_seqs * p.num_q_heads;
  return launch_overlapped(paged_decode_reduce_kernel<T, D>, dim3((pairs + 3) / 4), dim3(128),
                           0, stream, p);
}

template <typename T, int D, bool kPaged>
cudaError_t launch_for_group(const DecodeParams& p, int gt, cudaStream_t stream) {
  switch (gt) {
    case 1: return launch_typed<T, D, 1, kPaged>(p, stream);
    case 2: return launch_typed<T, D, 2, kPaged>(p, stream);
    default: return launch_typed<T, D, 4, kPaged>(p, stream);
  }
}

template <bool kPaged>
cudaError_t launch_any(const DecodeParams& p, int dtype, int head_dim, int gt,
                       cudaStream_t stream) {
  if (dtype == PKV_F16) {
    return head_dim == 64 ? launch_for_group<__half, 64, kPaged>(p, gt, stream)
                          : launch_for_group<__half, 128, kPaged>(p, gt, stream);
  }
  return head_dim == 64 ? launch_for_group<__nv_bfloat16, 64, kPaged>(p, gt, stream)
                        : launch_for_group<__nv_bfloat16, 128, kPaged>(p, gt, stream);
}

}  // namespace

int decode_ctas_per_sm(int head_dim, int gt) {
  // Occupancy depends on sizes only; both element types have the same.
  if (head_dim == 64) {
    return gt == 1 ? ctas_per_sm_typed<__half, 64, 1>()
                   : (gt == 2 ? ctas_per_sm_typed<__half, 64, 2>() : ctas_per_sm_typed<__half, 64, 4>());
  }
  return gt == 1 ? ctas_per_sm_typed<__half, 128, 1>()
                 : (gt == 2 ? ctas_per_sm_typed<__half, 128, 2>() : ctas_per_sm_typed<__half, 128, 4>());
}

int decode_heads_per_cta(int group) { return group == 1 ? 1 : (group == 2 ? 2 : 4); }

size_t decode_smem_bytes(int head_dim, int gt) {
  // The layout does not depend on the element type beyond its size (2 bytes).
  if (head_dim == 64) {
    return gt == 1 ? SmemLayout<__half, 64, 1>::kBytes
                   : (gt == 2 ? SmemLayout<__half, 64, 2>::kBytes : SmemLayout<__half, 64, 4>::kBytes);
  }
  return gt == 1 ? SmemLayout<__half, 128, 1>::kBytes
                 : (gt == 2 ? SmemLayout<__half, 128, 2>::kBytes : SmemLayout<__half, 128, 4>::kBytes);
}

cudaError_t launch_decode_reduce(const DecodeParams& p, int dtype, int head_dim,
                                 cudaStream_t stream) {
  const dim3 grid((p.num_seqs * p.num_q_heads + 3) / 4);
  if (dtype == PKV_F16) {
    return head_dim == 64
               ? launch_overlapped(paged_decode_reduce_kernel<__half, 64>, grid, dim3(128), 0,
                                   stream, p)
               : launch_overlapped(paged_decode_reduce_kernel<__half, 128>, grid, dim3(128), 0,
                                   stream, p);
  }
  return head_dim == 64
             ? launch_overlapped(paged_decode_reduce_kernel<__nv_bfloat16, 64>, grid, dim3(128), 0,
                                 stream, p)
             : launch_overlapped(paged_decode_reduce_kernel<__nv_bfloat16, 128>, grid, dim3(128),
                                 0, stream, p);
}

cudaError_t launch_paged_decode(const DecodeParams& p, int dtype, int head_dim, int gt,
                                cudaStream_t stream) {
  return launch_any<true>(p, dtype, head_dim, gt, stream);
}

cudaError_t launch_contiguous_decode(const DecodeParams& p, int dtype, int head_dim, int gt,
                                     cudaStream_t stream) {
  return launch_any<false>(p, dtype, head_dim, gt, stream);
}

}  // namespace pkv
