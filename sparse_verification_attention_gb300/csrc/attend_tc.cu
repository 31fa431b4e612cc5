// Split-KV sparse verification attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators), bf16, head dim 128, blocks of 64 tokens.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: every draft token
// attends to the same selected set of KV blocks, so the R = T*G query rows of
// one KV head are stacked into one MMA tile and each selected page is read
// from HBM once for all of them.
//
// Work split (one CTA per SM: the ring and all 512 TMEM columns are sized
// for a whole SM): the work units of a (b, h) pair are its selected blocks, a
// partial last block if any, and one draft tile. Three plans (chosen on the
// host): stream-K cuts the flattened (pair, unit) sequence into one equal run
// per CTA, so a CTA covers the tail of one pair and the head of the next at
// most (two segments: the first segment's Q in shared memory, the second's
// in TMEM); a cluster plan puts one thread-block cluster of 4..16 CTAs on
// each pair and splits its units evenly; otherwise a split map gives each
// pair whole splits.
//
// CTA roles (a 6-stage ring keeps ~192 KB of K/V in flight per SM):
//   * producer warp: loads the first segment's Q by 3-D TMA, takes each
//     selected block's pool row (written beside the selection by the top-k,
//     or looked up through the block table when the caller passes its own
//     selection; 32 at a time, one lane each) and issues 2-D TMA copies
//     (128-byte swizzle, L2 evict-first) of the page's K and V tiles into the
//     ring; the draft tile (the pair's draft K/V rows) comes the same way,
//     through a 4-D map over the draft tensors.
//   * MMA issue, split by role over two warps (one elected lane each): one
//     issues every S_i = Q K_i^T into TMEM (M=128 rows, N=64 tokens, K=128),
//     the other, after softmax, every O += P_i V_i with P read from TMEM
//     (M=128, N=128, K=64, V as an MN-major operand); the first P.V of each
//     softmax set in a segment starts a fresh accumulator; stages are
//     released by tcgen05 commits. The issuers poll their barriers with
//     test_wait (never suspended), so each issues as soon as a hand-off
//     lands.
//   * two softmax sets: set A takes the even tiles, set B the odd ones, each
//     with its own S, P and O in TMEM, so two independent softmax chains
//     overlap. In each set the warp owning TMEM lane quarter q holds stacked
//     rows 32q..32q+31, one row per thread (quarters past ceil(R/32) hold
//     only zero padding rows and stay idle). Each set keeps its own running
//     max (log2 domain; the accumulator is rescaled only when some row's max
//     grows by more than 2^8, decided per warp so that the warp-collective
//     TMEM loads/stores are taken by all lanes) and sum.
//   * partials and merge: a segment that ends mid-stream writes each set's
//     unnormalised (o, m, l) rows from registers; the final segment folds
//     the two sets straight out of TMEM (only (m, l) goes through shared
//     memory; each warp folds half the columns of its lane quarter's rows,
//     reading both sets' O). Cluster plans then merge the pair's
//     folded rows through distributed shared memory. Otherwise partials are
//     published in the workspace with an acquire-release arrival. When a
//     pair's merge is small, every segment takes a ticket as its stream ends
//     and the segment holding the last ticket merges alone: it keeps its own
//     folded rows in shared memory and waits only for the publications of
//     segments that took their tickets before it (so are past their streams
//     and wait on nothing). Larger merges go to the pair's last CTA to
//     arrive, which shares row slices with the pair's CTAs still waiting.
// Rows past R are padding: zero query rows whose outputs are never read.
#include <atomic>

#include "internal.h"
#include "ptx.h"
#include "tc.h"

namespace sva {
namespace {

constexpr int TD = 128;                       // head dim
constexpr int TBLK = 64;                      // tokens per block
constexpr int kBoxBytes = TBLK * 128;         // one 64-column box of a tile
constexpr int kTileBytes = 2 * kBoxBytes;     // K (or V) tile, 16 KB
constexpr int kStageBytes = 2 * kTileBytes;   // K + V, 32 KB
constexpr uint32_t kTmemCols = 512;
// threads per CTA: 8 softmax warps (two sets of four), the producer warp and
// two MMA-issuing warps (one issues every S, the other every P.V)
constexpr int kCtaThreads = 32 * 11;
// TMEM columns of set X in {0, 1}: S (64 fp32), O (128 fp32), P (32 x bf16x2)
__host__ __device__ constexpr uint32_t col_s(int x) { return x ? 64u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return x ? 256u : 128u; }
__host__ __device__ constexpr uint32_t col_p(int x) { return x ? 416u : 384u; }
// TMEM columns 448..511: the second segment's Q (128 rows x 128 bf16, two per
// column), the A operand of that segment's S = Q K^T
constexpr uint32_t kColQ1 = 448;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxSeg = 2;          // pair segments per CTA
#ifndef SVA_SPEC_UNITS
#define SVA_SPEC_UNITS 4
#endif
constexpr int kSpecUnits = SVA_SPEC_UNITS;  // units prefetched speculatively before the wait

constexpr int r1024(int x) { return (x + 1023) / 1024 * 1024; }

template <int NSW, int NS>
struct TcCfg {
  static constexpr int kThreads = kCtaThreads;
  static constexpr int kRows = 32 * NSW;          // stacked rows held in TMEM lanes (>= R)
  static constexpr int kQBox = 128 * 128;         // one 64-column Q box, 128 rows
  static constexpr int kQBytes = 2 * kQBox;       // the first segment's Q operand
  static constexpr int kRingOff = kQBytes;
  static constexpr int kOst = TD + 4;
  // epilogue area of the final segment: its folded o [kRows][kOst] (room is
  // kept for 2 kRows rows), both sets' (m, l) [2 kRows], the fold weights
  // [kRows] and the folded (M, L) [kRows]
  static constexpr int kMergeBytes = (2 * kRows * kOst + 4 * kRows * 2) * 4;
  static constexpr int kRingRaw = NS * kStageBytes;
  static constexpr int kRing = r1024(kMergeBytes > kRingRaw ? kMergeBytes : kRingRaw);
  static constexpr int kCtrlOff = kRingOff + kRing;
  static constexpr int kSmem = kCtrlOff + 256 + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  // a merge pass of two rows of the most slots a pair can have fits the ring
  static_assert(2 * kMaxSplits * (TD * 4 + 8) <= kRing, "merge staging");
};

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t swz128(int row, int chunk16) {
  return row * 128 + ((chunk16 ^ (row & 7)) << 4);
}

constexpr int kMergeRowBytes = TD * 4 + 8;  // a partial row's o and (m, l)
constexpr int kMaxCluster = 16;  // CTAs per pair in the cluster merge
constexpr int kMinCluster = 4;   // smallest cluster the plan uses
constexpr size_t kSoloMergeBytes = 128 * 1024;  // see launch_attend_tc
constexpr int kTicketWord = 1;  // word of a pair's attention count line holding merge tickets

// Log-sum-exp combine of rows [r0, r0 + nv) of one pair from partials staged
// in shared memory: o at so[(s * ld + r) * TD], (m, l) at sml[s * ld + r] for
// slots s < ns (r relative to r0). Eight threads per row, each with four
// float4 columns, so every load of a slot is independent of the others;
// the weights are formed in place (slot order, so the sums do not depend on
// which CTA merges). All threads of the CTA call it.
template <int NT>
__device__ __forceinline__ void combine_rows(const AttendArgs& a, int b, int h, int ns, int ld,
                                             int r0, int nv, const float* so, const float2* sml) {
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const int cg = threadIdx.x & 7;
  for (int r = threadIdx.x >> 3; r < nv; r += NT / 8) {
    float M = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (s0 + q < ns) M = fmaxf(M, sml[(s0 + q) * ld + r].x);
    }
    float L = 0.f;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (s0 + q < ns) {
          const float2 ml = sml[(s0 + q) * ld + r];
          const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
          L += w * ml.y;
          const float* orow = so + ((size_t)(s0 + q) * ld + r) * TD;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 o = *reinterpret_cast<const float4*>(orow + (cg + 8 * i) * 4);
            acc[i].x += w * o.x;
            acc[i].y += w * o.y;
            acc[i].z += w * o.z;
            acc[i].w += w * o.w;
          }
        }
      }
    }
    const float inv = 1.0f / L;
    const int rr = r0 + r, t = rr / a.G, gq = rr % a.G;
    __nv_bfloat16* dst = out + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * TD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst + (cg + 8 * i) * 4) = u;
    }
  }
}

// Bounded wait (thread scope, acquire at device scope) until the low 16 bits
// of *w reach `need`: false after kWaitBudgetNs, with `site` recorded in
// status[1].
__device__ __forceinline__ bool wait_count_at_least(const unsigned* w, unsigned need,
                                                    unsigned* status, unsigned site) {
  if ((load_acquire(w) & 0xFFFFu) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while ((load_acquire(w) & 0xFFFFu) < need) {
    if (globaltimer_ns() - t0 > kWaitBudgetNs) {
      atomicMax(status + 1, site);
      return false;
    }
  }
  return true;
}

// The work of one CTA: up to kMaxSeg segments, each a run of consecutive work
// units [u0, u1) of one (b, h) pair (units 0..n_sel-1 are the selected
// blocks, then the partial last block if the context has one, then the draft
// tile).
struct SegPlan {
  int n;
  int pair[kMaxSeg], u0[kMaxSeg], u1[kMaxSeg];
  int slot[kMaxSeg];  // this CTA's partial slot among the pair's segments
  int nseg[kMaxSeg];  // segments of the pair (over all CTAs)
  int mid[kMaxSeg];   // the pair's last segment ends mid-stream in its CTA
};

// Partial results of a pair: final segments (the CTA's last) fold both
// softmax sets and use their slot; a segment that ends mid-stream writes its
// two sets separately, set B in the extra slot nseg. Every segment counts one
// arrival at the end of its CTA.
__device__ SegPlan plan_segments(const AttendArgs& a) {
  SegPlan sp{};
  const int W = a.n_sel + (a.tail > 0 ? 1 : 0) + 1;
  const int c = blockIdx.x;
  if (a.streamk) {
    // stream-K: the flattened (pair, unit) sequence cut into gridDim.x equal
    // runs; the host guarantees every run is non-empty and no longer than a
    // pair, so a run spans at most two pairs
    const long long G = gridDim.x, U = (long long)a.B * a.Hkv * W;
    const long long f0 = (long long)c * U / G, f1 = (long long)(c + 1) * U / G;
    auto cta_of = [&](long long f) { return (int)(((f + 1) * G - 1) / U); };
    long long f = f0;
    while (f < f1 && sp.n < kMaxSeg) {
      const int p = (int)(f / W);
      const long long pbeg = (long long)p * W, pend = pbeg + W;
      const long long e = f1 < pend ? f1 : pend;
      const int first = cta_of(pbeg), last = cta_of(pend - 1);
      sp.pair[sp.n] = p;
      sp.u0[sp.n] = (int)(f - pbeg);
      sp.u1[sp.n] = (int)(e - pbeg);
      sp.slot[sp.n] = c - first;
      sp.nseg[sp.n] = last - first + 1;
      // the pair's last CTA carries on into the next pair
      sp.mid[sp.n] = ((long long)(last + 1) * U / G > pend) ? 1 : 0;
      ++sp.n;
      f = e;
    }
  } else {
    int pair, split, nsp;
    split_of_cta(c, a.n_splits, a.split_extra, &pair, &split, &nsp);
    // this pair's units (sequences may differ in selected blocks and tail)
    const int bq = pair / a.Hkv;
    const int Wp = n_of(a.vl, bq, a.n_sel) + (tail_of(a.vl, bq, a.tail) > 0 ? 1 : 0) + 1;
    const int bps = (Wp + nsp - 1) / nsp;
    sp.n = 1;
    sp.pair[0] = pair;
    sp.u0[0] = min(Wp, split * bps);
    sp.u1[0] = min(Wp, sp.u0[0] + bps);
    sp.slot[0] = split;
    sp.nseg[0] = nsp;
    sp.mid[0] = 0;
  }
  return sp;
}

template <int NSW, int NS>
__global__ void __launch_bounds__(kCtaThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDK,
                     const __grid_constant__ CUtensorMap tmDV, const __grid_constant__ AttendArgs a) {
  using C = TcCfg<NSW, NS>;
  constexpr int PRODUCER = 8, MMAW = 9, MMAW2 = 10;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qs = smem;  // [kMaxSeg][2 boxes]
  uint8_t* ring = smem + C::kRingOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kCtrlOff);
  uint64_t* empty = full + NS;
  uint64_t* s_full = empty + NS;   // [2] per set
  uint64_t* p_ready = s_full + 2;  // [2] per set, NSW warps each
  uint64_t* o_done = p_ready + 2;  // [2] per set
  uint64_t* mma_done = o_done + 2; // drain: every issued MMA has completed
  uint64_t* q_ready = mma_done + 1; // Q landed (TMA) and padding rows zeroed
  uint64_t* q1_ready = q_ready + 1; // second segment's Q written into TMEM
  uint64_t* mid_done = q1_ready + 1; // the mid-stream segment's partials are written
  uint64_t* merge_bar = mid_done + 1; // a merge's partials have landed (bulk copies)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(merge_bar + 1);
  int* stage_info = reinterpret_cast<int*>(tmem_slot + 1);  // bit0 valid, bit1 draft tile
  volatile int* abort_flag = stage_info + NS;
  volatile int* pair_done = abort_flag + 1;  // [kMaxSeg]: this CTA saw the pair complete
  volatile int* merge_got = pair_done + kMaxSeg;  // merge slices this CTA claimed
  // ancestor masks of the drafts, copied out of the parameter space with
  // warp-uniform indices (per-lane indices into it would serialize)
  __shared__ unsigned long long s_anc[kMaxT];

  // the CTA's segments, in shared memory: read again after the stream, where
  // a per-thread copy would come back from local memory through L2
  __shared__ SegPlan s_plan;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s_plan = plan_segments(a);
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&p_ready[i]), NSW);
      mbar_init(smem_u32(&o_done[i]), 1);
    }
    mbar_init(smem_u32(mma_done), 2);  // one arrival per MMA issuer
    mbar_init(smem_u32(q_ready), 5);  // producer's expect_tx + 4 zeroing warps
    mbar_init(smem_u32(q1_ready), 4);
    mbar_init(smem_u32(mid_done), 2 * NSW);
    mbar_init(smem_u32(merge_bar), 1);
    *abort_flag = 0;
    for (int j = 0; j < kMaxSeg; ++j) pair_done[j] = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmDK);
    prefetch_tensormap(&tmDV);
  }
  if (warp == MMAW) {
    tc::alloc(smem_u32(tmem_slot), kTmemCols);
    tc::relinquish();
  }
  if (warp == PRODUCER)
    for (int u = 0; u < a.T; ++u)
      if (lane == 0) s_anc[u] = a.anc[u];
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const SegPlan& sp = s_plan;
  const int n0 = sp.n > 0 ? sp.u1[0] - sp.u0[0] : 0;
  const int ntot = n0 + (sp.n > 1 ? sp.u1[1] - sp.u0[1] : 0);
  auto seg_of = [&](int i) { return i < n0 ? 0 : 1; };
  const uint32_t tmem = *tmem_slot;
  if (warp == PRODUCER) {
    // warm L2 with this CTA's block-table rows while earlier kernels finish
    // (a prefetch only: the lookups below still read after the wait)
    for (int j = 0; j < sp.n; ++j) {
      const int32_t* row = a.block_table + (size_t)(sp.pair[j] / a.Hkv) * a.nb_max;
      for (int e = 32 * lane; e < a.nb; e += 32 * 32) prefetch_l2(row + e);
    }
    if (a.spec_prefetch && lane < kSpecUnits && lane < ntot) {
      // Speculative: the pages of this CTA's first units, looked up with
      // relaxed reads that may see an earlier selection if the preceding
      // kernel rewrites it. Only L2 is touched, so a wrong guess costs
      // bandwidth and nothing else; the copies below re-read after the wait.
      const int j = lane < n0 ? 0 : 1;
      const int u = sp.u0[j] + lane - (j ? n0 : 0);
      const int pair = sp.pair[j], b = pair / a.Hkv, h = pair % a.Hkv;
      const int nsel = n_of(a.vl, b, a.n_sel), nbb = nb_of(a.vl, b, a.nb);
      int page = -1;
      if (u < nsel) {
        const int jb = a.sel ? load_relaxed(a.sel + (size_t)pair * a.sel_stride + u) : u;
        if (jb >= 0 && jb < nbb) page = load_relaxed(a.block_table + (size_t)b * a.nb_max + jb);
      } else if (u == nsel && tail_of(a.vl, b, a.tail) > 0) {
        page = load_relaxed(a.block_table + (size_t)b * a.nb_max + nbb);
      }
      if (page >= 0 && page < a.num_pages) {
        const size_t off = (size_t)((page * a.Hkv + h) * TBLK) * TD * 2;
        prefetch_bulk_l2(static_cast<const uint8_t*>(a.k_pool) + off, kTileBytes);
        prefetch_bulk_l2(static_cast<const uint8_t*>(a.v_pool) + off, kTileBytes);
      }
    }
  }
  if (warp == MMAW) {
    // touch every line of the parameter block while the previous kernel
    // drains, so that no role pays a cold parameter read after the wait
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(&a);
    uint32_t acc = 0;
    for (int w = lane * 16; w < (int)(sizeof(AttendArgs) / 4); w += 32 * 16) acc ^= pw[w];
    asm volatile("" ::"r"(acc));  // keeps the reads
  }
  pdl_wait();     // everything below may read what earlier kernels wrote
  pdl_trigger();  // let the next kernel launch and run its prologue

  // Q operand, 128 rows: rows r < R = the stacked query rows (draft t, head
  // g) = Q[b, t, h*G + g] in order r = t*G + g. The first segment's Q comes by
  // one 3-D TMA box per 64 dims (issued first by the producer) with rows
  // R..127 zeroed here; the second segment's Q is written by these four warps
  // into TMEM (lane = row), where the MMA reads it as a tensor-memory A operand.
  // zero the Q operand's padding rows R..127 and count this warp on q_ready
  auto zero_q_padding = [&]() {
    const int r = threadIdx.x;
    if (r >= a.R) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(qs + (c >> 3) * C::kQBox + swz128(r, c & 7)) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(q_ready));
  };
  if (warp < 4) {
    zero_q_padding();
    const int r = threadIdx.x;
    if (sp.n > 1) {
      const int b1 = sp.pair[1] / a.Hkv, h1 = sp.pair[1] % a.Hkv;
      const uint4* q1 = static_cast<const uint4*>(a.q) +
                        (((size_t)b1 * a.T + r / a.G) * a.Hq + h1 * a.G + r % a.G) * (TD / 8);
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u = (r < a.R) ? q1[half * 8 + c] : make_uint4(0, 0, 0, 0);
          qv[4 * c] = u.x;
          qv[4 * c + 1] = u.y;
          qv[4 * c + 2] = u.z;
          qv[4 * c + 3] = u.w;
        }
        tc::st32(tmem + lane_base + kColQ1 + 32 * half, qv);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(q1_ready));
    }
  }

  // per-thread softmax state (m, l of the final segment for the epilogue),
  // and a mid-stream segment's O row on its way to the workspace
  float o_row[TD];
  float m_run = -INFINITY, l_run = 0.f;
  // Narrow merges (the last CTA of a pair merges every row) go by tickets: a
  // segment takes its pair's ticket when its stream ends, and the segment
  // holding the last ticket merges; the others publish their partials.
  const bool ticketed = a.merge_wait_ns == 0 && !a.cluster_merge;
  unsigned final_ticket = 0u;  // thread 0: the final segment's ticket

  if (warp == PRODUCER) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && sp.n > 0) {
      // the first segment's query rows first, ahead of the K/V stream
      const uint32_t qb = smem_u32(q_ready);
      mbar_arrive_expect_tx(qb, (uint32_t)(a.R * TD * 2));
      const int b = sp.pair[0] / a.Hkv, h = sp.pair[0] % a.Hkv;
      tma_load_3d(smem_u32(qs), &tmQ, 0, h * a.G, b * a.T, qb);
      tma_load_3d(smem_u32(qs) + C::kQBox, &tmQ, 64, h * a.G, b * a.T, qb);
    }
    const int oob_row = a.num_pages * a.Hkv * TBLK;  // past the end: TMA zero-fills
    // pages are read once per call: first out of L2 (see l2_evict_first_policy)
    const uint64_t kv_policy = l2_evict_first_policy();
    int issued = 0;
    bool stop = false;
    int i = 0;  // ring index (a stage is i % NS, its phase parity (i / NS) & 1)
    for (int j = 0; j < sp.n && !stop; ++j) {
      const int pair = sp.pair[j], b = pair / a.Hkv, h = pair % a.Hkv;
      const int nsel = n_of(a.vl, b, a.n_sel), nbb = nb_of(a.vl, b, a.nb);
      const int tail = tail_of(a.vl, b, a.tail);
      const int ub = sp.u0[j];
      const int nblk = max(0, min(sp.u1[j], nsel) - ub);
      for (int base = 0; base < nblk && !stop; base += 32) {
        int row = oob_row, ok = 0;
        if (base + lane < nblk && a.rows) {
          // resolved by the select step (which flagged any bad page as -1)
          const int rr = __ldcg(a.rows + (size_t)pair * a.sel_stride + ub + base + lane);
          if (rr >= 0 && rr < oob_row) {
            row = rr;
            ok = 1;
          }
        } else if (base + lane < nblk) {
          const int jb = a.sel ? a.sel[(size_t)pair * a.sel_stride + ub + base + lane] : ub + base + lane;
          if (jb < 0 || jb >= nbb) {
            atomicOr(a.status, SV_FLAG_BAD_BLOCK_INDEX);
          } else {
            const int page = a.block_table[(size_t)b * a.nb_max + jb];
            if (page < 0 || page >= a.num_pages) {
              atomicOr(a.status, SV_FLAG_BAD_PAGE);
            } else {
              row = (page * a.Hkv + h) * TBLK;
              ok = 1;
            }
          }
        }
        const int cnt = min(32, nblk - base);
        for (int qq = 0; qq < cnt; ++qq, ++i) {
          const int rq = __shfl_sync(0xffffffffu, row, qq);
          const int okq = __shfl_sync(0xffffffffu, ok, qq);
          int fail = 0;
          if (lane == 0) {
            const int s = i % NS;
            if (i >= NS &&
                !mbar_wait_abortable(smem_u32(&empty[s]), ((i / NS) & 1) ^ 1, abort_flag, a.status, 1u)) {
              fail = 1;
            } else {
              stage_info[s] = okq;
              const uint32_t fb = smem_u32(&full[s]);
              mbar_arrive_expect_tx(fb, kStageBytes);
              const uint32_t kdst = smem_u32(ring + s * kStageBytes);
              const uint32_t vdst = kdst + kTileBytes;
              tma_load_2d_hint(kdst, &tmK, 0, rq, fb, kv_policy);
              tma_load_2d_hint(kdst + kBoxBytes, &tmK, 64, rq, fb, kv_policy);
              tma_load_2d_hint(vdst, &tmV, 0, rq, fb, kv_policy);
              tma_load_2d_hint(vdst + kBoxBytes, &tmV, 64, rq, fb, kv_policy);
              issued = i + 1;
            }
          }
          if (__shfl_sync(0xffffffffu, fail, 0)) {
            stop = true;
            break;
          }
        }
      }
      if (tail > 0 && sp.u0[j] <= nsel && nsel < sp.u1[j] && !stop) {
        // the partial last block: a full page copy, of which the softmax keeps
        // the first `tail` columns (stage_info bits 8..15)
        int rq = oob_row, okq = 0;
        if (lane == 0) {
          const int page = a.block_table[(size_t)b * a.nb_max + nbb];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, SV_FLAG_BAD_PAGE);
          } else {
            rq = (page * a.Hkv + h) * TBLK;
            okq = 1 | (tail << 8);
          }
        }
        int fail = 0;
        if (lane == 0) {
          const int s = i % NS;
          if (i >= NS &&
              !mbar_wait_abortable(smem_u32(&empty[s]), ((i / NS) & 1) ^ 1, abort_flag, a.status, 13u)) {
            fail = 1;
          } else {
            stage_info[s] = okq;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, kStageBytes);
            const uint32_t kdst = smem_u32(ring + s * kStageBytes);
            const uint32_t vdst = kdst + kTileBytes;
            tma_load_2d_hint(kdst, &tmK, 0, rq, fb, kv_policy);
            tma_load_2d_hint(kdst + kBoxBytes, &tmK, 64, rq, fb, kv_policy);
            tma_load_2d_hint(vdst, &tmV, 0, rq, fb, kv_policy);
            tma_load_2d_hint(vdst + kBoxBytes, &tmV, 64, rq, fb, kv_policy);
            issued = i + 1;
          }
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) stop = true;
        ++i;
      }
      const int ud = nsel + (tail > 0 ? 1 : 0);  // the draft tile's unit
      if (sp.u0[j] <= ud && ud < sp.u1[j] && !stop) {
        // draft tile: this pair's draft rows t < T by TMA like any page; rows
        // T..63 lie outside the draft tensor and arrive as zeros (the softmax
        // masks them as well)
        int fail = 0;
        if (lane == 0) {
          const int s = i % NS;
          if (i >= NS &&
              !mbar_wait_abortable(smem_u32(&empty[s]), ((i / NS) & 1) ^ 1, abort_flag, a.status, 2u)) {
            fail = 1;
          } else {
            stage_info[s] = 3;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, kStageBytes);
            const uint32_t kdst = smem_u32(ring + s * kStageBytes);
            const uint32_t vdst = kdst + kTileBytes;
            tma_load_4d(kdst, &tmDK, 0, h, 0, b, fb);
            tma_load_4d(kdst + kBoxBytes, &tmDK, 64, h, 0, b, fb);
            tma_load_4d(vdst, &tmDV, 0, h, 0, b, fb);
            tma_load_4d(vdst + kBoxBytes, &tmDV, 64, h, 0, b, fb);
            issued = i + 1;
          }
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) stop = true;
        ++i;
      }
    }
    // never leave with a bulk copy still writing into the ring
    if (lane == 0)
      for (int t = max(0, issued - NS); t < issued; ++t)
        mbar_wait_drain(smem_u32(&full[t % NS]), (t / NS) & 1);
    // The mid-stream segment's arrival, counted here while the CTA finishes
    // its last tiles: the softmax warps' mbarrier arrivals order their
    // partial stores before this thread's device-scope release.
    if (lane == 0 && sp.n > 1) {
      if (!mbar_wait_abortable(smem_u32(mid_done), 0, abort_flag, a.status, 12u))
        atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
      // the last arrival sees the pair complete (and acquires its partials);
      // with tickets, the last ticket merges (after every publication)
      unsigned* w = a.counters + sp.pair[0] * kPairWords;
      if (ticketed) {
        arrive_release(w);
        const unsigned t = atomicAdd(w + kTicketWord, 1u);
        if (t + 1u == (unsigned)sp.nseg[0]) pair_done[0] = 1;
        else if (t >= (unsigned)sp.nseg[0]) atomicOr(a.status, SV_FLAG_STALE_WORKSPACE);
      } else if ((arrive_acq_rel(w) & 0xFFFFu) + 1u == (unsigned)sp.nseg[0]) {
        pair_done[0] = 1;
      }
    }
  } else if (warp == MMAW || warp == MMAW2) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads, split by role: warp MMAW issues every S, warp
    // MMAW2 every P.V, each in tile order. A tcgen05.mma takes its issuing
    // thread tens of cycles (about 40 ns at these shapes), and a
    // tcgen05.commit tracks every earlier MMA of its thread: with one thread
    // issuing both, a set's next S waited for its P.V to be issued and then
    // to complete. Split by role, S(i) goes out as soon as tile i has landed
    // and the softmax of tile i-2 (same set) has read its S buffer, and its
    // commit waits for S MMAs only. (One issuer per softmax set instead was
    // measured 3-7% slower than one thread for both at 32 rows.)
    if (lane == 0 && ntot > 0) {
      constexpr uint32_t idq = tc::idesc_bf16(128, 64, false, false);
      constexpr uint32_t idp = tc::idesc_bf16(128, TD, false, true);
      const uint32_t rb = smem_u32(ring);
      const uint32_t qb = smem_u32(qs);
      bool q1_seen = false;
      // tile i (its set is i & 1) lives in ring stage rs(i) with phase rp(i)
      auto rs = [&](int t) { return t % NS; };
      auto rp = [&](int t) { return (uint32_t)((t / NS) & 1); };
      // Descriptors built once: a descriptor's address field is the byte
      // address >> 4, so a stage or k-step offset (a multiple of 16 bytes,
      // inside shared memory) is added to it directly.
      const uint64_t dq0 = tc::smem_desc(qb, 16, 1024);                      // Q (segment 0)
      const uint64_t dk0 = tc::smem_desc(rb, 16, 1024);                      // K of stage 0
      const uint64_t dv0 = tc::smem_desc(rb + kTileBytes, kBoxBytes, 1024);  // V of stage 0
      auto stage_off = [&](int t) { return (uint64_t)(rs(t) * (kStageBytes >> 4)); };
      auto issue_qk = [&](int i) {
        const uint64_t dk = dk0 + stage_off(i);
        const uint32_t d = tmem + col_s(i & 1);
        if (seg_of(i) == 0) {
#pragma unroll
          for (int kk = 0; kk < TD / 16; ++kk) {
            const uint64_t ad = dq0 + (uint64_t)(((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4);
            const uint64_t bd = dk + (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
            tc::mma_ss(d, ad, bd, idq, kk > 0 ? 1u : 0u);
          }
        } else {
          // second segment: A = Q from TMEM (16 dims = 8 columns per k-step)
#pragma unroll
          for (int kk = 0; kk < TD / 16; ++kk) {
            const uint64_t bd = dk + (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
            tc::mma_ts(d, tmem + kColQ1 + kk * 8, bd, idq, kk > 0 ? 1u : 0u);
          }
        }
        tc::commit(smem_u32(&s_full[i & 1]));
      };
      auto issue_pv = [&](int i) {
        const int first = seg_of(i) ? n0 : 0;  // the segment's first tile
        const uint64_t dv = dv0 + stage_off(i);
        const uint32_t pa = tmem + col_p(i & 1);
#pragma unroll
        for (int kt = 0; kt < TBLK / 16; ++kt) {
          // V tile as an MN-major operand: 64 head dims per 128-byte row (the
          // next 64 dims one box further, LBO), 8 tokens per 1024-byte group
          // (SBO); each k-step covers 16 tokens = two groups.
          const uint64_t bd = dv + (uint64_t)((kt * 2048) >> 4);
          tc::mma_ts(tmem + col_o(i & 1), pa + kt * 8, bd, idp, (i - first >= 2 || kt > 0) ? 1u : 0u);
        }
        tc::commit(smem_u32(&empty[rs(i)]));
        tc::commit(smem_u32(&o_done[i & 1]));
      };
      bool ok = mbar_wait_abortable(smem_u32(q_ready), 0, abort_flag, a.status, 3u);
      if (warp == MMAW) {
        // every S, in tile order: tile i landed, and its set's S buffer free
        // (the softmax of tile i-2 arrived on p_ready after reading it). The
        // softmax of tile i+2 cannot arrive before S(i+2) is issued, so the
        // phase waited for is never overtaken.
        for (int i = 0; ok && i < ntot; ++i) {
          if (i >= 2 && !mbar_spin_abortable(smem_u32(&p_ready[i & 1]), ((i - 2) >> 1) & 1,
                                             abort_flag, a.status, 6u)) {
            ok = false;
            break;
          }
          if (!mbar_spin_abortable(smem_u32(&full[rs(i)]), rp(i), abort_flag, a.status, 5u)) {
            ok = false;
            break;
          }
          if (seg_of(i) == 1 && !q1_seen) {
            if (!mbar_wait_abortable(smem_u32(q1_ready), 0, abort_flag, a.status, 7u)) {
              ok = false;
              break;
            }
            q1_seen = true;
          }
          tc::fence_after();
          issue_qk(i);
        }
      } else {
        // every P.V, in tile order, once the softmax of the tile has written
        // P; p_ready also says the set has read out its previous segment's O,
        // so the first P.V of a segment may overwrite it. The stage is
        // released after its P.V: its S had completed before the softmax
        // could write P.
        for (int i = 0; ok && i < ntot; ++i) {
          if (!mbar_spin_abortable(smem_u32(&p_ready[i & 1]), (i >> 1) & 1, abort_flag, a.status,
                                   6u)) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_pv(i);
        }
      }
      // tensor memory is released only after every issued MMA has finished
      // (every issuer arrives; one with no tiles arrives at once)
      tc::commit(smem_u32(mma_done));
      mbar_wait_drain(smem_u32(mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // set X = warp / 4 takes tiles X, X+2, ... over all segments; the warp
    // with lane quarter q owns stacked rows 32q..32q+31 (quarters >= NSW hold
    // only padding rows and stay idle)
    const int X = warp >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const bool active = q4 < NSW;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint32_t colS = col_s(X), colO = col_o(X), colP = col_p(X);
    // visible drafts of this row (bits < T only); padding rows see none
    const unsigned long long vis = (r < a.R) ? s_anc[r / a.G] : 0ull;
    bool ok = true;
    int i = X;  // this set's next tile
    int k = 0;  // this set's tiles so far (all segments): barrier phases
    for (int j = 0; j < sp.n && active; ++j) {
      const int seg_end = j == 0 ? n0 : ntot;
      m_run = -INFINITY;
      l_run = 0.f;
      int kseg = 0;  // this set's tiles in segment j
      for (; ok && i < seg_end; i += 2, ++k, ++kseg) {
        const int s = i % NS;
        // every branch that guards a warp-collective tcgen05 instruction must be
        // taken by all 32 lanes together: wait outcomes are made warp-uniform
        const bool got =
            mbar_wait_abortable(smem_u32(&s_full[X]), k & 1, abort_flag, a.status, 8u) &&
            mbar_wait_abortable(smem_u32(&full[s]), (i / NS) & 1, abort_flag, a.status, 9u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc::fence_after();
        float v[64];
#pragma unroll
        for (int h32 = 0; h32 < 2; ++h32) {
          uint32_t sr[32];
          tc::ld32(tmem + lane_base + colS + 32 * h32, sr);
          tc::wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[32 * h32 + jj] = __uint_as_float(sr[jj]);
        }
        const int info = stage_info[s];
        if (info != 1) {
          // invalid tile: nothing kept; draft tile: the row's visible drafts;
          // partial block: its first info >> 8 columns (branch-free: one
          // 64-bit keep mask, one select per column)
          const int lim = info >> 8;
          const unsigned long long keepb =
              (info & 1) ? ((info & 2) ? vis : (lim ? (1ull << lim) - 1ull : ~0ull)) : 0ull;
          const uint32_t klo = (uint32_t)keepb, khi = (uint32_t)(keepb >> 32);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            v[jj] = ((klo >> jj) & 1u) ? v[jj] : -INFINITY;
            v[32 + jj] = ((khi >> jj) & 1u) ? v[32 + jj] : -INFINITY;
          }
        }
        float mraw = v[0];
#pragma unroll
        for (int jj = 1; jj < 64; ++jj) mraw = fmaxf(mraw, v[jj]);
        const float mx = mraw * a.scale_log2;  // scale > 0: max commutes with it
        // This set's previous P.V must be done before P and (on a rescale) O
        // are touched again.
        if (k > 0) {
          const bool got2 = mbar_wait_abortable(smem_u32(&o_done[X]), (k - 1) & 1, abort_flag,
                                                a.status, 10u);
          if (!__all_sync(0xffffffffu, got2)) {
            ok = false;
            break;
          }
          tc::fence_after();
        }
        // Lazy rescale, decided per warp: when any row's max grew by more than
        // 2^8, every lane moves its reference to max(m_run, mx) (alpha = 1 for
        // rows whose max did not grow). A segment's first tile has no O yet.
        if (__any_sync(0xffffffffu, mx > m_run + kRescaleLog2)) {
          const float m_new = fmaxf(m_run, mx);
          const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);  // 0 if m_run = -inf
          if (kseg > 0) {
#pragma unroll
            for (int cc = 0; cc < TD / 32; ++cc) {
              uint32_t ov[32];
              tc::ld32(tmem + lane_base + colO + 32 * cc, ov);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tc::st32(tmem + lane_base + colO + 32 * cc, ov);
            }
          }
          l_run *= alpha;
          m_run = m_new;
        }
        const float nbase = (m_run == -INFINITY) ? 0.f : -m_run;
        uint32_t pk[32];
        float ls = 0.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const float p0 = exp2f(fmaf(v[2 * jj], a.scale_log2, nbase));
          const float p1 = exp2f(fmaf(v[2 * jj + 1], a.scale_log2, nbase));
          ls += p0 + p1;
          pk[jj] = pack_bf16(p0, p1);
        }
        l_run += ls;
        tc::st32(tmem + lane_base + colP, pk);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_ready[X]));
      }
      // the final segment's ticket, taken as its stream ends: the atomic's
      // round trip overlaps the read-out and staging below
      if (ticketed && threadIdx.x == 0 && j == sp.n - 1)
        final_ticket = atomicAdd(&a.counters[sp.pair[j] * kPairWords + kTicketWord], 1u);
      // this set's O of segment j is complete once its last P.V is (the final
      // segment's O stays in TMEM: the epilogue folds it from there)
      bool fin = ok && kseg > 0;
      if (fin)
        fin = mbar_wait_abortable(smem_u32(&o_done[X]), (k - 1) & 1, abort_flag, a.status, 11u);
      const bool ofin = __all_sync(0xffffffffu, fin);
      if (!ofin) {
        if (kseg > 0 || !ok) atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
        m_run = -INFINITY;  // weight 0 in every fold: its O is never read
        l_run = 0.f;
      }
      if (j + 1 < sp.n) {
        if (ofin) {
          tc::fence_after();
#pragma unroll
          for (int cc = 0; cc < TD / 32; ++cc) {
            uint32_t ov[32];
            tc::ld32(tmem + lane_base + colO + 32 * cc, ov);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o_row[32 * cc + e] = __uint_as_float(ov[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < TD; ++e) o_row[e] = 0.f;
        }
        // Mid-stream segment: this set's partial goes straight to the
        // workspace (set A in the segment's slot, set B in the pair's extra
        // slot nseg); the producer warp counts its arrival once every warp
        // has signalled mid_done. The next segment's first P.V overwrites O
        // only after this set's next p_ready arrival.
        const int pair = sp.pair[j];
        const int pslot = X == 0 ? sp.slot[j] : sp.nseg[j];
        const size_t row = ((size_t)pair * a.slot_stride + pslot) * a.rpad + r;
        if (r < a.R) {
#pragma unroll
          for (int c = 0; c < TD; c += 4)
            *reinterpret_cast<float4*>(a.part_o + row * TD + c) =
                make_float4(o_row[c], o_row[c + 1], o_row[c + 2], o_row[c + 3]);
          *reinterpret_cast<float2*>(a.part_ml + row * 2) = make_float2(m_run, l_run);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(mid_done));
      }
    }
  }

  tc::fence_before();
  __syncthreads();  // every MMA done (each set waited for its last P.V); the ring is idle

  // ---------------------------------------------------------------- epilogue
  // The final segment: both sets' (m, l) meet in shared memory (row r of set
  // X at X*kRows + r), and their O rows are folded with log-sum-exp weights
  // straight out of TMEM: the warp of lane quarter q in set X folds columns
  // [64X, 64X+64) of rows 32q..32q+31 (a warp reaches every column of its
  // lane quarter, so it reads both sets' O).
  constexpr int NT = C::kThreads;
  constexpr int OST = C::kOst;
  constexpr int KR = C::kRows;
  float* po = reinterpret_cast<float*>(ring);   // folded rows [KR][OST] (room for 2*KR)
  float* pml = po + (size_t)2 * KR * OST;       // [2*KR][2], then [KR][2] weights
  float* cml = pml + (size_t)6 * KR;            // [KR][2]: folded (M, L), cluster merge
  const int jf = sp.n - 1;  // final segment (none when the CTA has no work)
  if (jf >= 0) {
    const int pair = sp.pair[jf];
    const size_t slot = ((size_t)pair * a.slot_stride + sp.slot[jf]) * a.rpad;
    float* own_o = a.part_o + slot * TD;
    float2* own_ml = reinterpret_cast<float2*>(a.part_ml) + slot;
    if (warp < 8 && (warp & 3) < NSW) {
      const int row = (warp >> 2) * KR + 32 * (warp & 3) + lane;
      *reinterpret_cast<float2*>(pml + 2 * row) = make_float2(m_run, l_run);
    }
    // holding the pair's last ticket: merge with this partial kept here; a
    // ticket past the pair's count means a word left by an earlier call
    if (threadIdx.x == 0 && ticketed) {
      if (final_ticket + 1u == (unsigned)sp.nseg[jf]) pair_done[jf] = 2;
      else if (final_ticket >= (unsigned)sp.nseg[jf]) atomicOr(a.status, SV_FLAG_STALE_WORKSPACE);
    }
    __syncthreads();
    // the folded partial stays in shared memory for a cluster merge or for
    // this CTA's own merge
    const bool keep = a.cluster_merge || pair_done[jf] == 2;
    // per-row weights of the two sets (w_X = 2^(m_X - M)) and the folded (M, L)
    float* pw = pml + (size_t)4 * KR;  // [KR][2]
    for (int rr = threadIdx.x; rr < KR; rr += NT) {
      const float2 ma = *reinterpret_cast<const float2*>(pml + 2 * rr);
      const float2 mb = *reinterpret_cast<const float2*>(pml + 2 * (KR + rr));
      const float M = fmaxf(ma.x, mb.x);
      const float wa = (ma.x == -INFINITY) ? 0.f : exp2f(ma.x - M);
      const float wb = (mb.x == -INFINITY) ? 0.f : exp2f(mb.x - M);
      *reinterpret_cast<float2*>(pw + 2 * rr) = make_float2(wa, wb);
      if (keep)
        *reinterpret_cast<float2*>(cml + 2 * rr) = make_float2(M, wa * ma.y + wb * mb.y);
      else if (rr < a.rpad)
        own_ml[rr] = make_float2(M, wa * ma.y + wb * mb.y);
    }
    __syncthreads();
    if (warp < 8 && (warp & 3) < NSW) {
      // a set whose weight is 0 (no tile in this segment, or a wait gave up)
      // has an O that is never read: select, not multiply
      tc::fence_after();
      const int xs = warp >> 2, q4 = warp & 3, rr = 32 * q4 + lane;
      const float2 w = *reinterpret_cast<const float2*>(pw + 2 * rr);
      const uint32_t lb = (uint32_t)(32 * q4) << 16;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 64 * xs + 32 * hh;
        uint32_t oa[32], ob[32];
        tc::ld32(tmem + lb + col_o(0) + c0, oa);
        tc::ld32(tmem + lb + col_o(1) + c0, ob);
        tc::wait_ld();
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          f[e] = (w.x != 0.f ? w.x * __uint_as_float(oa[e]) : 0.f) +
                 (w.y != 0.f ? w.y * __uint_as_float(ob[e]) : 0.f);
        float* dst = keep ? po + (size_t)rr * OST + c0 : own_o + (size_t)rr * TD + c0;
        if (keep || rr < a.rpad) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        }
      }
    }
    // CTA barrier, then one thread's acquire-release arrival publishes
    // every thread's partial writes (the barrier orders them before it);
    // without tickets the arrival that completes a pair also acquires the
    // other partials. (A mid-stream segment arrived from the producer warp.)
    __syncthreads();
    if (threadIdx.x == 0 && !keep) {
      if (ticketed)
        arrive_release(&a.counters[pair * kPairWords]);
      else if ((arrive_acq_rel(&a.counters[pair * kPairWords]) & 0xFFFFu) + 1u ==
               (unsigned)sp.nseg[jf])
        pair_done[jf] = 1;
    }
  }
  tc::fence_before();
  __syncthreads();  // every TMEM read done
  if (warp == MMAW) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }

  if (a.cluster_merge) {
    // ------------------------------------------------------- cluster merge
    // The pair's CTAs are one cluster (rank = split); each has its folded
    // partial (o rows in po, (M, L) in cml) in its own shared memory. After
    // the cluster barrier, CTA `rank` merges rows [rank * share, ...) from
    // every CTA's shared memory, in rank order, with the formula below; the
    // second barrier keeps every CTA's shared memory alive until all reads
    // are done. Every CTA reaches both barriers on every path.
    cluster_sync_all();
    const int ncl = a.cluster_merge;
    const uint32_t rank = cluster_ctarank();
    const int pair = sp.pair[0], b = pair / a.Hkv, h = pair % a.Hkv;
    const int share = (a.R + ncl - 1) / ncl;
    const int r0 = min(a.R, (int)rank * share), r1 = min(a.R, r0 + share);
    const uint32_t po_s = smem_u32(po), ml_s = smem_u32(cml);
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);
    for (int idx = threadIdx.x; idx < (r1 - r0) * (TD / 4); idx += NT) {
      const int r = r0 + idx / (TD / 4), c4 = (idx % (TD / 4)) * 4;
      // every remote load of this (row, 4 columns) issued before any is used:
      // one round trip through the cluster's shared memory
      float2 ml[kMaxCluster];
      float4 o[kMaxCluster];
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q) {
        if (q < ncl) {
          ml[q] = ld_cluster_f2(cluster_map(ml_s + r * 8, q));
          o[q] = ld_cluster_f4(cluster_map(po_s + (r * OST + c4) * 4, q));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q)
        if (q < ncl) M = fmaxf(M, ml[q].x);
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q) {
        if (q < ncl && ml[q].x != -INFINITY) {  // a CTA without units adds nothing
          const float w = exp2f(ml[q].x - M);
          L += w * ml[q].y;
          acc.x += w * o[q].x;
          acc.y += w * o[q].y;
          acc.z += w * o[q].z;
          acc.w += w * o[q].w;
        }
      }
      const float inv = 1.0f / L;
      const int t = r / a.G, gq = r % a.G;
      __nv_bfloat16* dst = outp + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * TD + c4;
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst) = u;
    }
    cluster_sync_all();
    return;
  }

  // ----------------------------------------------------------------- merge
  //   M = max_s m_s, w_s = 2^(m_s - M), out = sum_s w_s o_s / sum_s w_s l_s,
  // summed in slot order whichever CTA merges, so results do not depend on
  // timing. The partials come into the idle ring by bulk copies (one per slot
  // and row range) and are combined from shared memory. The count word of a
  // pair holds its arrivals (low 16 bits) and the CTAs that finished their
  // merge share (high bits).
  uint32_t mphase = 0;
  // Staging of merge passes: with tickets it starts past the final
  // segment's folded partial (po, cml), which a merge may still read.
  const int stage_off = ticketed ? 2 * KR * OST + 8 * KR : 0;
  // bulk-copy rows [r0, r0 + nr) of the ns partial slots of `pair` (all but
  // slot `kept`, whose folded rows are in po and cml) into the ring (nr
  // even, so every (m, l) copy is a multiple of 16 bytes) and combine rows
  // [r0, r0 + nv) into out. With `pub`, the copies wait until its count
  // reaches `need` (acquire), while the other warps place the kept slot.
  auto merge_rows = [&](int pair, int ns, int r0, int nr, int nv, int kept, const unsigned* pub,
                        unsigned need) {
    const size_t pbase = (size_t)pair * a.slot_stride * a.rpad;
    float* so = reinterpret_cast<float*>(ring) + stage_off;               // [ns][nr][TD]
    float2* sml = reinterpret_cast<float2*>(so + (size_t)ns * nr * TD);   // [ns][nr]
    if (threadIdx.x < 32) {
      if (pub && threadIdx.x == 0 && !wait_count_at_least(pub, need, a.status, 14u))
        atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
      __syncwarp();  // the acquire above orders the warp's copies
      // the partials were written by other CTAs through the generic proxy
      // and acquired through the count word, and the staging area was last
      // used through the generic proxy; order both before the copy engine
      // runs. Lane 0 posts the byte count, then lane s issues slot s's copies.
      asm volatile("fence.proxy.async.global;" ::: "memory");
      fence_async_smem();
      const uint32_t mb = smem_u32(merge_bar);
      const int ncopy = ns - (kept >= 0 ? 1 : 0);
      if (threadIdx.x == 0) mbar_arrive_expect_tx(mb, (uint32_t)(ncopy * nr * kMergeRowBytes));
      __syncwarp();
      for (int sl = threadIdx.x; sl < ns; sl += 32) {
        if (sl == kept) continue;
        const size_t row0 = pbase + (size_t)sl * a.rpad + r0;
        bulk_load(smem_u32(so + (size_t)sl * nr * TD), a.part_o + row0 * TD, (uint32_t)(nr * TD * 4),
                  mb);
        bulk_load(smem_u32(sml + (size_t)sl * nr), a.part_ml + row0 * 2, (uint32_t)(nr * 8), mb);
      }
    }
    if (kept >= 0) {
      // this CTA's own slot: its folded rows, copied into place by warps
      // 1.. while warp 0 waits and the other slots land
      float* ko = so + (size_t)kept * nr * TD;
      for (int idx = threadIdx.x - 32; idx >= 0 && idx < nr * (TD / 4); idx += NT - 32) {
        const int rr = idx / (TD / 4), c4 = (idx % (TD / 4)) * 4;
        *reinterpret_cast<float4*>(ko + rr * TD + c4) =
            *reinterpret_cast<const float4*>(po + (r0 + rr) * OST + c4);
      }
      for (int rr = threadIdx.x - 32; rr >= 0 && rr < nr; rr += NT - 32)
        sml[(size_t)kept * nr + rr] = reinterpret_cast<const float2*>(cml)[r0 + rr];
    }
    __syncthreads();  // the kept slot is in place; warp 0 has issued every copy
    if (!mbar_wait_drain(smem_u32(merge_bar), mphase) && threadIdx.x == 0)
      atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
    mphase ^= 1u;
    combine_rows<NT>(a, pair / a.Hkv, pair % a.Hkv, ns, nr, r0, nv, so, sml);
    __syncthreads();  // the next copies overwrite the staging area
  };
  // Row slices of a pair, merged in parallel by the pair's CTAs: slice q
  // (q < nsl = min(segments, 32)) covers rows [q * share, (q + 1) * share)
  // and belongs to the CTA whose segment is the pair's q-th. A slice is
  // merged by whoever claims its bit in the pair's claim word first. Each CTA
  // waits (briefly, bounded) for the pair's last arrival and claims its own
  // slice; the CTA whose arrival completed the pair merges its own slice and
  // then claims, in one atomic, every slice still unclaimed: the slices of
  // CTAs that are slow, gave up waiting or are not resident. So every slice
  // is merged exactly once and no CTA depends on another to finish. The
  // count word's high half counts CTAs done with the pair; the last of them
  // returns the words to zero for the next call. With no wait
  // (merge_wait_ns == 0) the last CTA merges every row alone.
  for (int j = 0; j < sp.n; ++j) {
    const int pair = sp.pair[j];
    const int nseg = sp.nseg[j], ns = nseg + sp.mid[j];
    // rows per pass that the ring holds for ns slots (even; two always fit:
    // wide merges stage from the ring's start, and a narrow merge's slots
    // are few enough to fit past the folded partial)
    int rpp = ((C::kRing - stage_off * 4) / (ns * kMergeRowBytes)) & ~1;
    rpp = rpp < 2 ? 2 : (rpp > a.rpad ? a.rpad : rpp);
    // rows [r0, r1) (r0 even) in passes of rpp rows
    auto merge_range = [&](int r0, int r1, int kept, const unsigned* pub, unsigned need) {
      for (int q0 = r0; q0 < r1; q0 += rpp) {
        const int nv = min(rpp, r1 - q0);
        merge_rows(pair, ns, q0, min((nv + 1) & ~1, a.rpad - q0), nv, kept, q0 == r0 ? pub : nullptr,
                   need);
      }
    };
    const int pd = pair_done[j];  // the same in every thread
    if (ticketed) {
      // The narrow merge, by the pair's last ticket. Every other segment took
      // its ticket earlier, so it is past its stream and publishes without
      // waiting for anything: wait for those publications (every segment's,
      // or all but this one's when its partial stayed here), merge every
      // row, and return the pair's words to zero (nothing else touches them
      // any more).
      if (pd) {
        unsigned* w = a.counters + pair * kPairWords;
        merge_range(0, a.R, pd == 2 ? sp.slot[j] : -1, w, (unsigned)(pd == 2 ? nseg - 1 : nseg));
        if (threadIdx.x == 0) {
          w[0] = 0u;
          w[kTicketWord] = 0u;
        }
      }
      continue;
    }
    const bool last = pd != 0;
    const int nsl = nseg < 32 ? nseg : 32;
    const int share = ((a.R + nsl - 1) / nsl + 1) & ~1;
    const int own = sp.slot[j] < nsl ? sp.slot[j] : -1;
    if (threadIdx.x == 0) {
      int got = 0;
      if (own >= 0) {
        bool complete = last;
        if (!complete) {
          // a short bounded wait: the pair's CTAs normally finish together
          const uint64_t t0 = globaltimer_ns();
          unsigned nap = 64;
          while (!(complete = (load_acquire(&a.counters[pair * kPairWords]) & 0xFFFFu) >=
                              (unsigned)nseg)) {
            if (globaltimer_ns() - t0 > (uint64_t)a.merge_wait_ns) break;
            __nanosleep(nap);
            nap = nap < 512 ? 2 * nap : nap;
          }
        }
        if (complete) got = !(atomicOr(a.claim + pair * kPairWords, 1u << own) & (1u << own));
      }
      *merge_got = got;
    }
    __syncthreads();
    if (*merge_got) merge_range(min(a.R, own * share), min(a.R, (own + 1) * share), -1, nullptr, 0u);
    if (last) {
      if (threadIdx.x == 0) {
        const unsigned all = nsl == 32 ? 0xFFFFFFFFu : ((1u << nsl) - 1u);
        *merge_got = (int)(all & ~atomicOr(a.claim + pair * kPairWords, all));
      }
      __syncthreads();
      // each run of consecutive claimed slices is one row range, copied in
      // as few passes as the ring allows
      const unsigned mine = (unsigned)*merge_got;
      for (int q = 0; q < nsl;) {
        if (!(mine & (1u << q))) {
          ++q;
          continue;
        }
        int e = q + 1;
        while (e < nsl && (mine & (1u << e))) ++e;
        merge_range(min(a.R, q * share), min(a.R, e * share), -1, nullptr, 0u);
        q = e;
      }
    }
    if (threadIdx.x == 0) {
      if ((atomicAdd(&a.counters[pair * kPairWords], 1u << 16) >> 16) == (unsigned)nseg - 1u) {
        // every CTA of the pair is done with its words
        a.counters[pair * kPairWords] = 0u;
        a.claim[pair * kPairWords] = 0u;
      }
    }
    __syncthreads();
  }
}

template <int NSW>
struct TcKernel {
  static constexpr int NS = 6;
  using C = TcCfg<NSW, NS>;
  static void* fn() { return reinterpret_cast<void*>(attend_tc_kernel<NSW, NS>); }
};

template <int NSW>
cudaError_t launch_tc_cfg(const AttendArgs& a, cudaStream_t st) {
  using K = TcKernel<NSW>;
  CUtensorMap mk, mv;
  const char* why = nullptr;
  CUtensorMap mq, mdk, mdv;
  if (!encode_pool_map(&mk, a.k_pool, a.num_pages, a.Hkv, TBLK, TD, &why) ||
      !encode_pool_map(&mv, a.v_pool, a.num_pages, a.Hkv, TBLK, TD, &why) ||
      !encode_q_map(&mq, a.q, a.B, a.T, a.Hq, a.G, TD, &why) ||
      !encode_draft_map(&mdk, a.draft_k, a.B, a.T, a.Hkv, TD, TBLK, &why) ||
      !encode_draft_map(&mdv, a.draft_v, a.B, a.T, a.Hkv, TD, TBLK, &why))
    return cudaErrorInvalidValue;
  const int ctas = a.streamk ? a.n_splits : a.B * a.Hkv * a.n_splits + a.split_extra;
  if (a.cluster_merge)
    return launch_pdl_cluster(attend_tc_kernel<NSW, K::NS>, dim3(ctas), dim3(K::C::kThreads),
                              K::C::kSmem, a.cluster_merge, st, mk, mv, mq, mdk, mdv, a);
  return launch_pdl(attend_tc_kernel<NSW, K::NS>, dim3(ctas), dim3(K::C::kThreads), K::C::kSmem,
                    st, mk, mv, mq, mdk, mdv, a);
}

// Sets the kernel's shared-memory attributes and returns its resident CTAs
// per SM (one: the ring is sized for a whole SM); cached per device.
template <int NSW>
int occupancy_tc_cfg() {
  using K = TcKernel<NSW>;
  static std::atomic<int> cached[kMaxDevices];
  const int dev = current_device();
  const int c = cached[dev].load();
  if (c > 0) return c;
  if (cudaFuncSetAttribute(K::fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, K::C::kSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(K::fn(), cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      cudaFuncSetAttribute(K::fn(), cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K::fn(), K::C::kThreads, K::C::kSmem) !=
      cudaSuccess)
    return 0;
  if (n > 1) n = 1;
  cached[dev].store(n);
  return n;
}

}  // namespace

bool attend_tc_applies(const AttendArgs& a, int dtype) {
  if (dtype != SV_BF16 || a.d != TD || a.blk != TBLK) return false;
  if (a.R > 128 || a.T > TBLK) return false;
  if (a.num_pages < 1 || !a.k_pool || !a.v_pool) return false;
  if (reinterpret_cast<uintptr_t>(a.q) & 15) return false;
  if ((reinterpret_cast<uintptr_t>(a.k_pool) & 15) || (reinterpret_cast<uintptr_t>(a.v_pool) & 15))
    return false;
  if ((long long)(a.num_pages + 1) * a.Hkv * a.blk >= (1ll << 31)) return false;
  return true;
}

// Clusters of ncl CTAs that the device keeps resident at once.
template <int NSW>
int active_clusters_cfg(int ncl, int ctas) {
  using K = TcKernel<NSW>;
  if (occupancy_tc_cfg<NSW>() <= 0) return 0;  // sets the attributes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(K::C::kThreads);
  cfg.dynamicSmemBytes = K::C::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, K::fn(), &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

int attend_tc_cluster(const AttendArgs& a, int pairs) {
  constexpr int kMaxPairs = 64;
  if (pairs < 1 || pairs > kMaxPairs) return 0;
  const int nsw = (a.R + 31) / 32;
  const int cfgi = nsw <= 1 ? 0 : nsw <= 2 ? 1 : 2;
  // answers depend on the device, the kernel variant and the pair count only
  static std::atomic<int> cache[kMaxDevices][3][kMaxPairs + 1];
  const int dev = current_device();
  const int c = cache[dev][cfgi][pairs].load();
  if (c != 0) return c > 0 ? c : 0;
  // the largest cluster of 8..16 CTAs the device keeps `pairs` of resident
  // (16 is not always the best: how many fit depends on how the SMs are
  // grouped on the chip)
  int best = 0;
  for (int ncl = kMaxCluster; ncl >= kMinCluster; --ncl) {
    if (pairs * ncl > sm_count()) continue;
    const int n = cfgi == 0   ? active_clusters_cfg<1>(ncl, pairs * ncl)
                  : cfgi == 1 ? active_clusters_cfg<2>(ncl, pairs * ncl)
                              : active_clusters_cfg<4>(ncl, pairs * ncl);
    if (n >= pairs) {
      best = ncl;
      break;
    }
  }
  cache[dev][cfgi][pairs].store(best > 0 ? best : -1);
  return best;
}

bool attend_tc_narrow_merge(int slot_stride, int rpad) {
  // A narrow merge stages its passes past the merging CTA's folded partial:
  // two rows of every slot must fit there (they always do under the size
  // rule; checked rather than assumed).
  const int kr = rpad <= 32 ? 32 : rpad <= 64 ? 64 : 128;
  const size_t folded = ((size_t)2 * kr * TcCfg<4, 6>::kOst + 8 * kr) * 4;
  const size_t room = TcCfg<4, 6>::kRing - folded;
  return (size_t)slot_stride * rpad * kMergeRowBytes <= kSoloMergeBytes &&
         (size_t)2 * slot_stride * kMergeRowBytes <= room;
}

int attend_tc_ctas_per_sm(const AttendArgs& a) {
  const int nsw = (a.R + 31) / 32;
  if (nsw <= 1) return occupancy_tc_cfg<1>();
  if (nsw <= 2) return occupancy_tc_cfg<2>();
  return occupancy_tc_cfg<4>();
}

cudaError_t launch_attend_tc(AttendArgs a, cudaStream_t st) {
  const int nsw = (a.R + 31) / 32;
  // When one CTA would copy little (few slots of few rows), the pair's last
  // CTA merges it alone and the others leave at once, freeing their SMs for
  // the next kernel; otherwise the pair's CTAs share the rows.
  a.merge_wait_ns = attend_tc_narrow_merge(a.slot_stride, a.rpad) ? 0u : (unsigned)kMergeWaitNs;
  if (nsw <= 1) return launch_tc_cfg<1>(a, st);
  if (nsw <= 2) return launch_tc_cfg<2>(a, st);
  return launch_tc_cfg<4>(a, st);
}

}  // namespace sva
