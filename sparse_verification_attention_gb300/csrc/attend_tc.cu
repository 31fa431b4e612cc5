// Split-KV sparse verification attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators), bf16, head dim 128, blocks of 64 tokens.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: every draft token
// attends to the same selected set of KV blocks, so the R = T*G query rows of
// one KV head are stacked into one MMA tile and each selected page is read
// from HBM once for all of them.
//
// CTA roles (one CTA per SM, since tcgen05 kernels are scheduled one per SM
// here; a 6-stage ring keeps ~192 KB of K/V in flight per SM):
//   * producer warp: resolves selected block -> page through the block table
//     (32 at a time, one lane each) and issues 2-D TMA copies (128-byte
//     swizzle) of the page's K and V tiles into the ring; the draft tile (this
//     pair's draft K/V) is written into a ring stage directly.
//   * MMA warp (one elected lane): S_i = Q K_i^T into TMEM (M=128 rows, N=64
//     tokens, K=128), then after softmax O += P_i V_i with P read from TMEM
//     (M=128, N=128, K=64, V as an MN-major operand); stages are released by
//     tcgen05 commits.
//   * two softmax sets: set A takes the even work units, set B the odd ones,
//     each with its own S, P and O in TMEM, so two independent softmax
//     chains overlap. In each set the warp owning TMEM lane quarter q holds
//     stacked rows 32q..32q+31, one row per thread (quarters past ceil(R/32)
//     hold only zero padding rows and stay idle). Each set keeps its own
//     running max (log2 domain; the accumulator is rescaled only when some
//     row's max grows by more than 2^8, decided per warp so that the
//     warp-collective TMEM loads/stores are taken by all lanes) and sum: the
//     two sets are independent partials, folded with log-sum-exp weights in
//     the epilogue.
//   * epilogue: the split's unnormalised (o, m, l) rows go to the workspace;
//     the last CTA of each (b, h) to finish (an atomic arrival count in the
//     workspace, reset by that CTA) merges the pair's splits with log-sum-exp
//     weights and writes the output. The grid is 1-D with a non-uniform split
//     map so that every SM holds one CTA.
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
// TMEM columns of set X in {0, 1}: S (64 fp32), O (128 fp32), P (32 x bf16x2)
__host__ __device__ constexpr uint32_t col_s(int x) { return x ? 64u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return x ? 256u : 128u; }
__host__ __device__ constexpr uint32_t col_p(int x) { return x ? 416u : 384u; }
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxMergeSplits = 8;  // splits merged with all loads in flight

constexpr int r1024(int x) { return (x + 1023) / 1024 * 1024; }

template <int NSW, int NS>
struct TcCfg {
  static constexpr int kThreads = 32 * 10;        // 8 softmax + producer + MMA
  static constexpr int kRows = 32 * NSW;          // stacked rows held in TMEM lanes (>= R)
  static constexpr int kQBox = 128 * 128;         // one 64-column Q box, 128 rows
  static constexpr int kRingOff = 2 * kQBox;
  static constexpr int kOst = TD + 4;
  static constexpr int kMergeBytes = (2 * kRows * kOst + 2 * kRows * 2) * 4;
  static constexpr int kRingRaw = NS * kStageBytes;
  static constexpr int kRing = r1024(kMergeBytes > kRingRaw ? kMergeBytes : kRingRaw);
  static constexpr int kCtrlOff = kRingOff + kRing;
  static constexpr int kSmem = kCtrlOff + 256 + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t swz128(int row, int chunk16) {
  return row * 128 + ((chunk16 ^ (row & 7)) << 4);
}

template <int NSW, int NS>
__global__ void __launch_bounds__(32 * 10, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ AttendArgs a) {
  using C = TcCfg<NSW, NS>;
  constexpr int PRODUCER = 8, MMAW = 9;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* ring = smem + C::kRingOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kCtrlOff);
  uint64_t* empty = full + NS;
  uint64_t* s_full = empty + NS;   // [2] per set
  uint64_t* p_ready = s_full + 2;  // [2] per set, 4 warps each
  uint64_t* o_done = p_ready + 2;  // [2] per set
  uint64_t* mma_done = o_done + 2; // drain: every issued MMA has completed
  uint64_t* q_ready = mma_done + 1; // Q landed (TMA) and padding rows zeroed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_ready + 1);
  int* stage_info = reinterpret_cast<int*>(tmem_slot + 1);  // bit0 valid, bit1 draft tile
  volatile int* abort_flag = stage_info + NS;
  volatile int* last_flag = abort_flag + 1;
  // ancestor masks of the drafts, copied out of the parameter space with
  // warp-uniform indices (per-lane indices into it would serialize)
  __shared__ unsigned long long s_anc[kMaxT];

  int pair, split, nsp;
  split_of_cta(blockIdx.x, a.n_splits, a.split_extra, &pair, &split, &nsp);
  const int b = pair / a.Hkv, h = pair % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bps = (a.n_sel + 1 + nsp - 1) / nsp;
  const int u0 = split * bps;
  const int u1 = min(a.n_sel + 1, u0 + bps);
  const int nunits = max(0, u1 - u0);
  const int nblk = max(0, min(u1, a.n_sel) - u0);
  const bool has_draft = (u0 <= a.n_sel && a.n_sel < u1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&p_ready[i]), NSW);
      mbar_init(smem_u32(&o_done[i]), 1);
    }
    mbar_init(smem_u32(mma_done), 1);
    mbar_init(smem_u32(q_ready), 5);  // producer's expect_tx + 4 zeroing warps
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmQ);
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
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // everything below may read what earlier kernels wrote

  // Q operand, 128 rows: rows r < R = the stacked query rows (draft t, head
  // g) = Q[b, t, h*G + g] in order r = t*G + g, brought by one 3-D TMA box per
  // 64 dims (issued first by the producer); rows R..127 are zeroed here.
  if (warp < 4) {
    const int r = threadIdx.x;
    if (r >= a.R) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(qs + (c >> 3) * C::kQBox + swz128(r, c & 7)) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(q_ready));
  }

  // per-thread results for the epilogue (softmax threads)
  float o_row[TD];
  float m_run = -INFINITY, l_run = 0.f;

  if (warp == PRODUCER) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the query rows first, ahead of the K/V stream
      const uint32_t qb = smem_u32(q_ready);
      mbar_arrive_expect_tx(qb, (uint32_t)a.R * TD * 2);
      tma_load_3d(smem_u32(qs), &tmQ, 0, h * a.G, b * a.T, qb);
      tma_load_3d(smem_u32(qs) + C::kQBox, &tmQ, 64, h * a.G, b * a.T, qb);
    }
    const int oob_row = a.num_pages * a.Hkv * TBLK;  // past the end: TMA zero-fills
    int issued = 0;
    bool stop = false;
    for (int base = 0; base < nblk && !stop; base += 32) {
      int row = oob_row, ok = 0;
      if (base + lane < nblk) {
        const int j = a.sel ? a.sel[(size_t)pair * a.sel_stride + u0 + base + lane] : u0 + base + lane;
        if (j < 0 || j >= a.nb) {
          atomicOr(a.status, SV_FLAG_BAD_BLOCK_INDEX);
        } else {
          const int page = a.block_table[(size_t)b * a.nb_max + j];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, SV_FLAG_BAD_PAGE);
          } else {
            row = (page * a.Hkv + h) * TBLK;
            ok = 1;
          }
        }
      }
      const int cnt = min(32, nblk - base);
      for (int qq = 0; qq < cnt; ++qq) {
        const int i = base + qq;
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
            tma_load_2d(kdst, &tmK, 0, rq, fb);
            tma_load_2d(kdst + kBoxBytes, &tmK, 64, rq, fb);
            tma_load_2d(vdst, &tmV, 0, rq, fb);
            tma_load_2d(vdst + kBoxBytes, &tmV, 64, rq, fb);
            issued = i + 1;
          }
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) {
          stop = true;
          break;
        }
      }
    }
    if (has_draft && !stop) {
      // draft tile: rows u < T from this pair's draft K/V, rows T..63 zero
      const int i = nblk, s = i % NS;
      int fail = 0;
      if (lane == 0 && i >= NS &&
          !mbar_wait_abortable(smem_u32(&empty[s]), ((i / NS) & 1) ^ 1, abort_flag, a.status, 2u))
        fail = 1;
      if (!__shfl_sync(0xffffffffu, fail, 0)) {
        uint8_t* st = ring + s * kStageBytes;
        const uint4* dk = static_cast<const uint4*>(a.draft_k);
        const uint4* dv = static_cast<const uint4*>(a.draft_v);
        for (int idx = lane; idx < TBLK * 16; idx += 32) {
          const int u = idx >> 4, c = idx & 15;
          uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
          if (u < a.T) {
            const size_t off = (((size_t)b * a.T + u) * a.Hkv + h) * (TD / 8) + c;
            kv = dk[off];
            vv = dv[off];
          }
          const uint32_t o = (c >> 3) * kBoxBytes + swz128(u, c & 7);
          *reinterpret_cast<uint4*>(st + o) = kv;
          *reinterpret_cast<uint4*>(st + kTileBytes + o) = vv;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          stage_info[s] = 3;
          mbar_arrive(smem_u32(&full[s]));
        }
        issued = i + 1;
      }
    }
    // never leave with a bulk copy still writing into the ring
    if (lane == 0)
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_drain(smem_u32(&full[i % NS]), (i / NS) & 1);
  } else if (warp == MMAW) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && nunits > 0) {
      constexpr uint32_t idq = tc::idesc_bf16(128, 64, false, false);
      constexpr uint32_t idp = tc::idesc_bf16(128, TD, false, true);
      const uint32_t qb = smem_u32(qs);
      const uint32_t rb = smem_u32(ring);
      auto issue_qk = [&](int i) {
        const uint32_t kb = rb + (i % NS) * kStageBytes;
        const uint32_t d = tmem + col_s(i & 1);
#pragma unroll
        for (int kk = 0; kk < TD / 16; ++kk) {
          const uint64_t ad = tc::smem_desc(qb + (kk >> 2) * C::kQBox + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = tc::smem_desc(kb + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
          tc::mma_ss(d, ad, bd, idq, kk > 0 ? 1u : 0u);
        }
        tc::commit(smem_u32(&s_full[i & 1]));
      };
      bool ok = mbar_wait_abortable(smem_u32(q_ready), 0, abort_flag, a.status, 3u) &&
                mbar_wait_abortable(smem_u32(&full[0]), 0, abort_flag, a.status, 4u);
      tc::fence_after();
      if (ok) issue_qk(0);
      for (int i = 0; ok && i < nunits; ++i) {
        // S buffer of unit i+1's set is free: its previous reader (softmax of
        // unit i-1) arrived on p_ready before PV(i-1) was issued
        if (i + 1 < nunits) {
          if (!mbar_wait_abortable(smem_u32(&full[(i + 1) % NS]), ((i + 1) / NS) & 1, abort_flag,
                                   a.status, 5u)) {
            ok = false;
            break;
          }
          issue_qk(i + 1);
        }
        if (!mbar_wait_abortable(smem_u32(&p_ready[i & 1]), (i >> 1) & 1, abort_flag, a.status, 6u)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t vb = rb + (i % NS) * kStageBytes + kTileBytes;
        const uint32_t pa = tmem + col_p(i & 1);
#pragma unroll
        for (int kt = 0; kt < TBLK / 16; ++kt) {
          // V tile as an MN-major operand: 64 head dims per 128-byte row (the
          // next 64 dims one box further, LBO), 8 tokens per 1024-byte group
          // (SBO); each k-step covers 16 tokens = two groups.
          const uint64_t bd = tc::smem_desc(vb + kt * 2048, kBoxBytes, 1024);
          tc::mma_ts(tmem + col_o(i & 1), pa + kt * 8, bd, idp, (i >= 2 || kt > 0) ? 1u : 0u);
        }
        tc::commit(smem_u32(&empty[i % NS]));
        tc::commit(smem_u32(&o_done[i & 1]));
      }
      // tensor memory is released only after every issued MMA has finished
      tc::commit(smem_u32(mma_done));
      mbar_wait_drain(smem_u32(mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // set X = warp / 4 takes units X, X+2, ...; the warp with lane quarter q
    // owns stacked rows 32q..32q+31 (quarters >= NSW hold only padding rows
    // and stay idle)
    const int X = warp >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint32_t colS = col_s(X), colO = col_o(X), colP = col_p(X);
    // visible drafts of this row (bits < T only); padding rows see none
    const unsigned long long vis = (r < a.R) ? s_anc[r / a.G] : 0ull;
    const int nmine = (q4 < NSW && nunits > X) ? (nunits - X + 1) / 2 : 0;
    bool ok = true;
    for (int k = 0; k < nmine; ++k) {
      const int i = X + 2 * k;
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
        for (int j = 0; j < 32; ++j) v[32 * h32 + j] = __uint_as_float(sr[j]);
      }
      const int info = stage_info[s];
      if (info != 1) {
        // invalid tile: nothing kept; draft tile: the row's visible drafts
        // (branch-free: one 64-bit keep mask, one select per column)
        const unsigned long long keepb = (info & 1) ? ((info & 2) ? vis : ~0ull) : 0ull;
        const uint32_t klo = (uint32_t)keepb, khi = (uint32_t)(keepb >> 32);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = ((klo >> j) & 1u) ? v[j] : -INFINITY;
          v[32 + j] = ((khi >> j) & 1u) ? v[32 + j] : -INFINITY;
        }
      }
      float mraw = v[0];
#pragma unroll
      for (int j = 1; j < 64; ++j) mraw = fmaxf(mraw, v[j]);
      const float mx = mraw * a.scale_log2;  // scale > 0: max commutes with it
      // This set's previous P.V must be done before P and (on a rescale) O are
      // touched again.
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
      // rows whose max did not grow).
      if (__any_sync(0xffffffffu, mx > m_run + kRescaleLog2)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);  // 0 if m_run = -inf
        if (k > 0) {
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
      for (int j = 0; j < 32; ++j) {
        const float p0 = exp2f(fmaf(v[2 * j], a.scale_log2, nbase));
        const float p1 = exp2f(fmaf(v[2 * j + 1], a.scale_log2, nbase));
        ls += p0 + p1;
        pk[j] = pack_bf16(p0, p1);
      }
      l_run += ls;
      tc::st32(tmem + lane_base + colP, pk);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_ready[X]));
    }
    bool fin = ok && nmine > 0;
    if (fin)
      fin = mbar_wait_abortable(smem_u32(&o_done[X]), (nmine - 1) & 1, abort_flag, a.status, 11u);
    if (__all_sync(0xffffffffu, fin)) {
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
      if (nmine > 0) atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
#pragma unroll
      for (int e = 0; e < TD; ++e) o_row[e] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }
  }
  pdl_trigger();

  tc::fence_before();
  __syncthreads();  // all TMEM reads and MMAs done; the ring is idle
  if (warp == MMAW) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }

  // ---------------------------------------------------------------- epilogue
  // Stage both sets' (o, m, l) for the kRows real lanes; fold set B into set A
  // with log-sum-exp weights (row r of set X staged at X*kRows + r).
  constexpr int NT = 32 * 10;
  constexpr int OST = C::kOst;
  constexpr int KR = C::kRows;
  float* po = reinterpret_cast<float*>(ring);   // [2*KR][OST]
  float* pml = po + (size_t)2 * KR * OST;       // [2*KR][2]
  if (warp < 8 && (warp & 3) < NSW) {
    const int row = (warp >> 2) * KR + 32 * (warp & 3) + lane;
#pragma unroll
    for (int c = 0; c < TD; c += 4)
      *reinterpret_cast<float4*>(po + row * OST + c) =
          make_float4(o_row[c], o_row[c + 1], o_row[c + 2], o_row[c + 3]);
    *reinterpret_cast<float2*>(pml + 2 * row) = make_float2(m_run, l_run);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < KR * (TD / 4); idx += NT) {
    const int r = idx / (TD / 4), c4 = (idx % (TD / 4)) * 4;
    const float2 ma = *reinterpret_cast<const float2*>(pml + 2 * r);
    const float2 mb = *reinterpret_cast<const float2*>(pml + 2 * (KR + r));
    const float M = fmaxf(ma.x, mb.x);
    const float wa = (ma.x == -INFINITY) ? 0.f : exp2f(ma.x - M);
    const float wb = (mb.x == -INFINITY) ? 0.f : exp2f(mb.x - M);
    const float4 oa = *reinterpret_cast<const float4*>(po + r * OST + c4);
    const float4 ob = *reinterpret_cast<const float4*>(po + (KR + r) * OST + c4);
    // (r, c4) is read and written by this thread only
    *reinterpret_cast<float4*>(po + r * OST + c4) =
        make_float4(wa * oa.x + wb * ob.x, wa * oa.y + wb * ob.y, wa * oa.z + wb * ob.z,
                    wa * oa.w + wb * ob.w);
  }
  __syncthreads();
  for (int r = threadIdx.x; r < KR; r += NT) {
    const float2 ma = *reinterpret_cast<const float2*>(pml + 2 * r);
    const float2 mb = *reinterpret_cast<const float2*>(pml + 2 * (KR + r));
    const float M = fmaxf(ma.x, mb.x);
    const float wa = (ma.x == -INFINITY) ? 0.f : exp2f(ma.x - M);
    const float wb = (mb.x == -INFINITY) ? 0.f : exp2f(mb.x - M);
    *reinterpret_cast<float2*>(pml + 2 * r) = make_float2(M, wa * ma.y + wb * mb.y);
  }
  __syncthreads();

  // ---------------------------------------- split partial, then last-CTA merge
  const size_t pbase = (size_t)pair * a.slot_stride * a.rpad;
  const size_t slot = pbase + (size_t)split * a.rpad;
  for (int idx = threadIdx.x; idx < a.rpad * (TD / 4); idx += NT) {
    const int r = idx / (TD / 4), c = (idx % (TD / 4)) * 4;
    *reinterpret_cast<float4*>(a.part_o + (slot + r) * TD + c) =
        *reinterpret_cast<const float4*>(po + r * OST + c);
  }
  for (int r = threadIdx.x; r < a.rpad; r += NT)
    *reinterpret_cast<float2*>(a.part_ml + (slot + r) * 2) = *reinterpret_cast<const float2*>(pml + 2 * r);
  // The last split of this (b, h) to arrive combines all of them:
  //   M = max_s m_s, w_s = 2^(m_s - M), out = sum_s w_s o_s / sum_s w_s l_s.
  // CTA barrier, then one thread's device-scope fence publishes every
  // thread's partial writes before the arrival count (the barrier orders
  // them before the fence); the last arrival fences again before reading.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(&a.counters[pair], 1u) == (unsigned)nsp - 1u;
    if (last) __threadfence();
    *last_flag = last;
  }
  __syncthreads();
  if (*last_flag) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    // this CTA's own split is still staged in shared memory (rows < KR)
    auto merge_item = [&](int idx, float2 (&ml)[kMaxMergeSplits], float4 (&o)[kMaxMergeSplits]) {
      const int r = idx / (TD / 4), c = (idx % (TD / 4)) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < kMaxMergeSplits; ++s) M = fmaxf(M, ml[s].x);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float Lsum = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxMergeSplits; ++s) {
        const float w = (ml[s].x == -INFINITY) ? 0.f : exp2f(ml[s].x - M);
        Lsum += w * ml[s].y;
        acc.x += w * o[s].x; acc.y += w * o[s].y; acc.z += w * o[s].z; acc.w += w * o[s].w;
      }
      // pairs with more splits than the unrolled window add the rest
      for (int s = kMaxMergeSplits; s < nsp; ++s) {
        const size_t row = pbase + (size_t)s * a.rpad + r;
        const float2 m2 = __ldcg(reinterpret_cast<const float2*>(a.part_ml + row * 2));
        const float4 o2 = __ldcg(reinterpret_cast<const float4*>(a.part_o + row * TD + c));
        if (m2.x > M) {
          const float sc = (M == -INFINITY) ? 0.f : exp2f(M - m2.x);
          acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
          Lsum *= sc;
          M = m2.x;
        }
        const float w = (m2.x == -INFINITY) ? 0.f : exp2f(m2.x - M);
        Lsum += w * m2.y;
        acc.x += w * o2.x; acc.y += w * o2.y; acc.z += w * o2.z; acc.w += w * o2.w;
      }
      const float inv = 1.0f / Lsum;
      const int t = r / a.G, gq = r % a.G;
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * TD + c) = u;
    };
    auto load_item = [&](int idx, float2 (&ml)[kMaxMergeSplits], float4 (&o)[kMaxMergeSplits]) {
      const int r = idx / (TD / 4), c = (idx % (TD / 4)) * 4;
#pragma unroll
      for (int s = 0; s < kMaxMergeSplits; ++s) {
        ml[s] = make_float2(-INFINITY, 0.f);
        o[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s == split) {
          ml[s] = *reinterpret_cast<const float2*>(pml + 2 * r);
          o[s] = *reinterpret_cast<const float4*>(po + r * OST + c);
        } else if (s < nsp) {
          const size_t row = pbase + (size_t)s * a.rpad + r;
          ml[s] = __ldcg(reinterpret_cast<const float2*>(a.part_ml + row * 2));
          o[s] = __ldcg(reinterpret_cast<const float4*>(a.part_o + row * TD + c));
        }
      }
    };
    const int nitems = a.R * (TD / 4);
    for (int idx = threadIdx.x; idx < nitems; idx += 2 * NT) {
      // two items' loads in flight before either is combined
      float2 ml0[kMaxMergeSplits], ml1[kMaxMergeSplits];
      float4 o0[kMaxMergeSplits], o1[kMaxMergeSplits];
      const int idx1 = idx + NT;
      load_item(idx, ml0, o0);
      if (idx1 < nitems) load_item(idx1, ml1, o1);
      merge_item(idx, ml0, o0);
      if (idx1 < nitems) merge_item(idx1, ml1, o1);
    }
    if (threadIdx.x == 0) a.counters[pair] = 0;  // ready for the next call
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
  CUtensorMap mq;
  if (!encode_pool_map(&mk, a.k_pool, a.num_pages, a.Hkv, TBLK, TD, &why) ||
      !encode_pool_map(&mv, a.v_pool, a.num_pages, a.Hkv, TBLK, TD, &why) ||
      !encode_q_map(&mq, a.q, a.B, a.T, a.Hq, a.G, TD, &why))
    return cudaErrorInvalidValue;
  const int ctas = a.B * a.Hkv * a.n_splits + a.split_extra;
  return launch_pdl(attend_tc_kernel<NSW, K::NS>, dim3(ctas), dim3(K::C::kThreads), K::C::kSmem,
                    st, mk, mv, mq, a);
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
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
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

int attend_tc_ctas_per_sm(const AttendArgs& a) {
  const int nsw = (a.R + 31) / 32;
  if (nsw <= 1) return occupancy_tc_cfg<1>();
  if (nsw <= 2) return occupancy_tc_cfg<2>();
  return occupancy_tc_cfg<4>();
}

cudaError_t launch_attend_tc(const AttendArgs& a, cudaStream_t st) {
  const int nsw = (a.R + 31) / 32;
  if (nsw <= 1) return launch_tc_cfg<1>(a, st);
  if (nsw <= 2) return launch_tc_cfg<2>(a, st);
  return launch_tc_cfg<4>(a, st);
}

}  // namespace sva
