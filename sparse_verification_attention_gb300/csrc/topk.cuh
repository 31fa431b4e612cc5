// CTA-wide top-k block selection, shared by the standalone select kernel and
// the fused score+select kernel.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: the blocks with the
// highest representative scores are kept, one set shared by every draft.
// [SV-Tut1] tutorial page, core technique 1: the number kept is the budget.
// Ties go to the lower block index (this library's reading); the kept set is
// written in ascending block order.
//
// Method: scores become order-preserving 32-bit keys, held in registers (each
// thread owns a contiguous run of block indices; shared memory when nb is
// too large). The k-th largest key is found bit by bit from the most
// significant bit: a candidate with the next bit set is kept when at least k
// keys are >= it; each pass is one CTA-wide count (register compares, a warp
// reduction, one shared atomic per warp, one barrier). Two CTA-wide prefix
// scans in index order then rank the keys equal to the threshold (lower
// index first) and compact the kept indices in ascending order.
#pragma once

#include "internal.h"

namespace sva {

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) f = 0.0f;  // -0 and +0 tie
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int NT>
struct TopkSmem {
  uint32_t cnt[3];  // per-pass CTA count, triple-buffered (reset two passes ahead)
  uint32_t warp_tot[NT / 32 + 1];
};

// Exclusive prefix sum over the CTA in thread order.
template <int NT>
__device__ __forceinline__ uint32_t cta_exclusive_scan(uint32_t v, uint32_t* warp_tot) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < NW ? warp_tot[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < NW) warp_tot[lane] = wi - w;
  }
  __syncthreads();
  const uint32_t res = warp_tot[warp] + incl - v;
  __syncthreads();
  return res;
}

// CTA-wide count of predicate hits (all NT threads call it; pass index p
// selects the buffer; one barrier).
template <int NT>
__device__ __forceinline__ uint32_t cta_count(uint32_t c, int p, TopkSmem<NT>& sm) {
  c = __reduce_add_sync(0xffffffffu, c);
  if (threadIdx.x == 0) sm.cnt[(p + 1) % 3] = 0;  // last read two passes ago
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(&sm.cnt[p % 3], c);
  __syncthreads();
  return sm.cnt[p % 3];
}

// All NT threads of the CTA call this. sc: nb scores (global; read through
// L2 only, they may have been written by other CTAs of this grid); keys: nb
// words of shared memory (used only when nb > NT * KPT); out: kmax entries
// (k kept indices ascending, then -1).
template <int NT, int KPT>
__device__ void cta_topk(const float* sc, int nb, int k_req, int32_t* out, int kmax,
                         uint32_t* keys, TopkSmem<NT>& sm) {
  const int tid = threadIdx.x;
  const int k = k_req < nb ? k_req : nb;
  for (int i = k + tid; i < kmax; i += NT) out[i] = -1;
  if (k == 0) return;
  if (k == nb) {
    for (int i = tid; i < nb; i += NT) out[i] = i;
    return;
  }
  // thread t owns block indices [j0, j1) in order
  const int per = (nb + NT - 1) / NT;
  const int j0 = min(nb, tid * per);
  const int j1 = min(nb, j0 + per);
  const bool in_regs = per <= KPT;
  uint32_t rk[KPT];
  if (in_regs) {
#pragma unroll
    for (int e = 0; e < KPT; ++e) rk[e] = (j0 + e < j1) ? order_key(__ldcg(sc + j0 + e)) : 0u;
  } else {
    for (int j = tid; j < nb; j += NT) keys[j] = order_key(__ldcg(sc + j));
  }
  if (tid == 0) sm.cnt[0] = sm.cnt[1] = sm.cnt[2] = 0;
  __syncthreads();
  // padding slots hold key 0, the smallest possible key: counting keys >= a
  // candidate with its top bit set never counts them, and the candidate 0 is
  // never tested.
  auto count_ge = [&](uint32_t cand) {
    uint32_t c = 0;
    if (in_regs) {
#pragma unroll
      for (int e = 0; e < KPT; ++e) c += (rk[e] >= cand);
    } else {
      for (int j = j0; j < j1; ++j) c += (keys[j] >= cand);
    }
    return c;
  };
  // k-th largest key: the largest v with #(key >= v) >= k, built bit by bit.
  uint32_t thr = 0;
  int p = 0;
  for (int bit = 31; bit >= 0; --bit, ++p) {
    const uint32_t cand = thr | (1u << bit);
    if (cta_count<NT>(count_ge(cand), p, sm) >= (uint32_t)k) thr = cand;
  }
  // keys strictly above the threshold are all kept; `need` keys equal to it
  uint32_t above = 0, ties = 0;
  if (in_regs) {
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if (j0 + e < j1) {
        above += (rk[e] > thr);
        ties += (rk[e] == thr);
      }
    }
  } else {
    for (int j = j0; j < j1; ++j) {
      above += (keys[j] > thr);
      ties += (keys[j] == thr);
    }
  }
  const uint32_t need = (uint32_t)k - cta_count<NT>(above, p, sm);
  const uint32_t tie_rank = cta_exclusive_scan<NT>(ties, sm.warp_tot);
  // kept entries of this thread's run, in index order (ties: lower index first)
  auto keep = [&](uint32_t key, uint32_t& tr) {
    if (key > thr) return true;
    if (key == thr) return tr++ < need;
    return false;
  };
  uint32_t kept = 0;
  {
    uint32_t tr = tie_rank;
    if (in_regs) {
#pragma unroll
      for (int e = 0; e < KPT; ++e)
        if (j0 + e < j1) kept += keep(rk[e], tr);
    } else {
      for (int j = j0; j < j1; ++j) kept += keep(keys[j], tr);
    }
  }
  uint32_t pos = cta_exclusive_scan<NT>(kept, sm.warp_tot);
  {
    uint32_t tr = tie_rank;
    if (in_regs) {
#pragma unroll
      for (int e = 0; e < KPT; ++e)
        if (j0 + e < j1 && keep(rk[e], tr)) out[pos++] = j0 + e;
    } else {
      for (int j = j0; j < j1; ++j)
        if (keep(keys[j], tr)) out[pos++] = j;
    }
  }
}

}  // namespace sva
