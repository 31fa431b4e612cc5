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
// Method. Scores become order-preserving 32-bit keys held in registers. Warp
// w owns the index range [w*32*per, (w+1)*32*per); lane l holds the indices
// w*32*per + 32*e + l for e < per, so every load is coalesced and index order
// inside a warp is (e, lane) order. The k-th largest key is found two bits
// per pass from the most significant end: each warp counts its keys at or
// above the three candidates that extend the current prefix, the per-warp
// counts meet in shared memory behind one barrier, and every warp picks the
// same digit from them. The search stops as soon as exactly k keys lie at or
// above the prefix found so far (the kept set is then known and has no
// ties). Otherwise the keys above the k-th largest are kept, and keys equal
// to it are kept in index order until k are kept. Tie ranks and output
// positions come from warp ballots plus per-warp totals (one barrier each).
#pragma once

#include <type_traits>

#include "internal.h"

namespace sva {

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) f = 0.0f;  // -0 and +0 tie
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkRadixBits = 2;
constexpr int kTopkCands = (1 << kTopkRadixBits) - 1;  // candidates per pass

template <int NT>
struct TopkSmem {
  uint32_t cnt[2][kTopkCands][NT / 32];  // per-pass per-candidate per-warp counts
  uint32_t above[NT / 32], ties[NT / 32], kept[NT / 32];
};

// All NT threads of the CTA call this once. sc: nb scores (global, read
// through L2 only: other CTAs of the grid may have just written them);
// nb <= NT * KPT. out: kmax entries, the k kept indices ascending then -1.
template <int NT, int KPT>
__device__ void cta_topk(const float* sc, int nb, int k_req, int32_t* out, int kmax,
                         TopkSmem<NT>& sm) {
  constexpr int NW = NT / 32;
  using Mask = std::conditional_t<(KPT > 32), unsigned long long, uint32_t>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = k_req < nb ? k_req : nb;
  for (int i = k + tid; i < kmax; i += NT) out[i] = -1;
  if (k == 0) return;
  if (k == nb) {
    for (int i = tid; i < nb; i += NT) out[i] = i;
    return;
  }
  const int per = (nb + NT - 1) / NT;
  const int wbase = warp * 32 * per;
  // padding entries hold key 0, below every candidate tested
  uint32_t rk[KPT];
  Mask valid = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const int j = wbase + 32 * e + lane;
    const bool ok = e < per && j < nb;
    rk[e] = ok ? order_key(__ldcg(sc + j)) : 0u;
    valid |= (Mask)(ok ? 1u : 0u) << e;
  }

  // k-th largest key, two bits per pass: thr holds the digits found so far
  // (lower bits zero), cnt = #keys >= thr.
  uint32_t thr = 0, cnt = (uint32_t)nb;
  bool exact = false;
  int p = 0;
  for (int shift = 32 - kTopkRadixBits; shift >= 0; shift -= kTopkRadixBits, ++p) {
    const uint32_t P = thr >> shift;  // low kTopkRadixBits bits are zero
    uint32_t c[kTopkCands];
#pragma unroll
    for (int v = 0; v < kTopkCands; ++v) c[v] = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if (e >= per) break;
      const uint32_t dk = rk[e] >> shift;
#pragma unroll
      for (int v = 0; v < kTopkCands; ++v) c[v] += (dk >= P + (uint32_t)(v + 1));
    }
    uint32_t mine = 0;
#pragma unroll
    for (int v = 0; v < kTopkCands; ++v) {
      const uint32_t s = __reduce_add_sync(0xffffffffu, c[v]);
      if (lane == v) mine = s;
    }
    // double-buffered: a warp can only rewrite this buffer two passes on,
    // after every warp has passed the next barrier (and so read this one)
    if (lane < kTopkCands) sm.cnt[p & 1][lane][warp] = mine;
    __syncthreads();
    uint32_t tot = 0;
    if (lane < kTopkCands) {
#pragma unroll
      for (int w = 0; w < NW; ++w) tot += sm.cnt[p & 1][lane][w];
    }
    // counts fall with the candidate: the lanes meeting k form a prefix
    const int dig = __popc(__ballot_sync(0xffffffffu, lane < kTopkCands && tot >= (uint32_t)k));
    const uint32_t tdig = __shfl_sync(0xffffffffu, tot, dig > 0 ? dig - 1 : 0);
    if (dig) {
      thr |= (uint32_t)dig << shift;
      cnt = tdig;
    }
    if (cnt == (uint32_t)k) {  // same decision in every thread
      exact = true;
      break;
    }
  }

  const unsigned lt = (1u << lane) - 1u;
  Mask keep = 0;
  if (exact) {  // exactly the keys >= thr
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if (e >= per) break;
      const bool kp = ((valid >> e) & 1u) && rk[e] >= thr;
      keep |= (Mask)(kp ? 1u : 0u) << e;
    }
  } else {  // thr is the k-th largest key: keys above it, then ties by index
    uint32_t a_w = 0, t_w = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if (e >= per) break;
      const bool v = (valid >> e) & 1u;
      a_w += __popc(__ballot_sync(0xffffffffu, v && rk[e] > thr));
      t_w += __popc(__ballot_sync(0xffffffffu, v && rk[e] == thr));
    }
    if (lane == 0) {
      sm.above[warp] = a_w;
      sm.ties[warp] = t_w;
    }
    __syncthreads();
    uint32_t above = 0, rank = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      above += sm.above[w];
      rank += (w < warp) ? sm.ties[w] : 0u;
    }
    const uint32_t need = (uint32_t)k - above;  // >= 1: thr is the k-th largest
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if (e >= per) break;
      const bool v = (valid >> e) & 1u;
      const bool tie = v && rk[e] == thr;
      const unsigned b = __ballot_sync(0xffffffffu, tie);
      const bool kp = (v && rk[e] > thr) || (tie && rank + __popc(b & lt) < need);
      keep |= (Mask)(kp ? 1u : 0u) << e;
      rank += __popc(b);
    }
  }
  // compaction in index order: exactly k entries are kept
  uint32_t k_w = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if (e >= per) break;
    k_w += __popc(__ballot_sync(0xffffffffu, (keep >> e) & 1u));
  }
  if (lane == 0) sm.kept[warp] = k_w;
  __syncthreads();
  uint32_t pos = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) pos += (w < warp) ? sm.kept[w] : 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if (e >= per) break;
    const bool kp = (keep >> e) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, kp);
    if (kp) out[pos + __popc(b & lt)] = wbase + 32 * e + lane;
    pos += __popc(b);
  }
}

}  // namespace sva
