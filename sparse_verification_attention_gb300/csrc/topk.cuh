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
// Method. Scores become order-preserving 32-bit keys held in registers, KPT
// per thread. Warp w owns the index range [w*32*KPT, (w+1)*32*KPT); lane l
// holds the indices w*32*KPT + 32*e + l for e < KPT, so every load is
// coalesced and index order inside a warp is (e, lane) order. KPT is a
// compile-time constant (cta_topk_fit picks the smallest that holds nb), so
// every per-key loop unrolls without branches and the independent loads and
// latency chains of a thread's keys overlap.
//
// Bucketed path (tried first). The scores are binned linearly over
// [min, max] into kTopkBins bins. The binning is monotone: a higher bin only
// holds strictly larger scores. One shared histogram and a suffix scan give
// the bin b* holding the k-th largest score. Every key above b* is kept, and
// every key below it is dropped. Order keys by the composite
// (key << 32 | ~index): a larger score first, then the lower index. The keys
// of b* (at most kTopkMaxCand) are ranked against each other by that
// composite. The one of rank k - (keys above b*) - 1 is the threshold T, and
// a key is kept if and only if its composite is >= T. Keys above b* pass and
// keys below it fail automatically. A boundary bin with more keys, equal
// scores everywhere, or non-finite extremes fall back to the radix search
// below.
//
// Radix search. The k-th largest key is found two bits
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

// The score an order key stands for (-0 comes back as +0).
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

constexpr int kTopkRadixBits = 2;
constexpr int kTopkCands = (1 << kTopkRadixBits) - 1;  // candidates per pass
constexpr int kTopkBins = 1024;                        // bucketed path: histogram bins
constexpr int kTopkMaxCand = 256;                      // largest boundary bin it ranks

// Bin of a key for scores in [lo, lo + kTopkBins / scale]: monotone in the
// key (rounded subtraction and multiplication are monotone, truncation of a
// non-negative value is a floor), and the same instructions wherever used.
__device__ __forceinline__ int key_bin(uint32_t key, float lo, float scale) {
  const float x = __fmul_rn(__fsub_rn(key_value(key), lo), scale);  // >= 0
  const int i = __float2int_rz(x);  // NaN gives 0; the clamps keep any value in range
  return i <= 0 ? 0 : (i < kTopkBins - 1 ? i : kTopkBins - 1);
}

template <int NT, int KPT>
struct TopkSmem {
  uint32_t cnt[2][kTopkCands][NT / 32];  // per-pass per-candidate per-warp counts
  uint32_t above[NT / 32], ties[NT / 32], kept[NT / 32];
  uint32_t wmin[NT / 32], wmax[NT / 32], wsum[NT / 32];
  uint32_t hist[kTopkBins];
  unsigned long long cand[kTopkMaxCand];  // composites of the boundary bin's keys
  unsigned long long thr;                 // the threshold composite T
  int bstar;
  uint32_t bstar_above, ncand;
};

// Optional second output of a selection: the pool row of every kept block,
// row = (page * Hkv + h) * blk with page = bt[index] (the first token row of
// that block's tile for KV head h), written beside the index; -1 (and
// SV_FLAG_BAD_PAGE) for a page outside [0, num_pages). The attention then
// needs one load per block instead of two dependent ones. bt == nullptr:
// no rows.
struct TopkRows {
  const int32_t* bt;  // block-table row of the sequence
  int32_t* out;       // kmax entries, beside the indices
  int Hkv, h, blk, num_pages;
  unsigned* status;   // may be null
};

__device__ __forceinline__ int32_t topk_row(const TopkRows& tr, int page) {
  if (page < 0 || page >= tr.num_pages) {
    if (tr.status) atomicOr(tr.status, SV_FLAG_BAD_PAGE);
    return -1;
  }
  return (page * tr.Hkv + tr.h) * tr.blk;
}

// Larger score first, then the lower index: (key << 32) | ~index.
__device__ __forceinline__ unsigned long long topk_composite(uint32_t key, int idx) {
  return ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)idx;
}

// All NT threads of the CTA call this once. sc: nb scores (global, read
// through L2 only: other CTAs of the grid may have just written them);
// nb <= NT * KPT <= NT * KMAX. out: kmax entries, the k kept indices
// ascending then -1.
template <int NT, int KPT, int KMAX>
__device__ void cta_topk(const float* sc, int nb, int k_req, int32_t* out, int kmax,
                         TopkSmem<NT, KMAX>& sm, const TopkRows& tr) {
  static_assert(KPT <= KMAX, "shared memory sized for fewer keys");
  constexpr int NW = NT / 32;
  constexpr int BPT = kTopkBins / NT;  // histogram bins per thread in the scan
  static_assert(kTopkBins % NT == 0 && NT >= kTopkMaxCand, "bucketed top-k layout");
  using Mask = std::conditional_t<(KPT > 32), unsigned long long, uint32_t>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = k_req < nb ? k_req : nb;
  for (int i = k + tid; i < kmax; i += NT) {
    out[i] = -1;
    if (tr.bt) tr.out[i] = -1;
  }
  if (k == 0) return;
  if (k == nb) {
    for (int i = tid; i < nb; i += NT) {
      out[i] = i;
      if (tr.bt) tr.out[i] = topk_row(tr, tr.bt[i]);
    }
    return;
  }
  const int wbase = warp * 32 * KPT;
  // With few keys per thread, every key's page is loaded beside its score (the
  // same round trip); with more, a kept key's page is loaded at the end.
  constexpr bool kPagesInRegs = KPT <= 8;
  int32_t pg[kPagesInRegs ? KPT : 1];
  // padding entries hold key 0, below every candidate tested
  uint32_t rk[KPT];
  Mask valid = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const int j = wbase + 32 * e + lane;
    const bool ok = j < nb;
    rk[e] = ok ? order_key(__ldcg(sc + j)) : 0u;
    if constexpr (kPagesInRegs) pg[e] = (ok && tr.bt) ? tr.bt[j] : -1;
    valid |= (Mask)(ok ? 1u : 0u) << e;
  }

  const unsigned lt = (1u << lane) - 1u;
  Mask keep = 0;
  bool done = false;

  // ---- bucketed path
  {
    uint32_t lmin = 0xffffffffu, lmax = 0u;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      if ((valid >> e) & 1u) {
        lmin = min(lmin, rk[e]);
        lmax = max(lmax, rk[e]);
      }
    }
    lmin = __reduce_min_sync(0xffffffffu, lmin);
    lmax = __reduce_max_sync(0xffffffffu, lmax);
    if (lane == 0) {
      sm.wmin[warp] = lmin;
      sm.wmax[warp] = lmax;
    }
    for (int i = tid; i < kTopkBins; i += NT) sm.hist[i] = 0u;
    if (tid == 0) {
      sm.ncand = 0u;
      sm.bstar = 0;  // overwritten below; a valid index whatever happens
      sm.bstar_above = 0u;
    }
    __syncthreads();
    uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      kmn = min(kmn, sm.wmin[w]);
      kmx = max(kmx, sm.wmax[w]);
    }
    const float lo = key_value(kmn);
    const float range = __fsub_rn(key_value(kmx), lo);
    const float scale = (float)kTopkBins / range;
    // the same decision in every thread: a finite, non-zero spread
    if (range > 0.f && scale > 0.f && scale <= 3.0e38f) {
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        if ((valid >> e) & 1u) atomicAdd(&sm.hist[key_bin(rk[e], lo, scale)], 1u);
      }
      __syncthreads();
      // suffix counts: thread t scans bins kTopkBins-1-BPT*t-j (j < BPT), so
      // thread order runs from the highest bin down
      uint32_t hb[BPT], s = 0;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        hb[j] = sm.hist[kTopkBins - 1 - BPT * tid - j];
        s += hb[j];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) sm.wsum[warp] = incl;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < NW; ++w) incl += (w < warp) ? sm.wsum[w] : 0u;
      uint32_t cum = incl - s;  // keys in bins above this thread's
      if (cum < (uint32_t)k && (uint32_t)k <= incl) {  // exactly one thread
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
          if (cum + hb[j] >= (uint32_t)k) {
            sm.bstar = kTopkBins - 1 - BPT * tid - j;
            sm.bstar_above = cum;
            break;
          }
          cum += hb[j];
        }
      }
      __syncthreads();
      const int bstar = sm.bstar;
      const uint32_t above = sm.bstar_above;
      if (sm.hist[bstar] <= (uint32_t)kTopkMaxCand) {  // same value in every thread
        // the keys of the boundary bin, in any order
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
          if (((valid >> e) & 1u) && key_bin(rk[e], lo, scale) == bstar) {
            const uint32_t slot = atomicAdd(&sm.ncand, 1u);
            if (slot < (uint32_t)kTopkMaxCand)
              sm.cand[slot] = topk_composite(rk[e], wbase + 32 * e + lane);
          }
        }
        __syncthreads();
        // the composites are distinct, so exactly one candidate has rank
        // need - 1 (need <= the bin's count)
        const uint32_t need = (uint32_t)k - above;  // >= 1
        const int nc = (int)min(sm.ncand, (uint32_t)kTopkMaxCand);
        if (tid < nc) {
          const unsigned long long c = sm.cand[tid];
          uint32_t rank = 0;
#pragma unroll 4
          for (int j = 0; j < nc; ++j) rank += (sm.cand[j] > c) ? 1u : 0u;
          if (rank == need - 1) sm.thr = c;
        }
        __syncthreads();
        const unsigned long long thr_c = sm.thr;
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
          const bool kp = ((valid >> e) & 1u) &&
                          topk_composite(rk[e], wbase + 32 * e + lane) >= thr_c;
          keep |= (Mask)(kp ? 1u : 0u) << e;
        }
        done = true;
      }
    }
  }

  if (!done) {
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

  if (exact) {  // exactly the keys >= thr
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool kp = ((valid >> e) & 1u) && rk[e] >= thr;
      keep |= (Mask)(kp ? 1u : 0u) << e;
    }
  } else {  // thr is the k-th largest key: keys above it, then ties by index
    uint32_t a_w = 0, t_w = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
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
      const bool v = (valid >> e) & 1u;
      const bool tie = v && rk[e] == thr;
      const unsigned b = __ballot_sync(0xffffffffu, tie);
      const bool kp = (v && rk[e] > thr) || (tie && rank + __popc(b & lt) < need);
      keep |= (Mask)(kp ? 1u : 0u) << e;
      rank += __popc(b);
    }
  }
  }  // radix search
  // compaction in index order: exactly k entries are kept
  uint32_t k_w = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    k_w += __popc(__ballot_sync(0xffffffffu, (keep >> e) & 1u));
  }
  if (lane == 0) sm.kept[warp] = k_w;
  __syncthreads();
  uint32_t pos = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) pos += (w < warp) ? sm.kept[w] : 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const bool kp = (keep >> e) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, kp);
    if (kp) {
      const int j = wbase + 32 * e + lane;
      const int at = pos + __popc(b & lt);
      out[at] = j;
      if (tr.bt) {
        if constexpr (kPagesInRegs) tr.out[at] = topk_row(tr, pg[e]);
        else tr.out[at] = topk_row(tr, tr.bt[j]);
      }
    }
    pos += __popc(b);
  }
}

// cta_topk with the fewest keys per thread that hold nb scores (the same
// choice in every thread of the CTA).
template <int NT, int KMAX>
__device__ void cta_topk_fit(const float* sc, int nb, int k_req, int32_t* out, int kmax,
                             TopkSmem<NT, KMAX>& sm, const TopkRows& tr) {
  if (KMAX > 4 && nb <= NT * 4)
    cta_topk<NT, (KMAX > 4 ? 4 : KMAX), KMAX>(sc, nb, k_req, out, kmax, sm, tr);
  else if (KMAX > 8 && nb <= NT * 8)
    cta_topk<NT, (KMAX > 8 ? 8 : KMAX), KMAX>(sc, nb, k_req, out, kmax, sm, tr);
  else
    cta_topk<NT, KMAX, KMAX>(sc, nb, k_req, out, kmax, sm, tr);
}

}  // namespace sva
