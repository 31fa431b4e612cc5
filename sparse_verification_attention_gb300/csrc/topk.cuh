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
// Bucketed path (tried first). The keys are binned by their offset from
// the smallest key, (key - min key) >> shift, with shift the smallest that
// leaves at most kTopkBins bins. Order keys follow the float bit patterns, so
// the bins are about logarithmic in the score: a few far-out scores (an
// attention sink, strongly planted blocks) do not squeeze the bulk of the
// scores into a handful of bins, as bins linear in the score would. The
// binning is monotone: a higher bin only holds strictly larger keys. One
// shared histogram and a suffix scan give the bin b* holding the k-th
// largest key. Every key above b* is kept, and every key below it is
// dropped. Order keys by the composite (key << 32 | ~index): a larger score
// first, then the lower index. The keys of b* (at most kTopkMaxCand) are
// ranked against each other by that composite. The one of rank
// k - (keys above b*) - 1 is the threshold T, and a key is kept if and only
// if its composite is >= T. Keys above b* pass and keys below it fail
// automatically. A boundary bin with more than kTopkRankCand keys is
// refined first: its key range becomes the next histogram's range (bins
// 2^10 times narrower), and so on down to single keys. A boundary bin that
// still holds more than kTopkMaxCand keys (many equal scores), or equal keys
// everywhere, falls back to the radix search below.
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
constexpr int kTopkRankCand = 48;                      // larger boundary bins are refined
constexpr int kTopkBinBits = 10;                       // kTopkBins = 2^kTopkBinBits

// Bin of a key k >= kmin: (k - kmin) >> shift, monotone in the key.
__device__ __forceinline__ int key_bin(uint32_t key, uint32_t kmin, int shift) {
  return (int)((key - kmin) >> shift);
}

// Smallest shift that maps [0, span] into kTopkBins bins.
__device__ __forceinline__ int key_bin_shift(uint32_t span) {
  static_assert((1 << kTopkBinBits) == kTopkBins, "bin count is a power of two");
  const int bits = 32 - __clz(span);  // significant bits of span (0 for span 0)
  return bits > kTopkBinBits ? bits - kTopkBinBits : 0;
}

template <int NT, int KPT>
struct TopkSmem {
  uint32_t cnt[2][kTopkCands][NT / 32];  // per-pass per-candidate per-warp counts
  uint32_t above[NT / 32], ties[NT / 32], kept[NT / 32];
  uint32_t wmin[NT / 32], wmax[NT / 32], wsum[NT / 32];
  uint32_t hist[2][kTopkBins];  // two levels in flight: one filled, one zeroed
  unsigned long long cand[kTopkMaxCand];  // composites of the boundary bin's keys
  unsigned long long thr;                 // the threshold composite T
  int bstar;
  uint32_t bstar_above, bstar_cnt, ncand;
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
    if constexpr (kPagesInRegs) {
      // issued here, beside the scores, and not where the pages are used
      pg[e] = -1;
      if (ok && tr.bt) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(pg[e]) : "l"(tr.bt + j));
    }
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
    for (int i = tid; i < kTopkBins; i += NT) sm.hist[0][i] = 0u;
    if (tid == 0) {
      sm.ncand = 0u;
      sm.bstar = 0;  // overwritten below; valid values whatever happens
      sm.bstar_above = 0u;
      sm.bstar_cnt = 0xffffffffu;
    }
    __syncthreads();
    uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      kmn = min(kmn, sm.wmin[w]);
      kmx = max(kmx, sm.wmax[w]);
    }
    // the same decision in every thread: keys that are not all equal
    if (kmx > kmn) {
      // window of keys [lo, lo + (kTopkBins << shift)); `above` keys lie
      // above it; the k-th largest key is inside it
      uint32_t lo = kmn, above = 0u, cnt = 0u;
      int shift = key_bin_shift(kmx - kmn), bstar = 0;
      for (int level = 0;; ++level) {
        uint32_t* hist = sm.hist[level & 1];
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
          if (((valid >> e) & 1u) && rk[e] >= lo) {
            const uint32_t bin = (rk[e] - lo) >> shift;
            if (bin < (uint32_t)kTopkBins) atomicAdd(&hist[bin], 1u);
          }
        }
        // the other histogram is free (its last reader passed the barrier
        // that published the previous level's boundary bin)
        for (int i = tid; i < kTopkBins; i += NT) sm.hist[(level + 1) & 1][i] = 0u;
        __syncthreads();
        // suffix counts: thread t scans bins kTopkBins-1-BPT*t-j (j < BPT), so
        // thread order runs from the highest bin down
        uint32_t hb[BPT], s = 0;
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
          hb[j] = hist[kTopkBins - 1 - BPT * tid - j];
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
        uint32_t cum = incl - s;  // window keys in bins above this thread's
        const uint32_t need = (uint32_t)k - above;  // >= 1, <= the window's keys
        if (cum < need && need <= incl) {  // exactly one thread
#pragma unroll
          for (int j = 0; j < BPT; ++j) {
            if (cum + hb[j] >= need) {
              sm.bstar = kTopkBins - 1 - BPT * tid - j;
              sm.bstar_above = above + cum;
              sm.bstar_cnt = hb[j];
              break;
            }
            cum += hb[j];
          }
        }
        __syncthreads();
        bstar = sm.bstar;
        above = sm.bstar_above;
        cnt = sm.bstar_cnt;
        // refine while the boundary bin is too full to rank cheaply
        if (cnt <= (uint32_t)kTopkRankCand || shift == 0) break;
        lo += (uint32_t)bstar << shift;
        shift = shift > kTopkBinBits ? shift - kTopkBinBits : 0;
      }
      if (cnt <= (uint32_t)kTopkMaxCand) {  // same value in every thread
        // the keys of the boundary bin, in any order: one shared-memory
        // atomic per warp reserves all of the warp's places
        unsigned bal[KPT];
        uint32_t nw = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
          bal[e] = __ballot_sync(0xffffffffu, ((valid >> e) & 1u) && rk[e] >= lo &&
                                                  ((rk[e] - lo) >> shift) == (uint32_t)bstar);
          nw += (uint32_t)__popc(bal[e]);
        }
        if (nw) {
          uint32_t base = 0;
          if (lane == 0) base = atomicAdd(&sm.ncand, nw);
          base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
          for (int e = 0; e < KPT; ++e) {
            const uint32_t slot = base + __popc(bal[e] & lt);
            if (((bal[e] >> lane) & 1u) && slot < (uint32_t)kTopkMaxCand)
              sm.cand[slot] = topk_composite(rk[e], wbase + 32 * e + lane);
            base += (uint32_t)__popc(bal[e]);
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
