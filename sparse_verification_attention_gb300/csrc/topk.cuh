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
// Method: scores become order-preserving 32-bit keys in shared memory; a
// 4-pass MSB-first radix select (8-bit digits, shared histogram, warp-parallel
// suffix scan) finds the k-th largest key and how many keys equal to it are
// still needed; two CTA-wide prefix scans in index order then rank the ties
// (lower index first) and compact the kept indices in ascending order.
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
  uint32_t hist[256];
  uint32_t warp_tot[NT / 32 + 1];
  uint32_t digit, need;
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

// All NT threads of the CTA call this. sc: nb scores (global; read through
// L2 only, they may have been written by other CTAs of this grid); keys: nb
// words of shared memory; out: kmax entries (k kept indices ascending, then
// -1).
template <int NT>
__device__ void cta_topk(const float* sc, int nb, int k_req, int32_t* out, int kmax,
                         uint32_t* keys, TopkSmem<NT>& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = k_req < nb ? k_req : nb;
  for (int i = k + tid; i < kmax; i += NT) out[i] = -1;
  if (k == 0) return;
  if (k == nb) {
    for (int i = tid; i < nb; i += NT) out[i] = i;
    return;
  }
  for (int j = tid; j < nb; j += NT) keys[j] = order_key(__ldcg(sc + j));
  __syncthreads();

  uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) sm.hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < nb; j += NT) {
      const uint32_t key = keys[j];
      if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane L owns digits 255-8L-i (i = 0..7), highest digits first.
      uint32_t c[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = sm.hist[255 - 8 * lane - i];
        local += c[i];
      }
      uint32_t incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const uint32_t excl = incl - local;
      if (excl < need && need <= incl) {
        uint32_t cum = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + c[i] >= need) {
            sm.digit = 255u - 8u * lane - i;
            sm.need = need - cum;
            break;
          }
          cum += c[i];
        }
      }
    }
    __syncthreads();
    prefix |= sm.digit << shift;
    mask |= 0xFFu << shift;
    need = sm.need;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // key of the k-th largest score

  const int per = (nb + NT - 1) / NT;
  const int j0 = tid * per;
  const int j1 = min(nb, j0 + per);
  uint32_t ties = 0;
  for (int j = j0; j < j1; ++j) ties += (keys[j] == thr);
  const uint32_t tie_rank = cta_exclusive_scan<NT>(ties, sm.warp_tot);
  uint32_t kept = 0;
  {
    uint32_t tr = tie_rank;
    for (int j = j0; j < j1; ++j) {
      const uint32_t key = keys[j];
      if (key > thr) ++kept;
      else if (key == thr) { kept += (tr < need); ++tr; }
    }
  }
  uint32_t pos = cta_exclusive_scan<NT>(kept, sm.warp_tot);
  {
    uint32_t tr = tie_rank;
    for (int j = j0; j < j1; ++j) {
      const uint32_t key = keys[j];
      bool take = false;
      if (key > thr) take = true;
      else if (key == thr) { take = tr < need; ++tr; }
      if (take) out[pos++] = j;
    }
  }
}

}  // namespace sva
