// Top-k block selection per (sequence, kv head).
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: the most relevant
// blocks by representative score are kept and shared by every draft token.
// [SV-Tut1] tutorial page, core technique 1: the number kept is the budget.
// Ties go to the lower block index (this library's reading); the kept set is
// written in ascending block order.
//
// Method: one CTA per (b, h). Scores become order-preserving 32-bit keys in
// shared memory; a 4-pass MSB-first radix select (8-bit digits, shared
// histogram, warp-parallel suffix scan) finds the k-th largest key and how
// many keys equal to it are still needed; two block-wide prefix scans in
// index order then rank the ties (lower index first) and compact the kept
// indices in ascending order.
#include <atomic>

#include "internal.h"

namespace sva {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.0f) f = 0.0f;  // -0 and +0 tie
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the CTA in thread order; also returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t* total) {
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
    uint32_t w = lane < kSelWarps ? warp_tot[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kSelWarps) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == kSelWarps - 1) warp_tot[kSelWarps] = wi;
  }
  __syncthreads();
  const uint32_t res = warp_tot[warp] + incl - v;
  *total = warp_tot[kSelWarps];
  __syncthreads();  // warp_tot is reused by the next scan
  return res;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[kSelWarps + 1];
  __shared__ uint32_t s_digit, s_need;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x;
  const int nb = a.nb;
  const int k = a.k < nb ? a.k : nb;
  const float* sc = a.scores + (size_t)pair * nb;
  int32_t* out = a.sel + (size_t)pair * a.kmax;

  for (int i = k + tid; i < a.kmax; i += kSelThreads) out[i] = -1;
  if (k == 0) return;
  if (k == nb) {
    for (int i = tid; i < nb; i += kSelThreads) out[i] = i;
    return;
  }
  for (int j = tid; j < nb; j += kSelThreads) keys[j] = order_key(sc[j]);
  __syncthreads();

  uint32_t prefix = 0, mask = 0;
  uint32_t need = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < nb; j += kSelThreads) {
      const uint32_t key = keys[j];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane L owns digits 255-8L-i (i = 0..7), highest digits first.
      uint32_t c[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
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
            s_digit = 255u - 8u * lane - i;
            s_need = need - cum;
            break;
          }
          cum += c[i];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 0xFFu << shift;
    need = s_need;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // key of the k-th largest score

  // Contiguous chunk per thread keeps the scans in index order.
  const int per = (nb + kSelThreads - 1) / kSelThreads;
  const int j0 = tid * per;
  const int j1 = min(nb, j0 + per);
  uint32_t ties = 0;
  for (int j = j0; j < j1; ++j) ties += (keys[j] == thr);
  uint32_t total;
  uint32_t tie_rank = block_exclusive_scan(ties, warp_tot, &total);
  uint32_t kept = 0;
  {
    uint32_t tr = tie_rank;
    for (int j = j0; j < j1; ++j) {
      const uint32_t key = keys[j];
      if (key > thr) ++kept;
      else if (key == thr) { kept += (tr < need); ++tr; }
    }
  }
  uint32_t pos = block_exclusive_scan(kept, warp_tot, &total);
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

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  if (a.pairs == 0) return cudaSuccess;
  const size_t smem = (size_t)(a.nb > 0 ? a.nb : 1) * sizeof(uint32_t);
  static std::atomic<int> attr_set[kMaxDevices];
  const int dev = current_device();
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kMaxNB * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1);
  }
  select_kernel<<<a.pairs, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sva
