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
#include "ptx.h"
#include "topk.cuh"

namespace sva {
namespace {

constexpr int kSelThreads = 512;

__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelectArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ TopkSmem<kSelThreads> tsm;
  pdl_wait();
  const int pair = blockIdx.x;
  cta_topk<kSelThreads, 8>(a.scores + (size_t)pair * a.nb, a.nb, a.k,
                           a.sel + (size_t)pair * a.kmax, a.kmax, keys, tsm);
  pdl_trigger();
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
  return launch_pdl(select_kernel, dim3(a.pairs), dim3(kSelThreads), smem, st, a);
}

}  // namespace sva
