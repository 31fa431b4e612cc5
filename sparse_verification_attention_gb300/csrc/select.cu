// Top-k block selection per (sequence, kv head).
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: the most relevant
// blocks by representative score are kept and shared by every draft token.
// [SV-Tut1] tutorial page, core technique 1: the number kept is the budget.
// Ties go to the lower block index (this library's reading); the kept set is
// written in ascending block order.
//
// Method: one CTA per (b, h) running the CTA top-k of topk.cuh with every
// score held in registers (512 threads x 32 keys covers the largest block
// count the library accepts; smaller counts take 4 or 8 keys per thread).
#include "internal.h"
#include "ptx.h"
#include "topk.cuh"

namespace sva {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelKeys = kMaxNB / kSelThreads;  // keys per thread
static_assert(kSelThreads * kSelKeys >= kMaxNB, "select must hold every score");

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const __grid_constant__ SelectArgs a) {
  __shared__ TopkSmem<kSelThreads, kSelKeys> tsm;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  const int pair = blockIdx.x, b = pair / a.Hkv;
  const TopkRows tr{a.block_table ? a.block_table + (size_t)b * a.nb_max : nullptr,
                    a.rows ? a.rows + (size_t)pair * a.kmax : nullptr, a.Hkv, pair % a.Hkv,
                    a.blk, a.num_pages, a.status};
  cta_topk_fit<kSelThreads, kSelKeys>(a.scores + (size_t)pair * a.nb, nb_of(a.vl, b, a.nb),
                                  n_of(a.vl, b, a.k), a.sel + (size_t)pair * a.kmax, a.kmax, tsm,
                                  tr);
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  if (a.pairs == 0) return cudaSuccess;
  return launch_pdl(select_kernel, dim3(a.pairs), dim3(kSelThreads), 0, st, a);
}

}  // namespace sva
