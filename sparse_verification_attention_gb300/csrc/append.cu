// Acceptance write-back: after verification, each sequence's accepted drafts
// become ordinary context. Not a step the pages describe; it closes the
// verification loop (the next step's context is the old one plus the
// accepted drafts, and blocks that fill get representatives).
#include "internal.h"
#include "ptx.h"

namespace sva {
namespace {

constexpr int kAppendThreads = 64;

// grid (B, T, Hkv): CTA (b, i, h) copies draft accept_idx[b][i]'s K and V
// row of kv head h to position seq_ctx[b] + i of sequence b (i < n_accept[b]).
// Bad indices are skipped and flagged.
template <typename T>
__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const __grid_constant__ AppendArgs a) {
  const int b = blockIdx.x, i = blockIdx.y, h = blockIdx.z;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  const int n = min(max(a.n_accept[b], 0), a.T);
  if (i >= n) return;
  const int ctx = a.seq_ctx[b];
  const int u = a.accept_idx[(size_t)b * a.T + i];
  const int pos = ctx + i;
  const int j = pos / a.blk;
  int page = -1;
  if (ctx >= 0 && j < a.nb_max) page = a.block_table[(size_t)b * a.nb_max + j];
  const bool bad_idx = u < 0 || u >= a.T;
  const bool bad_page = page < 0 || page >= a.num_pages;
  if (bad_idx || bad_page) {
    if (a.status && threadIdx.x == 0)
      atomicOr(a.status, bad_idx ? SV_FLAG_BAD_BLOCK_INDEX : SV_FLAG_BAD_PAGE);
    return;
  }
  constexpr int VEC = 16 / sizeof(T);
  const size_t src = (((size_t)b * a.T + u) * a.Hkv + h) * a.d;
  const size_t dst = (((size_t)page * a.Hkv + h) * a.blk + pos % a.blk) * a.d;
  const uint4* sk = reinterpret_cast<const uint4*>(static_cast<const T*>(a.draft_k) + src);
  const uint4* sv = reinterpret_cast<const uint4*>(static_cast<const T*>(a.draft_v) + src);
  uint4* dk = reinterpret_cast<uint4*>(static_cast<T*>(a.k_pool) + dst);
  uint4* dv = reinterpret_cast<uint4*>(static_cast<T*>(a.v_pool) + dst);
  for (int c = threadIdx.x; c < a.d / VEC; c += kAppendThreads) {
    dk[c] = sk[c];
    dv[c] = sv[c];
  }
}

}  // namespace

cudaError_t launch_append_kv(const AppendArgs& a, int dtype, cudaStream_t st) {
  if (a.B == 0 || a.T == 0) return cudaSuccess;
  dim3 grid(a.B, a.T, a.Hkv);
  if (dtype == SV_BF16)
    return launch_pdl(append_kv_kernel<__nv_bfloat16>, grid, dim3(kAppendThreads), 0, st, a);
  return launch_pdl(append_kv_kernel<float>, grid, dim3(kAppendThreads), 0, st, a);
}

}  // namespace sva
