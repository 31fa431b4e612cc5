// Overlap of the block sets that each draft's own query would select: the
// measurement behind the figure that follows the Figure 1 caption on the
// paper summary page of "Accelerate Speculative Decoding with Sparse
// Computation in Verification" (the overlap ratio of the KV block selection
// for draft-token pairs at different position distances). It is the
// evidence that one shared set (draft 0's) serves every draft.
//
// One CTA per (sequence, KV head) pair. Every thread takes draft pairs (t, u)
// and counts |S_t ∩ S_u| with a two-pointer walk over the two ascending index
// lists. Sums are kept as integer counts, so the result does not depend on
// the order in which threads add them.
#include "internal.h"
#include "ptx.h"

namespace sva {
namespace {

constexpr int kOvThreads = 256;

__device__ int intersect_sorted(const int32_t* a, const int32_t* b, int n) {
  int i = 0, j = 0, c = 0;
  while (i < n && j < n) {
    const int x = a[i], y = b[j];
    c += (x == y) ? 1 : 0;
    i += (x <= y) ? 1 : 0;
    j += (y <= x) ? 1 : 0;
  }
  return c;
}

__global__ void __launch_bounds__(kOvThreads) overlap_kernel(const __grid_constant__ OverlapArgs a) {
  __shared__ unsigned long long csum[kMaxT];
  __shared__ unsigned cnt[kMaxT];
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x;
  for (int i = threadIdx.x; i < a.T; i += kOvThreads) {
    csum[i] = 0ull;
    cnt[i] = 0u;
  }
  __syncthreads();
  const size_t tstride = (size_t)a.pairs * a.kmax;
  const int32_t* base = a.sels + (size_t)p * a.kmax;
  for (int idx = threadIdx.x; idx < a.T * a.T; idx += kOvThreads) {
    const int t = idx / a.T, u = idx % a.T;
    if (t != 0 && u <= t) continue;  // draft 0 against every u, then pairs t < u
    const int c = intersect_sorted(base + t * tstride, base + u * tstride, a.k);
    if (t == 0) a.overlap0[(size_t)p * a.T + u] = (float)c / (float)a.k;
    if (t < u) {
      const int dd = a.depth[t] - a.depth[u];
      const int delta = dd < 0 ? -dd : dd;
      atomicAdd(&csum[delta], (unsigned long long)c);
      atomicAdd(&cnt[delta], 1u);
    }
  }
  __syncthreads();
  for (int dl = threadIdx.x; dl < a.T; dl += kOvThreads)
    a.by_distance[(size_t)p * a.T + dl] =
        cnt[dl] ? (float)((double)csum[dl] / ((double)cnt[dl] * a.k)) : __int_as_float(0x7fc00000);
}

}  // namespace

cudaError_t launch_overlap(const OverlapArgs& a, cudaStream_t st) {
  if (a.pairs == 0) return cudaSuccess;
  return launch_pdl(overlap_kernel, dim3(a.pairs), dim3(kOvThreads), 0, st, a);
}

}  // namespace sva
