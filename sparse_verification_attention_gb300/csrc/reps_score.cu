// Block representatives and block importance scores.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: blocks are chosen by
// the dot product between the first draft token's query and a representative
// value of each KV block. The representative is read here as the mean of the
// block's keys, accumulated in fp32.
#include <atomic>

#include "internal.h"
#include "ptx.h"
#include "topk.cuh"

namespace sva {
namespace {

// Loads 4 consecutive elements as fp32 (8 bytes for bf16, 16 for fp32).
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}

// ------------------------------------------------------------------ reps
// One CTA of kRepThreads per (logical block, kv head, sequence). Thread t owns
// one 16-byte chunk of the head dimension (c = t % chunks) and one group of
// tokens (g = t / chunks); each group sums its tokens in order, then the
// groups are added in order through shared memory. All of a page's 16-byte
// loads are independent, so the block is read in one memory round trip.
constexpr int kRepThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kRepThreads) build_reps_kernel(RepsArgs a) {
  constexpr int VEC = 16 / sizeof(T);  // elements per 16-byte chunk
  __shared__ float part[kRepThreads * VEC];
  const int j = a.first_block + blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int chunks = a.d / VEC;
  const int groups = kRepThreads / chunks;  // >= 1 since d <= 256
  const int c = threadIdx.x % chunks, g = threadIdx.x / chunks;
  pdl_wait();
  const int page = a.block_table[(size_t)b * a.nb_max + j];
  float* dst = a.reps + (((size_t)b * a.Hkv + h) * a.nb_max + j) * a.d;
  if (page < 0 || page >= a.num_pages) {
    if (a.status && threadIdx.x == 0) atomicOr(a.status, SV_FLAG_BAD_PAGE);
    for (int i = threadIdx.x; i < a.d; i += kRepThreads) dst[i] = 0.f;
    return;
  }
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  if (g < groups) {
    const T* src = static_cast<const T*>(a.k_pool) + ((size_t)page * a.Hkv + h) * a.blk * a.d;
    const int per = (a.blk + groups - 1) / groups;
    const int t0 = g * per, t1 = min(a.blk, t0 + per);
    for (int t = t0; t < t1; ++t) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + (size_t)t * a.d) + c);
      const T* v = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        if constexpr (sizeof(T) == 2) acc[e] += __bfloat162float(v[e]);
        else acc[e] += v[e];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) part[threadIdx.x * VEC + e] = acc[e];
  __syncthreads();
  const float inv = 1.0f / (float)a.blk;
  for (int i = threadIdx.x; i < a.d; i += kRepThreads) {
    const int ci = i / VEC, ei = i % VEC;
    float sum = 0.f;
    for (int gg = 0; gg < groups; ++gg) sum += part[(gg * chunks + ci) * VEC + ei];
    dst[i] = sum * inv;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------ scores
// grid = (ceil(nb / kRowsPerCta), B*Hkv). Each warp streams whole fp32
// representative rows with 128-bit loads (lane c holds dims 4c..4c+3), dots
// them with the group-summed draft-0 query held in registers, and reduces
// across the warp. Rows are processed kUnroll at a time so that every lane
// keeps several independent 16-byte loads in flight.
constexpr int kScoreWarps = 8;
constexpr int kUnroll = 8;
constexpr int kRowsPerWarp = 8;
constexpr int kRowsPerCta = kScoreWarps * kRowsPerWarp;
constexpr int kMaxChunks = kMaxD / 4 / 32;  // float4 chunks per lane (d <= 256)

template <typename T>
__global__ void __launch_bounds__(kScoreWarps * 32) score_kernel(const __grid_constant__ ScoreArgs a) {
  const int pair = blockIdx.y;  // b * Hkv + h
  const int b = pair / a.Hkv, h = pair % a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunk = a.d / 4;
  pdl_wait();

  // qhat = sum over the G query heads of KV head h of draft 0's query.
  float4 qh[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    qh[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int ch = lane + 32 * c;
    if (ch < nchunk) {
      const T* q0 = static_cast<const T*>(a.q) + ((size_t)b * a.T * a.Hq + (size_t)h * a.G) * a.d;
      for (int g = 0; g < a.G; ++g) {
        float4 v = load4<T>(q0 + (size_t)g * a.d + ch * 4);
        qh[c].x += v.x; qh[c].y += v.y; qh[c].z += v.z; qh[c].w += v.w;
      }
    }
  }

  const float* rep0 = a.reps + (size_t)pair * a.nb_max * a.d;
  const int row0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
#pragma unroll
  for (int it = 0; it < kRowsPerWarp; it += kUnroll) {
    float acc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      acc[u] = 0.f;
      const int j = row0 + it + u;
      if (j < a.nb) {
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          const int ch = lane + 32 * c;
          if (ch < nchunk) {
            float4 r = __ldg(reinterpret_cast<const float4*>(rep0 + (size_t)j * a.d) + ch);
            acc[u] = fmaf(qh[c].x, r.x, acc[u]);
            acc[u] = fmaf(qh[c].y, r.y, acc[u]);
            acc[u] = fmaf(qh[c].z, r.z, acc[u]);
            acc[u] = fmaf(qh[c].w, r.w, acc[u]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
      const int j = row0 + it + u;
      if (lane == 0 && j < a.nb) a.scores[(size_t)pair * a.nb + j] = acc[u];
    }
  }
  if (!a.sel) {
    pdl_trigger();
    return;
  }

  // Fused selection: the last CTA to finish scoring this (b, h) selects.
  __shared__ unsigned s_last;
  __shared__ TopkSmem<kScoreWarps * 32> tsm;
  extern __shared__ uint32_t keys[];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.counters[pair], 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    cta_topk<kScoreWarps * 32, 16>(a.scores + (size_t)pair * a.nb, a.nb, a.k,
                                   a.sel + (size_t)pair * a.kmax, a.kmax, keys, tsm);
    if (threadIdx.x == 0) a.counters[pair] = 0;  // ready for the next call
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_build_reps(const RepsArgs& a, int dtype, cudaStream_t st) {
  if (a.n_blocks == 0) return cudaSuccess;
  dim3 grid(a.n_blocks, a.Hkv, a.B);
  if (dtype == SV_BF16)
    return launch_pdl(build_reps_kernel<__nv_bfloat16>, grid, dim3(kRepThreads), 0, st, a);
  return launch_pdl(build_reps_kernel<float>, grid, dim3(kRepThreads), 0, st, a);
}

cudaError_t launch_score(const ScoreArgs& a, int dtype, cudaStream_t st) {
  if (a.nb == 0) return cudaSuccess;
  dim3 grid((a.nb + kRowsPerCta - 1) / kRowsPerCta, a.B * a.Hkv);
  const size_t smem = a.sel ? (size_t)a.nb * sizeof(uint32_t) : 0;
  auto kern = (dtype == SV_BF16) ? score_kernel<__nv_bfloat16> : score_kernel<float>;
  static std::atomic<int> attr_set[kMaxDevices][2];
  const int dev = current_device();
  const int which = dtype == SV_BF16 ? 0 : 1;
  if (!attr_set[dev][which].load()) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kMaxNB * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set[dev][which].store(1);
  }
  return launch_pdl(kern, grid, dim3(kScoreWarps * 32), smem, st, a);
}

}  // namespace sva
