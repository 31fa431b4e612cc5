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
// groups are added in order through shared memory. A thread issues the loads
// of up to kRepBatch tokens before summing them, so a block of up to
// kRepBatch tokens per group is read in one memory round trip.
constexpr int kRepThreads = 128;
constexpr int kRepBatch = 8;  // token loads in flight per thread

// Representative of logical block j of (sequence b, kv head h); all
// kRepThreads threads of the CTA call it (part: kRepThreads * VEC floats of
// shared memory).
template <typename T>
__device__ void block_rep(const RepsArgs& a, int b, int h, int j, float* part) {
  constexpr int VEC = 16 / sizeof(T);  // elements per 16-byte chunk
  const int chunks = a.d / VEC;
  const int groups = kRepThreads / chunks;  // >= 1 since d <= 256
  const int c = threadIdx.x % chunks, g = threadIdx.x / chunks;
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
    // kRepBatch tokens' loads are issued before any is summed, so a group
    // of up to kRepBatch tokens costs one memory round trip
    for (int tb = t0; tb < t1; tb += kRepBatch) {
      uint4 u[kRepBatch];
#pragma unroll
      for (int i = 0; i < kRepBatch; ++i)
        u[i] = (tb + i < t1) ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)(tb + i) * a.d) + c)
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < kRepBatch; ++i) {
        if (tb + i >= t1) break;
        const T* v = reinterpret_cast<const T*>(&u[i]);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          if constexpr (sizeof(T) == 2) acc[e] += __bfloat162float(v[e]);
          else acc[e] += v[e];
        }
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
}

template <typename T>
__global__ void __launch_bounds__(kRepThreads) build_reps_kernel(RepsArgs a) {
  __shared__ float part[kRepThreads * (16 / sizeof(T))];
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  const int b = blockIdx.z, j = a.first_block + blockIdx.x;
  if (a.vl.on && j >= a.vl.nb[b]) return;  // past this sequence's full blocks
  block_rep<T>(a, b, blockIdx.y, j, part);
}

// After an append: grid (B, most blocks one append can complete, Hkv); CTA
// (b, f, h) rebuilds block ctx_b / blk + f of sequence b if the append made
// it full.
template <typename T>
__global__ void __launch_bounds__(kRepThreads) append_reps_kernel(RepsArgs a, AppendArgs ap) {
  __shared__ float part[kRepThreads * (16 / sizeof(T))];
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  const int b = blockIdx.x, h = blockIdx.z;
  const int ctx = ap.seq_ctx[b];
  const int n = min(max(ap.n_accept[b], 0), ap.T);
  if (ctx < 0) return;  // flagged by the copy kernel
  const int j = ctx / a.blk + blockIdx.y;
  if (j >= (ctx + n) / a.blk) return;
  if (j >= a.nb_max) return;  // flagged by the copy kernel
  block_rep<T>(a, b, h, j, part);
}

// ------------------------------------------------------------------ scores
// grid = (CTAs per pair, B*Hkv); CTA x of a pair scores blocks
// [x*rows_per_cta, (x+1)*rows_per_cta), sized on the host so that the whole
// grid is resident at once. Each warp streams whole fp32 representative rows
// with 128-bit loads (lane c holds dims 4c..4c+3 of each 128-dim chunk),
// R rows at a time: all of a group's loads are issued before its dot
// products, and the first group's loads are in flight while the warp forms
// the group-summed draft-0 query. The R row sums are reduced together by a
// transposing butterfly (each exchange halves the values a lane holds).
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreKeys = kFusedSelectMaxNB / kScoreThreads;  // top-k keys per thread

template <int CH>
__host__ __device__ constexpr int score_rows() { return 16 / CH; }

template <typename T, int CH>  // CH: 128-dim chunks per row (d <= 128 * CH)
__global__ void __launch_bounds__(kScoreThreads, 2) score_kernel(const __grid_constant__ ScoreArgs a) {
  constexpr int R = score_rows<CH>();  // rows in flight per warp
  constexpr int S = 32 / R;            // lanes per row after the butterfly
  const int pair = blockIdx.y;         // b * Hkv + h
  const int b = pair / a.Hkv, h = pair % a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunk = a.d / 4;
  const int nbb = nb_of(a.vl, b, a.nb);  // this sequence's blocks (rows keep stride nb)
  const int r0 = blockIdx.x * a.rows_per_cta;
  const int r1 = min(nbb, r0 + a.rows_per_cta);
  const float* rep0 = a.reps + (size_t)pair * a.nb_max * a.d;
  float* srow = a.scores + (size_t)pair * a.nb;
  if (threadIdx.x < 32 && r0 < r1) {
    // Warm L2 with this CTA's representative rows (contiguous) while the
    // previous kernel finishes: a prefetch only, so it cannot expose data
    // that kernel is still writing (L2 is where every write lands); the
    // loads below still come after the wait. 16 KB per lane and copy.
    const uint8_t* base = reinterpret_cast<const uint8_t*>(rep0 + (size_t)r0 * a.d);
    const size_t bytes = (size_t)(r1 - r0) * a.d * sizeof(float);  // a multiple of 16
    constexpr size_t kChunk = 16384;
    for (size_t off = (size_t)threadIdx.x * kChunk; off < bytes; off += 32 * kChunk)
      prefetch_bulk_l2(base + off, (uint32_t)(bytes - off < kChunk ? bytes - off : kChunk));
  }
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  if (r0 >= nbb) {
    // past this sequence's blocks: no rows, no arrival; a sequence without
    // full blocks gets an empty selection from its first CTA
    if (nbb == 0 && blockIdx.x == 0 && a.sel && a.nb <= kFusedSelectMaxNB)
      for (int i = threadIdx.x; i < a.kmax; i += kScoreThreads) a.sel[(size_t)pair * a.kmax + i] = -1;
    return;
  }

  if (a.sel && a.block_table) {
    // warm L2 with the block-table entries of these rows: the selecting CTA
    // reads the kept blocks' pages from there
    const int32_t* bt = a.block_table + (size_t)b * a.nb_max;
    for (int e = r0 + 32 * threadIdx.x; e < r1; e += 32 * kScoreThreads) prefetch_l2(bt + e);
  }
  const uint64_t pol = l2_evict_first_policy();  // representatives are read once per call
  float4 qh[CH];
  bool have_q = false;
  for (int base = r0 + warp * R; base < r1; base += kScoreWarps * R) {
    float4 rv[R][CH];
#pragma unroll
    for (int u = 0; u < R; ++u) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int ch = lane + 32 * c;
        rv[u][c] = (base + u < r1 && ch < nchunk)
                       ? ld_stream_f4(reinterpret_cast<const float4*>(rep0 + (size_t)(base + u) * a.d) + ch,
                                      pol)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (!have_q) {  // qhat = sum over the G query heads of kv head h, draft 0
      const T* q0 = static_cast<const T*>(a.q) + ((size_t)b * a.T * a.Hq + (size_t)h * a.G) * a.d;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        qh[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int ch = lane + 32 * c;
        if (ch < nchunk) {
          for (int g = 0; g < a.G; ++g) {
            const float4 v = load4<T>(q0 + (size_t)g * a.d + ch * 4);
            qh[c].x += v.x; qh[c].y += v.y; qh[c].z += v.z; qh[c].w += v.w;
          }
        }
      }
      have_q = true;
    }
    float acc[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      acc[u] = 0.f;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        acc[u] = fmaf(qh[c].x, rv[u][c].x, acc[u]);
        acc[u] = fmaf(qh[c].y, rv[u][c].y, acc[u]);
        acc[u] = fmaf(qh[c].z, rv[u][c].z, acc[u]);
        acc[u] = fmaf(qh[c].w, rv[u][c].w, acc[u]);
      }
    }
    // transposing butterfly: after the exchange at offset o a lane keeps the
    // half of its values selected by bit o of its lane index; lane l ends
    // with row l / S summed over the lanes that share l / S
#pragma unroll
    for (int n = R, o = 16; n > 1; n >>= 1, o >>= 1) {
      const bool hi = lane & o;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = hi ? acc[i] : acc[i + n / 2];
        const float keep = hi ? acc[i + n / 2] : acc[i];
        acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
#pragma unroll
    for (int o = S / 2; o > 0; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
    const int j = base + lane / S;
    if ((lane % S) == 0 && j < r1) srow[j] = acc[0];
  }
  if (!a.sel || a.nb > kFusedSelectMaxNB) {
    return;
  }

  // Fused selection: the last CTA to finish scoring this (b, h) selects. The
  // barrier orders every thread's score stores before thread 0's
  // acquire-release arrival; the last arrival thereby sees every score.
  __shared__ unsigned s_last;
  __shared__ TopkSmem<kScoreThreads, kScoreKeys> tsm;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned ctas = (unsigned)((nbb + a.rows_per_cta - 1) / a.rows_per_cta);
    const bool last = arrive_acq_rel(&a.counters[pair * kPairWords]) == ctas - 1;
    s_last = last;
  }
  __syncthreads();
  if (s_last) {
    const TopkRows tr{a.block_table ? a.block_table + (size_t)b * a.nb_max : nullptr,
                      a.rows ? a.rows + (size_t)pair * a.kmax : nullptr, a.Hkv, h, a.blk,
                      a.num_pages, a.status};
    cta_topk_fit<kScoreThreads, kScoreKeys>(srow, nbb, n_of(a.vl, b, a.k), a.sel + (size_t)pair * a.kmax,
                                        a.kmax, tsm, tr);
    if (threadIdx.x == 0) a.counters[pair * kPairWords] = 0;  // ready for the next call
  }
}

}  // namespace

cudaError_t launch_append_reps(const RepsArgs& a, const AppendArgs& ap, int dtype,
                               cudaStream_t st) {
  // appending at most T tokens completes at most (blk - 1 + T) / blk blocks
  const int most = (a.blk - 1 + ap.T) / a.blk;
  if (a.B == 0 || most == 0) return cudaSuccess;
  dim3 grid(a.B, most, a.Hkv);
  if (dtype == SV_BF16)
    return launch_pdl(append_reps_kernel<__nv_bfloat16>, grid, dim3(kRepThreads), 0, st, a, ap);
  return launch_pdl(append_reps_kernel<float>, grid, dim3(kRepThreads), 0, st, a, ap);
}

cudaError_t launch_build_reps(const RepsArgs& a, int dtype, cudaStream_t st) {
  if (a.n_blocks == 0) return cudaSuccess;
  dim3 grid(a.n_blocks, a.Hkv, a.B);
  if (dtype == SV_BF16)
    return launch_pdl(build_reps_kernel<__nv_bfloat16>, grid, dim3(kRepThreads), 0, st, a);
  return launch_pdl(build_reps_kernel<float>, grid, dim3(kRepThreads), 0, st, a);
}

template <typename T, int CH>
static cudaError_t launch_score_t(ScoreArgs a, cudaStream_t st) {
  auto kern = score_kernel<T, CH>;
  // resident CTAs per SM, queried once per device
  static std::atomic<int> occ_cache[kMaxDevices];
  const int dev = current_device();
  int occ = occ_cache[dev].load();
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kScoreThreads, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    occ_cache[dev].store(occ);
  }
  // one resident wave: spread sm_count * occ CTAs over the pairs
  const int pairs = a.B * a.Hkv;
  constexpr int R = score_rows<CH>();
  int cpp = sm_count() * occ / pairs;
  const int max_cpp = (a.nb + kScoreWarps * R - 1) / (kScoreWarps * R);
  cpp = cpp < 1 ? 1 : cpp > max_cpp ? max_cpp : cpp;
  a.rows_per_cta = (a.nb + cpp - 1) / cpp;
  cpp = (a.nb + a.rows_per_cta - 1) / a.rows_per_cta;
  return launch_pdl(kern, dim3(cpp, pairs), dim3(kScoreThreads), 0, st, a);
}

cudaError_t launch_score(ScoreArgs a, int dtype, cudaStream_t st) {
  if (a.nb == 0) return cudaSuccess;
  const bool wide = a.d > 128;
  if (dtype == SV_BF16)
    return wide ? launch_score_t<__nv_bfloat16, 2>(a, st) : launch_score_t<__nv_bfloat16, 1>(a, st);
  return wide ? launch_score_t<float, 2>(a, st) : launch_score_t<float, 1>(a, st);
}

}  // namespace sva
