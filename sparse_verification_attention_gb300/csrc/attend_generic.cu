// Split-KV sparse verification attention, CUDA-core path for shapes the
// tensor-core path does not take (fp32 inputs, d not in {64,128}, blk not in
// {32,64}, more than 128 stacked rows, more drafts than a block holds), and
// the log-sum-exp merge of split partials shared by both paths.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: every draft attends to
// the one selected block set; drafts additionally see themselves and their
// ancestors (tree or chain mask among drafts).
#include "internal.h"
#include "ptx.h"

namespace sva {
namespace {

constexpr int kPer = kMaxD / 32;  // dims per lane

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

struct RowState {
  float q[kPer], o[kPer], m, l;
};

// One key/value row into a warp's running softmax (log2 domain).
template <typename T>
__device__ __forceinline__ void absorb(RowState& st, const T* krow, const T* vrow, int d,
                                       float scale_log2, int lane) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int i = lane + 32 * e;
    if (i < d) s = fmaf(st.q[e], ldf<T>(krow + i), s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  s *= scale_log2;
  const float mn = fmaxf(st.m, s);
  const float alpha = exp2f(st.m - mn);  // 0 when st.m == -inf
  const float p = exp2f(s - mn);
  st.l = st.l * alpha + p;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int i = lane + 32 * e;
    if (i < d) st.o[e] = st.o[e] * alpha + p * ldf<T>(vrow + i);
  }
  st.m = mn;
}

// grid = (splits, Hkv, B); each warp walks whole rows (one stacked query row
// at a time) over the split's selected blocks and, on the last split, the
// drafts the row may see.
template <typename T>
__global__ void __launch_bounds__(128) attend_generic_kernel(const __grid_constant__ AttendArgs a) {
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int pair = b * a.Hkv + h;
  // work units: the n_sel selected blocks, the partial last block (unit
  // n_sel, if any), then the draft tile
  const int nsel = n_of(a.vl, b, a.n_sel), nbb = nb_of(a.vl, b, a.nb);
  const int tail = tail_of(a.vl, b, a.tail);
  const int ntail = tail > 0 ? 1 : 0;
  const int u0 = split * a.bps;
  const int u1 = min(nsel + ntail + 1, u0 + a.bps);
  const int j0 = u0, j1 = min(u1, nsel);
  const bool has_tail = ntail && u0 <= nsel && nsel < u1;
  const bool has_draft = (u0 <= nsel + ntail && nsel + ntail < u1);
  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);
  const T* q = static_cast<const T*>(a.q);
  const T* dk = static_cast<const T*>(a.draft_k);
  const T* dv = static_cast<const T*>(a.draft_v);
  const size_t slot = ((size_t)pair * a.slot_stride + split) * a.rpad;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish

  for (int r = warp; r < a.R; r += nw) {
    const int t = r / a.G, gq = r % a.G;
    RowState st;
    const T* qrow = q + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * a.d;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = lane + 32 * e;
      st.q[e] = (i < a.d) ? ldf<T>(qrow + i) : 0.f;
      st.o[e] = 0.f;
    }
    st.m = -INFINITY;
    st.l = 0.f;
    for (int jj = j0; jj < j1; ++jj) {
      const int j = a.sel ? a.sel[(size_t)pair * a.sel_stride + jj] : jj;
      if (j < 0 || j >= nbb) {
        if (lane == 0) atomicOr(a.status, SV_FLAG_BAD_BLOCK_INDEX);
        continue;
      }
      const int page = a.block_table[(size_t)b * a.nb_max + j];
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) atomicOr(a.status, SV_FLAG_BAD_PAGE);
        continue;
      }
      const size_t base = ((size_t)page * a.Hkv + h) * a.blk * a.d;
      for (int x = 0; x < a.blk; ++x)
        absorb<T>(st, kp + base + (size_t)x * a.d, vp + base + (size_t)x * a.d, a.d,
                  a.scale_log2, lane);
    }
    if (has_tail) {
      const int page = a.block_table[(size_t)b * a.nb_max + nbb];
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) atomicOr(a.status, SV_FLAG_BAD_PAGE);
      } else {
        const size_t base = ((size_t)page * a.Hkv + h) * a.blk * a.d;
        for (int x = 0; x < tail; ++x)
          absorb<T>(st, kp + base + (size_t)x * a.d, vp + base + (size_t)x * a.d, a.d,
                    a.scale_log2, lane);
      }
    }
    if (has_draft) {
      const unsigned long long vis = a.anc[t];
      for (int u = 0; u < a.T; ++u) {
        if (!((vis >> u) & 1ull)) continue;
        const size_t off = (((size_t)b * a.T + u) * a.Hkv + h) * a.d;
        absorb<T>(st, dk + off, dv + off, a.d, a.scale_log2, lane);
      }
    }
    float* po = a.part_o + (slot + r) * a.d;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = lane + 32 * e;
      if (i < a.d) po[i] = st.o[e];
    }
    if (lane == 0) {
      a.part_ml[(slot + r) * 2] = st.m;
      a.part_ml[(slot + r) * 2 + 1] = st.l;
    }
  }
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// Log-sum-exp merge of the split partials, one thread per 4 output columns
// of one stacked row (a warp covers 128 columns of one row, so the (m, l)
// loads are warp broadcasts):
//   M = max_s m_s,  w_s = 2^(m_s - M),  out = sum_s w_s o_s / sum_s w_s l_s.
// The split loops are unrolled so the independent loads overlap.
constexpr int kMergeThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ AttendArgs a) {
  const int c4n = a.d / 4;
  const long long gid = (long long)blockIdx.x * kMergeThreads + threadIdx.x;
  const long long total = (long long)a.B * a.Hkv * a.R * c4n;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish
  if (gid < total) {
    const int c = (int)(gid % c4n) * 4;
    const long long pr = gid / c4n;
    const int r = (int)(pr % a.R);
    const int pair = (int)(pr / a.R);
    const int b = pair / a.Hkv, h = pair % a.Hkv;
    const int nsp = a.n_splits + (pair < a.split_extra ? 1 : 0);
    const size_t base = (size_t)pair * a.slot_stride * a.rpad + r;
    float M = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < nsp; ++s) M = fmaxf(M, a.part_ml[(base + (size_t)s * a.rpad) * 2]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
#pragma unroll 8
    for (int s = 0; s < nsp; ++s) {
      const size_t row = base + (size_t)s * a.rpad;
      const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + row * 2);
      const float4 o = *reinterpret_cast<const float4*>(a.part_o + row * a.d + c);
      const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
      L += w * ml.y;
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
    const float inv = 1.0f / L;
    const int t = r / a.G, gq = r % a.G;
    T* out = static_cast<T*>(a.out) + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * a.d;
    store4<T>(out + c, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
}

}  // namespace

cudaError_t launch_attend_generic(const AttendArgs& a, int dtype, cudaStream_t st) {
  dim3 grid(a.n_splits, a.Hkv, a.B);
  if (dtype == SV_BF16) return launch_pdl(attend_generic_kernel<__nv_bfloat16>, grid, dim3(128), 0, st, a);
  return launch_pdl(attend_generic_kernel<float>, grid, dim3(128), 0, st, a);
}

cudaError_t launch_merge(const AttendArgs& a, int dtype, cudaStream_t st) {
  const long long total = (long long)a.B * a.Hkv * a.R * (a.d / 4);
  dim3 grid((unsigned)((total + kMergeThreads - 1) / kMergeThreads));
  if (dtype == SV_BF16)
    return launch_pdl(merge_kernel<__nv_bfloat16>, grid, dim3(kMergeThreads), 0, st, a);
  return launch_pdl(merge_kernel<float>, grid, dim3(kMergeThreads), 0, st, a);
}

}  // namespace sva
