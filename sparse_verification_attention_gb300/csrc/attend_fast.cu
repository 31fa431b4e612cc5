// Split-KV sparse verification attention, bf16 tensor-core path.
//
// [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
// Verification", paper summary page, Figure 1 caption: all draft tokens use
// the same selected set of KV blocks. That is what makes this kernel
// bandwidth-efficient: the T*G query rows that share a KV head are stacked
// into one tile (R = T*G rows) and every selected KV page is read from HBM
// exactly once for all of them.
//
// Design (GB300):
//   * grid = (splits, Hkv, B); each CTA owns a contiguous run of the selected
//     blocks of one (b, kv head); the last split also owns the draft tile.
//   * warp 0 is the producer: one lane walks the selection, resolves the page
//     through the block table and issues 2-D bulk tensor copies (TMA, 128-byte
//     swizzle) of the page's K and V tiles into an NS-stage shared-memory ring
//     guarded by mbarriers (full: transaction bytes; empty: consumer warps).
//   * warps 1..NWC are consumers, 16 stacked rows each: S = Q K^T and O += P V
//     on tensor cores (m16n8k16 bf16, fp32 accumulate), operands fetched with
//     ldmatrix from the swizzled tiles, online softmax in registers (log2
//     domain), P re-packed to bf16 straight from the accumulator registers.
//   * the CTA writes an unnormalised partial (o, m, l) per row; a small merge
//     kernel combines the splits with log-sum-exp weights.
//   * every wait is bounded: on timeout a status flag is raised and the CTA
//     drains its own copies before leaving; no spin can hang the GPU.
#include <cooperative_groups.h>

#include <atomic>

#include "internal.h"
#include "ptx.h"

namespace sva {
namespace {

template <int D, int BLK, int NWC, int NS, bool CLUSTER>
struct FastCfg {
  static constexpr int kBoxes = D / 64;           // 128-byte-wide TMA boxes per tile
  static constexpr int kBoxBytes = BLK * 128;     // BLK rows x 64 bf16
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
  static constexpr int kThreads = 32 * (NWC + 1);
  // The cluster merge stages the partial (o, m, l) and merge weights in the
  // ring once the ring is idle; the ring is sized to hold them.
  static constexpr int kOst = D + 4;              // padded fp32 row stride of the staged o
  static constexpr int kRows = 16 * NWC;
  static constexpr int kMergeBytes = (kRows * kOst + kRows * 2 + kRows * 16) * 4;
  static constexpr int kRingRaw = NS * kStageBytes;
  static constexpr int kRing =
      ((CLUSTER && kMergeBytes > kRingRaw ? kMergeBytes : kRingRaw) + 1023) / 1024 * 1024;
  static constexpr int kSmem = kRing + 1024 + 256;  // + alignment slack + barriers
  static_assert(BLK % 16 == 0 && D % 64 == 0, "tile shape");
};

__device__ __forceinline__ uint32_t ld_bf16x2(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int D, int BLK>
__device__ __forceinline__ uint32_t swz(int row, int dcol) {
  // byte offset of (row, dcol) inside a K or V tile laid out as D/64 boxes of
  // [BLK][64] bf16 with the 128-byte TMA swizzle (16-byte chunk c of row r at
  // chunk c ^ (r & 7)).
  const int box = dcol >> 6;
  const int c = (dcol & 63) >> 3;
  return box * (BLK * 128) + row * 128 + ((c ^ (row & 7)) << 4);
}

template <int D, int BLK, int NWC>
struct Consumer {
  uint32_t qf[D / 16][4];
  float o[D / 8][4];
  float m_lo, m_hi, l_lo, l_hi;
  int r_lo, r_hi;
  unsigned long long vis_lo, vis_hi;  // visible drafts of rows r_lo, r_hi

  // draft: mask columns by the rows' ancestor bits; limit: columns past it
  // (a partial last block) are masked
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, const AttendArgs& a,
                                       bool draft, int limit, int lane) {
    const int t4 = lane & 3;
    float s[BLK / 8][4];
#pragma unroll
    for (int nt = 0; nt < BLK / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;

    // S = Q K^T: B fragments of two 8-token n-tiles per ldmatrix.x4.
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int ntp = 0; ntp < BLK / 16; ++ntp) {
        const int mi = lane >> 3;
        const int tok = 16 * ntp + 8 * (mi >> 1) + (lane & 7);
        const int dcol = 16 * kk + 8 * (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz<D, BLK>(tok, dcol), b0, b1, b2, b3);
        mma_bf16(s[2 * ntp], qf[kk], b0, b1);
        mma_bf16(s[2 * ntp + 1], qf[kk], b2, b3);
      }
    }

    // Scale into the log2 domain, mask (draft tile, partial block), online
    // softmax.
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < BLK / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nt][e] * a.scale_log2;
        const int u = 8 * nt + 2 * t4 + (e & 1);
        if (draft) {
          // bit u of the row's ancestor mask (zero for padding rows)
          const unsigned long long vis = (e < 2) ? vis_lo : vis_hi;
          if (!((vis >> u) & 1ull)) v = -INFINITY;
        } else if (u >= limit) {
          v = -INFINITY;
        }
        s[nt][e] = v;
      }
      mx_lo = fmaxf(mx_lo, fmaxf(s[nt][0], s[nt][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(s[nt][2], s[nt][3]));
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float base_lo = (mn_lo == -INFINITY) ? 0.f : mn_lo;
    const float base_hi = (mn_hi == -INFINITY) ? 0.f : mn_hi;
    const float al_lo = exp2f(m_lo - base_lo), al_hi = exp2f(m_hi - base_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    l_lo *= al_lo;
    l_hi *= al_hi;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= al_lo; o[nd][1] *= al_lo;
      o[nd][2] *= al_hi; o[nd][3] *= al_hi;
    }
    uint32_t pa[BLK / 16][4];
#pragma unroll
    for (int nt = 0; nt < BLK / 8; ++nt) {
      const float p0 = exp2f(s[nt][0] - base_lo), p1 = exp2f(s[nt][1] - base_lo);
      const float p2 = exp2f(s[nt][2] - base_hi), p3 = exp2f(s[nt][3] - base_hi);
      l_lo += p0 + p1;
      l_hi += p2 + p3;
      // C fragment of n-tile nt -> A fragment of k-step nt/2 (FA2 register reuse).
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }

    // O += P V: V is token-major, so its B fragments come from ldmatrix.trans.
#pragma unroll
    for (int kt = 0; kt < BLK / 16; ++kt) {
#pragma unroll
      for (int ndp = 0; ndp < D / 16; ++ndp) {
        const int mi = lane >> 3;
        const int tok = 16 * kt + 8 * (mi & 1) + (lane & 7);
        const int dcol = 8 * (2 * ndp + (mi >> 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz<D, BLK>(tok, dcol), b0, b1, b2, b3);
        mma_bf16(o[2 * ndp], pa[kt], b0, b1);
        mma_bf16(o[2 * ndp + 1], pa[kt], b2, b3);
      }
    }
  }
};

template <int D, int BLK, int NWC, int NS, bool CLUSTER>
__global__ void __launch_bounds__(32 * (NWC + 1))
    attend_fast_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ AttendArgs a) {
  using C = FastCfg<D, BLK, NWC, NS, CLUSTER>;
  constexpr int NT = 32 * (NWC + 1);
  constexpr int OST = C::kOst;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRing);
  uint64_t* empty = full + NS;
  int* stage_ok = reinterpret_cast<int*>(empty + NS);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = b * a.Hkv + h;
  // Work units of this (b, h): the n_sel selected blocks, the partial last
  // block (unit n_sel, if any), then the draft tile.
  const int nsel = n_of(a.vl, b, a.n_sel), nbb = nb_of(a.vl, b, a.nb);
  const int tail = tail_of(a.vl, b, a.tail);
  const int ntail = tail > 0 ? 1 : 0;
  const int u0 = split * a.bps;
  const int u1 = min(nsel + ntail + 1, u0 + a.bps);
  const int j0 = u0;
  const int nblk = max(0, min(u1, nsel) - u0);
  const bool has_tail = ntail && u0 <= nsel && nsel < u1;
  const bool has_draft = (u0 <= nsel + ntail && nsel + ntail < u1);
  const int nring = nblk + (has_tail ? 1 : 0);  // tiles through the ring

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), NWC);
    }
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  pdl_wait();  // everything below may read what earlier kernels wrote
  pdl_trigger();  // the next kernel may launch; it still waits for this grid to finish

  Consumer<D, BLK, NWC> cs;
  const int g = lane >> 2, t4 = lane & 3;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp resolves 32 selected blocks at a time (selection entry,
    // then block-table page) so that these dependent global loads overlap;
    // lane 0 then issues the copies in order.
    const int oob_row = a.num_pages * a.Hkv * BLK;  // past the end: TMA zero-fills
    int issued = 0;
    bool stop = false;
    for (int base = 0; base < nring && !stop; base += 32) {
      int row = oob_row, ok = 0;
      if (base + lane < nring) {
        // the partial last block rides after the selected ones (stage_ok 2)
        const bool tailu = base + lane == nblk;
        const int j = tailu ? nbb
                            : a.sel ? a.sel[(size_t)pair * a.sel_stride + j0 + base + lane]
                                    : j0 + base + lane;
        if (!tailu && (j < 0 || j >= nbb)) {
          atomicOr(a.status, SV_FLAG_BAD_BLOCK_INDEX);
        } else {
          const int page = a.block_table[(size_t)b * a.nb_max + j];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, SV_FLAG_BAD_PAGE);
          } else {
            row = (page * a.Hkv + h) * BLK;
            ok = tailu ? 2 : 1;
          }
        }
      }
      const int cnt = min(32, nring - base);
      for (int qq = 0; qq < cnt; ++qq) {
        const int i = base + qq;
        const int rq = __shfl_sync(0xffffffffu, row, qq);
        const int okq = __shfl_sync(0xffffffffu, ok, qq);
        int fail = 0;
        if (lane == 0) {
          const int s = i % NS;
          if (i >= NS && !mbar_wait(smem_u32(&empty[s]), ((i / NS) & 1) ^ 1, kSpinLimit)) {
            atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
            fail = 1;
          } else {
            stage_ok[s] = okq;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            const uint32_t kdst = smem_u32(smem + s * C::kStageBytes);
            const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x) {
              tma_load_2d(kdst + x * C::kBoxBytes, &tmK, 64 * x, rq, fb);
              tma_load_2d(vdst + x * C::kBoxBytes, &tmV, 64 * x, rq, fb);
            }
            issued = i + 1;
          }
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) {
          stop = true;
          break;
        }
      }
    }
    // Never leave the ring with a bulk copy still writing into it.
    if (lane == 0)
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait(smem_u32(&full[i % NS]), (i / NS) & 1, kSpinLimit);
  } else {
    // -------------------------------------------------------------- consumers
    const int cw = warp - 1;
    cs.r_lo = 16 * cw + g;
    cs.r_hi = cs.r_lo + 8;
    cs.vis_lo = cs.vis_hi = 0ull;
    for (int t = 0; t < a.T; ++t) {  // warp-uniform index into the parameters
      const unsigned long long m = a.anc[t];
      if (cs.r_lo < a.R && cs.r_lo / a.G == t) cs.vis_lo = m;
      if (cs.r_hi < a.R && cs.r_hi / a.G == t) cs.vis_hi = m;
    }
    {
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
      const __nv_bfloat16* qlo = nullptr;
      const __nv_bfloat16* qhi = nullptr;
      if (cs.r_lo < a.R)
        qlo = q + (((size_t)b * a.T + cs.r_lo / a.G) * a.Hq + h * a.G + cs.r_lo % a.G) * D;
      if (cs.r_hi < a.R)
        qhi = q + (((size_t)b * a.T + cs.r_hi / a.G) * a.Hq + h * a.G + cs.r_hi % a.G) * D;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int col = 16 * kk + 2 * t4;
        cs.qf[kk][0] = qlo ? ld_bf16x2(qlo + col) : 0u;
        cs.qf[kk][1] = qhi ? ld_bf16x2(qhi + col) : 0u;
        cs.qf[kk][2] = qlo ? ld_bf16x2(qlo + col + 8) : 0u;
        cs.qf[kk][3] = qhi ? ld_bf16x2(qhi + col + 8) : 0u;
      }
    }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) cs.o[nd][0] = cs.o[nd][1] = cs.o[nd][2] = cs.o[nd][3] = 0.f;
    cs.m_lo = cs.m_hi = -INFINITY;
    cs.l_lo = cs.l_hi = 0.f;

    const uint32_t sbase = smem_u32(smem);
    for (int i = 0; i < nring; ++i) {
      const int s = i % NS;
      // warp-uniform outcome: ldmatrix/mma.sync below need all 32 lanes
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s]), (i / NS) & 1, kSpinLimit))) {
        atomicOr(a.status, SV_FLAG_WAIT_TIMEOUT);
        break;
      }
      if (stage_ok[s]) {
        const uint32_t kb = sbase + s * C::kStageBytes;
        cs.tile(kb, kb + C::kTileBytes, a, false, stage_ok[s] == 2 ? tail : BLK, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

    if (has_draft) {
      // Draft tile: draft K/V rows u < T (rows T..BLK-1 zero) written into
      // stage 0 in the same swizzled layout, then one masked tile.
      asm volatile("bar.sync 1, %0;" ::"r"(NWC * 32) : "memory");
      const int ctid = threadIdx.x - 32;
      const uint4* dk = static_cast<const uint4*>(a.draft_k);
      const uint4* dv = static_cast<const uint4*>(a.draft_v);
      for (int idx = ctid; idx < BLK * (D / 8); idx += NWC * 32) {
        const int u = idx / (D / 8), c = idx % (D / 8);
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (u < a.T) {
          const size_t off = (((size_t)b * a.T + u) * a.Hkv + h) * (D / 8) + c;
          kv = dk[off];
          vv = dv[off];
        }
        const uint32_t o = swz<D, BLK>(u, 8 * c);
        *reinterpret_cast<uint4*>(smem + o) = kv;
        *reinterpret_cast<uint4*>(smem + C::kTileBytes + o) = vv;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NWC * 32) : "memory");
      cs.tile(sbase, sbase + C::kTileBytes, a, true, BLK, lane);
    }
    cs.l_lo += __shfl_xor_sync(0xffffffffu, cs.l_lo, 1);
    cs.l_lo += __shfl_xor_sync(0xffffffffu, cs.l_lo, 2);
    cs.l_hi += __shfl_xor_sync(0xffffffffu, cs.l_hi, 1);
    cs.l_hi += __shfl_xor_sync(0xffffffffu, cs.l_hi, 2);
  }

  if constexpr (CLUSTER) {
    // ------------------------------------------------ in-cluster merge (DSMEM)
    // Every CTA of the cluster holds one split of the same (b, h). Each stages
    // its unnormalised partial (o, m, l) in its own shared memory; after a
    // cluster barrier, CTA r combines rows [r*rows, (r+1)*rows) across all
    // peers with log-sum-exp weights and writes the output.
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int nsplit = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    float* po = reinterpret_cast<float*>(smem);                 // [rpad][OST]
    float* pml = po + (size_t)a.rpad * OST;                     // [rpad][2]
    float* wgt = pml + (size_t)a.rpad * 2;                      // [rows][nsplit]
    __syncthreads();  // ring and draft tile no longer read by anyone
    if (warp > 0) {
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = 8 * nd + 2 * t4;
        if (cs.r_lo < a.rpad)
          *reinterpret_cast<float2*>(po + cs.r_lo * OST + col) = make_float2(cs.o[nd][0], cs.o[nd][1]);
        if (cs.r_hi < a.rpad)
          *reinterpret_cast<float2*>(po + cs.r_hi * OST + col) = make_float2(cs.o[nd][2], cs.o[nd][3]);
      }
      if (t4 == 0) {
        if (cs.r_lo < a.rpad) *reinterpret_cast<float2*>(pml + 2 * cs.r_lo) = make_float2(cs.m_lo, cs.l_lo);
        if (cs.r_hi < a.rpad) *reinterpret_cast<float2*>(pml + 2 * cs.r_hi) = make_float2(cs.m_hi, cs.l_hi);
      }
    }
    cl.sync();
    const int rows = (a.R + nsplit - 1) / nsplit;
    const int r0 = rank * rows;
    const int r1 = min(a.R, r0 + rows);
    for (int r = r0 + threadIdx.x; r < r1; r += NT) {
      float M = -INFINITY;
      for (int s = 0; s < nsplit; ++s) M = fmaxf(M, cl.map_shared_rank(pml, s)[2 * r]);
      float L = 0.f;
      for (int s = 0; s < nsplit; ++s) {
        const float2 ml = *reinterpret_cast<const float2*>(cl.map_shared_rank(pml, s) + 2 * r);
        const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
        wgt[(r - r0) * nsplit + s] = w;
        L += w * ml.y;
      }
      const float inv = 1.0f / L;
      for (int s = 0; s < nsplit; ++s) wgt[(r - r0) * nsplit + s] *= inv;
    }
    __syncthreads();
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    for (int idx = threadIdx.x; idx < (r1 - r0) * (D / 4); idx += NT) {
      const int r = r0 + idx / (D / 4), c = (idx % (D / 4)) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < nsplit; ++s) {
        const float w = wgt[(r - r0) * nsplit + s];
        const float4 o = *reinterpret_cast<const float4*>(cl.map_shared_rank(po, s) + r * OST + c);
        acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
      }
      const int t = r / a.G, gq = r % a.G;
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + (((size_t)b * a.T + t) * a.Hq + h * a.G + gq) * D + c) = u;
    }
    cl.sync();  // peers may still be reading this CTA's shared memory
  } else {
    // -------------------------------------------- partials for the merge kernel
    if (warp > 0) {
      const size_t slot = ((size_t)pair * a.slot_stride + split) * a.rpad;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = 8 * nd + 2 * t4;
        if (cs.r_lo < a.rpad)
          *reinterpret_cast<float2*>(a.part_o + (slot + cs.r_lo) * D + col) =
              make_float2(cs.o[nd][0], cs.o[nd][1]);
        if (cs.r_hi < a.rpad)
          *reinterpret_cast<float2*>(a.part_o + (slot + cs.r_hi) * D + col) =
              make_float2(cs.o[nd][2], cs.o[nd][3]);
      }
      if (t4 == 0) {
        if (cs.r_lo < a.rpad)
          *reinterpret_cast<float2*>(a.part_ml + (slot + cs.r_lo) * 2) = make_float2(cs.m_lo, cs.l_lo);
        if (cs.r_hi < a.rpad)
          *reinterpret_cast<float2*>(a.part_ml + (slot + cs.r_hi) * 2) = make_float2(cs.m_hi, cs.l_hi);
      }
    }
  }
}

template <int D, int BLK, int NWC, bool CLUSTER>
struct FastKernel {
  static constexpr int NS = 3;
  using C = FastCfg<D, BLK, NWC, NS, CLUSTER>;
  static void* fn() { return reinterpret_cast<void*>(attend_fast_kernel<D, BLK, NWC, NS, CLUSTER>); }
};

template <int D, int BLK, int NWC, bool CLUSTER>
cudaError_t launch_cfg(const AttendArgs& a, int cluster, cudaStream_t st) {
  using K = FastKernel<D, BLK, NWC, CLUSTER>;
  CUtensorMap mk, mv;
  const char* why = nullptr;
  if (!encode_pool_map(&mk, a.k_pool, a.num_pages, a.Hkv, BLK, D, &why) ||
      !encode_pool_map(&mv, a.v_pool, a.num_pages, a.Hkv, BLK, D, &why))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.Hkv, a.B);
  cfg.blockDim = dim3(K::C::kThreads);
  cfg.dynamicSmemBytes = K::C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (CLUSTER) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, attend_fast_kernel<D, BLK, NWC, K::NS, CLUSTER>, mk, mv, a);
}

template <int D, int BLK, bool CLUSTER>
cudaError_t launch_rows(const AttendArgs& a, int cluster, cudaStream_t st) {
  const int nwc = a.rpad / 16;
  if (nwc <= 1) return launch_cfg<D, BLK, 1, CLUSTER>(a, cluster, st);
  if (nwc <= 2) return launch_cfg<D, BLK, 2, CLUSTER>(a, cluster, st);
  if (nwc <= 4) return launch_cfg<D, BLK, 4, CLUSTER>(a, cluster, st);
  return launch_cfg<D, BLK, 8, CLUSTER>(a, cluster, st);
}

// Sets the kernel's shared-memory attribute and returns its resident CTAs per
// SM; computed once per device and cached.
template <int D, int BLK, int NWC, bool CLUSTER>
int occupancy_cfg() {
  using K = FastKernel<D, BLK, NWC, CLUSTER>;
  static std::atomic<int> cached[kMaxDevices];
  const int dev = current_device();
  const int c = cached[dev].load();
  if (c > 0) return c;
  const int smem = K::C::kSmem;
  if (cudaFuncSetAttribute(K::fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(K::fn(), cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K::fn(), K::C::kThreads, smem) !=
      cudaSuccess)
    return 0;
  cached[dev].store(n);
  return n;
}

template <int D, int BLK, bool CLUSTER>
int occupancy_rows(const AttendArgs& a) {
  const int nwc = a.rpad / 16;
  if (nwc <= 1) return occupancy_cfg<D, BLK, 1, CLUSTER>();
  if (nwc <= 2) return occupancy_cfg<D, BLK, 2, CLUSTER>();
  if (nwc <= 4) return occupancy_cfg<D, BLK, 4, CLUSTER>();
  return occupancy_cfg<D, BLK, 8, CLUSTER>();
}

template <bool CLUSTER>
int occupancy_any(const AttendArgs& a) {
  if (a.d == 128 && a.blk == 64) return occupancy_rows<128, 64, CLUSTER>(a);
  if (a.d == 128 && a.blk == 32) return occupancy_rows<128, 32, CLUSTER>(a);
  if (a.d == 64 && a.blk == 64) return occupancy_rows<64, 64, CLUSTER>(a);
  return occupancy_rows<64, 32, CLUSTER>(a);
}

}  // namespace

bool attend_fast_applies(const AttendArgs& a, int dtype) {
  if (dtype != SV_BF16) return false;
  if (!(a.d == 64 || a.d == 128)) return false;
  if (!(a.blk == 32 || a.blk == 64)) return false;
  if (a.rpad > 128 || a.T > a.blk) return false;
  // an empty cache (no pages) has no tensor map to encode
  if (a.num_pages < 1 || !a.k_pool || !a.v_pool) return false;
  if ((reinterpret_cast<uintptr_t>(a.k_pool) & 15) || (reinterpret_cast<uintptr_t>(a.v_pool) & 15))
    return false;
  if ((long long)(a.num_pages + 1) * a.Hkv * a.blk >= (1ll << 31)) return false;
  return true;
}

int attend_fast_ctas_per_sm(const AttendArgs& a, bool cluster) {
  return cluster ? occupancy_any<true>(a) : occupancy_any<false>(a);
}

cudaError_t launch_attend_fast(const AttendArgs& a, int cluster, cudaStream_t st) {
  const bool cl = cluster > 0;
  if (a.d == 128 && a.blk == 64)
    return cl ? launch_rows<128, 64, true>(a, cluster, st) : launch_rows<128, 64, false>(a, 0, st);
  if (a.d == 128 && a.blk == 32)
    return cl ? launch_rows<128, 32, true>(a, cluster, st) : launch_rows<128, 32, false>(a, 0, st);
  if (a.d == 64 && a.blk == 64)
    return cl ? launch_rows<64, 64, true>(a, cluster, st) : launch_rows<64, 64, false>(a, 0, st);
  if (a.d == 64 && a.blk == 32)
    return cl ? launch_rows<64, 32, true>(a, cluster, st) : launch_rows<64, 32, false>(a, 0, st);
  return cudaErrorInvalidValue;
}

}  // namespace sva
