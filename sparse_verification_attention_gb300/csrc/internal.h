// Internal declarations shared by the translation units of libsva.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "sva.h"

namespace sva {

constexpr int kMaxT = 64;          // draft tokens (ancestor masks are 64-bit)
constexpr int kMaxD = 256;
constexpr int kMaxNB = 16384;      // blocks per sequence (top-k keys fit in smem)
constexpr int kMaxSplits = 64;     // split-KV partial slots per (b, kv head)
constexpr int kStatusBytes = 256;  // workspace head: device status word

// Bounded spin for every device-side wait: after this many polls the waiter
// sets SV_FLAG_WAIT_TIMEOUT and gives up instead of hanging the GPU.
constexpr uint32_t kSpinLimit = 1u << 22;

// Every kernel is launched with programmatic stream serialization: it may
// begin launching while the previous kernel in the stream drains, and calls
// pdl_wait() before it touches any global memory that a predecessor might
// read or write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch_pdl with the grid cut into thread-block clusters of `cluster` CTAs
// (x dimension).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cluster, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Per-(b, h) words that CTAs poll or count on (arrival counts, claim words)
// sit one per 128-byte line, so that polling one pair's word
// does not queue behind every other pair's at the same L2 slice.
constexpr int kPairWords = 32;  // stride of such arrays, in 32-bit words
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace carve-up (offsets in bytes from the workspace base).
struct WsLayout {
  size_t status, ctr_score, ctr_attend, claim, scores, rows, part_o, part_ml, total;
  int rpad, slots;
};
WsLayout ws_layout(const sv_shape& s, int nb_max, int kmax);

// ---------------------------------------------------------------- kernels
// Per-sequence counts of a call whose sequences have different contexts
// (on = 0: every sequence uses the call's uniform values).
constexpr int kMaxVarB = 64;  // sequences of such a call
struct VarLen {
  int on;
  int nb[kMaxVarB];    // full blocks of sequence b
  int tail[kMaxVarB];  // tokens of its partial last block
  int n[kMaxVarB];     // blocks it selects / attends
};

struct RepsArgs {
  const void* k_pool;
  const int32_t* block_table;
  float* reps;
  int B, Hkv, d, blk, nb_max, num_pages, first_block, n_blocks;
  unsigned* status;  // may be null (sv_build_reps has no workspace)
  VarLen vl;         // per-sequence full blocks: blocks past them are skipped
};
cudaError_t launch_build_reps(const RepsArgs& a, int dtype, cudaStream_t st);

// Acceptance write-back: sequence b appends the drafts accept_idx[b][0, n)
// (n = n_accept[b], clamped to [0, T]) at positions seq_ctx[b], ... of its
// paged cache.
struct AppendArgs {
  void* k_pool;
  void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_ctx;     // [B] device
  const int32_t* n_accept;    // [B] device
  const int32_t* accept_idx;  // [B, T] device
  const void* draft_k;        // [B, T, Hkv, d]
  const void* draft_v;
  unsigned* status;           // may be null
  int B, T, Hkv, d, blk, nb_max, num_pages;
};
cudaError_t launch_append_kv(const AppendArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_append_reps(const RepsArgs& a, const AppendArgs& ap, int dtype,
                               cudaStream_t st);

struct ScoreArgs {
  const void* q;
  const float* reps;
  float* scores;
  int B, T, Hq, Hkv, G, d, nb, nb_max;
  int rows_per_cta;  // blocks scored by one CTA (set by launch_score)
  // fused selection (sel == nullptr: scores only): the last scoring CTA of
  // each (b, h) selects k blocks into sel[b][h][0..kmax)
  int32_t* sel;
  int k, kmax;
  unsigned* counters;  // [B*Hkv], zero between calls
  VarLen vl;           // per-sequence nb (rows) and k; score rows keep stride nb
  // optional pool rows of the kept blocks (rows[b][h][0..kmax), beside sel)
  const int32_t* block_table;  // null: no rows
  int32_t* rows;
  int blk, num_pages;
  unsigned* status;
};
cudaError_t launch_score(ScoreArgs a, int dtype, cudaStream_t st);
// Largest block count whose selection the score kernel fuses (its 256
// threads hold 32 keys each); beyond it scoring and selection are two launches.
constexpr int kFusedSelectMaxNB = 8192;

struct SelectArgs {
  const float* scores;
  int32_t* sel;
  int pairs, nb, k, kmax;
  int Hkv;             // pairs are (b, h) with b = pair / Hkv
  VarLen vl;           // per-sequence nb and k; score rows keep stride nb
  // optional pool rows of the kept blocks, as in ScoreArgs
  const int32_t* block_table;
  int32_t* rows;
  int nb_max, blk, num_pages;
  unsigned* status;
};
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

struct AttendArgs {
  const void* q;        // [B,T,Hq,d]
  const void* k_pool;   // [P,Hkv,blk,d]
  const void* v_pool;
  const void* draft_k;  // [B,T,Hkv,d]
  const void* draft_v;
  const int32_t* block_table;
  const int32_t* sel;   // null: identity selection over NB blocks
  // optional pool rows of the selected blocks ([pairs][sel_stride], written by
  // the select step of the same call): the producer reads them instead of
  // resolving sel through the block table
  const int32_t* rows;
  float* part_o;        // [B,Hkv,S,Rpad,d]
  float* part_ml;       // [B,Hkv,S,Rpad,2]
  void* out;            // [B,T,Hq,d]
  unsigned* counters;   // [B*Hkv] segment arrivals (tcgen05 path), zero between calls
  unsigned* claim;      // [B*Hkv] merge slices claimed (tcgen05 path), zero between calls
  unsigned* status;
  int B, T, Hq, Hkv, G, d, blk, R, rpad;
  int nb, nb_max, num_pages, n_sel, sel_stride;
  // tokens of a partial last block (logical block nb), 0 if none: always
  // attended, as work unit n_sel (the draft tile follows it)
  int tail;
  // Work units of a (b, h): the n_sel selected blocks, then the draft tile
  // (unit n_sel). Split s covers units [s*bps, min(n_sel+1, (s+1)*bps)).
  int n_splits, bps;
  // Non-uniform split map (1-D grids): pairs [0, split_extra) have
  // n_splits + 1 splits, the others n_splits; partial slots of a pair are
  // slot_stride apart. Uniform plans: split_extra = 0, slot_stride = n_splits.
  int split_extra, slot_stride;
  // tcgen05 path: 1 = stream-K (n_splits CTAs, each an equal run of the
  // flattened (pair, unit) sequence; split_extra unused)
  int streamk;
  // 1: before the dependency wait, the producer may read sel and the block
  // table (relaxed; possibly stale) and prefetch the first pages into L2.
  // Set only when this call's selection was not just written by the
  // preceding kernel; a stale guess only costs bandwidth, never results.
  int spec_prefetch;
  // How long (ns) a CTA that finished its units waits for the rest of its
  // pair so that the pair's CTAs share the merge in row slices; whatever is
  // unclaimed when the wait ends is merged by the pair's last CTA to arrive.
  // 0: the last CTA merges every row and nothing waits.
  unsigned merge_wait_ns;
  // > 0 (tcgen05 path, one segment per CTA): the n_splits = cluster_merge CTAs of
  // a pair form one thread-block cluster and merge the pair's partials
  // through distributed shared memory at the end; no workspace partials,
  // counts or waits on other clusters.
  int cluster_merge;
  float scale_log2;     // log2(e) / sqrt(d)
  unsigned long long anc[kMaxT];  // bit u of anc[t]: draft t sees draft u
  VarLen vl;  // per-sequence nb, tail and n_sel (on = 0: the uniform ones)
};

// Overlap of per-draft selections (the shared-set diagnostic).
struct OverlapArgs {
  const int32_t* sels;  // [T][pairs][kmax], each row ascending in its first k
  float* overlap0;      // [pairs][T]: |S_0 ∩ S_t| / k
  float* by_distance;   // [pairs][T]: mean |S_t ∩ S_u| / k over t < u at each depth distance
  int T, pairs, kmax, k;
  int depth[kMaxT];     // depth of each draft in its tree
};
cudaError_t launch_overlap(const OverlapArgs& a, cudaStream_t st);

// The contexts of one call: uniform (var = false) or per sequence.
struct Ctxs {
  bool var;
  int nb, nb_min;  // largest and smallest full-block counts over sequences
  int tail;        // partial-block tokens (uniform contexts)
  VarLen vl;       // per sequence: nb and tail (n left to the caller)
};

// The counts of sequence b under a VarLen block (uniform values when off).
__host__ __device__ inline int nb_of(const VarLen& v, int b, int uniform) {
  return v.on ? v.nb[b] : uniform;
}
__host__ __device__ inline int tail_of(const VarLen& v, int b, int uniform) {
  return v.on ? v.tail[b] : uniform;
}
__host__ __device__ inline int n_of(const VarLen& v, int b, int uniform) {
  return v.on ? v.n[b] : uniform;
}

// CTA c of a 1-D grid under the non-uniform split map -> (pair, split, splits
// of that pair).
__host__ __device__ inline void split_of_cta(int c, int S, int extra, int* pair, int* split,
                                             int* nsp) {
  const int big = extra * (S + 1);
  if (c < big) {
    *pair = c / (S + 1);
    *split = c % (S + 1);
    *nsp = S + 1;
  } else {
    c -= big;
    *pair = extra + c / S;
    *split = c % S;
    *nsp = S;
  }
}

// Tensor-core path availability: bf16, d in {64,128}, blk in {32,64},
// rpad <= 128, T <= blk, 16-byte aligned pools, a non-empty pool.
bool attend_fast_applies(const AttendArgs& a, int dtype);
// Resident CTAs per SM of the tensor-core kernel (cluster-merge variant or
// global-partials variant) for this row count.
int attend_fast_ctas_per_sm(const AttendArgs& a, bool cluster);
// cluster > 0: splits of one (b, h) form a thread-block cluster of that size
// (== n_splits) and merge through distributed shared memory; cluster == 0:
// splits write global partials for launch_merge.
cudaError_t launch_attend_fast(const AttendArgs& a, int cluster, cudaStream_t st);
// tcgen05 path: bf16, d == 128, blk == 64, R <= 128, T <= 64.
// Merges each (b, h)'s split partials into out inside the same launch: with
// a.cluster_merge through distributed shared memory in the pair's cluster;
// otherwise from global partials (stream-K runs, or the split map above),
// by the pair's last CTA to arrive (alone when its copy is small, else
// sharing row slices with the pair's CTAs still waiting, for a bounded wait).
bool attend_tc_applies(const AttendArgs& a, int dtype);
int attend_tc_ctas_per_sm(const AttendArgs& a);
cudaError_t launch_attend_tc(AttendArgs a, cudaStream_t st);
// Largest cluster size in 4..16 (CTAs per pair, one pair per cluster) for
// which all `pairs` clusters of the tcgen05 kernel are resident at once, 0 if
// none.
int attend_tc_cluster(const AttendArgs& a, int pairs);
// True when one CTA merging a pair's slot_stride partial slots of rpad rows
// copies little enough that the pair's last CTA should merge it alone.
bool attend_tc_narrow_merge(int slot_stride, int rpad);
cudaError_t launch_attend_generic(const AttendArgs& a, int dtype, cudaStream_t st);
// Log-sum-exp merge of the global split partials into out (any path; honours
// the non-uniform split map).
cudaError_t launch_merge(const AttendArgs& a, int dtype, cudaStream_t st);


// Per-device once-only setup results (kernel attributes, occupancy), so that
// steady-state calls only launch kernels and can be captured in CUDA graphs.
int current_device();
int sm_count();  // SMs of the current device (cached per device)
constexpr int kMaxDevices = 64;

// TMA descriptor encoding through the driver entry point (no -lcuda).
bool encode_pool_map(CUtensorMap* map, const void* pool, int num_pages, int Hkv, int blk,
                     int d, const char** why);
// Q [B, T, Hq, d] bf16 viewed as (d, Hq, B*T) with boxes of (64, G, T): one
// box is the T*G stacked query rows of one kv head, 64 dims wide.
bool encode_draft_map(CUtensorMap* map, const void* dkv, int B, int T, int Hkv, int d, int rows,
                      const char** why);
bool encode_q_map(CUtensorMap* map, const void* q, int B, int T, int Hq, int G, int d,
                  const char** why);

}  // namespace sva
