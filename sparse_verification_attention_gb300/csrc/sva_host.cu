// C ABI of libsva.so: argument validation, workspace carve-up, split-KV
// planning and kernel launches. Declarations and contracts: include/sva.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace sva {

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    int c = cached[dev].load();
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cached[dev].store(n);
  return n;
}

namespace {

thread_local std::string g_err;

sv_status fail(sv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

sv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

sv_status check_shape(const sv_shape* s) {
  if (!s) return fail(SV_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->d < 1 || s->blk < 1 || s->T < 1)
    return fail(SV_ERR_INVALID_ARG, "shape fields must be >= 1 (B=%d Hq=%d Hkv=%d d=%d blk=%d T=%d)",
                s->B, s->Hq, s->Hkv, s->d, s->blk, s->T);
  if (s->Hq % s->Hkv) return fail(SV_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", s->Hq, s->Hkv);
  if (s->dtype != SV_BF16 && s->dtype != SV_F32)
    return fail(SV_ERR_INVALID_ARG, "unknown dtype %d", s->dtype);
  if (s->d % 8 || s->d > kMaxD)
    return fail(SV_ERR_UNSUPPORTED, "head dim %d must be a multiple of 8 and <= %d", s->d, kMaxD);
  if (s->T > kMaxT) return fail(SV_ERR_UNSUPPORTED, "T=%d drafts exceeds %d", s->T, kMaxT);
  if ((long long)s->T * (s->Hq / s->Hkv) > 4096)
    return fail(SV_ERR_UNSUPPORTED, "T*G=%d stacked rows exceeds 4096", s->T * (s->Hq / s->Hkv));
  return SV_OK;
}

sv_status check_kv(const sv_shape* s, const sv_kv* kv, bool need_v) {
  if (!kv) return fail(SV_ERR_INVALID_ARG, "kv is NULL");
  int nb = 0, nblocks = 0;  // the largest over the sequences
  if (kv->seq_ctx) {
    if (s->B > kMaxVarB)
      return fail(SV_ERR_UNSUPPORTED, "B=%d sequences with per-sequence ctx exceeds %d", s->B,
                  kMaxVarB);
    for (int b = 0; b < s->B; ++b) {
      const int c = kv->seq_ctx[b];
      if (c < 0) return fail(SV_ERR_INVALID_ARG, "seq_ctx[%d]=%d is negative", b, c);
      nb = std::max(nb, c / s->blk);
      nblocks = std::max(nblocks, (c + s->blk - 1) / s->blk);
    }
  } else {
    if (kv->ctx < 0) return fail(SV_ERR_INVALID_ARG, "ctx=%d is negative", kv->ctx);
    nb = kv->ctx / s->blk;                        // full blocks
    nblocks = (kv->ctx + s->blk - 1) / s->blk;    // with a partial last one
  }
  if (nb > kMaxNB) return fail(SV_ERR_UNSUPPORTED, "NB=%d blocks exceeds %d", nb, kMaxNB);
  if (kv->nb_max < nblocks)
    return fail(SV_ERR_INVALID_ARG, "nb_max=%d < %d blocks holding the context", kv->nb_max,
                nblocks);
  if (nblocks > 0) {
    if (!kv->k_pool || (need_v && !kv->v_pool) || !kv->block_table)
      return fail(SV_ERR_INVALID_ARG, "k_pool/v_pool/block_table is NULL");
    if (kv->num_pages < 1) return fail(SV_ERR_INVALID_ARG, "num_pages=%d", kv->num_pages);
    if (!aligned(kv->k_pool, 16) || (need_v && !aligned(kv->v_pool, 16)))
      return fail(SV_ERR_INVALID_ARG, "k_pool/v_pool must be 16-byte aligned");
    if ((long long)(kv->num_pages + 1) * s->Hkv * s->blk >= (1ll << 31))
      return fail(SV_ERR_UNSUPPORTED, "pool of %d pages is too large", kv->num_pages);
  }
  return SV_OK;
}

// Full blocks and partial-block tokens of every sequence of a (validated)
// cache: uniform, or per sequence when kv->seq_ctx is given.
Ctxs ctxs_of(const sv_shape* s, const sv_kv* kv) {
  Ctxs c{};
  c.var = kv->seq_ctx != nullptr;
  c.vl.on = c.var ? 1 : 0;
  if (!c.var) {
    c.nb = c.nb_min = kv->ctx / s->blk;
    c.tail = kv->ctx % s->blk;
    return c;
  }
  c.nb_min = 1 << 30;
  for (int b = 0; b < s->B; ++b) {
    const int x = kv->seq_ctx[b];
    c.vl.nb[b] = x / s->blk;
    c.vl.tail[b] = x % s->blk;
    c.nb = std::max(c.nb, c.vl.nb[b]);
    c.nb_min = std::min(c.nb_min, c.vl.nb[b]);
  }
  if (s->B == 0) c.nb_min = 0;
  return c;
}

// The smooth curve: a keep-rate of 1 per context token up to short_ctx,
// frac_mid up to long_ctx and frac_long beyond; the kept tokens are its
// integral and k = min(nb, max(floor, ceil(kept / ctx * nb))). Fractions are
// taken as decimals of nine places, so the rounding up is exact.
static int smooth_budget_blocks(const sv_budget* bd, int ctx, int nb) {
  if (bd->short_ctx < 0 || bd->long_ctx < bd->short_ctx) return -1;
  if (ctx <= bd->short_ctx) return nb;
  const long long kDec = 1000000000LL;
  const long long fm = std::llround(bd->frac_mid * 1e9), fl = std::llround(bd->frac_long * 1e9);
  const long long mid = std::min<long long>(ctx, bd->long_ctx) - bd->short_ctx;
  const long long lng = std::max<long long>((long long)ctx - bd->long_ctx, 0);
  const __int128 kept = (__int128)bd->short_ctx * kDec + (__int128)fm * mid + (__int128)fl * lng;
  const __int128 num = kept * nb, den = (__int128)kDec * ctx;
  const long long want = (long long)((num + den - 1) / den);
  const long long k = want > bd->floor_blocks ? want : bd->floor_blocks;
  return (int)(k < nb ? k : nb);
}

int budget_blocks(const sv_budget* bd, int ctx, int nb) {
  if (!bd || ctx < 0 || nb < 0) return -1;
  if (bd->mode == SV_BUDGET_FIXED) {
    if (bd->fixed_blocks < 0) return -1;
    return nb < bd->fixed_blocks ? nb : bd->fixed_blocks;
  }
  if (bd->mode != SV_BUDGET_PIECEWISE && bd->mode != SV_BUDGET_SMOOTH) return -1;
  if (bd->floor_blocks < 0 || !(bd->frac_mid >= 0.0 && bd->frac_mid <= 1.0) ||
      !(bd->frac_long >= 0.0 && bd->frac_long <= 1.0))
    return -1;
  if (bd->mode == SV_BUDGET_SMOOTH) return smooth_budget_blocks(bd, ctx, nb);
  if (ctx <= bd->short_ctx) return nb;
  const double frac = (ctx <= bd->long_ctx) ? bd->frac_mid : bd->frac_long;
  // ceil(frac * nb) with a guard against products like 0.125*960 landing a
  // hair above an integer through rounding.
  const double prod = frac * (double)nb;
  long long want = (long long)std::ceil(prod - 1e-9 * (prod > 1.0 ? prod : 1.0));
  long long k = want > bd->floor_blocks ? want : bd->floor_blocks;
  return (int)(k < nb ? k : nb);
}


// Split planning for the global-partials path: enough CTAs to fill every SM
// `per_sm` deep in one wave, at most one split per work unit (a selected
// block or the draft tile), at most `max_splits`.
void plan_splits(int pairs, int n_units, int per_sm, int max_splits, int* n_splits, int* bps) {
  const int slots = sm_count() * (per_sm > 0 ? per_sm : 1);
  int s = slots / (pairs > 0 ? pairs : 1);
  if (s < 1) s = 1;
  if (s > max_splits) s = max_splits;
  if (s > n_units) s = n_units;
  const int per = (n_units + s - 1) / s;
  *bps = per;
  *n_splits = (n_units + per - 1) / per;
}

// Cluster size for the in-cluster merge path, or 0 when that path would leave
// more than half of the GPU idle (few (b, h) pairs): the largest cluster of
// at most 8 CTAs whose grid still fits in one wave.
// The whole grid must be resident at once: max_clusters(c) is how many
// clusters of c CTAs fit on the GPU.
template <typename MaxClusters>
int plan_cluster(int pairs, int n_units, int per_sm, int* bps, MaxClusters max_clusters) {
  const int slots = sm_count() * (per_sm > 0 ? per_sm : 1);
  int c = 8;
  while (c > 1 && pairs * c > slots) c >>= 1;
  if (c > n_units) c = n_units;
  if ((long long)pairs * c * 2 < slots) return 0;
  while (c > 1 && max_clusters(c) < pairs) --c;
  if (c <= 1) return 0;
  const int per = (n_units + c - 1) / c;
  *bps = per;
  return (n_units + per - 1) / per;
}

void fill_ancestors(const int32_t* parent, int T, unsigned long long* anc) {
  for (int t = 0; t < kMaxT; ++t) anc[t] = 0ull;
  for (int t = 0; t < T; ++t) {
    unsigned long long m = 0ull;
    int u = t;
    while (u >= 0) {
      m |= 1ull << u;
      u = parent ? parent[u] : u - 1;
    }
    anc[t] = m;
  }
}

sv_status check_parents(const int32_t* parent, int T) {
  if (!parent) return SV_OK;
  if (parent[0] != -1) return fail(SV_ERR_INVALID_ARG, "draft_parent[0]=%d must be -1", parent[0]);
  for (int t = 1; t < T; ++t)
    if (parent[t] < 0 || parent[t] >= t)
      return fail(SV_ERR_INVALID_ARG, "draft_parent[%d]=%d must be in [0,%d)", t, parent[t], t);
  return SV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encoded tensor maps, kept by what the encoding depends on (which map,
// base address, sizes): a map describes only an address range and its
// layout, so it stays valid for any later call on the same tensor, and the
// driver call that encodes it is skipped. A small set, replaced round-robin.
struct MapKey {
  int kind;
  const void* base;
  int v[6];
  bool operator==(const MapKey& o) const {
    if (kind != o.kind || base != o.base) return false;
    for (int i = 0; i < 6; ++i)
      if (v[i] != o.v[i]) return false;
    return true;
  }
};

template <typename Encode>
bool cached_map(const MapKey& key, CUtensorMap* map, Encode&& encode) {
  constexpr int kSlots = 64;
  static MapKey keys[kSlots];
  static CUtensorMap maps[kSlots];
  static bool used[kSlots];
  static int next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < kSlots; ++i)
      if (used[i] && keys[i] == key) {
        *map = maps[i];
        return true;
      }
  }
  if (!encode(map)) return false;
  std::lock_guard<std::mutex> g(mu);
  keys[next] = key;
  maps[next] = *map;
  used[next] = true;
  next = (next + 1) % kSlots;
  return true;
}

}  // namespace

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

WsLayout ws_layout(const sv_shape& s, int nb_max, int kmax) {
  WsLayout L;
  const int G = s.Hq / s.Hkv;
  L.rpad = round_up(s.T * G, 16);
  // one partial slot per work unit (selected blocks, a partial last block,
  // the draft tile), plus one for a stream-K run that leaves a pair
  // mid-stream
  const int units = (kmax < 0 ? 0 : kmax) + 2;
  L.slots = units + 1 > kMaxSplits ? kMaxSplits : units + 1;
  const size_t pairs = (size_t)s.B * s.Hkv;
  L.status = 0;
  const size_t words = align256(pairs * kPairWords * sizeof(uint32_t));  // one line per pair
  L.ctr_score = kStatusBytes;
  L.ctr_attend = L.ctr_score + words;
  L.claim = L.ctr_attend + words;
  L.scores = L.claim + words;
  L.rows = L.scores + align256(pairs * (size_t)(nb_max > 0 ? nb_max : 1) * sizeof(float));
  L.part_o = L.rows + align256(pairs * (size_t)(kmax > 0 ? kmax : 1) * sizeof(int32_t));
  L.part_ml = L.part_o + align256(pairs * L.slots * (size_t)L.rpad * s.d * sizeof(float));
  L.total = L.part_ml + align256(pairs * L.slots * (size_t)L.rpad * 2 * sizeof(float));
  return L;
}

static bool encode_pool_map_now(CUtensorMap* map, const void* pool, int num_pages, int Hkv,
                                int blk, int d, const char** why);
static bool encode_draft_map_now(CUtensorMap* map, const void* dkv, int B, int T, int Hkv, int d,
                                 int rows, const char** why);
static bool encode_q_map_now(CUtensorMap* map, const void* q, int B, int T, int Hq, int G, int d,
                             const char** why);

bool encode_pool_map(CUtensorMap* map, const void* pool, int num_pages, int Hkv, int blk, int d,
                     const char** why) {
  return cached_map(MapKey{0, pool, {num_pages, Hkv, blk, d, 0, 0}}, map, [&](CUtensorMap* m) {
    return encode_pool_map_now(m, pool, num_pages, Hkv, blk, d, why);
  });
}

bool encode_draft_map(CUtensorMap* map, const void* dkv, int B, int T, int Hkv, int d, int rows,
                      const char** why) {
  return cached_map(MapKey{1, dkv, {B, T, Hkv, d, rows, 0}}, map, [&](CUtensorMap* m) {
    return encode_draft_map_now(m, dkv, B, T, Hkv, d, rows, why);
  });
}

bool encode_q_map(CUtensorMap* map, const void* q, int B, int T, int Hq, int G, int d,
                  const char** why) {
  return cached_map(MapKey{2, q, {B, T, Hq, G, d, 0}}, map, [&](CUtensorMap* m) {
    return encode_q_map_now(m, q, B, T, Hq, G, d, why);
  });
}

static bool encode_pool_map_now(CUtensorMap* map, const void* pool, int num_pages, int Hkv,
                                int blk, int d, const char** why) {
  auto enc = get_encode();
  if (!enc) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)num_pages * Hkv * blk};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)blk};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed";
    return false;
  }
  return true;
}

static bool encode_draft_map_now(CUtensorMap* map, const void* dkv, int B, int T, int Hkv, int d,
                                 int rows, const char** why) {
  auto enc = get_encode();
  if (!enc) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  // [B, T, Hkv, d] viewed as (d, Hkv, T, B): one box = `rows` draft rows of
  // one kv head of one sequence, 64 dims wide; rows t >= T lie outside the
  // tensor and arrive as zeros
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2, (cuuint64_t)T * Hkv * d * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(dkv), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (draft) failed";
    return false;
  }
  return true;
}

static bool encode_q_map_now(CUtensorMap* map, const void* q, int B, int T, int Hq, int G, int d,
                             const char** why) {
  auto enc = get_encode();
  if (!enc) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)B * T};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)T};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (q) failed";
    return false;
  }
  return true;
}

// Path and split plan of one attention call (shared by the launch and by
// sv_attend_plan).
struct AttendPlan {
  int path;      // SV_PATH_*
  int cluster;   // > 0: in-cluster merge with this many CTAs per (b, h)
  int n_splits, bps, per_sm;
  int extra, slot_stride;  // non-uniform split map (tcgen05 path)
  int streamk;             // tcgen05 path: n_splits CTAs share the flattened units
};

// Stream-K plan of the tcgen05 path: G CTAs, CTA c covering flattened units
// [c*U/G, (c+1)*U/G) of U = pairs * W. Usable when every run is non-empty
// and no longer than one pair (so a run touches at most two pairs). Returns
// the largest number of partial slots a pair needs (its segments, plus one
// when its last segment ends mid-run), or 0 when stream-K does not apply.
static int streamk_slots(int pairs, int W, int G) {
  const long long U = (long long)pairs * W;
  if (G < 1 || U < G || (U + G - 1) / G > W) return 0;
  auto cta_of = [&](long long f) { return (int)(((f + 1) * G - 1) / U); };
  int most = 0;
  for (int p = 0; p < pairs; ++p) {
    const long long pend = (long long)(p + 1) * W;
    const int first = cta_of(pend - W), last = cta_of(pend - 1);
    const int mid = ((long long)(last + 1) * U / G > pend) ? 1 : 0;
    most = std::max(most, last - first + 1 + mid);
  }
  return most;
}

static AttendPlan make_plan(AttendArgs& a, int dtype, int pairs, int n_sel, int max_slots) {
  AttendPlan p{};
  // units of the largest pair: blocks, partial block, drafts
  int n_units = n_sel + (a.tail > 0 ? 1 : 0) + 1;
  if (a.vl.on) {
    n_units = 1;
    for (int b = 0; b < a.B; ++b)
      n_units = std::max(n_units, a.vl.n[b] + (a.vl.tail[b] > 0 ? 1 : 0) + 1);
  }
  const bool tcp = attend_tc_applies(a, dtype);
  const bool fast = !tcp && attend_fast_applies(a, dtype);
  p.path = tcp ? SV_PATH_TCGEN05 : fast ? SV_PATH_MMA_SYNC : SV_PATH_CUDA_CORES;
  if (tcp) {
    // one CTA per SM: spread exactly one wave of CTAs over the (b, h) pairs,
    // some pairs getting one split more than others
    p.per_sm = attend_tc_ctas_per_sm(a);
    const int slots = sm_count() * (p.per_sm > 0 ? p.per_sm : 1);
    // stream-K cuts equal runs of equal-length pairs: uniform contexts only
    const int sk = a.vl.on ? 0 : streamk_slots(pairs, n_units, slots);
    const bool sk_ok = sk > 0 && sk <= max_slots;
    // Stream-K uses every SM; it is kept when the pair's last CTA can merge
    // the pair alone (few partial slots of few rows). Otherwise -- few pairs
    // (many slots each), or 128-row tiles -- one cluster of 4 to 16 CTAs per
    // pair, the pair's units split evenly over it and merged through
    // distributed shared memory, when the device keeps all of them resident.
    const bool narrow = sk_ok && attend_tc_narrow_merge(sk, a.rpad);
    const int ncl = narrow ? 0 : attend_tc_cluster(a, pairs);
    if (ncl > 0 && n_units >= ncl) {
      p.cluster = ncl;
      p.n_splits = ncl;
      p.slot_stride = ncl;
      p.bps = (n_units + ncl - 1) / ncl;
      return p;
    }
    if (sk_ok) {
      p.streamk = 1;
      p.n_splits = slots;
      p.bps = (int)(((long long)pairs * n_units + slots - 1) / slots);
      p.slot_stride = sk;
      return p;
    }
    int S = slots / pairs, extra = slots % pairs;
    if (S < 1) {
      S = 1;
      extra = 0;
    }
    const int cap = n_units < max_slots ? n_units : max_slots;
    if (S + (extra ? 1 : 0) > cap) {
      S = cap;
      extra = 0;
    }
    p.n_splits = S;
    p.extra = extra;
    p.slot_stride = S + (extra ? 1 : 0);
    p.bps = (n_units + S - 1) / S;
    return p;
  }
  auto per_sm = [&](bool cl) { return fast ? attend_fast_ctas_per_sm(a, cl) : 4; };
  if (fast) {
    p.per_sm = per_sm(true);
    p.cluster = plan_cluster(pairs, n_units, p.per_sm, &p.bps, [](int) { return 1 << 30; });
  }
  if (p.cluster > 0) {
    p.n_splits = p.cluster;
  } else {
    p.per_sm = per_sm(false);
    plan_splits(pairs, n_units, p.per_sm, max_slots, &p.n_splits, &p.bps);
  }
  p.slot_stride = p.n_splits;
  return p;
}

static void fill_args(AttendArgs& a, const sv_shape* s, const void* q, const sv_kv* kv,
                      const int32_t* sel, int n_sel, int sel_stride, const void* dk,
                      const void* dv, const int32_t* parent, void* ws, const WsLayout& L);

static void set_nsel(AttendArgs& a, const int* nsel_b) {
  // per-sequence selected counts: given, else the call's n_sel (a selection
  // passed in) or every full block (sel == NULL)
  if (!a.vl.on) return;
  for (int b = 0; b < a.B; ++b) a.vl.n[b] = nsel_b ? nsel_b[b] : a.sel ? a.n_sel : a.vl.nb[b];
}

// fresh_sel: the selection was written by the kernel launched just before
// (score + select in the same call), so no speculative prefetch from it.
// rows: pool rows of sel written by the select step of this call (then no
// speculative prefetch either: the selection is fresh).
static sv_status run_attend(const sv_shape* s, const void* q, const sv_kv* kv, const int32_t* sel,
                            int n_sel, int sel_stride, const void* dk, const void* dv,
                            const int32_t* parent, void* out, void* ws, const WsLayout& L,
                            cudaStream_t st, const int* nsel_b = nullptr,
                            const int32_t* rows = nullptr) {
  AttendArgs a{};
  fill_args(a, s, q, kv, sel, n_sel, sel_stride, dk, dv, parent, ws, L);
  set_nsel(a, nsel_b);
  a.rows = rows;
  a.spec_prefetch = rows ? 0 : 1;
  a.out = out;
  const AttendPlan p = make_plan(a, s->dtype, s->B * s->Hkv, n_sel, L.slots);
  a.n_splits = p.n_splits;
  a.bps = p.bps;
  a.split_extra = p.extra;
  a.slot_stride = p.slot_stride;
  a.streamk = p.streamk;
  cudaError_t e;
  if (p.cluster > 0 && p.path != SV_PATH_TCGEN05) {
    e = launch_attend_fast(a, p.cluster, st);
    if (e != cudaSuccess) return cuda_fail(e, "attend launch");
    return SV_OK;
  }
  if (p.path == SV_PATH_TCGEN05) {  // merges in the same launch
    a.cluster_merge = p.cluster;
    e = launch_attend_tc(a, st);
    return e == cudaSuccess ? SV_OK : cuda_fail(e, "attend launch");
  }
  e = p.path == SV_PATH_MMA_SYNC ? launch_attend_fast(a, 0, st)
                                 : launch_attend_generic(a, s->dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "attend launch");
  e = launch_merge(a, s->dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return SV_OK;
}

static void fill_args(AttendArgs& a, const sv_shape* s, const void* q, const sv_kv* kv,
                      const int32_t* sel, int n_sel, int sel_stride, const void* dk,
                      const void* dv, const int32_t* parent, void* ws, const WsLayout& L) {
  a.q = q;
  a.k_pool = kv->k_pool;
  a.v_pool = kv->v_pool;
  a.draft_k = dk;
  a.draft_v = dv;
  a.block_table = kv->block_table;
  a.sel = sel;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.part_o = w ? reinterpret_cast<float*>(w + L.part_o) : nullptr;
  a.part_ml = w ? reinterpret_cast<float*>(w + L.part_ml) : nullptr;
  a.status = w ? reinterpret_cast<unsigned*>(w + L.status) : nullptr;
  a.counters = w ? reinterpret_cast<unsigned*>(w + L.ctr_attend) : nullptr;
  a.claim = w ? reinterpret_cast<unsigned*>(w + L.claim) : nullptr;
  a.B = s->B;
  a.T = s->T;
  a.Hq = s->Hq;
  a.Hkv = s->Hkv;
  a.G = s->Hq / s->Hkv;
  a.d = s->d;
  a.blk = s->blk;
  a.R = s->T * a.G;
  a.rpad = L.rpad;
  const Ctxs c = ctxs_of(s, kv);
  a.nb = c.nb;      // the largest sequence's full blocks
  a.tail = c.tail;  // uniform contexts (per sequence in a.vl otherwise)
  a.vl = c.vl;
  a.nb_max = kv->nb_max;
  a.num_pages = kv->num_pages;
  a.n_sel = n_sel;
  a.sel_stride = sel_stride;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s->d));
  fill_ancestors(parent, s->T, a.anc);
}

static sv_status check_ws(const sv_shape* s, int nb_max, int kmax, const void* ws, size_t bytes,
                          WsLayout* L) {
  *L = ws_layout(*s, nb_max, kmax);
  if (!ws) return fail(SV_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(SV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (bytes < L->total)
    return fail(SV_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, L->total);
  return SV_OK;
}

// Scores, budget and selection into sel; with `rows`, the kept blocks' pool
// rows too (the attention of the same call reads those instead of resolving
// sel through the block table).
static sv_status do_score_select(const sv_shape* s, const void* q, const float* reps,
                                 const sv_kv* kv, int k, int32_t* sel, int kmax, void* ws,
                                 const WsLayout& L, cudaStream_t st, const int* k_b = nullptr,
                                 int32_t* rows = nullptr) {
  Ctxs c = ctxs_of(s, kv);
  const int nb = c.nb;  // the largest sequence's (score rows keep this stride)
  if (c.vl.on)
    for (int b = 0; b < s->B; ++b) c.vl.n[b] = k_b[b];
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* scores = reinterpret_cast<float*>(w + L.scores);
  unsigned* status = reinterpret_cast<unsigned*>(w + L.status);
  const int32_t* bt = rows ? kv->block_table : nullptr;
  cudaError_t e;
  if (nb == 0) {
    // nothing to score: the selection is empty
    SelectArgs se{scores, sel, s->B * s->Hkv, 0, 0, kmax, s->Hkv, c.vl,
                  nullptr, nullptr, kv->nb_max, s->blk, kv->num_pages, status};
    e = launch_select(se, st);
  } else {
    ScoreArgs sa{q, reps, scores, s->B, s->T, s->Hq, s->Hkv, s->Hq / s->Hkv, s->d, nb, kv->nb_max,
                 0, sel, k, kmax, reinterpret_cast<unsigned*>(w + L.ctr_score), c.vl,
                 nb > kFusedSelectMaxNB ? nullptr : bt, rows, s->blk, kv->num_pages, status};
    e = launch_score(sa, s->dtype, st);
    if (e == cudaSuccess && nb > kFusedSelectMaxNB) {  // too many keys to fuse
      SelectArgs se{scores, sel, s->B * s->Hkv, nb, k, kmax, s->Hkv, c.vl,
                    bt, rows, kv->nb_max, s->blk, kv->num_pages, status};
      e = launch_select(se, st);
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "score/select launch");
  return SV_OK;
}

// ------------------------------------------------------------ allocation-free attend
// Scratch of sv_sparse_attend_noalloc. It is for callers that cannot hand the
// library a workspace: an operation hosted inside another runtime (a plugin
// or callback that receives only its input and output tensors) after that
// runtime's memory planner has claimed the device memory. Such a caller has
// no allocator to draw scratch from, and a cudaMalloc at call time would
// synchronise the whole device inside the host runtime's schedule. The
// scratch is module memory, reserved on each device when the library's
// device code is loaded there and held until the process exits; no call
// allocates anything. In host code the array's name is only a host-side
// stand-in for the symbol: kernels get its device address, looked up below.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device, looked up with that
// device current and cached per (device, context): a device reset or a
// re-created primary context loads the module again, possibly elsewhere, so
// a new context means a new lookup.
static std::mutex g_noalloc_mu;
static void* g_noalloc_ctx[kMaxDevices];
static void* g_noalloc_ptr[kMaxDevices];

static void* current_context() {
  using GetCurrent = int (*)(void**);  // cuCtxGetCurrent(CUcontext*)
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrent>(p);
  });
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

static sv_status noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(SV_ERR_UNSUPPORTED, "device %d: at most %d devices", dev, kMaxDevices);
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!ctx || ctx != g_noalloc_ctx[dev] || !g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (static scratch)");
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = current_context();  // the lookup may have made the context current
  }
  *ptr = g_noalloc_ptr[dev];
  return SV_OK;
}

// Status word, attend arrival counters (both zeroed by every call: the
// prefix [0, part_o)), then the split partials of the plan actually launched:
// slot_stride splits per pair rather than a workspace's worst case.
static WsLayout noalloc_layout(const sv_shape& s, int rpad, int slot_stride) {
  WsLayout L{};
  const size_t pairs = (size_t)s.B * s.Hkv;
  const size_t rows = pairs * (size_t)slot_stride * rpad;
  L.rpad = rpad;
  L.slots = slot_stride;
  L.status = 0;
  L.ctr_attend = kStatusBytes;
  L.ctr_score = L.ctr_attend;  // unused: this entry does not score
  const size_t words = align256(pairs * kPairWords * sizeof(uint32_t));  // one line per pair
  L.claim = L.ctr_attend + words;
  L.part_o = L.claim + words;
  L.scores = L.part_o;  // unused
  L.rows = L.part_o;    // unused
  L.part_ml = L.part_o + align256(rows * s.d * sizeof(float));
  L.total = L.part_ml + align256(rows * 2 * sizeof(float));
  return L;
}

// Digest of what a computed selection depends on beyond the inputs'
// values: batch and head layout, block size, row length, every sequence's
// context length and budget (FNV-1a, 64 bit; never 0, which marks a slot
// that no computing call has written).
static uint64_t selection_stamp(const sv_shape* s, const sv_kv* kv, const Ctxs& c, int kmax, int k,
                                const int* k_b) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](long long v) {
    for (int i = 0; i < 8; ++i) {
      h ^= (uint64_t)((v >> (8 * i)) & 0xff);
      h *= 1099511628211ull;
    }
  };
  mix(s->B);
  mix(s->Hkv);
  mix(s->blk);
  mix(kmax);
  mix(c.var ? 1 : 0);
  if (c.var) {
    for (int b = 0; b < s->B; ++b) {
      mix(kv->seq_ctx[b]);
      mix(k_b[b]);
    }
  } else {
    mix(kv->ctx);
    mix(k);
  }
  return h ? h : 1ull;
}

// The budget of every sequence (k_b[b], per-sequence contexts only) and
// the largest one; -1 for an invalid rule.
static int budgets_of(const sv_budget* bd, const sv_kv* kv, const Ctxs& c, int B, int* k_b) {
  if (!c.var) return budget_blocks(bd, kv->ctx, c.nb);
  int k = 0;
  for (int b = 0; b < B; ++b) {
    k_b[b] = budget_blocks(bd, kv->seq_ctx[b], c.vl.nb[b]);
    if (k_b[b] < 0) return -1;
    k = std::max(k, k_b[b]);
  }
  return k;
}

}  // namespace sva

using namespace sva;

namespace {
// An NVTX range named after the C-ABI call, around its whole host side
// (validation, planning, launches), for timeline tools; a no-op without one.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
}  // namespace

extern "C" {

int sv_abi_version(void) { return SV_ABI_VERSION; }

const char* sv_last_error(void) { return g_err.c_str(); }

int sv_budget_blocks(const sv_budget* budget, int ctx, int nb) {
  return budget_blocks(budget, ctx, nb);
}

size_t sv_workspace_bytes(const sv_shape* shape, int nb_max, int kmax) {
  if (check_shape(shape) != SV_OK || nb_max < 0 || kmax < 0) return 0;
  return ws_layout(*shape, nb_max, kmax).total;
}

sv_status sv_clear_status(void* workspace, void* stream) {
  const CallRange range("sv_clear_status");
  if (!workspace) return fail(SV_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "cudaMemsetAsync");
}

sv_status sv_reset_workspace(const sv_shape* shape, int nb_max, int kmax, void* workspace,
                             size_t ws_bytes, void* stream) {
  const CallRange range("sv_reset_workspace");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if (nb_max < 0 || kmax < 0)
    return fail(SV_ERR_INVALID_ARG, "nb_max=%d / kmax=%d is negative", nb_max, kmax);
  WsLayout L;
  if ((r = check_ws(shape, nb_max, kmax, workspace, ws_bytes, &L)) != SV_OK) return r;
  // the status word and the per-(b, h) words lie in front of the scores
  cudaError_t e = cudaMemsetAsync(workspace, 0, L.scores, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "cudaMemsetAsync");
}

sv_status sv_read_status(const void* workspace, uint32_t* flags, void* stream) {
  const CallRange range("sv_read_status");
  if (!workspace || !flags) return fail(SV_ERR_INVALID_ARG, "workspace/flags is NULL");
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *flags = v;
  if (v) return fail(SV_ERR_DEVICE_FAULT, "device status flags 0x%x", v);
  return SV_OK;
}

sv_status sv_build_reps(const sv_shape* shape, const sv_kv* kv, int first_block, int n_blocks,
                        float* reps, void* stream) {
  const CallRange range("sv_build_reps");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, false)) != SV_OK) return r;
  const Ctxs c = ctxs_of(shape, kv);
  const int nb = c.nb;  // blocks past a shorter sequence's own are skipped
  if (first_block < 0 || n_blocks < 0 || first_block + n_blocks > nb)
    return fail(SV_ERR_INVALID_ARG, "blocks [%d, %d) outside [0, %d)", first_block,
                first_block + n_blocks, nb);
  if (n_blocks == 0) return SV_OK;
  if (!reps || !aligned(reps, 16)) return fail(SV_ERR_INVALID_ARG, "reps NULL or not 16-byte aligned");
  RepsArgs a{kv->k_pool, kv->block_table, reps, shape->B, shape->Hkv, shape->d, shape->blk,
             kv->nb_max, kv->num_pages, first_block, n_blocks, nullptr, c.vl};
  cudaError_t e = launch_build_reps(a, shape->dtype, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "build_reps launch");
}

sv_status sv_append_kv(const sv_shape* shape, void* k_pool, void* v_pool, const int32_t* block_table,
                       int nb_max, int num_pages, const int32_t* seq_ctx, const int32_t* n_accept,
                       const int32_t* accept_idx, const void* draft_k, const void* draft_v,
                       float* reps, void* workspace, void* stream) {
  const CallRange range("sv_append_kv");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if (!k_pool || !v_pool || !block_table || !seq_ctx || !n_accept || !accept_idx || !draft_k ||
      !draft_v)
    return fail(SV_ERR_INVALID_ARG, "a pool, table, index array or draft tensor is NULL");
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(draft_k, 16) || !aligned(draft_v, 16))
    return fail(SV_ERR_INVALID_ARG, "pools and draft tensors must be 16-byte aligned");
  if (nb_max < 1 || num_pages < 1)
    return fail(SV_ERR_INVALID_ARG, "nb_max=%d / num_pages=%d", nb_max, num_pages);
  if (reps && !aligned(reps, 16)) return fail(SV_ERR_INVALID_ARG, "reps must be 16-byte aligned");
  if (workspace && !aligned(workspace, 256))
    return fail(SV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  unsigned* status = static_cast<unsigned*>(workspace);
  const AppendArgs ap{k_pool, v_pool, block_table, seq_ctx, n_accept, accept_idx, draft_k, draft_v,
                      status, shape->B, shape->T, shape->Hkv, shape->d, shape->blk, nb_max, num_pages};
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_append_kv(ap, shape->dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  if (reps) {
    const RepsArgs ra{k_pool, block_table, reps, shape->B, shape->Hkv, shape->d, shape->blk, nb_max,
                      num_pages, 0, 0, status};
    e = launch_append_reps(ra, ap, shape->dtype, st);
    if (e != cudaSuccess) return cuda_fail(e, "append reps launch");
  }
  return SV_OK;
}

sv_status sv_score_blocks(const sv_shape* shape, const void* q, const float* reps, const sv_kv* kv,
                          float* scores, void* stream) {
  const CallRange range("sv_score_blocks");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, false)) != SV_OK) return r;
  const Ctxs c = ctxs_of(shape, kv);
  const int nb = c.nb;
  if (nb == 0) return SV_OK;
  if (!q || !reps || !scores) return fail(SV_ERR_INVALID_ARG, "q/reps/scores is NULL");
  if (!aligned(q, 16) || !aligned(reps, 16))
    return fail(SV_ERR_INVALID_ARG, "q and reps must be 16-byte aligned");
  ScoreArgs sa{q, reps, scores, shape->B, shape->T, shape->Hq, shape->Hkv,
               shape->Hq / shape->Hkv, shape->d, nb, kv->nb_max, 0, nullptr, 0, 0, nullptr, c.vl,
               nullptr, nullptr, shape->blk, kv->num_pages, nullptr};
  cudaError_t e = launch_score(sa, shape->dtype, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "score launch");
}

sv_status sv_select_blocks(const sv_shape* shape, const float* scores, int nb, int k, int32_t* sel,
                           int kmax, void* stream) {
  const CallRange range("sv_select_blocks");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if (nb < 0 || nb > kMaxNB) return fail(SV_ERR_UNSUPPORTED, "nb=%d outside [0, %d]", nb, kMaxNB);
  if (k < 0 || k > kmax) return fail(SV_ERR_INVALID_ARG, "k=%d outside [0, kmax=%d]", k, kmax);
  if (kmax == 0) return SV_OK;
  if (!sel || (nb > 0 && !scores)) return fail(SV_ERR_INVALID_ARG, "scores/sel is NULL");
  SelectArgs se{scores, sel, shape->B * shape->Hkv, nb, k, kmax, shape->Hkv, VarLen{},
                nullptr, nullptr, 0, shape->blk, 0, nullptr};
  cudaError_t e = launch_select(se, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "select launch");
}

sv_status sv_score_select(const sv_shape* shape, const void* q, const float* reps, const sv_kv* kv,
                          const sv_budget* budget, int32_t* sel, int kmax, int* k_out,
                          void* workspace, size_t ws_bytes, void* stream) {
  const CallRange range("sv_score_select");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, false)) != SV_OK) return r;
  const Ctxs c = ctxs_of(shape, kv);
  const int nb = c.nb;
  int k_b[kMaxVarB];
  const int k = budgets_of(budget, kv, c, shape->B, k_b);
  if (k < 0) return fail(SV_ERR_INVALID_ARG, "invalid budget");
  if (k > kmax) return fail(SV_ERR_INVALID_ARG, "budget k=%d exceeds kmax=%d", k, kmax);
  if (kmax > 0 && !sel) return fail(SV_ERR_INVALID_ARG, "sel is NULL");
  if (nb > 0 && (!q || !reps)) return fail(SV_ERR_INVALID_ARG, "q/reps is NULL");
  if (nb > 0 && (!aligned(q, 16) || !aligned(reps, 16)))
    return fail(SV_ERR_INVALID_ARG, "q and reps must be 16-byte aligned");
  WsLayout L;
  if ((r = check_ws(shape, kv->nb_max, kmax, workspace, ws_bytes, &L)) != SV_OK) return r;
  if (k_out) *k_out = k;
  if (kmax == 0) return SV_OK;
  return do_score_select(shape, q, reps, kv, k, sel, kmax, workspace, L, (cudaStream_t)stream,
                         k_b);
}

sv_status sv_sparse_attend(const sv_shape* shape, const void* q, const sv_kv* kv, const int32_t* sel,
                           int n_sel, int sel_stride, const void* draft_k, const void* draft_v,
                           const int32_t* draft_parent, void* out, void* workspace,
                           size_t ws_bytes, void* stream) {
  const CallRange range("sv_sparse_attend");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, true)) != SV_OK) return r;
  const int nb = ctxs_of(shape, kv).nb;  // sel == NULL: each sequence's own blocks
  if (!sel) {
    n_sel = nb;
    sel_stride = nb;
  } else if (n_sel < 0 || n_sel > sel_stride) {
    return fail(SV_ERR_INVALID_ARG, "n_sel=%d outside [0, sel_stride=%d]", n_sel, sel_stride);
  }
  if (!q || !draft_k || !draft_v || !out)
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out is NULL");
  if (!aligned(q, 16) || !aligned(draft_k, 16) || !aligned(draft_v, 16) || !aligned(out, 16))
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out must be 16-byte aligned");
  if ((r = check_parents(draft_parent, shape->T)) != SV_OK) return r;
  WsLayout L;
  if ((r = check_ws(shape, kv->nb_max, n_sel, workspace, ws_bytes, &L)) != SV_OK) return r;
  return run_attend(shape, q, kv, sel, n_sel, sel_stride, draft_k, draft_v, draft_parent, out,
                    workspace, L, (cudaStream_t)stream);
}

sv_status sv_attend_plan(const sv_shape* shape, const sv_kv* kv, int n_sel, sv_plan* out) {
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, true)) != SV_OK) return r;
  if (!out) return fail(SV_ERR_INVALID_ARG, "out is NULL");
  if (n_sel < 0) return fail(SV_ERR_INVALID_ARG, "n_sel=%d is negative", n_sel);
  const WsLayout L = ws_layout(*shape, kv->nb_max, n_sel);
  AttendArgs a{};
  fill_args(a, shape, nullptr, kv, nullptr, n_sel, n_sel, nullptr, nullptr, nullptr, nullptr, L);
  if (a.vl.on)
    for (int b = 0; b < a.B; ++b) a.vl.n[b] = std::min(n_sel, a.vl.nb[b]);
  const AttendPlan p = make_plan(a, shape->dtype, shape->B * shape->Hkv, n_sel, L.slots);
  out->path = p.path;
  out->cluster = p.cluster;
  out->n_splits = p.n_splits;
  out->blocks_per_split = p.bps;
  out->ctas_per_sm = p.per_sm;
  out->split_extra = p.extra;
  out->streamk = p.streamk;
  return SV_OK;
}

namespace {

// The host side of sv_verify_layer_host: per-token inputs copied in before
// the first launch, the output copied back after the last.
struct HostIO {
  const void *q, *dk, *dv;
  void* out;
  size_t q_bytes, dkv_bytes;
  cudaStream_t in_st, out_st;  // null: the compute stream
};

// Events that order copy streams against the compute stream: a pool per
// device, created on first use and reused round-robin (an event may be
// recorded again once the waits on its earlier record have been enqueued,
// which happens within the same call).
cudaError_t pool_event(cudaEvent_t* ev) {
  constexpr int kEvents = 64;
  static cudaEvent_t pool[kMaxDevices][kEvents];
  static std::once_flag once[kMaxDevices];
  static std::atomic<unsigned> next[kMaxDevices];
  static cudaError_t made[kMaxDevices];
  const int dev = current_device();
  std::call_once(once[dev], [dev] {
    made[dev] = cudaSuccess;
    for (int i = 0; i < kEvents && made[dev] == cudaSuccess; ++i)
      made[dev] = cudaEventCreateWithFlags(&pool[dev][i], cudaEventDisableTiming);
  });
  if (made[dev] != cudaSuccess) return made[dev];
  *ev = pool[dev][next[dev].fetch_add(1) % kEvents];
  return cudaSuccess;
}

// Make `waiter` wait for the work enqueued so far on `producer`.
cudaError_t stream_after(cudaStream_t waiter, cudaStream_t producer) {
  cudaEvent_t ev;
  cudaError_t e = pool_event(&ev);
  if (e == cudaSuccess) e = cudaEventRecord(ev, producer);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
  return e;
}

sv_status stage_in(const HostIO* io, const void* q, const void* dk, const void* dv,
                   cudaStream_t st) {
  if (!io) return SV_OK;
  const cudaStream_t cs = io->in_st ? io->in_st : st;
  cudaError_t e = cudaMemcpyAsync(const_cast<void*>(q), io->q, io->q_bytes,
                                  cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<void*>(dk), io->dk, io->dkv_bytes, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<void*>(dv), io->dv, io->dkv_bytes, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess && io->in_st) e = stream_after(st, io->in_st);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "input copy");
}

sv_status stage_out(const HostIO* io, const void* out, cudaStream_t st) {
  if (!io) return SV_OK;
  cudaError_t e = cudaSuccess;
  if (io->out_st) e = stream_after(io->out_st, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(io->out, out, io->q_bytes, cudaMemcpyDeviceToHost,
                        io->out_st ? io->out_st : st);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "output copy");
}

sv_status verify_layer(const sv_shape* shape, const void* q, const sv_kv* kv, const float* reps,
                       const sv_budget* budget, const void* draft_k, const void* draft_v,
                       const int32_t* draft_parent, int reuse, sv_sel_slot* slot, int* k_out,
                       void* out, void* workspace, size_t ws_bytes, void* stream,
                       const HostIO* io) {
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, true)) != SV_OK) return r;
  if (reuse < 0 || reuse > 2)
    return fail(SV_ERR_INVALID_ARG, "reuse=%d must be 0, 1 or 2", reuse);
  if (reuse != 2 && !slot) return fail(SV_ERR_INVALID_ARG, "selection slot is NULL");
  const int kmax = slot ? slot->kmax : 0;
  int32_t* sel_cache = slot ? slot->sel : nullptr;
  if (kmax < 0) return fail(SV_ERR_INVALID_ARG, "slot kmax=%d is negative", kmax);
  const Ctxs c = ctxs_of(shape, kv);
  const int nb = c.nb;
  if (reuse == 2) {
    // full verification: every block, no scoring, selection or budget
    if (!q || !draft_k || !draft_v || !out)
      return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out is NULL");
    if (!aligned(q, 16) || !aligned(draft_k, 16) || !aligned(draft_v, 16) || !aligned(out, 16))
      return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out must be 16-byte aligned");
    if ((r = check_parents(draft_parent, shape->T)) != SV_OK) return r;
    // partial slots for all nb blocks when the workspace holds them (as
    // sv_sparse_attend with sel == NULL), else for the slot's kmax
    WsLayout L;
    const int kws = ws_layout(*shape, kv->nb_max, std::max(kmax, nb)).total <= ws_bytes
                        ? std::max(kmax, nb) : kmax;
    if ((r = check_ws(shape, kv->nb_max, kws, workspace, ws_bytes, &L)) != SV_OK) return r;
    if (k_out) *k_out = nb;
    const cudaStream_t st = (cudaStream_t)stream;
    if ((r = stage_in(io, q, draft_k, draft_v, st)) != SV_OK) return r;
    r = run_attend(shape, q, kv, nullptr, nb, nb, draft_k, draft_v, draft_parent, out, workspace,
                   L, st);
    return r == SV_OK ? stage_out(io, out, st) : r;
  }
  int k_b[kMaxVarB];
  const int k = budgets_of(budget, kv, c, shape->B, k_b);
  if (k < 0) return fail(SV_ERR_INVALID_ARG, "invalid budget");
  if (k > kmax) return fail(SV_ERR_INVALID_ARG, "budget k=%d exceeds kmax=%d", k, kmax);
  if (kmax > 0 && !sel_cache) return fail(SV_ERR_INVALID_ARG, "sel_cache is NULL");
  if (!q || !draft_k || !draft_v || !out)
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out is NULL");
  if (!aligned(q, 16) || !aligned(draft_k, 16) || !aligned(draft_v, 16) || !aligned(out, 16))
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out must be 16-byte aligned");
  if (!reuse && nb > 0 && (!reps || !aligned(reps, 16)))
    return fail(SV_ERR_INVALID_ARG, "reps NULL or not 16-byte aligned");
  if ((r = check_parents(draft_parent, shape->T)) != SV_OK) return r;
  WsLayout L;
  if ((r = check_ws(shape, kv->nb_max, kmax, workspace, ws_bytes, &L)) != SV_OK) return r;
  const uint64_t stamp = selection_stamp(shape, kv, c, kmax, k, k_b);
  if (reuse == 1 && slot->stamp != stamp)
    return fail(SV_ERR_INVALID_ARG,
                slot->stamp ? "reuse of a selection computed for another shape, context or budget"
                            : "reuse of a selection slot that no computing call has written");
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = stage_in(io, q, draft_k, draft_v, st)) != SV_OK) return r;
  int32_t* rows = nullptr;
  if (!reuse && kmax > 0) {
    rows = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + L.rows);
    r = do_score_select(shape, q, reps, kv, k, sel_cache, kmax, workspace, L, st, k_b, rows);
    if (r != SV_OK) return r;
  }
  if (k_out) *k_out = k;
  r = run_attend(shape, q, kv, sel_cache, k, kmax, draft_k, draft_v, draft_parent, out, workspace,
                 L, st, c.var ? k_b : nullptr, rows);
  if (r == SV_OK && reuse == 0) slot->stamp = stamp;
  return r == SV_OK ? stage_out(io, out, st) : r;
}

}  // namespace

sv_status sv_verify_layer(const sv_shape* shape, const void* q, const sv_kv* kv, const float* reps,
                          const sv_budget* budget, const void* draft_k, const void* draft_v,
                          const int32_t* draft_parent, int reuse, sv_sel_slot* slot, int* k_out,
                          void* out, void* workspace, size_t ws_bytes, void* stream) {
  const CallRange range("sv_verify_layer");
  return verify_layer(shape, q, kv, reps, budget, draft_k, draft_v, draft_parent, reuse, slot,
                      k_out, out, workspace, ws_bytes, stream, nullptr);
}

sv_status sv_verify_layer_host(const sv_shape* shape, const void* q_host, void* q_dev,
                               const sv_kv* kv, const float* reps, const sv_budget* budget,
                               const void* draft_k_host, const void* draft_v_host,
                               void* draft_k_dev, void* draft_v_dev,
                               const int32_t* draft_parent, int reuse, sv_sel_slot* slot,
                               int* k_out, void* out_host, void* out_dev, void* workspace,
                               size_t ws_bytes, void* stream, void* copy_in_stream,
                               void* copy_out_stream) {
  const CallRange range("sv_verify_layer_host");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if (!q_host || !draft_k_host || !draft_v_host || !out_host)
    return fail(SV_ERR_INVALID_ARG, "q_host/draft_k_host/draft_v_host/out_host is NULL");
  const size_t es = shape->dtype == SV_BF16 ? 2 : 4;
  const size_t rows = (size_t)shape->B * shape->T;
  const HostIO io{q_host, draft_k_host, draft_v_host, out_host,
                  rows * shape->Hq * shape->d * es, rows * shape->Hkv * shape->d * es,
                  (cudaStream_t)copy_in_stream, (cudaStream_t)copy_out_stream};
  return verify_layer(shape, q_dev, kv, reps, budget, draft_k_dev, draft_v_dev, draft_parent,
                      reuse, slot, k_out, out_dev, workspace, ws_bytes, stream, &io);
}

sv_status sv_sparse_attend_noalloc(const sv_shape* shape, const void* q, const sv_kv* kv,
                                   const int32_t* sel, int n_sel, int sel_stride,
                                   const void* draft_k, const void* draft_v,
                                   const int32_t* draft_parent, void* out, uint32_t* flags_out,
                                   void* stream) {
  const CallRange range("sv_sparse_attend_noalloc");
  sv_status r = check_shape(shape);
  if (r != SV_OK) return r;
  if ((r = check_kv(shape, kv, true)) != SV_OK) return r;
  const int nb = ctxs_of(shape, kv).nb;  // sel == NULL: each sequence's own blocks
  if (!sel) {
    n_sel = nb;
    sel_stride = nb;
  } else if (n_sel < 0 || n_sel > sel_stride) {
    return fail(SV_ERR_INVALID_ARG, "n_sel=%d outside [0, sel_stride=%d]", n_sel, sel_stride);
  }
  if (!q || !draft_k || !draft_v || !out)
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out is NULL");
  if (!aligned(q, 16) || !aligned(draft_k, 16) || !aligned(draft_v, 16) || !aligned(out, 16))
    return fail(SV_ERR_INVALID_ARG, "q/draft_k/draft_v/out must be 16-byte aligned");
  if (flags_out && !aligned(flags_out, 4))
    return fail(SV_ERR_INVALID_ARG, "flags_out must be 4-byte aligned");
  if ((r = check_parents(draft_parent, shape->T)) != SV_OK) return r;
  // the same plan sv_sparse_attend makes for this call
  const WsLayout W = ws_layout(*shape, kv->nb_max, n_sel);
  AttendArgs a{};
  fill_args(a, shape, q, kv, sel, n_sel, sel_stride, draft_k, draft_v, draft_parent, nullptr, W);
  set_nsel(a, nullptr);
  a.out = out;
  a.spec_prefetch = 1;
  const AttendPlan p = make_plan(a, shape->dtype, shape->B * shape->Hkv, n_sel, W.slots);
  const WsLayout L = noalloc_layout(*shape, W.rpad, p.slot_stride);
  if (L.total > kNoAllocScratchBytes)
    return fail(SV_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch; the static scratch holds %zu "
                "(use sv_sparse_attend with a workspace)",
                L.total, kNoAllocScratchBytes);
  void* base = nullptr;
  if ((r = noalloc_scratch(&base)) != SV_OK) return r;
  uint8_t* w = static_cast<uint8_t*>(base);
  a.status = reinterpret_cast<unsigned*>(w + L.status);
  a.counters = reinterpret_cast<unsigned*>(w + L.ctr_attend);
  a.claim = reinterpret_cast<unsigned*>(w + L.claim);
  a.part_o = reinterpret_cast<float*>(w + L.part_o);
  a.part_ml = reinterpret_cast<float*>(w + L.part_ml);
  a.n_splits = p.n_splits;
  a.bps = p.bps;
  a.split_extra = p.extra;
  a.slot_stride = p.slot_stride;
  a.streamk = p.streamk;
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: zero the status word and
  // the arrival counters (the partials are fully written before being read)
  cudaError_t e = cudaMemsetAsync(base, 0, L.part_o, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (static scratch)");
  if (p.cluster > 0 && p.path != SV_PATH_TCGEN05) {
    e = launch_attend_fast(a, p.cluster, st);
  } else if (p.path == SV_PATH_TCGEN05) {
    a.cluster_merge = p.cluster;
    e = launch_attend_tc(a, st);
  } else {
    e = p.path == SV_PATH_MMA_SYNC ? launch_attend_fast(a, 0, st)
                                   : launch_attend_generic(a, shape->dtype, st);
    if (e == cudaSuccess) e = launch_merge(a, shape->dtype, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attend launch");
  if (flags_out) {
    e = cudaMemcpyAsync(flags_out, base, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
  }
  return SV_OK;
}

sv_status sv_selection_overlap(const int32_t* sels, int T, int pairs, int kmax, int k,
                               const int32_t* draft_parent, float* overlap0, float* by_distance,
                               void* stream) {
  const CallRange range("sv_selection_overlap");
  if (T < 1 || T > kMaxT) return fail(SV_ERR_UNSUPPORTED, "T=%d outside [1, %d]", T, kMaxT);
  if (pairs < 0 || kmax < 1 || k < 1 || k > kmax)
    return fail(SV_ERR_INVALID_ARG, "pairs=%d, k=%d, kmax=%d: need pairs >= 0, 1 <= k <= kmax",
                pairs, k, kmax);
  if (pairs > 0 && (!sels || !overlap0 || !by_distance))
    return fail(SV_ERR_INVALID_ARG, "sels/overlap0/by_distance is NULL");
  sv_status r = check_parents(draft_parent, T);
  if (r != SV_OK) return r;
  OverlapArgs a{sels, overlap0, by_distance, T, pairs, kmax, k, {}};
  for (int t = 0; t < T; ++t)
    a.depth[t] = t == 0 ? 0 : a.depth[draft_parent ? draft_parent[t] : t - 1] + 1;
  const cudaError_t e = launch_overlap(a, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "overlap launch");
}

}  // extern "C"
