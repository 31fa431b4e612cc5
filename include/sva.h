/*
 * sva.h -- C ABI of the sparse verification attention library (libsva.so).
 *
 * The method: a target LLM verifying T draft tokens against a long, paged KV
 * cache keeps only a budgeted set of KV blocks. Each block has a
 * representative; the first draft token's query is dotted with every
 * representative; a piecewise budget fixes how many top-scoring blocks are
 * kept; all T drafts attend to that ONE shared set plus the drafts the mask
 * lets them see; adjacent layers may reuse a previous layer's selection.
 *
 * Sources, cited by page title and part of the page:
 *   [SV-Fig1] "Accelerate Speculative Decoding with Sparse Computation in
 *             Verification" (paper summary page), Figure 1 caption.
 *   [SV-Abs]  same page, Abstract (inter-draft and inter-layer reuse).
 *   [SV-Tut1] same title, tutorial page, section "core technique 1" on sparse
 *             attention for multiple tokens: importance-based block choice,
 *             piecewise budget control, inter-layer retrieval reuse.
 *   [SpecPV]  "SpecPV: Improving self-speculative decoding for long-context
 *             generation via partial verification", introduction (full
 *             verification as the baseline).
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is caller-owned DEVICE memory unless the argument
 *     says "host". The library never allocates device memory.
 *   - Layouts are dense row-major (C order) with the shapes given.
 *   - dtype SV_BF16: q, k/v pools, draft k/v and out are bf16;
 *     SV_F32: all of them fp32. Representatives and scores are always fp32.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). The return value covers host-side validation and
 *     launch errors only. Device-side index checks (a block-table entry or a
 *     selected block out of range) skip the bad access and OR a flag into
 *     the workspace status word; read it with sv_read_status().
 *   - Validation happens before anything is launched: a call that returns
 *     SV_ERR_INVALID_ARG or SV_ERR_UNSUPPORTED has launched nothing.
 *   - Nothing throws across the ABI. sv_last_error() describes the last
 *     non-OK status of the calling thread.
 *   - Every call that enqueues GPU work is wrapped, on the host, in an NVTX
 *     range named after the call (visible to timeline tools; no cost
 *     without one).
 *   - Limits: 1 <= T <= 64; Hq % Hkv == 0; d % 8 == 0 and 8 <= d <= 256;
 *     NB = ctx/blk full blocks <= 16384; a partial last block (ctx % blk
 *     tokens) is allowed; B <= 64 when the cache gives per-sequence
 *     lengths (sv_kv.seq_ctx).
 */
#ifndef SVA_H_
#define SVA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_ABI_VERSION 4

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shape   */
  SV_ERR_UNSUPPORTED = 2,   /* valid but outside the limits above           */
  SV_ERR_WORKSPACE = 3,     /* workspace smaller than sv_workspace_bytes()  */
  SV_ERR_CUDA = 4,          /* a CUDA runtime call failed                   */
  SV_ERR_DEVICE_FAULT = 5   /* sv_read_status() found a device-side flag    */
} sv_status;

typedef enum { SV_BF16 = 0, SV_F32 = 1 } sv_dtype;

/* Device-side status flags (OR-ed into the workspace status word). */
#define SV_FLAG_BAD_BLOCK_INDEX 0x1u  /* selected block index outside [0, NB)  */
#define SV_FLAG_BAD_PAGE 0x2u         /* block_table entry outside [0, pages)  */
#define SV_FLAG_WAIT_TIMEOUT 0x4u     /* a pipeline wait gave up (never hangs) */
#define SV_FLAG_STALE_WORKSPACE 0x8u  /* a per-(b, h) merge word held a count left by an
                                         earlier call (sv_reset_workspace repairs it) */

/* Problem shape. Stacked query rows per KV head: R = T * (Hq / Hkv). */
typedef struct {
  int B;      /* sequences in the batch                                  */
  int Hq;     /* query heads                                             */
  int Hkv;    /* KV heads (grouped-query attention: G = Hq / Hkv)        */
  int d;      /* head dimension                                          */
  int blk;    /* tokens per KV block (page)                              */
  int T;      /* draft tokens being verified                             */
  int dtype;  /* sv_dtype                                                */
} sv_shape;

/* Piecewise budget control [SV-Tut1]. The pages give the shape of the rule
 * (more blocks kept at short context, harder sparsification at long context)
 * but no constants; the caller supplies them. */
#define SV_BUDGET_FIXED 0
#define SV_BUDGET_PIECEWISE 1
/* SMOOTH: the same page says the piecewise control makes the transition from
 * short to long context smooth. This library's reading of a curve without
 * jumps: a keep-rate of 1 per context token up to short_ctx, frac_mid up to
 * long_ctx and frac_long beyond, kept = its integral over [0, ctx), and
 * k = min(NB, max(floor, ceil(kept / ctx * NB))) (all NB up to short_ctx).
 * k never falls as ctx grows. Needs long_ctx >= short_ctx >= 0. Fractions are
 * read as decimals of up to nine places (0.1 is exactly one tenth). */
#define SV_BUDGET_SMOOTH 2
typedef struct {
  int mode;           /* SV_BUDGET_FIXED, SV_BUDGET_PIECEWISE or SMOOTH    */
  int fixed_blocks;   /* FIXED: k = min(NB, fixed_blocks)                  */
  int short_ctx;      /* PIECEWISE: ctx <= short_ctx keeps all NB blocks   */
  int floor_blocks;   /* otherwise k = min(NB, max(floor, ceil(frac*NB)))  */
  double frac_mid;    /*   frac = frac_mid when ctx <= long_ctx            */
  int long_ctx;
  double frac_long;   /*   frac = frac_long when ctx > long_ctx            */
} sv_budget;

/* Paged KV cache, caller-owned device memory. Page p of head h holds blk
 * consecutive tokens: k_pool[p][h][0..blk)[0..d). Every sequence has ctx
 * prefix tokens, or seq_ctx[b] when seq_ctx is given: NB = ctx/blk full
 * blocks and, when ctx % blk != 0, a partial last block (logical block NB,
 * its first ctx % blk tokens). Logical
 * block j of sequence b lives in page block_table[b * nb_max + j]. Only full
 * blocks have representatives and compete for the budget; a partial last
 * block is always attended, outside the budget (this library's reading of
 * the method for the step after drafts are accepted). Pool base addresses
 * must be 16-byte aligned. */
typedef struct {
  const void* k_pool;       /* [num_pages, Hkv, blk, d]                    */
  const void* v_pool;       /* [num_pages, Hkv, blk, d]                    */
  const int32_t* block_table; /* [B, nb_max]                              */
  int nb_max;               /* row stride of block_table, >= ceil(ctx/blk) */
  int num_pages;
  int ctx;                  /* prefix tokens per sequence (same for all)   */
  /* Per-sequence prefix lengths, HOST memory, B entries (B <= 64), or NULL
   * for the uniform ctx above (which is then ignored when non-NULL). Read
   * during the call only; the caller keeps ownership. With per-sequence
   * lengths every budget is taken per sequence (the piecewise rule of each
   * sequence's own ctx), sel rows hold k_b valid entries followed by -1, and
   * nb_max must cover the longest sequence. */
  const int32_t* seq_ctx;
} sv_kv;

/* ABI version (SV_ABI_VERSION of the built library). Host only. */
int sv_abi_version(void);

/* Thread-local description of the calling thread's last non-OK status. */
const char* sv_last_error(void);

/* Piecewise budget control [SV-Tut1]: number of blocks kept for a context of
 * ctx tokens in nb blocks. Pure host function, no GPU needed. Returns -1 on
 * an invalid budget (NULL, unknown mode, negative sizes, fractions outside
 * [0, 1], long_ctx < short_ctx in SMOOTH mode). */
int sv_budget_blocks(const sv_budget* budget, int ctx, int nb);

/* Bytes of workspace that score/select/attend/verify calls with this shape
 * need, for selections of up to kmax blocks over up to nb_max blocks. The
 * first 256 bytes hold the device status word; after it come three arrays
 * of per-(b, h) words, one 128-byte line each (the scoring count; the
 * attention's count of published partials and its merge tickets; a merge
 * claim word), then scores, pool rows and split partials. The whole workspace
 * must be zero before its first use (allocate it zeroed). Every call that
 * completes returns the per-(b, h) words to zero; the status word keeps its
 * flags until sv_clear_status. A call that raised SV_FLAG_WAIT_TIMEOUT may
 * leave those words non-zero: call sv_reset_workspace before the workspace
 * is used again. A call that finds a merge ticket beyond its pair's count
 * (a word left non-zero) raises SV_FLAG_STALE_WORKSPACE and leaves that
 * pair's output unwritten; the same reset repairs it. Returns 0 on an
 * invalid shape. Host only. */
size_t sv_workspace_bytes(const sv_shape* shape, int nb_max, int kmax);

/* Zero the workspace status word (async on stream). */
sv_status sv_clear_status(void* workspace, void* stream);

/* Zero the status word and every per-(b, h) count and flag of a workspace
 * laid out for (shape, nb_max, kmax) (async on stream): what a workspace
 * needs after a call that raised SV_FLAG_WAIT_TIMEOUT. Scores, rows and
 * partials need no reset (every call writes them before it reads them). */
sv_status sv_reset_workspace(const sv_shape* shape, int nb_max, int kmax, void* workspace,
                             size_t ws_bytes, void* stream);

/* Synchronously read the workspace status word into *flags (host). Returns
 * SV_ERR_DEVICE_FAULT when any flag is set. */
sv_status sv_read_status(const void* workspace, uint32_t* flags, void* stream);

/* Block representatives [SV-Fig1] (mean of a block's keys; the pages do not
 * define the representative, the mean is this library's reading):
 *   reps[b][h][j][:] = (1/blk) * sum_t K[page(b,j)][h][t][:],  fp32,
 * for logical blocks j in [first_block, first_block + n_blocks) of every
 * sequence. reps: [B, Hkv, nb_max, d] fp32, written only at those j. Call it
 * over all full blocks after prefill and again for each block that fills
 * up. Requires first_block >= 0, n_blocks >= 0, first_block + n_blocks <=
 * ctx/blk (with per-sequence lengths: the longest sequence's full blocks;
 * blocks at or past a shorter sequence's own ctx_b/blk are skipped for it). */
sv_status sv_build_reps(const sv_shape* shape, const sv_kv* kv, int first_block,
                        int n_blocks, float* reps, void* stream);

/* Block importance scores [SV-Fig1]: for every sequence b, KV head h and
 * block j < NB,
 *   scores[b][h][j] = sum_{g<G} < Q[b][0][h*G+g][:], reps[b][h][j][:] >
 * (draft 0's query; a KV head's score sums its G query heads' dot products;
 * no 1/sqrt(d), which does not change the ranking).
 * q: [B, T, Hq, d]; reps: [B, Hkv, nb_max, d]; scores: [B, Hkv, NB] fp32.
 * With per-sequence lengths NB is the longest sequence's full blocks (the
 * row stride); entries at or past sequence b's own ctx_b/blk are not
 * written. */
sv_status sv_score_blocks(const sv_shape* shape, const void* q, const float* reps,
                          const sv_kv* kv, float* scores, void* stream);

/* Top-k block selection [SV-Fig1], [SV-Tut1]: for every (b, h), the k
 * highest of scores[b][h][0..nb), ties to the lower block index, written in
 * ascending block order to sel[b][h][0..k); sel[b][h][k..kmax) = -1.
 * scores: [B, Hkv, nb] fp32; sel: [B, Hkv, kmax] int32; 0 <= k <= kmax;
 * k > nb keeps all nb blocks. Scores must be finite (NaN order undefined);
 * -0.0 and +0.0 tie. */
sv_status sv_select_blocks(const sv_shape* shape, const float* scores, int nb, int k,
                           int32_t* sel, int kmax, void* stream);

/* Score + budget + select in one call [SV-Fig1], [SV-Tut1]:
 * k = sv_budget_blocks(budget, kv->ctx, NB); scores go to the workspace;
 * sel as in sv_select_blocks; *k_out (host, may be NULL) receives k. With
 * per-sequence lengths (kv->seq_ctx), sequence b keeps
 * k_b = sv_budget_blocks(budget, seq_ctx[b], seq_ctx[b] / blk) blocks, its
 * sel rows hold k_b indices and then -1, and *k_out receives the largest k_b.
 * SV_ERR_INVALID_ARG if k (the largest k_b) > kmax. */
sv_status sv_score_select(const sv_shape* shape, const void* q, const float* reps,
                          const sv_kv* kv, const sv_budget* budget, int32_t* sel,
                          int kmax, int* k_out, void* workspace, size_t ws_bytes,
                          void* stream);

/* Sparse multi-token verification attention [SV-Fig1]: every draft row
 * (t, query head qh, KV head h = qh / G) attends, with softmax scale
 * 1/sqrt(d), to
 *   - every token of the n_sel blocks sel[b][h][0..n_sel) (logical block
 *     indices, the SAME set for all T drafts and all G heads of h), and
 *   - the drafts u that t may see: u = t and the ancestors of t.
 * draft_parent: HOST int[T] with draft_parent[0] = -1 and
 * 0 <= draft_parent[t] < t for t > 0 (a tree); NULL = linear chain.
 * sel == NULL selects all NB blocks in order: dense full verification
 * attention [SpecPV], the comparison baseline (n_sel is then ignored).
 * A partial last block (ctx % blk tokens) is attended in every case.
 * With per-sequence lengths, sel == NULL takes each sequence's own full
 * blocks, and a given sel must hold n_sel valid blocks of that sequence in
 * every row (the same n_sel for all; sv_verify_layer instead uses each
 * sequence's own budget).
 * sel: [B, Hkv, sel_stride] int32 with n_sel <= sel_stride.
 * q: [B, T, Hq, d]; draft_k, draft_v: [B, T, Hkv, d]; out: [B, T, Hq, d].
 * The workspace holds the split-KV partial results (its size from
 * sv_workspace_bytes with kmax >= n_sel, or >= NB when sel == NULL). */
sv_status sv_sparse_attend(const sv_shape* shape, const void* q, const sv_kv* kv,
                           const int32_t* sel, int n_sel, int sel_stride,
                           const void* draft_k, const void* draft_v,
                           const int32_t* draft_parent, void* out, void* workspace,
                           size_t ws_bytes, void* stream);

/* Which attention kernel and split plan sv_sparse_attend (and sv_verify_layer)
 * uses for this shape, cache and number of selected blocks: path
 * SV_PATH_TCGEN05 (bf16, d = 128, blk = 64, T*G <= 128: 5th-generation tensor
 * cores with TMEM accumulators), SV_PATH_MMA_SYNC (bf16, d in {64,128},
 * blk in {32,64}, T*G <= 128, T <= blk), else SV_PATH_CUDA_CORES; cluster > 0
 * when the splits of one (b, h) merge inside a thread-block cluster of that
 * size (on the tcgen05 path: 4 to 16 CTAs per (b, h) pair, merged through
 * distributed shared memory, when stream-K's merge would be wide: few pairs,
 * or 128-row tiles); split_extra > 0 when that many (b, h) pairs get n_splits + 1 splits;
 * streamk = 1 when n_splits CTAs instead share the work units of all pairs
 * in equal runs (the tcgen05 path when there are at least as many units as
 * CTAs and a run fits in one pair).
 * Queries the current device (occupancy); launches nothing. */
#define SV_PATH_CUDA_CORES 0
#define SV_PATH_MMA_SYNC 1
#define SV_PATH_TCGEN05 2
typedef struct {
  int path;
  int cluster;
  int n_splits;          /* CTAs per (b, h)                            */
  int blocks_per_split;  /* work units (selected blocks, draft tile)   */
  int ctas_per_sm;       /* resident CTAs per SM the plan assumed      */
  int split_extra;       /* pairs [0, split_extra) have n_splits + 1   */
  int streamk;           /* 1: n_splits CTAs each take an equal run of
                            the flattened (pair, unit) sequence, at
                            most two pairs per CTA (tcgen05 path)      */
} sv_plan;
sv_status sv_attend_plan(const sv_shape* shape, const sv_kv* kv, int n_sel, sv_plan* out);

/* Selection cache slot for inter-layer retrieval reuse [SV-Tut1] (core
 * technique 1, the paragraph on letting some layers reuse the previous
 * layer's retrieval): a layer may reuse only a selection that a computing
 * layer actually wrote for the same problem.
 *   sel:   DEVICE int32 [B, Hkv, kmax], caller-owned;
 *   kmax:  its row length (>= every budget it will hold);
 *   stamp: HOST-side digest, written by sv_verify_layer when it computes a
 *          selection into the slot (reuse == 0): a digest of B, Hkv, blk,
 *          kmax, the context length of every sequence and the budget k of
 *          every sequence. A reuse call (reuse == 1) computes the same digest
 *          for its own arguments and returns SV_ERR_INVALID_ARG, launching
 *          nothing, when the slot's stamp differs (a slot never written, or
 *          written for another context length, budget or shape). Set it to 0
 *          when the slot is created; copy it with the device contents when
 *          the slot is copied. */
typedef struct {
  int32_t* sel;
  int kmax;
  uint64_t stamp;
} sv_sel_slot;

/* One layer of sparse verification [SV-Fig1], [SV-Tut1], [SV-Abs]:
 *   reuse == 0: sv_score_select into slot->sel, then sv_sparse_attend on it,
 *               and slot->stamp set for this call;
 *   reuse == 1: inter-layer retrieval reuse -- no scoring or selection; the
 *               selection already in slot->sel, written by an earlier
 *               reuse == 0 call for the same shape, context lengths and
 *               budget (checked through slot->stamp), is attended to as is.
 *   reuse == 2: full verification [SpecPV] -- every block of the context is
 *               attended (as sv_sparse_attend with sel == NULL), for the
 *               periodic full-verification steps that partial verification
 *               interleaves; reps, budget and the slot are not used (slot may
 *               be NULL) and the slot keeps its contents and stamp.
 * reps may be NULL when reuse != 0. *k_out (host, may be NULL) receives the
 * number of blocks attended. */
sv_status sv_verify_layer(const sv_shape* shape, const void* q, const sv_kv* kv,
                          const float* reps, const sv_budget* budget,
                          const void* draft_k, const void* draft_v,
                          const int32_t* draft_parent, int reuse, sv_sel_slot* slot,
                          int* k_out, void* out, void* workspace, size_t ws_bytes,
                          void* stream);

/* sv_verify_layer with the step's per-token tensors in HOST memory: the
 * call a serving loop makes once the KV pool, representatives and slot live
 * on the device. On `stream` it enqueues, in order: the copies of q_host
 * [B, T, Hq, d], draft_k_host and draft_v_host [B, T, Hkv, d] into the
 * caller's device buffers q_dev, draft_k_dev, draft_v_dev (same shapes); the
 * verification exactly as sv_verify_layer (reuse, slot, k_out, workspace
 * alike); and the copy of the result out_dev [B, T, Hq, d] into out_host.
 * Element type: the shape's dtype. All of it is asynchronous: the host
 * buffers must stay valid, and unchanged, until the stream reaches the copies
 * (page-locked host memory makes the copies truly asynchronous). When
 * copy_in_stream / copy_out_stream are not NULL the input copies go on
 * copy_in_stream and the output copy on copy_out_stream, ordered against
 * `stream` by events the library records (one pool of events per device,
 * created on first use), so that the next call's inputs and this call's
 * output move while other work computes; the caller then must not reuse
 * the device buffers of a call before its output copy has completed
 * (rotating sets of buffers, as a serving loop double-buffers, is enough).
 * Validation is the same as sv_verify_layer's, done before anything is
 * enqueued; q_host, draft_k_host, draft_v_host and out_host must not be
 * NULL. */
sv_status sv_verify_layer_host(const sv_shape* shape, const void* q_host, void* q_dev,
                               const sv_kv* kv, const float* reps, const sv_budget* budget,
                               const void* draft_k_host, const void* draft_v_host,
                               void* draft_k_dev, void* draft_v_dev,
                               const int32_t* draft_parent, int reuse, sv_sel_slot* slot,
                               int* k_out, void* out_host, void* out_dev, void* workspace,
                               size_t ws_bytes, void* stream, void* copy_in_stream,
                               void* copy_out_stream);

/* Acceptance write-back: the step after verification. The pages have no
 * formula for it; it closes the loop that [SV-Fig1] verifies one step of:
 * the accepted drafts become context for the next step. Sequence b (ctx_b =
 * seq_ctx[b] tokens before the call) appends the K/V rows of drafts
 * accept_idx[b][0 .. n) in that order, n = n_accept[b] clamped to [0, T], at
 * token positions ctx_b, ctx_b + 1, ... (page block_table[b][pos / blk],
 * slot pos % blk), for every KV head. When reps is not NULL, every block the
 * append makes full (blocks ctx_b / blk .. (ctx_b + n) / blk - 1) gets its
 * representative rebuilt as in sv_build_reps.
 * k_pool, v_pool: [num_pages, Hkv, blk, d], written; block_table: [B, nb_max]
 * with the pages for the new positions already assigned; seq_ctx, n_accept:
 * DEVICE int32 [B]; accept_idx: DEVICE int32 [B, T]; draft_k, draft_v:
 * [B, T, Hkv, d]; reps: [B, Hkv, nb_max, d] fp32 or NULL; workspace (may be
 * NULL): a workspace whose status word receives SV_FLAG_BAD_BLOCK_INDEX for
 * a draft index outside [0, T) and SV_FLAG_BAD_PAGE for a position without a
 * valid page (those rows are skipped). Rows of different sequences must not
 * share pages. Asynchronous on stream. */
sv_status sv_append_kv(const sv_shape* shape, void* k_pool, void* v_pool,
                       const int32_t* block_table, int nb_max, int num_pages,
                       const int32_t* seq_ctx, const int32_t* n_accept,
                       const int32_t* accept_idx, const void* draft_k, const void* draft_v,
                       float* reps, void* workspace, void* stream);

/* Overlap of per-draft block selections: the measurement behind the figure
 * that follows the Figure 1 caption of [SV-Fig1] (overlap of the KV block
 * selection for draft-token pairs at different position distances), which
 * is the evidence that draft 0's set can serve every draft. The caller
 * scores and selects once per draft t with draft t's own query (for
 * example sv_score_blocks and sv_select_blocks on a T = 1 view of q) and
 * passes the T selections:
 *   sels: DEVICE int32 [T, pairs, kmax]; row (t, p) holds draft t's k kept
 *         blocks of pair p in ascending order (entries past k are ignored);
 *   draft_parent: HOST int[T] as in sv_sparse_attend (NULL = chain). A
 *         draft's position is ctx + its depth in the tree, so the position
 *         distance of drafts t and u is |depth(t) - depth(u)| (|t - u| in a
 *         chain); this is the library's reading of "position distance".
 * Writes (DEVICE float32):
 *   overlap0[p][t]    = |S_0 ∩ S_t| / k;
 *   by_distance[p][d] = mean of |S_t ∩ S_u| / k over draft pairs t < u at
 *                       distance d, NaN where no pair has distance d.
 * 1 <= T <= 64, 1 <= k <= kmax. Asynchronous on stream. */
sv_status sv_selection_overlap(const int32_t* sels, int T, int pairs, int kmax, int k,
                               const int32_t* draft_parent, float* overlap0,
                               float* by_distance, void* stream);

/* sv_sparse_attend without a workspace. The paper has no counterpart: this
 * entry exists for callers that cannot allocate device memory, such as an
 * operation hosted by another runtime (a plugin or callback handed only its
 * tensors) after that runtime's memory planner has claimed the device; such
 * a caller has no allocator to ask for a workspace, and a cudaMalloc at call
 * time would synchronise the device under the host runtime's schedule.
 *
 * Arguments q, kv, sel, n_sel, sel_stride, draft_k, draft_v, draft_parent
 * and out are those of sv_sparse_attend, and the result is the same (same
 * kernels, same split plan). flags_out: DEVICE uint32 (may be NULL) that
 * receives this call's device status flags (SV_FLAG_*), written on stream
 * after the attention.
 *
 * Scratch: a 16 MiB array in the library's device code, which every device
 * that loads the library holds until the process exits. No call allocates
 * (no cudaMalloc, no cudaFree, no allocating library routine). A call whose
 * split partials need more than 16 MiB returns SV_ERR_WORKSPACE and launches
 * nothing; sv_sparse_attend with a workspace handles it instead.
 * Set-up: the first call made with a given device current looks up the
 * array's device address there (cudaGetSymbolAddress), which may load the
 * library's device code; make that first call before any stream capture.
 * Every call zeroes the status word and arrival counters it uses on
 * `stream`. All calls on one device share the one array: two calls whose
 * work overlaps on the GPU (different streams, or different host threads,
 * without ordering between them) race and corrupt each other's results;
 * order them on one stream or with events. */
sv_status sv_sparse_attend_noalloc(const sv_shape* shape, const void* q, const sv_kv* kv,
                                   const int32_t* sel, int n_sel, int sel_stride,
                                   const void* draft_k, const void* draft_v,
                                   const int32_t* draft_parent, void* out, uint32_t* flags_out,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SVA_H_ */
