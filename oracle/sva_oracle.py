"""CPU oracle for sparse verification attention (TEST INFRASTRUCTURE ONLY).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this module. The CUDA library never calls it, and it imports nothing
from the CUDA path: it is a plain, slow, fp64 restatement of the method, step
by step, so that a reader can check it against the pages by eye.

Sources (page title, then the part of the page):
  [SV-Fig1]  "Accelerate Speculative Decoding with Sparse Computation in
             Verification", paper summary page, Figure 1 caption.
  [SV-Abs]   the same page, Abstract.
  [SV-Tut1]  the same title, tutorial page, section "Core technique 1: sparse
             attention for multiple tokens" (the piecewise budget and the
             inter-layer retrieval reuse paragraphs belong to it).
  [SpecPV]   "SpecPV: Improving self-speculative decoding for long-context
             generation via partial verification", introduction (full vs.
             partial verification).

Readings where the pages are silent, ambiguous or garbled:
  R1 block representative = mean of the block's keys (the pages never define
     it); computed in fp64.
  R2 the scoring query is draft 0's (tree root's) query; with grouped-query
     attention a KV head's score is the SUM over its G query heads of the
     per-head dot products; no 1/sqrt(d) (it does not change the ranking).
  R3 budget: all blocks when ctx <= short_ctx; otherwise
     min(NB, max(floor, ceil(frac * NB))) with frac = frac_mid up to long_ctx
     and frac_long beyond; FIXED mode gives min(NB, fixed).
  R3b smooth budget (SMOOTH mode, a variant of R3): the pages say the
     piecewise control gives a smooth transition from short to long context.
     Reading: the keep-rate per context token is piecewise constant (1 up to
     short_ctx, frac_mid up to long_ctx, frac_long beyond), and the kept
     budget is its integral, so it is continuous and never falls as ctx
     grows. As a fraction of the blocks, k = min(NB, max(floor,
     ceil(kept_tokens / ctx * NB))).
  R4 top-k ties go to the lower block index; the selected set is reported in
     ascending block order.
  R5 draft-to-draft mask: draft t sees itself and its ancestors (a chain is
     the special case parent[t] = t-1). Prefix tokens of selected blocks are
     visible to every draft.
  R6 softmax scale 1/sqrt(d); Q and K are post-positional-encoding inputs.
  R7 reuse: a reuse layer takes the selection of the previous computing layer
     unchanged and does no scoring or selection of its own.
  R8 a context that ends in a partial block: only the ctx // blk full blocks
     get representatives and compete for the budget; the partial block's
     ctx % blk tokens are always attended, outside the budget. Accepted drafts
     are appended at positions ctx, ctx+1, ... in the order accepted.
  R10 the position distance of two drafts (the overlap diagnostic) is the
     difference of their depths in the draft tree: a draft sits at position
     ctx + depth; in a chain that is |t - u|.

Parity status: every function here is pinned by tests/test_oracle_pins.py
against closed forms, brute force, invariants or torch SDPA, except R1's
choice of *mean* as the representative, which the pages leave open
("parity unpinned" for that reading; the mean itself is pinned).
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Optional, Sequence

import torch

F64 = torch.float64

BUDGET_FIXED = 0
BUDGET_PIECEWISE = 1
BUDGET_SMOOTH = 2


# --------------------------------------------------------------------------
# C1  block representatives  [SV-Fig1]; reading R1
# --------------------------------------------------------------------------
def block_representatives(k_pool: torch.Tensor, block_table: torch.Tensor,
                          n_blocks: int, blk: int) -> torch.Tensor:
    """rep[b, h, j, :] = (1/blk) * sum of the blk keys of logical block j.

    k_pool: [P, Hkv, blk, d] (any float dtype); block_table: [B, >=n_blocks].
    Returns fp64 [B, Hkv, n_blocks, d].
    """
    B = block_table.shape[0]
    P, Hkv, blk_, d = k_pool.shape
    assert blk_ == blk
    reps = torch.zeros(B, Hkv, n_blocks, d, dtype=F64)
    for b in range(B):
        for j in range(n_blocks):
            page = int(block_table[b, j])
            keys = k_pool[page].to(F64)          # [Hkv, blk, d]
            reps[b, :, j, :] = keys.sum(dim=1) / blk
    return reps


# --------------------------------------------------------------------------
# C2  block scores  [SV-Fig1], [SV-Tut1]; reading R2
# --------------------------------------------------------------------------
def block_scores(q: torch.Tensor, reps: torch.Tensor, G: int) -> torch.Tensor:
    """s[b, h, j] = sum_{g<G} < Q[b, 0, h*G+g, :], rep[b, h, j, :] >.

    q: [B, T, Hq, d]; reps: [B, Hkv, NB, d]. Returns fp64 [B, Hkv, NB].
    """
    B, T, Hq, d = q.shape
    Hkv = reps.shape[1]
    assert Hq == Hkv * G
    s = torch.zeros(B, Hkv, reps.shape[2], dtype=F64)
    for b in range(B):
        for h in range(Hkv):
            R = reps[b, h].to(F64)               # [NB, d]
            for g in range(G):
                q0 = q[b, 0, h * G + g].to(F64)   # draft 0's query, one head
                s[b, h] += R @ q0
    return s


# --------------------------------------------------------------------------
# C3  piecewise budget  [SV-Tut1]; reading R3
# --------------------------------------------------------------------------
def budget_blocks(ctx: int, nb: int, mode: int, fixed_blocks: int = 0,
                  short_ctx: int = 0, floor_blocks: int = 0, frac_mid: float = 0.0,
                  long_ctx: int = 0, frac_long: float = 0.0) -> int:
    """Number of KV blocks kept for a context of ctx tokens in nb full blocks."""
    if mode == BUDGET_FIXED:
        return min(nb, fixed_blocks)
    if mode == BUDGET_SMOOTH:
        return smooth_budget_blocks(ctx, nb, short_ctx, floor_blocks, frac_mid, long_ctx,
                                    frac_long)
    if ctx <= short_ctx:
        return nb                                # short context: keep everything
    # fractions are decimal percentages (12.5% = 0.125): ceil of the exact
    # decimal product, not of its binary floating-point approximation
    frac = Fraction(repr(frac_mid)) if ctx <= long_ctx else Fraction(repr(frac_long))
    want = math.ceil(frac * nb)
    return min(nb, max(floor_blocks, want))


def smooth_kept_tokens(ctx: int, short_ctx: int, frac_mid: float, long_ctx: int,
                       frac_long: float) -> Fraction:
    """Reading R3b: the context tokens' worth of budget kept at length ctx,
    the integral of a keep-rate of 1 on [0, short_ctx], frac_mid on
    (short_ctx, long_ctx] and frac_long beyond (fractions as decimals)."""
    fm, fl = Fraction(repr(frac_mid)), Fraction(repr(frac_long))
    short_part = min(ctx, short_ctx)
    mid_part = min(max(ctx - short_ctx, 0), long_ctx - short_ctx)
    long_part = max(ctx - long_ctx, 0)
    return short_part + fm * mid_part + fl * long_part


def smooth_budget_blocks(ctx: int, nb: int, short_ctx: int, floor_blocks: int,
                         frac_mid: float, long_ctx: int, frac_long: float) -> int:
    """Blocks kept under reading R3b: the kept fraction of the context,
    kept_tokens / ctx, applied to the nb full blocks and rounded up, then
    at least floor and at most nb. Everything is kept up to short_ctx."""
    if ctx <= short_ctx:
        return nb
    kept = smooth_kept_tokens(ctx, short_ctx, frac_mid, long_ctx, frac_long)
    want = math.ceil(kept / ctx * nb)
    return min(nb, max(floor_blocks, want))


def budget_from(budget, ctx: int, nb: int) -> int:
    """budget_blocks() with the fields of a workloads.Budget-like object."""
    return budget_blocks(ctx, nb, budget.mode, budget.fixed_blocks, budget.short_ctx,
                         budget.floor_blocks, budget.frac_mid, budget.long_ctx,
                         budget.frac_long)


# --------------------------------------------------------------------------
# C4  top-k selection  [SV-Fig1], [SV-Tut1]; reading R4
# --------------------------------------------------------------------------
def select_blocks(scores_row: Sequence[float], k: int) -> list[int]:
    """Indices of the k highest scores (lower index first on ties), ascending."""
    vals = [float(x) for x in scores_row]
    order = sorted(range(len(vals)), key=lambda j: (-vals[j], j))
    return sorted(order[:k])


def select_all(scores: torch.Tensor, k: int) -> torch.Tensor:
    """select_blocks() for every (b, h): [B, Hkv, NB] -> int64 [B, Hkv, k]."""
    B, Hkv, NB = scores.shape
    sel = torch.empty(B, Hkv, k, dtype=torch.int64)
    for b in range(B):
        for h in range(Hkv):
            sel[b, h] = torch.tensor(select_blocks(scores[b, h].tolist(), k),
                                     dtype=torch.int64)
    return sel


def boundary_gap(scores_row: Sequence[float], k: int) -> Optional[float]:
    """Relative gap between the k-th and (k+1)-th highest scores, or None when
    k == 0 or k >= NB (no boundary exists)."""
    vals = sorted((float(x) for x in scores_row), reverse=True)
    if k <= 0 or k >= len(vals):
        return None
    a, b = vals[k - 1], vals[k]
    return (a - b) / max(abs(a), 1e-30)


# --------------------------------------------------------------------------
# C5/C6  sparse multi-token attention  [SV-Fig1]; readings R5, R6
# --------------------------------------------------------------------------
def ancestors(parents: Sequence[int], t: int) -> list[int]:
    """Draft t itself and all its ancestors, ascending."""
    out = []
    u = t
    while u >= 0:
        out.append(u)
        u = parents[u]
    return sorted(out)


def _softmax_weighted_sum(scores: torch.Tensor, values: torch.Tensor) -> torch.Tensor:
    m = scores.max()
    w = torch.exp(scores - m)
    return (w @ values) / w.sum()


def sparse_attend(q, k_pool, v_pool, block_table, sel, draft_k, draft_v,
                  parents: Sequence[int], tail_block: int = 0,
                  tail_len: int = 0) -> torch.Tensor:
    """Attention of every draft row over the ONE shared block set plus the
    drafts it may see.

    q [B,T,Hq,d]; pools [P,Hkv,blk,d]; block_table [B,>=NB]; sel [B,Hkv,k]
    (logical block indices; the same set for all T drafts and all G query
    heads of a KV head); draft_k/v [B,T,Hkv,d]. With tail_len > 0 the first
    tail_len tokens of logical block tail_block (the partial last block of
    the context) are attended as well, outside the selection (reading R8).
    Returns fp64 [B,T,Hq,d].
    """
    B, T, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d)
    out = torch.zeros(B, T, Hq, d, dtype=F64)
    for b in range(B):
        for h in range(Hkv):
            pages = [int(block_table[b, int(j)]) for j in sel[b, h].tolist()]
            Ks = [k_pool[p, h].to(F64) for p in pages]
            Vs = [v_pool[p, h].to(F64) for p in pages]
            if tail_len > 0:
                tp = int(block_table[b, tail_block])
                Ks.append(k_pool[tp, h, :tail_len].to(F64))
                Vs.append(v_pool[tp, h, :tail_len].to(F64))
            Kp = torch.cat(Ks) if Ks else torch.zeros(0, d, dtype=F64)   # [k*blk (+tail), d]
            Vp = torch.cat(Vs) if Vs else torch.zeros(0, d, dtype=F64)
            for t in range(T):
                vis = ancestors(parents, t)
                Kt = torch.cat([Kp, draft_k[b, vis, h].to(F64)])
                Vt = torch.cat([Vp, draft_v[b, vis, h].to(F64)])
                for g in range(G):
                    qv = q[b, t, h * G + g].to(F64)
                    out[b, t, h * G + g] = _softmax_weighted_sum((Kt @ qv) * scale, Vt)
    return out


# --------------------------------------------------------------------------
# C8  dense full verification attention  [SpecPV]; readings R5, R6
# --------------------------------------------------------------------------
def dense_verify_attention(q, k_ctx, v_ctx, draft_k, draft_v,
                           parents: Sequence[int]) -> torch.Tensor:
    """Full verification: every draft attends to the whole prefix plus the
    drafts the mask allows, written as one masked softmax over ctx+T keys.

    q [B,T,Hq,d]; k_ctx/v_ctx [B,ctx,Hkv,d] (logical order); draft_k/v
    [B,T,Hkv,d]. Returns fp64 [B,T,Hq,d].
    """
    B, T, Hq, d = q.shape
    ctx = k_ctx.shape[1]
    Hkv = k_ctx.shape[2]
    G = Hq // Hkv
    allowed = torch.zeros(T, ctx + T, dtype=torch.bool)
    allowed[:, :ctx] = True
    for t in range(T):
        for u in ancestors(parents, t):
            allowed[t, ctx + u] = True
    out = torch.zeros(B, T, Hq, d, dtype=F64)
    for b in range(B):
        for qh in range(Hq):
            h = qh // G
            K = torch.cat([k_ctx[b, :, h], draft_k[b, :, h]]).to(F64)   # [ctx+T, d]
            V = torch.cat([v_ctx[b, :, h], draft_v[b, :, h]]).to(F64)
            logits = (q[b, :, qh].to(F64) @ K.T) / math.sqrt(d)       # [T, ctx+T]
            logits = logits.masked_fill(~allowed, float("-inf"))
            w = torch.exp(logits - logits.max(dim=1, keepdim=True).values)
            out[b, :, qh] = (w @ V) / w.sum(dim=1, keepdim=True)
    return out


def logical_kv_tokens(pool: torch.Tensor, block_table: torch.Tensor, ctx: int) -> torch.Tensor:
    """The first ctx tokens of every sequence in logical order [B, ctx, Hkv, d]
    (the last block may be partial)."""
    blk = pool.shape[2]
    nblk = (ctx + blk - 1) // blk
    return logical_kv(pool, block_table, nblk)[:, :ctx]


def logical_kv(pool: torch.Tensor, block_table: torch.Tensor, n_blocks: int) -> torch.Tensor:
    """Gather a paged pool [P,Hkv,blk,d] into logical order [B, n_blocks*blk, Hkv, d]."""
    B = block_table.shape[0]
    P, Hkv, blk, d = pool.shape
    out = torch.empty(B, n_blocks * blk, Hkv, d, dtype=pool.dtype)
    for b in range(B):
        for j in range(n_blocks):
            out[b, j * blk:(j + 1) * blk] = pool[int(block_table[b, j])].transpose(0, 1)
    return out


# --------------------------------------------------------------------------
# One verification layer, and a stack with inter-layer reuse  [SV-Tut1]; R7
# --------------------------------------------------------------------------
def verify_layer(q, k_pool, v_pool, block_table, draft_k, draft_v, parents,
                 ctx: int, blk: int, budget, reps: Optional[torch.Tensor] = None,
                 reuse_sel: Optional[torch.Tensor] = None):
    """Score -> budget -> select -> attend for one layer.

    With reuse_sel given, the layer reuses that selection and does no scoring
    or selection (inter-layer retrieval reuse). Returns (out, sel, scores);
    scores is None on a reuse layer.
    """
    NB = ctx // blk              # full blocks: the candidates for selection
    tail = ctx - NB * blk        # tokens of a partial last block, always attended
    G = q.shape[2] // k_pool.shape[1]
    if reuse_sel is not None:
        sel, scores = reuse_sel, None
    else:
        if reps is None:
            reps = block_representatives(k_pool, block_table, NB, blk)
        scores = block_scores(q, reps, G)
        k = budget_from(budget, ctx, NB)
        sel = select_all(scores, k)
    out = sparse_attend(q, k_pool, v_pool, block_table, sel, draft_k, draft_v, parents,
                        tail_block=NB, tail_len=tail)
    return out, sel, scores


def verify_stack(layers, parents, ctx: int, blk: int, budget, compute_every: int):
    """Run verify_layer over a list of per-layer input tuples
    (q, k_pool, v_pool, block_table, draft_k, draft_v); layer l recomputes the
    selection when l % compute_every == 0 and otherwise reuses the last one."""
    outs, sels = [], []
    sel = None
    for l, (q, kp, vp, bt, dk, dv) in enumerate(layers):
        reuse = None if l % compute_every == 0 else sel
        out, sel, _ = verify_layer(q, kp, vp, bt, dk, dv, parents, ctx, blk, budget,
                                   reuse_sel=reuse)
        outs.append(out)
        sels.append(sel)
    return outs, sels


# --------------------------------------------------------------------------
# The shared-set diagnostic  [SV-Fig1]: how much each draft's own block set
# overlaps the first draft's (the set every draft actually uses)
# --------------------------------------------------------------------------
def draft_selection_overlap(q: torch.Tensor, reps: torch.Tensor, G: int, k: int) -> torch.Tensor:
    """overlap[b, h, t] = |S_t ∩ S_0| / k, where S_t is the top-k block set
    that draft t's own query would select (same scoring and tie rule as
    draft 0's). q [B,T,Hq,d]; reps [B,Hkv,NB,d]. Returns fp64 [B,Hkv,T]."""
    B, T = q.shape[0], q.shape[1]
    Hkv, NB = reps.shape[1], reps.shape[2]
    kk = min(k, NB)
    sets = [select_all(block_scores(q[:, t:t + 1], reps, G), kk) for t in range(T)]
    out = torch.zeros(B, Hkv, T, dtype=F64)
    for b in range(B):
        for h in range(Hkv):
            s0 = set(sets[0][b, h].tolist())
            for t in range(T):
                out[b, h, t] = len(s0 & set(sets[t][b, h].tolist())) / kk if kk else 1.0
    return out


def draft_depths(parents: Sequence[int]) -> list[int]:
    """Depth of every draft in its tree (root 0); a chain's draft t has depth t."""
    depth = []
    for t, p in enumerate(parents):
        depth.append(0 if p < 0 else depth[p] + 1)
    return depth


def draft_overlap_by_distance(q: torch.Tensor, reps: torch.Tensor, G: int, k: int,
                              parents: Sequence[int]) -> torch.Tensor:
    """The figure after [SV-Fig1]'s caption plots, for pairs of draft tokens, how much
    the block sets their own queries would select overlap, against the pairs'
    position distance. For every unordered pair of drafts t != u this takes
    |S_t ∩ S_u| / k (S_t: the top-k blocks of draft t's own query, same
    scoring and tie rule as draft 0's) and averages it over the pairs whose
    distance is delta = |depth(t) - depth(u)| (reading R10: a draft sits at
    position ctx + depth in its tree; in a chain delta = |t - u|).

    q [B,T,Hq,d]; reps [B,Hkv,NB,d]. Returns fp64 [B, Hkv, T]: entry delta is
    the mean overlap at that distance, NaN where no pair has it."""
    B, T = q.shape[0], q.shape[1]
    Hkv, NB = reps.shape[1], reps.shape[2]
    kk = min(k, NB)
    depth = draft_depths(parents)
    sets = [select_all(block_scores(q[:, t:t + 1], reps, G), kk) for t in range(T)]
    out = torch.full((B, Hkv, T), float("nan"), dtype=F64)
    for b in range(B):
        for h in range(Hkv):
            sums, counts = [0.0] * T, [0] * T
            for t in range(T):
                st = set(sets[t][b, h].tolist())
                for u in range(t + 1, T):
                    delta = abs(depth[t] - depth[u])
                    su = set(sets[u][b, h].tolist())
                    sums[delta] += len(st & su) / kk if kk else 1.0
                    counts[delta] += 1
            for delta in range(T):
                if counts[delta]:
                    out[b, h, delta] = sums[delta] / counts[delta]
    return out


# --------------------------------------------------------------------------
# Acceptance write-back: the step after verification (not on the pages)
# --------------------------------------------------------------------------
def append_accepted(k_pool, v_pool, block_table, ctx: Sequence[int], n_accept: Sequence[int],
                    accept_idx, draft_k, draft_v):
    """Append the accepted drafts' K/V to each sequence's paged cache.

    Sequence b accepted the drafts accept_idx[b][0:n_accept[b]] (draft indices
    along the accepted path, in order); their K/V rows go to logical positions
    ctx[b], ctx[b]+1, ... (page block_table[b, pos // blk], slot pos % blk).
    Returns updated copies of the pools and, per sequence, the logical blocks
    that became full (reps to rebuild).
    """
    k_new, v_new = k_pool.clone(), v_pool.clone()
    blk = k_pool.shape[2]
    filled = []
    for b in range(len(ctx)):
        for i in range(n_accept[b]):
            pos = ctx[b] + i
            page = int(block_table[b, pos // blk])
            k_new[page, :, pos % blk] = draft_k[b, int(accept_idx[b][i])]
            v_new[page, :, pos % blk] = draft_v[b, int(accept_idx[b][i])]
        first, last = ctx[b] // blk, (ctx[b] + n_accept[b]) // blk
        filled.append(list(range(first, last)))
    return k_new, v_new, filled
