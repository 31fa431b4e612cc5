"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each pin takes the oracle module as an argument so that
tests/test_oracle_mutations.py can plant a mistake in the oracle (on the CPU)
and show that some pin catches it. None of the expected values below comes
from the CUDA path: they are hand-worked fixtures under tests/golden/, closed
forms, brute force on tiny inputs, invariants, or torch's own
scaled_dot_product_attention.
"""
from __future__ import annotations

import itertools
import math
import os

import torch
import torch.nn.functional as F

from sparse_verification_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F64 = torch.float64


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split("#")[0].rstrip() for ln in f if ln.split("#")[0].strip()]


def small_inputs(B=2, Hq=4, Hkv=2, d=16, blk=4, NB=6, T=3, parents=None, seed=0,
                 permute=True):
    g = torch.Generator().manual_seed(seed)
    P = B * NB
    q = torch.randn(B, T, Hq, d, generator=g, dtype=F64)
    kp = torch.randn(P, Hkv, blk, d, generator=g, dtype=F64)
    vp = torch.randn(P, Hkv, blk, d, generator=g, dtype=F64)
    dk = torch.randn(B, T, Hkv, d, generator=g, dtype=F64)
    dv = torch.randn(B, T, Hkv, d, generator=g, dtype=F64)
    perm = torch.randperm(P, generator=g) if permute else torch.arange(P)
    bt = perm.view(B, NB).to(torch.int32)
    if parents is None:
        parents = [t - 1 for t in range(T)]
    return q, kp, vp, bt, dk, dv, list(parents)


# ------------------------------------------------------------------ C1 reps
def pin_rep_golden(O):
    ln = _lines("rep_mean_example.txt")
    keys = [list(map(float, x.split())) for x in ln[1:5]]
    want = list(map(float, ln[5].split(":")[1].split()))
    kp = torch.tensor(keys, dtype=F64).view(1, 1, 4, 3)
    rep = O.block_representatives(kp, torch.zeros(1, 1, dtype=torch.int32), 1, 4)
    assert rep.view(-1).tolist() == want, (rep, want)


def pin_rep_constant_block(O):
    q, kp, vp, bt, dk, dv, par = small_inputs()
    B, NB = bt.shape
    consts = torch.randn(kp.shape[0], kp.shape[1], 1, kp.shape[3], dtype=F64)
    kc = consts.expand_as(kp).clone()
    rep = O.block_representatives(kc, bt, NB, kp.shape[2])
    for b in range(B):
        for j in range(NB):
            p = int(bt[b, j])
            assert torch.equal(rep[b, :, j], consts[p, :, 0]), (b, j)


# ------------------------------------------------------------------ C2 scores
def pin_score_onehot(O):
    """Draft 0's query = unit vector e_i(h) on every head of group h, other
    drafts random: the score must be G * rep[..., i(h)] (sum over the group,
    draft 0 only, no scale, head h*G+g belongs to KV head h)."""
    B, Hq, Hkv, d, T, NB = 2, 6, 3, 8, 4, 5
    G = Hq // Hkv
    g = torch.Generator().manual_seed(7)
    q = torch.randn(B, T, Hq, d, generator=g, dtype=F64)
    axis = {0: 1, 1: 5, 2: 2}
    for h in range(Hkv):
        for gg in range(G):
            q[:, 0, h * G + gg] = 0.0
            q[:, 0, h * G + gg, axis[h]] = 1.0
    reps = torch.randn(B, Hkv, NB, d, generator=g, dtype=F64)
    s = O.block_scores(q, reps, G)
    for h in range(Hkv):
        assert torch.allclose(s[:, h], G * reps[:, h, :, axis[h]], rtol=0, atol=1e-12), h


def pin_score_first_draft_only(O):
    q, kp, vp, bt, dk, dv, par = small_inputs(T=4)
    reps = torch.randn(bt.shape[0], kp.shape[1], bt.shape[1], kp.shape[3], dtype=F64)
    G = q.shape[2] // kp.shape[1]
    s0 = O.block_scores(q, reps, G)
    q2 = q.clone()
    q2[:, 1:] = torch.randn_like(q2[:, 1:])
    assert torch.equal(O.block_scores(q2, reps, G), s0)
    q3 = q.clone()
    q3[:, 0] += 1.0
    assert not torch.allclose(O.block_scores(q3, reps, G), s0)


# ------------------------------------------------------------------ C3 budget
def pin_budget_table(O):
    for ln in _lines("budget_table.txt"):
        lhs, want = ln.split("->") if "->" in ln else (ln.rsplit(None, 1)[0], ln.rsplit(None, 1)[1])
        f = lhs.split()
        ctx, nb, mode, fixed, short, floor = map(int, f[:6])
        frac_mid, long_ctx, frac_long = float(f[6]), int(f[7]), float(f[8])
        got = O.budget_blocks(ctx, nb, mode, fixed, short, floor, frac_mid, long_ctx, frac_long)
        assert got == int(want), (ln, got)


def pin_budget_properties(O):
    b = W.PIECEWISE_6P25_ABOVE_32K
    for blk in (16, 64):
        prev_frac = 2.0
        for ctx in range(0, 300_000, 4096):
            nb = ctx // blk
            k = O.budget_from(b, ctx, nb)
            assert 0 <= k <= nb
            if ctx <= b.short_ctx:
                assert k == nb
            else:
                assert k >= min(nb, b.floor_blocks)
                frac = k / nb
                # the kept fraction never grows as the context grows
                assert frac <= prev_frac + 1e-12, (ctx, frac, prev_frac)
                prev_frac = frac


def pin_smooth_budget_properties(O):
    """Reading R3b: with ctx a whole number of blocks and no floor, one more
    block of context adds at most one kept block and never removes one
    (the curve has no jumps), everything is kept up to short_ctx, and the
    kept fraction tends to frac_long."""
    b = W.Budget(W.BUDGET_SMOOTH, 0, 4096, 0, 0.125, 32768, 0.0625)
    for blk in (16, 64):
        prev = None
        for nb in range(0, 200_000 // blk + 1, 7):
            ctx = nb * blk
            k = O.budget_from(b, ctx, nb)
            assert 0 <= k <= nb
            if ctx <= b.short_ctx:
                assert k == nb
            if prev is not None:
                pnb, pk = prev
                assert pk <= k <= pk + (nb - pnb), (ctx, pk, k)
            prev = (nb, k)
    # far beyond long_ctx the kept fraction approaches frac_long from above
    nb = 10**7
    k = O.budget_from(b, nb * 64, nb)
    assert 0.0625 < k / nb < 0.0625 * 1.01
    # all rates 1: every block kept at any length
    one = W.Budget(W.BUDGET_SMOOTH, 0, 100, 0, 1.0, 1000, 1.0)
    assert all(O.budget_from(one, n * 16, n) == n for n in range(0, 500, 13))


# ------------------------------------------------------------------ C4 select
def pin_select_golden(O):
    for ln in _lines("topk_ties.txt"):
        k, sc, want = (x.strip() for x in ln.split("|"))
        got = O.select_blocks([float(x) for x in sc.split()], int(k))
        assert got == [int(x) for x in want.split()], (ln, got)


def pin_select_bruteforce(O):
    """Counting definition: block j is kept iff fewer than k blocks beat it
    (a higher score, or an equal score at a lower index)."""
    g = torch.Generator().manual_seed(3)
    for trial in range(300):
        nb = int(torch.randint(1, 12, (1,), generator=g))
        k = int(torch.randint(0, nb + 2, (1,), generator=g))
        s = torch.randint(-3, 4, (nb,), generator=g).tolist()
        want = [j for j in range(nb)
                if sum(1 for i in range(nb) if s[i] > s[j] or (s[i] == s[j] and i < j)) < k]
        assert O.select_blocks(s, k) == want, (s, k)
    # and on distinct scores, the kept set is the k-subset of maximum total
    for trial in range(40):
        nb = int(torch.randint(1, 9, (1,), generator=g))
        k = int(torch.randint(0, nb + 1, (1,), generator=g))
        s = torch.randn(nb, generator=g).tolist()
        best = max(itertools.combinations(range(nb), k), key=lambda c: sum(s[i] for i in c))
        assert O.select_blocks(s, k) == sorted(best)


def pin_planted_blocks_selected(O):
    wl = W.WORKLOADS["tiny_f32"]
    x = W.make_layer(wl)
    _, sel, scores = O.verify_layer(x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k,
                                    x.draft_v, x.parents, wl.ctx, wl.blk, wl.budget)
    for b in range(wl.B):
        for h in range(wl.Hkv):
            assert set(x.planted[b, h].tolist()) <= set(sel[b, h].tolist()), (b, h)


# ------------------------------------------------------------------ C6 attend
def pin_two_key_golden(O):
    want = list(map(float, _lines("two_key_softmax.txt")[0].split(":")[1].split()))
    l3, l4 = math.log(3.0), math.log(4.0)
    q = torch.tensor([1.0, 0, 0, 0], dtype=F64).view(1, 1, 1, 4)
    kp = torch.tensor([[0.0, 0, 0, 0], [2 * l3, 0, 0, 0]], dtype=F64).view(1, 1, 2, 4)
    vp = torch.tensor([[8.0, 0, 0, 0], [0, 8.0, 0, 0]], dtype=F64).view(1, 1, 2, 4)
    dk = torch.tensor([2 * l4, 0, 0, 0], dtype=F64).view(1, 1, 1, 4)
    dv = torch.tensor([0, 0, 8.0, 0], dtype=F64).view(1, 1, 1, 4)
    sel = torch.zeros(1, 1, 1, dtype=torch.int64)
    out = O.sparse_attend(q, kp, vp, torch.zeros(1, 1, dtype=torch.int32), sel, dk, dv, [-1])
    assert torch.allclose(out.view(-1), torch.tensor(want, dtype=F64), atol=1e-12), out


def pin_tree_ancestors(O):
    ln = _lines("tree16_ancestors.txt")
    parents = [int(x) for x in ln[0].split(":")[1].split()]
    assert tuple(parents) == W.TREE16_PARENTS
    for row in ln[1:]:
        t, anc = row.split(":")
        assert O.ancestors(parents, int(t)) == [int(x) for x in anc.split()], row
    chain = [t - 1 for t in range(6)]
    for t in range(6):
        assert O.ancestors(chain, t) == list(range(t + 1))


def _uniform_check(O, parents, T):
    """Q = 0 makes attention uniform: each output is the plain mean of the V
    rows the draft may see (all selected prefix tokens + its visible drafts)."""
    q, kp, vp, bt, dk, dv, par = small_inputs(T=T, parents=parents)
    q = torch.zeros_like(q)
    B, NB = bt.shape
    Hkv, blk = kp.shape[1], kp.shape[2]
    G = q.shape[2] // Hkv
    sel = torch.tensor([[[1, 4], [0, 5]]] * B, dtype=torch.int64)
    out = O.sparse_attend(q, kp, vp, bt, sel, dk, dv, parents)
    for b in range(B):
        for h in range(Hkv):
            rows = [vp[int(bt[b, j]), h, i] for j in sel[b, h].tolist() for i in range(blk)]
            for t in range(T):
                vis = [t]
                u = parents[t]
                while u >= 0:
                    vis.append(u)
                    u = parents[u]
                allr = rows + [dv[b, u, h] for u in vis]
                mean = torch.stack(allr).mean(0)
                for gg in range(G):
                    assert torch.allclose(out[b, t, h * G + gg], mean, atol=1e-12), (b, h, t)


def pin_uniform_attention_chain(O):
    _uniform_check(O, [t - 1 for t in range(4)], 4)


def pin_uniform_attention_tree(O):
    _uniform_check(O, list(W.TREE16_PARENTS), 16)


def pin_value_ones(O):
    q, kp, vp, bt, dk, dv, par = small_inputs(T=5, parents=[-1, 0, 0, 1, 2])
    sel = torch.tensor([[[0, 2, 3], [1, 2, 5]]] * 2, dtype=torch.int64)
    out = O.sparse_attend(q * 3, kp, torch.ones_like(vp), bt, sel, dk, torch.ones_like(dv), par)
    assert torch.allclose(out, torch.ones_like(out), atol=1e-12)


def pin_full_budget_equals_dense(O):
    """With every block kept, sparse verification is full verification."""
    for parents, T in (([t - 1 for t in range(4)], 4), ([-1, 0, 0, 1, 1, 2], 6)):
        q, kp, vp, bt, dk, dv, par = small_inputs(T=T, parents=parents)
        B, NB = bt.shape
        Hkv, blk = kp.shape[1], kp.shape[2]
        sel = torch.arange(NB).expand(B, Hkv, NB)
        sp = O.sparse_attend(q, kp, vp, bt, sel, dk, dv, parents)
        dn = O.dense_verify_attention(q, O.logical_kv(kp, bt, NB), O.logical_kv(vp, bt, NB),
                                      dk, dv, parents)
        assert torch.allclose(sp, dn, atol=1e-12), (sp - dn).abs().max()


def pin_dense_vs_sdpa(O):
    """The dense routine against torch's scaled_dot_product_attention (a
    library routine) with an explicit boolean mask and repeated KV heads."""
    parents = [-1, 0, 0, 1, 2]
    q, kp, vp, bt, dk, dv, par = small_inputs(T=5, parents=parents)
    B, NB = bt.shape
    Hkv, blk = kp.shape[1], kp.shape[2]
    Hq = q.shape[2]
    G = Hq // Hkv
    kc, vc = O.logical_kv(kp, bt, NB), O.logical_kv(vp, bt, NB)
    ctx = NB * blk
    dn = O.dense_verify_attention(q, kc, vc, dk, dv, parents)
    Kall = torch.cat([kc, dk], 1).repeat_interleave(G, dim=2).transpose(1, 2)  # [B,Hq,S,d]
    Vall = torch.cat([vc, dv], 1).repeat_interleave(G, dim=2).transpose(1, 2)
    mask = torch.zeros(5, ctx + 5, dtype=torch.bool)
    mask[:, :ctx] = True
    for t, anc in enumerate([[0], [0, 1], [0, 2], [0, 1, 3], [0, 2, 4]]):
        mask[t, [ctx + a for a in anc]] = True
    ref = F.scaled_dot_product_attention(q.transpose(1, 2), Kall, Vall, attn_mask=mask)
    assert torch.allclose(dn, ref.transpose(1, 2), atol=1e-10)


def pin_decode_special_case(O):
    """T=1, G=1, all blocks: textbook single-query decode attention."""
    q, kp, vp, bt, dk, dv, par = small_inputs(Hq=2, Hkv=2, T=1)
    B, NB = bt.shape
    sel = torch.arange(NB).expand(B, 2, NB)
    sp = O.sparse_attend(q, kp, vp, bt, sel, dk, dv, [-1])
    kc = torch.cat([O.logical_kv(kp, bt, NB), dk], 1).transpose(1, 2)
    vc = torch.cat([O.logical_kv(vp, bt, NB), dv], 1).transpose(1, 2)
    ref = F.scaled_dot_product_attention(q.transpose(1, 2), kc, vc)
    assert torch.allclose(sp, ref.transpose(1, 2), atol=1e-10)


def pin_selected_equals_dense_on_gathered(O):
    """Sparse attention over a set = dense attention over a context made of
    only the selected blocks (in ascending block order)."""
    parents = [-1, 0, 1]
    q, kp, vp, bt, dk, dv, par = small_inputs(Hq=2, Hkv=1, T=3, parents=parents)
    B = bt.shape[0]
    sel = torch.tensor([[[0, 3, 4]]] * B, dtype=torch.int64)
    sp = O.sparse_attend(q, kp, vp, bt, sel, dk, dv, parents)
    bt_sub = torch.stack([bt[b, sel[b, 0]] for b in range(B)]).to(torch.int32)
    dn = O.dense_verify_attention(q, O.logical_kv(kp, bt_sub, 3), O.logical_kv(vp, bt_sub, 3),
                                  dk, dv, parents)
    assert torch.allclose(sp, dn, atol=1e-12)


def pin_page_permutation_invariance(O):
    q, kp, vp, bt, dk, dv, par = small_inputs(permute=False)
    P = kp.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(11))
    inv = torch.argsort(perm)
    kp2, vp2 = kp[perm], vp[perm]          # page p of the new pool = old page perm[p]
    bt2 = inv[bt.long()].to(torch.int32)
    sel = torch.tensor([[[0, 2], [1, 5]]] * bt.shape[0], dtype=torch.int64)
    a = O.sparse_attend(q, kp, vp, bt, sel, dk, dv, par)
    b = O.sparse_attend(q, kp2, vp2, bt2, sel, dk, dv, par)
    assert torch.allclose(a, b, atol=1e-12)


# --------------------------------------------------------- C5 shared set, C7
def pin_shared_set(O):
    """One selection per (b, kv head), whatever the later drafts' queries."""
    q, kp, vp, bt, dk, dv, par = small_inputs(T=4)
    B, NB = bt.shape
    budget = W.Budget(W.BUDGET_FIXED, 3, 0, 0, 0.0, 0, 0.0)
    ctx, blk = NB * kp.shape[2], kp.shape[2]
    _, sel, _ = O.verify_layer(q, kp, vp, bt, dk, dv, par, ctx, blk, budget)
    q2 = q.clone()
    q2[:, 1:] = torch.randn_like(q2[:, 1:]) * 10
    _, sel2, _ = O.verify_layer(q2, kp, vp, bt, dk, dv, par, ctx, blk, budget)
    assert torch.equal(sel, sel2)
    assert sel.shape == (B, kp.shape[1], 3)


def pin_reuse(O):
    wl = W.scaled(W.WORKLOADS["llama8b_60k_32layer"], ctx=1024, blk=16, Hq=4, Hkv=2, d=16,
                  layers=4, n_planted=4, budget=W.Budget(W.BUDGET_FIXED, 6, 0, 0, 0, 0, 0))
    ps = W.planted_sets(wl)
    layers = []
    for l in range(wl.layers):
        x = W.make_layer(wl, l, planted=ps[l])
        layers.append((x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k, x.draft_v))
    outs, sels = O.verify_stack(layers, wl.parent_list(), wl.ctx, wl.blk, wl.budget, 2)
    assert torch.equal(sels[1], sels[0]) and torch.equal(sels[3], sels[2])
    assert not torch.equal(sels[2], sels[0])
    ref1 = O.sparse_attend(*layers[1][:4], sels[0], *layers[1][4:], wl.parent_list())
    assert torch.equal(outs[1], ref1)


# ------------------------------------------------- partial tail block (R8)
def _fixed(nblocks):
    from types import SimpleNamespace
    return SimpleNamespace(mode=O_FIXED, fixed_blocks=nblocks, short_ctx=0, floor_blocks=0,
                           frac_mid=0.0, long_ctx=0, frac_long=0.0)


O_FIXED = 0


def pin_tail_full_budget_equals_dense(O):
    """A context ending in a partial block: keeping every full block and
    always attending the partial one is full verification over exactly ctx
    tokens (dense attention, which knows nothing of blocks)."""
    for ctx, parents, T in ((4 * 5 + 3, [-1, 0, 1, 2], 4), (4 * 2 + 1, [-1, 0, 0, 1, 1], 5),
                            (3, [-1, 0], 2)):
        q, kp, vp, bt, dk, dv, par = small_inputs(T=T, parents=parents, NB=6)
        blk = kp.shape[2]
        nfull = ctx // blk
        out, sel, _ = O.verify_layer(q, kp, vp, bt, dk, dv, parents, ctx, blk, _fixed(nfull))
        dn = O.dense_verify_attention(q, O.logical_kv_tokens(kp, bt, ctx),
                                      O.logical_kv_tokens(vp, bt, ctx), dk, dv, parents)
        assert sel.shape[-1] == nfull
        assert torch.allclose(out, dn, atol=1e-12), (ctx, (out - dn).abs().max())


def pin_tail_outside_budget(O):
    """The partial block is attended even with a budget of zero blocks:
    then each row attends to the tail tokens and its visible drafts only."""
    q, kp, vp, bt, dk, dv, par = small_inputs(T=3, NB=6)
    blk = kp.shape[2]
    ctx = 4 * blk + 2
    out, sel, _ = O.verify_layer(q, kp, vp, bt, dk, dv, par, ctx, blk, _fixed(0))
    B, T, Hq, d = q.shape
    Hkv = kp.shape[1]
    G = Hq // Hkv
    for b in range(B):
        page = int(bt[b, 4])
        for h in range(Hkv):
            for t in range(T):
                vis = O.ancestors(par, t)
                K = torch.cat([kp[page, h, :2], dk[b, vis, h]])
                V = torch.cat([vp[page, h, :2], dv[b, vis, h]])
                for g in range(G):
                    s = (K @ q[b, t, h * G + g]) / math.sqrt(d)
                    want = torch.softmax(s, 0) @ V
                    assert torch.allclose(out[b, t, h * G + g], want, atol=1e-12)


def pin_append_accepted(O):
    """Acceptance write-back: the accepted drafts' rows land at positions
    ctx, ctx+1, ... of their sequence in the order accepted; every other
    position is unchanged; the blocks reported full are exactly those that
    the append completed."""
    q, kp, vp, bt, dk, dv, par = small_inputs(T=5, NB=6)
    blk = kp.shape[2]
    ctx = [blk * 2 + 3, blk * 3]
    n_acc = [3, 5]
    acc = [[0, 1, 3, -1, -1], [0, 2, 4, 1, 3]]
    kn, vn, filled = O.append_accepted(kp, vp, bt, ctx, n_acc, acc, dk, dv)
    for b in range(2):
        before_k = O.logical_kv_tokens(kp, bt, ctx[b] + n_acc[b])[b]
        after_k = O.logical_kv_tokens(kn, bt, ctx[b] + n_acc[b])[b]
        after_v = O.logical_kv_tokens(vn, bt, ctx[b] + n_acc[b])[b]
        assert torch.equal(after_k[:ctx[b]], before_k[:ctx[b]])
        for i in range(n_acc[b]):
            assert torch.equal(after_k[ctx[b] + i], dk[b, acc[b][i]])
            assert torch.equal(after_v[ctx[b] + i], dv[b, acc[b][i]])
    # 11 + 3 = 14 tokens fill block 2 (tokens 8..11 and 12..13 do not fill 3)
    assert filled == [[2], [3]]
    # pages not touched by the append are bit-identical
    touched = {int(bt[b, (ctx[b] + i) // blk]) for b in range(2) for i in range(n_acc[b])}
    for p in range(kp.shape[0]):
        if p not in touched:
            assert torch.equal(kn[p], kp[p]) and torch.equal(vn[p], vp[p])


# ------------------------------------------------- shared-set diagnostic
def pin_draft_overlap_closed_form(O):
    """One-hot representatives: block j's rep is e_(j mod d) scaled by
    (j + 1), so a query equal to e_i scores block j by (j + 1) [j = i mod d].
    Draft t's query e_(t) with d = 4, NB = 8, k = 2 picks blocks {t, t + 4};
    the overlap with draft 0's {0, 4} is 1 for t = 0 and 0 otherwise; a draft
    that repeats draft 0's query overlaps fully."""
    B, T, Hkv, G, d, NB = 1, 5, 1, 1, 4, 8
    reps = torch.zeros(B, Hkv, NB, d, dtype=F64)
    for j in range(NB):
        reps[0, 0, j, j % d] = j + 1.0
    q = torch.zeros(B, T, Hkv * G, d, dtype=F64)
    for t in range(4):
        q[0, t, 0, t] = 1.0
    q[0, 4, 0, 0] = 3.0  # same direction as draft 0
    ov = O.draft_selection_overlap(q, reps, G, 2)
    assert ov[0, 0].tolist() == [1.0, 0.0, 0.0, 0.0, 1.0]


def _onehot_reps(NB=8, d=4):
    reps = torch.zeros(1, 1, NB, d, dtype=F64)
    for j in range(NB):
        reps[0, 0, j, j % d] = j + 1.0
    return reps


def pin_overlap_by_distance_chain(O):
    """One-hot representatives as above: a query e_i keeps blocks {i, i + 4}
    (k = 2). Chain drafts with queries e0, e0, e1, e0: the pairs at distance
    1 are (0,1) -> 1, (1,2) -> 0, (2,3) -> 0, mean 1/3; at distance 2 (0,2)
    -> 0 and (1,3) -> 1, mean 1/2; at distance 3 (0,3) -> 1. No pair has
    distance 0."""
    q = torch.zeros(1, 4, 1, 4, dtype=F64)
    for t, i in enumerate([0, 0, 1, 0]):
        q[0, t, 0, i] = 1.0
    got = O.draft_overlap_by_distance(q, _onehot_reps(), 1, 2, [-1, 0, 1, 2])[0, 0]
    assert math.isnan(got[0])
    assert torch.allclose(got[1:], torch.tensor([1 / 3, 1 / 2, 1.0], dtype=F64))


def pin_overlap_by_distance_tree(O):
    """Tree drafts (parents -1, 0, 0, 1: depths 0, 1, 1, 2) with queries
    e0, e0, e1, e1. By depth difference: distance 0 is the sibling pair
    (1,2) -> 0; distance 1 is (0,1) -> 1, (0,2) -> 0, (1,3) -> 0, (2,3) -> 1,
    mean 1/2; distance 2 is (0,3) -> 0. (Index distance would give 2/3 at
    distance 1.)"""
    q = torch.zeros(1, 4, 1, 4, dtype=F64)
    for t, i in enumerate([0, 0, 1, 1]):
        q[0, t, 0, i] = 1.0
    got = O.draft_overlap_by_distance(q, _onehot_reps(), 1, 2, [-1, 0, 0, 1])[0, 0]
    assert torch.allclose(got[:3], torch.tensor([0.0, 0.5, 0.0], dtype=F64))
    assert math.isnan(got[3])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
