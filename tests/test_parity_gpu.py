"""CUDA path (through the C ABI) against the CPU oracle.

Oracle-sized cases span several split tiles and ragged tails; the full-size
workloads are checked on sampled (sequence, kv head) pairs that the oracle
recomputes one by one, in the same launch configuration the benchmark uses.
"""
import pytest
import torch

from oracle import sva_oracle as O
from sparse_verification_attention_gb300 import api, build_lib
from sparse_verification_attention_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    build_lib.build()
    api.lib()
    torch.cuda.set_device(0)


def small_wl(dtype="bf16", **kw):
    base = dict(name="small", B=2, Hq=8, Hkv=2, d=128, blk=64, ctx=64 * 40, T=8, dtype=dtype,
                budget=W.Budget(W.BUDGET_FIXED, 13, 0, 0, 0, 0, 0), seed=21, n_planted=4,
                permute_pages=True)
    base.update(kw)
    return W.Workload(**base)


def random_sel(B, H, NB, k, seed):
    g = torch.Generator().manual_seed(seed)
    sel = torch.full((B, H, max(k, 1)), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            if k:
                sel[b, h, :k] = torch.sort(torch.randperm(NB, generator=g)[:k]).values.to(torch.int32)
    return sel


# ------------------------------------------------------------------ reps
@pytest.mark.parametrize("dtype,d,blk", [("bf16", 128, 64), ("f32", 64, 16), ("bf16", 96, 32)])
def test_build_reps(dtype, d, blk):
    wl = small_wl(dtype, d=d, blk=blk, ctx=blk * 37)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    shape = api.make_shape(wl.B, wl.Hq, wl.Hkv, wl.d, wl.blk, wl.T, wl.torch_dtype)
    kv = api.make_kv(xd.k_pool, xd.v_pool, xd.block_table, wl.ctx)
    reps = torch.full((wl.B, wl.Hkv, wl.NB, wl.d), float("nan"), device="cuda")
    # incremental: two ranges, a gap left untouched in between
    api.sv_build_reps(shape, kv, 0, 20, reps)
    api.sv_build_reps(shape, kv, 25, wl.NB - 25, reps)
    torch.cuda.synchronize()
    ref = O.block_representatives(x.k_pool, x.block_table, wl.NB, wl.blk)
    got = reps.cpu().double()
    assert torch.isnan(got[:, :, 20:25]).all()
    keep = torch.cat([torch.arange(20), torch.arange(25, wl.NB)])
    assert torch.allclose(got[:, :, keep], ref[:, :, keep], rtol=0, atol=1e-5)


# ------------------------------------------------------------------ scores / select
@pytest.mark.parametrize("dtype,d,G", [("bf16", 128, 4), ("f32", 64, 2), ("bf16", 256, 8)])
def test_score_blocks(dtype, d, G):
    wl = small_wl(dtype, d=d, Hkv=2, Hq=2 * G, blk=32, ctx=32 * 301)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    shape = api.make_shape(wl.B, wl.Hq, wl.Hkv, wl.d, wl.blk, wl.T, wl.torch_dtype)
    kv = api.make_kv(xd.k_pool, xd.v_pool, xd.block_table, wl.ctx)
    reps_ref = O.block_representatives(x.k_pool, x.block_table, wl.NB, wl.blk)
    reps = reps_ref.float().cuda()  # exact oracle reps, rounded to the fp32 the ABI takes
    scores = torch.empty(wl.B, wl.Hkv, wl.NB, device="cuda")
    api.sv_score_blocks(shape, xd.q, reps, kv, scores)
    torch.cuda.synchronize()
    ref = O.block_scores(x.q, reps.cpu().double(), wl.G)
    assert torch.allclose(scores.cpu().double(), ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("nb,k", [(64, 8), (512, 64), (2048, 128), (1000, 999), (37, 37), (37, 50),
                                  (1, 1), (16384, 1024), (300, 0), (3000, 200), (4096, 4000),
                                  (5000, 1)])
def test_select_blocks_exact(nb, k):
    """Host-made scores with many ties (small integers), +-0 and negatives:
    the GPU selection must equal the oracle's, bit for bit."""
    g = torch.Generator().manual_seed(nb * 7 + k)
    B, H = 2, 3
    scores = torch.randint(-20, 21, (B, H, nb), generator=g).float() * 0.25
    scores[0, 0, ::7] = -0.0
    scores[1, 2] = torch.randn(nb, generator=g)  # one row without ties
    shape = api.make_shape(B, 4 * H, H, 64, 64, 4, torch.bfloat16)
    kmax = max(k, 1) + 3
    sel = torch.zeros(B, H, kmax, dtype=torch.int32, device="cuda")
    api.sv_select_blocks(shape, scores.cuda(), nb, k, sel, kmax)
    torch.cuda.synchronize()
    s = sel.cpu()
    for b in range(B):
        for h in range(H):
            want = O.select_blocks(scores[b, h].tolist(), k)
            kk = len(want)
            assert s[b, h, :kk].tolist() == want, (b, h)
            assert (s[b, h, kk:] == -1).all()


def _score_patterns(nb, g):
    """Score rows that stress the selection: outliers, many ties, extreme
    and tiny ranges, signed zeros, one-ulp steps, a wide plateau at the
    boundary, all equal."""
    rows = []
    rows.append(torch.randn(nb, generator=g) * 3)
    x = torch.randn(nb, generator=g)
    x[torch.randint(0, nb, (17,), generator=g)] += 40.0
    rows.append(x)
    rows.append(torch.randint(-20, 21, (nb,), generator=g).float() * 0.25)
    x = torch.randn(nb, generator=g)
    x[0], x[1] = 3e37, -3e37
    rows.append(x)
    rows.append(torch.full((nb,), 1.5))
    rows.append(torch.randn(nb, generator=g) * 1e-30)
    x = torch.zeros(nb)
    x[::3] = -0.0
    x[5] = 1.0
    rows.append(x)
    rows.append(1.0 + torch.randint(0, 4, (nb,), generator=g).float() * 2.0**-23)
    x = torch.randn(nb, generator=g)
    x[: nb // 2] = 7.0
    rows.append(x)
    return torch.stack(rows).float()


@pytest.mark.parametrize("nb,k", [(2048, 128), (2048, 1), (8192, 512), (300, 299), (9000, 700)])
def test_score_select_adversarial_scores(nb, k):
    """Scores planted exactly through the representatives (one non-zero
    dimension, draft-0 queries of 1.0, so score = G * value in fp32) run
    through the fused score + select kernel (nb <= 8192) or the score
    kernel and the standalone select: the selection must equal the
    oracle's bit for bit."""
    g = torch.Generator().manual_seed(nb + k)
    vals = _score_patterns(nb, g)                  # [H, nb]
    H, G, d, blk = vals.shape[0], 4, 64, 16
    shape = api.make_shape(1, H * G, H, d, blk, 2, torch.bfloat16)
    q = torch.zeros(1, 2, H * G, d, dtype=torch.bfloat16)
    q[0, 0, :, 0] = 1.0
    reps = torch.zeros(1, H, nb, d)
    reps[0, :, :, 0] = vals
    pool = torch.zeros(1, H, blk, d, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, nb, dtype=torch.int32, device="cuda")
    kv = api.make_kv(pool, pool, bt, nb * blk)
    kmax = k + 2
    sel = torch.full((1, H, kmax), 7, dtype=torch.int32, device="cuda")
    ws = api.alloc_workspace(shape, nb, kmax)
    got_k = api.sv_score_select(shape, q.cuda(), reps.cuda(), kv,
                                W.Budget(W.BUDGET_FIXED, k, 0, 0, 0, 0, 0), sel, kmax, ws)
    torch.cuda.synchronize()
    assert got_k == k and api.sv_read_status(ws) == 0
    s = sel.cpu()
    for h in range(H):
        want = O.select_blocks((vals[h] * G).tolist(), k)
        assert s[0, h, :k].tolist() == want, (h, nb, k)
        assert (s[0, h, k:] == -1).all()


def test_score_select_vs_oracle():
    wl = small_wl(ctx=64 * 150, budget=W.Budget(W.BUDGET_FIXED, 21, 0, 0, 0, 0, 0))
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    k = api.sv_score_select(st.shape, xd.q, st.reps, st.kv, wl.budget, st.sel, st.kmax, st.ws)
    torch.cuda.synchronize()
    assert k == 21
    reps_ref = O.block_representatives(x.k_pool, x.block_table, wl.NB, wl.blk)
    ref_scores = O.block_scores(x.q, reps_ref, wl.G)
    U.compare_selection(st.sel.cpu(), ref_scores, k)
    # the kernel's top-k is exact on its own fp32 scores
    scores = torch.empty(wl.B, wl.Hkv, wl.NB, device="cuda")
    api.sv_score_blocks(st.shape, xd.q, st.reps, st.kv, scores)
    torch.cuda.synchronize()
    U.check_topk_property(st.sel.cpu(), scores.cpu(), k)
    for b in range(wl.B):
        for h in range(wl.Hkv):
            assert set(x.planted[b, h].tolist()) <= set(st.sel[b, h].cpu().tolist())


# ------------------------------------------------------------------ attend
ATTEND_CASES = [
    # name (path prefix: tc = tcgen05, mma = legacy mma.sync, generic = CUDA
    # cores), workload overrides, number of selected blocks
    ("tc_d128_blk64_R32", dict(), 13),
    ("tc_R32_ragged", dict(B=3, ctx=64 * 77), 61),
    ("tc_tree16_G8_R128", dict(Hq=16, Hkv=2, T=16, parents=W.TREE16_PARENTS), 29),
    ("tc_R48", dict(Hq=8, Hkv=2, T=12, ctx=64 * 45), 9),
    ("tc_T1_G1", dict(Hq=2, Hkv=2, T=1), 5),
    ("tc_nsel0_drafts_only", dict(), 0),
    ("tc_all_blocks", dict(ctx=64 * 24), 24),
    ("tc_T64_chain", dict(T=64, Hq=2, Hkv=1, ctx=64 * 30), 7),
    # many (b, h) pairs: non-uniform split map (some pairs get one more split)
    ("tc_many_pairs_B8_H8_R32", dict(B=8, Hq=32, Hkv=8, ctx=64 * 24), 13),
    ("tc_many_pairs_tree16_R128", dict(B=8, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                       ctx=64 * 20), 11),
    ("tc_many_pairs_few_units", dict(B=8, Hq=32, Hkv=8, ctx=64 * 24), 2),
    ("tc_many_pairs_all_blocks", dict(B=8, Hq=32, Hkv=8, ctx=64 * 10), 10),
    ("tc_more_pairs_than_sms", dict(B=40, Hq=16, Hkv=4, ctx=64 * 6), 3),
    # stream-K: every CTA takes an equal run of the flattened (pair, unit)
    # sequence, crossing at most one pair boundary
    ("tc_sk_32pairs_129units", dict(B=4, Hq=32, Hkv=8, ctx=64 * 200), 128),
    ("tc_sk_tree16_R128", dict(B=10, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                               ctx=64 * 40), 29),
    ("tc_sk_one_unit_per_cta", dict(B=19, Hq=8, Hkv=2, ctx=64 * 30), 3),
    ("tc_sk_runs_cross_pairs", dict(B=23, Hq=4, Hkv=1, T=4, ctx=64 * 12), 8),
    ("tc_sk_two_unit_pairs", dict(B=75, Hq=4, Hkv=2, T=2, ctx=64 * 4), 1),
    # few pairs: one cluster of 8 to 16 CTAs per pair (as many as the device
    # keeps resident for that many pairs), merged through distributed shared
    # memory
    ("tc_cluster_B1_H8", dict(B=1, Hq=32, Hkv=8, ctx=64 * 100), 64),
    ("tc_cluster_tree16_R128_tail", dict(B=1, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                         ctx=64 * 60 + 5), 40),
    ("tc_cluster_12pairs", dict(B=3, Hq=32, Hkv=4, ctx=64 * 40), 30),
    # 128-row tiles over 32 pairs: a wide merge, so clusters of 4
    ("tc_cluster_tree16_32pairs", dict(B=8, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                       ctx=64 * 40 + 9), 29),
    ("tc_cluster_idle_ctas", dict(B=1, Hq=32, Hkv=8, ctx=64 * 20), 16),
    # contexts ending in a partial block: its tokens are always attended
    ("tc_tail_split", dict(ctx=64 * 20 + 17), 7),
    ("tc_sk_tail", dict(B=4, Hq=32, Hkv=8, ctx=64 * 100 + 40), 50),
    ("tc_tail_only", dict(ctx=37), 0),
    ("tc_sk_tail_tree16_R128", dict(B=10, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                    ctx=64 * 30 + 63), 20),
    ("mma_R16_pad", dict(Hq=4, Hkv=2, T=4, d=64, blk=32, ctx=32 * 50), 17),
    ("mma_R48_rows_pad", dict(Hq=8, Hkv=2, T=12, blk=32, ctx=32 * 45), 9),
    ("mma_d64_blk64", dict(d=64, ctx=64 * 30), 11),
    ("mma_cluster_d64_blk32_R16", dict(B=16, Hq=16, Hkv=8, d=64, blk=32, ctx=32 * 40), 9),
    ("mma_cluster_blk32_R32", dict(B=8, Hq=32, Hkv=8, blk=32, ctx=32 * 40), 9),
    ("generic_f32", dict(dtype="f32", d=64, blk=16, ctx=16 * 64, Hq=4, Hkv=2, T=4), 8),
    ("generic_d96", dict(d=96, blk=32, ctx=32 * 40), 11),
    ("generic_T_gt_blk", dict(T=40, Hq=2, Hkv=1, blk=32, ctx=32 * 30), 7),
    ("generic_R256", dict(T=32, Hq=16, Hkv=2, ctx=64 * 20), 6),
    ("generic_blk16_bf16", dict(blk=16, ctx=16 * 90), 19),
    ("mma_tail", dict(Hq=4, Hkv=2, T=4, d=64, blk=32, ctx=32 * 50 + 5), 17),
    ("mma_many_tail", dict(B=8, Hq=32, Hkv=8, blk=32, ctx=32 * 40 + 31), 9),
    ("generic_tail_f32", dict(dtype="f32", d=64, blk=16, ctx=16 * 64 + 9, Hq=4, Hkv=2, T=4), 8),
    ("generic_tail_R256", dict(T=32, Hq=16, Hkv=2, ctx=64 * 20 + 63), 6),
]


@pytest.mark.parametrize("name,over,n_sel", ATTEND_CASES, ids=[c[0] for c in ATTEND_CASES])
def test_sparse_attend(name, over, n_sel):
    over = dict(over)
    dtype = over.pop("dtype", "bf16")
    wl = small_wl(dtype, **over)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd, kmax=max(n_sel, 1), build_reps=False)
    sel = random_sel(wl.B, wl.Hkv, wl.NB, n_sel, seed=len(name))
    plan = api.sv_attend_plan(st.shape, st.kv, n_sel)
    want_path = {"tc": api.SV_PATH_TCGEN05, "mma": api.SV_PATH_MMA_SYNC,
                 "generic": api.SV_PATH_CUDA_CORES}[name.split("_")[0]]
    assert plan.path == want_path, (plan.path, want_path)
    if "cluster" in name:
        assert plan.cluster >= (4 if want_path == api.SV_PATH_TCGEN05 else 1), plan.cluster
    if "_sk_" in name:
        assert plan.streamk == 1, (plan.n_splits, plan.blocks_per_split)
    out = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, sel.cuda(), n_sel, sel.shape[-1], xd.draft_k,
                         xd.draft_v, st.parents, out, st.ws)
    torch.cuda.synchronize()
    words = st.ws[:8].view(torch.int32).tolist()
    assert api.sv_read_status(st.ws) == 0, f"status words {words} plan {plan.cluster} {plan.n_splits}"
    ref = O.sparse_attend(x.q, x.k_pool, x.v_pool, x.block_table, sel[:, :, :n_sel].long(),
                          x.draft_k, x.draft_v, wl.parent_list(), tail_block=wl.NB,
                          tail_len=wl.ctx % wl.blk)
    U.compare_out(out, ref, U.out_atol(wl.torch_dtype))


def test_tc_late_rescale_divergent_rows():
    """One CTA per (b, h) walks 41 work units; a late selected block has keys
    boosted along the group's query, so the running max of some rows (not
    all) jumps by far more than 2^8 mid-stream: the accumulator rescale must
    be taken by the whole warp and stay exact."""
    wl = small_wl(B=19, Hq=32, Hkv=8, ctx=64 * 48, n_planted=0, sink_alpha=None)
    x = W.make_layer(wl)
    G = wl.G
    n_sel = 40
    sel = random_sel(wl.B, wl.Hkv, wl.NB, n_sel, seed=99)
    for b in range(wl.B):
        for h in range(wl.Hkv):
            j = int(sel[b, h, 33])  # a late block of this pair's selection
            page = int(x.block_table[b, j])
            q0 = x.q[b, :, h * G].float().mean(0)  # the group's mean query direction
            boost = (x.k_pool[page, h].float() + 6.0 * q0).to(x.k_pool.dtype)
            x.k_pool[page, h] = boost
    xd = x.to("cuda")
    st = api.LayerState(wl, xd, kmax=n_sel, build_reps=False)
    plan = api.sv_attend_plan(st.shape, st.kv, n_sel)
    assert plan.path == api.SV_PATH_TCGEN05
    # one CTA walks a whole pair: a split map with one split, or (152 pairs on
    # 152 SMs) stream-K runs of exactly one pair's 41 units
    whole_pair = (plan.n_splits == 1 if not plan.streamk else
                  wl.B * wl.Hkv * (n_sel + 1) == plan.n_splits * plan.blocks_per_split)
    assert whole_pair, (plan.streamk, plan.n_splits, plan.blocks_per_split)
    out = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, sel.cuda(), n_sel, sel.shape[-1], xd.draft_k,
                         xd.draft_v, None, out, st.ws)
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    ref = O.sparse_attend(x.q, x.k_pool, x.v_pool, x.block_table, sel.long(), x.draft_k,
                          x.draft_v, wl.parent_list())
    U.compare_out(out, ref, U.BF16_ATOL)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "bf16_many_pairs", "bf16_tail", "f32_tail"])
def test_dense_attend(dtype):
    if dtype == "bf16":
        over = dict(ctx=64 * 33)
    elif dtype == "bf16_many_pairs":
        dtype, over = "bf16", dict(B=8, Hq=32, Hkv=8, ctx=64 * 21)
    elif dtype == "bf16_tail":
        dtype, over = "bf16", dict(B=4, Hq=32, Hkv=8, ctx=64 * 21 + 50)
    elif dtype == "f32_tail":
        dtype, over = "f32", dict(d=64, blk=16, ctx=16 * 70 + 3, T=5, parents=(-1, 0, 0, 1, 2))
    else:
        over = dict(d=64, blk=16, ctx=16 * 70, T=5, parents=(-1, 0, 0, 1, 2))
    wl = small_wl(dtype, **over)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd, build_reps=False)
    out = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, None, 0, 0, xd.draft_k, xd.draft_v, st.parents,
                         out, st.ws)
    torch.cuda.synchronize()
    ref = O.dense_verify_attention(x.q, O.logical_kv_tokens(x.k_pool, x.block_table, wl.ctx),
                                   O.logical_kv_tokens(x.v_pool, x.block_table, wl.ctx), x.draft_k,
                                   x.draft_v, wl.parent_list())
    U.compare_out(out, ref, U.out_atol(wl.torch_dtype))


def test_value_ones_gives_ones():
    wl = small_wl(ctx=64 * 30)
    x = W.make_layer(wl)
    x.v_pool = torch.ones_like(x.v_pool)
    x.draft_v = torch.ones_like(x.draft_v)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    out = st.verify()
    torch.cuda.synchronize()
    assert (out.float() - 1).abs().max().item() <= 2 ** -8


# ------------------------------------------------------------------ verify layer
def _verify_vs_oracle(wl, x, xd, pairs=None):
    """Run sv_verify_layer on the device, recompute (b, h) pairs on the CPU
    oracle (all pairs by default) and compare selection and outputs.

    The selection must equal the oracle's bit for bit, except inside a
    boundary band (oracle boundary gap below 1e-4 relative), where either
    choice is correct. Outputs are then compared element by element for
    every pair against the oracle's attention over the set the GPU actually
    used: that set is the oracle's own wherever the two agree, so no pair
    goes unchecked. Returns (max abs error, pairs whose set differed)."""
    st = api.LayerState(wl, xd)
    out = st.verify()
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    k = st.k
    if pairs is None:
        pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
    gsel = st.sel.cpu()
    gout = out.cpu()
    by_b = {}
    for b, h in pairs:
        by_b.setdefault(b, []).append(h)
    worst, n_differ = 0.0, 0
    for b, hs in by_b.items():
        qb = x.q[b:b + 1]
        btb = x.block_table[b:b + 1]
        reps = O.block_representatives(x.k_pool, btb, wl.NB, wl.blk)
        scores = O.block_scores(qb, reps, wl.G)
        n_differ += len(U.compare_selection(gsel[b:b + 1, hs], scores[:, hs], k))
        used = gsel[b:b + 1, :, :k].long()
        ref = O.sparse_attend(qb, x.k_pool, x.v_pool, btb, used, x.draft_k[b:b + 1],
                              x.draft_v[b:b + 1], wl.parent_list(), tail_block=wl.NB,
                              tail_len=wl.ctx % wl.blk)
        for h in hs:
            cols = slice(h * wl.G, (h + 1) * wl.G)
            err = (gout[b:b + 1, :, cols].double() - ref[:, :, cols]).abs().max().item()
            worst = max(worst, err)
            assert err <= U.out_atol(wl.torch_dtype), (b, h, err)
    return worst, n_differ


def test_repeated_calls_identical():
    """Scoring, selection and attention leave the workspace ready for the
    next call: repeated calls give bit-identical selections and outputs."""
    for over in (dict(), dict(B=8, Hq=32, Hkv=8, ctx=64 * 40)):
        wl = small_wl(**over)
        x = W.make_layer(wl)
        st = api.LayerState(wl, x.to("cuda"))
        outs, sels = [], []
        for _ in range(3):
            st.out.zero_()
            st.sel.fill_(-7)
            st.verify()
            torch.cuda.synchronize()
            outs.append(st.out.clone())
            sels.append(st.sel.clone())
        assert all(torch.equal(outs[0], o) for o in outs[1:])
        assert all(torch.equal(sels[0], s) for s in sels[1:])
        assert api.sv_read_status(st.ws) == 0


def test_verify_tiny_f32():
    wl = W.WORKLOADS["tiny_f32"]
    x = W.make_layer(wl)
    _verify_vs_oracle(wl, x, x.to("cuda"))


def test_verify_llama8b_32k_full():
    wl = W.WORKLOADS["llama8b_32k"]
    x = W.make_layer(wl)
    _verify_vs_oracle(wl, x, x.to("cuda"))


def test_verify_llama8b_32k_partial_last_block():
    """A 32K context plus 40 tokens: 512 full blocks compete for the budget,
    the 40-token block is always attended."""
    from dataclasses import replace
    wl = replace(W.WORKLOADS["llama8b_32k"], ctx=32768 + 40)
    x = W.make_layer(wl)
    _verify_vs_oracle(wl, x, x.to("cuda"))


def test_verify_empty_context():
    wl = small_wl(ctx=0)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    out = st.verify()
    torch.cuda.synchronize()
    ref = O.sparse_attend(x.q, x.k_pool, x.v_pool, x.block_table,
                          torch.zeros(wl.B, wl.Hkv, 0, dtype=torch.int64), x.draft_k, x.draft_v,
                          wl.parent_list())
    U.compare_out(out, ref, U.BF16_ATOL)


def test_verify_short_context_keeps_all_blocks():
    wl = small_wl(ctx=64 * 48, budget=W.PIECEWISE_6P25_ABOVE_32K)  # 3072 <= 4096: all blocks
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    out = st.verify()
    torch.cuda.synchronize()
    assert st.k == wl.NB
    assert (st.sel.cpu()[:, :, :wl.NB] == torch.arange(wl.NB, dtype=torch.int32)).all()
    ref = O.dense_verify_attention(x.q, O.logical_kv(x.k_pool, x.block_table, wl.NB),
                                   O.logical_kv(x.v_pool, x.block_table, wl.NB), x.draft_k,
                                   x.draft_v, wl.parent_list())
    U.compare_out(out, ref, U.BF16_ATOL)


@pytest.mark.slow
def test_verify_llama8b_128k_b4_all_pairs():
    """The benchmark workload (B4, 128K context, 128 of 2048 blocks), every
    (sequence, KV head) pair against the oracle."""
    wl = W.WORKLOADS["llama8b_128k_b4"]
    xd = W.make_layer(wl, device="cuda")
    x = xd.to("cpu")
    _verify_vs_oracle(wl, x, xd)


@pytest.mark.slow
def test_verify_qwen3moe_tree_all_pairs():
    """Qwen3-MoE-shaped tree workload (B8, G8, T16 tree, 128 of 1024 blocks),
    every pair against the oracle."""
    wl = W.WORKLOADS["qwen3moe_64k_b8_tree16"]
    xd = W.make_layer(wl, device="cuda")
    x = xd.to("cpu")
    _verify_vs_oracle(wl, x, xd)


@pytest.mark.slow
def test_stack_llama8b_60k_reuse():
    """32-layer stack with the selection recomputed every 2nd layer, every
    layer against the oracle: a computing layer's selection against the
    oracle's top-k of that layer (bit-exact outside a boundary band), a reuse
    layer's selection bit-identical to the computing layer's, and every
    layer's output against the oracle layer (oracle.verify_layer, which is
    what oracle.verify_stack runs per layer) attending over that selection."""
    wl = W.WORKLOADS["llama8b_60k_32layer"]
    ps = W.planted_sets(wl)
    prev = None
    oracle_sel = None
    for l in range(wl.layers):
        xd = W.make_layer(wl, l, device="cuda", planted=ps[l])
        st = api.LayerState(wl, xd)
        reuse = l % wl.compute_every != 0
        if reuse:
            st.slot = prev.slot.copy()
        st.verify(reuse=int(reuse))
        torch.cuda.synchronize()
        assert api.sv_read_status(st.ws) == 0
        gsel, gout = st.sel.cpu(), st.out.cpu()
        x = xd.to("cpu")
        if reuse:
            assert torch.equal(gsel, prev_sel), l
            ref, _, _ = O.verify_layer(x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k,
                                       x.draft_v, wl.parent_list(), wl.ctx, wl.blk, wl.budget,
                                       reuse_sel=used)
        else:
            ref, oracle_sel, scores = O.verify_layer(x.q, x.k_pool, x.v_pool, x.block_table,
                                                     x.draft_k, x.draft_v, wl.parent_list(),
                                                     wl.ctx, wl.blk, wl.budget)
            k = oracle_sel.shape[-1]
            differ = U.compare_selection(gsel, scores, k)
            used = gsel[:, :, :k].long()
            if differ:  # the oracle's attention over the set the GPU used
                ref, _, _ = O.verify_layer(x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k,
                                           x.draft_v, wl.parent_list(), wl.ctx, wl.blk,
                                           wl.budget, reuse_sel=used)
        U.compare_out(gout, ref, U.BF16_ATOL)
        prev, prev_sel = st, gsel
        del xd, x


# ------------------------------------------------------------------ device-side checks
def test_bad_indices_flagged_not_faulting():
    """A selected block outside [0, NB) and a block-table entry outside the
    pool are skipped and reported through the status word."""
    wl = small_wl(ctx=64 * 20)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd, kmax=4, build_reps=False)
    sel = torch.tensor([[[0, 3, 5, wl.NB + 7]] * wl.Hkv] * wl.B, dtype=torch.int32).cuda()
    out = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, sel, 4, 4, xd.draft_k, xd.draft_v, None, out, st.ws)
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) & api.SV_FLAG_BAD_BLOCK_INDEX
    api.sv_clear_status(st.ws)
    bt = xd.block_table.clone()
    bt[0, 3] = x.k_pool.shape[0] + 100
    kv = api.make_kv(xd.k_pool, xd.v_pool, bt, wl.ctx)
    sel2 = torch.tensor([[[0, 3, 5, 6]] * wl.Hkv] * wl.B, dtype=torch.int32).cuda()
    api.sv_sparse_attend(st.shape, xd.q, kv, sel2, 4, 4, xd.draft_k, xd.draft_v, None, out, st.ws)
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) & api.SV_FLAG_BAD_PAGE
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------------ acceptance write-back
def _append_case(dtype, blk, ctx, n_acc, acc, T=6, Hkv=2, d=128, seed=3):
    B = len(ctx)
    nbt = max((c + T + blk - 1) // blk for c in ctx)  # room for every appended token
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    P = B * nbt
    kp = torch.randn(P, Hkv, blk, d, generator=g).to(dt)
    vp = torch.randn(P, Hkv, blk, d, generator=g).to(dt)
    dk = torch.randn(B, T, Hkv, d, generator=g).to(dt)
    dv = torch.randn(B, T, Hkv, d, generator=g).to(dt)
    bt = torch.randperm(P, generator=g).view(B, nbt).to(torch.int32)
    accept = torch.full((B, T), -1, dtype=torch.int32)
    for b in range(B):
        accept[b, :len(acc[b])] = torch.tensor(acc[b], dtype=torch.int32)
    return kp, vp, dk, dv, bt, accept


@pytest.mark.parametrize("dtype,blk", [("bf16", 64), ("bf16", 16), ("f32", 16)])
def test_append_kv_vs_oracle(dtype, blk):
    ctx = [blk * 3 + 5, blk * 2, blk * 4 + blk - 1]
    n_acc = [3, 6, 2]
    acc = [[0, 1, 3], [0, 2, 4, 5, 1, 3], [0, 5]]
    T, Hkv, d = 6, 2, 128
    kp, vp, dk, dv, bt, accept = _append_case(dtype, blk, ctx, n_acc, acc, T=T, Hkv=Hkv, d=d)
    B, nbt = bt.shape
    shape = api.make_shape(B, 4, Hkv, d, blk, T, kp.dtype)
    reps_before = torch.randn(B, Hkv, nbt, d)  # stand-ins: only filled blocks may change
    kpd, vpd, reps = kp.cuda(), vp.cuda(), reps_before.clone().cuda()
    ws = api.alloc_workspace(shape, nbt, 4)
    api.sv_append_kv(shape, kpd, vpd, bt.cuda(), torch.tensor(ctx, dtype=torch.int32).cuda(),
                     torch.tensor(n_acc, dtype=torch.int32).cuda(), accept.cuda(), dk.cuda(),
                     dv.cuda(), reps, ws)
    torch.cuda.synchronize()
    assert api.sv_read_status(ws) == 0
    kn, vn, filled = O.append_accepted(kp, vp, bt, ctx, n_acc, accept.tolist(), dk, dv)
    assert torch.equal(kpd.cpu(), kn) and torch.equal(vpd.cpu(), vn)  # a copy: bit-exact
    new_reps = O.block_representatives(kn, bt, nbt, blk)
    got = reps.cpu()
    for b in range(B):
        for j in range(nbt):
            if j in filled[b]:
                assert torch.allclose(got[b, :, j].double(), new_reps[b, :, j], atol=1e-5), (b, j)
            else:
                assert torch.equal(got[b, :, j], reps_before[b, :, j]), (b, j)
    assert any(filled)  # the case completes blocks


def test_append_kv_bad_index_skipped_and_flagged():
    ctx, n_acc, acc = [64 + 3, 64], [2, 2], [[0, 7], [1, 0]]  # draft 7 does not exist (T = 6)
    kp, vp, dk, dv, bt, accept = _append_case("bf16", 64, ctx, n_acc, acc)
    B, nbt = bt.shape
    shape = api.make_shape(B, 4, 2, 128, 64, 6, kp.dtype)
    kpd, vpd = kp.cuda(), vp.cuda()
    ws = api.alloc_workspace(shape, nbt, 4)
    api.sv_append_kv(shape, kpd, vpd, bt.cuda(), torch.tensor(ctx, dtype=torch.int32).cuda(),
                     torch.tensor(n_acc, dtype=torch.int32).cuda(), accept.cuda(), dk.cuda(),
                     dv.cuda(), None, ws)
    torch.cuda.synchronize()
    assert api.sv_read_status(ws) & api.SV_FLAG_BAD_BLOCK_INDEX
    # the bad row is skipped, the others land
    good = [[0], [1, 0]]
    kn, vn, _ = O.append_accepted(kp, vp, bt, ctx, [1, 2], good, dk, dv)
    assert torch.equal(kpd.cpu(), kn) and torch.equal(vpd.cpu(), vn)


def test_verify_append_verify_loop():
    """Two steps of the speculative loop on the device against the oracle:
    verify at ctx, append n accepted drafts (the same n for every sequence),
    then verify the next step's drafts at ctx + n, whose last block is
    partial."""
    from dataclasses import replace
    wl = replace(small_wl(B=3, Hq=8, Hkv=2, ctx=64 * 24, T=8), ctx=64 * 24)
    n = 5
    x = W.make_layer(replace(wl, ctx=wl.ctx + 64))  # pages for the appended tokens
    x0 = W.LayerInputs(x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k, x.draft_v, x.planted,
                       parents=x.parents)
    xd = x0.to("cuda")
    st = api.LayerState(wl, xd)
    out1 = st.verify()
    torch.cuda.synchronize()
    # accept the first n drafts of the chain
    accept = torch.tensor([list(range(n)) + [-1] * (wl.T - n)] * wl.B, dtype=torch.int32)
    ctx_t = torch.full((wl.B,), wl.ctx, dtype=torch.int32)
    nacc_t = torch.full((wl.B,), n, dtype=torch.int32)
    api.sv_append_kv(st.shape, xd.k_pool, xd.v_pool, xd.block_table, ctx_t.cuda(), nacc_t.cuda(),
                     accept.cuda(), xd.draft_k, xd.draft_v, st.reps, st.ws)
    # next step: new drafts and queries over the longer context
    wl2 = replace(wl, ctx=wl.ctx + n)
    g = torch.Generator().manual_seed(77)
    q2 = torch.randn(x.q.shape, generator=g).to(x.q.dtype)
    dk2 = torch.randn(x.draft_k.shape, generator=g).to(x.q.dtype)
    dv2 = torch.randn(x.draft_v.shape, generator=g).to(x.q.dtype)
    st2 = api.LayerState(wl2, W.LayerInputs(q2.cuda(), xd.k_pool, xd.v_pool, xd.block_table,
                                            dk2.cuda(), dv2.cuda(), x.planted, parents=x.parents),
                         build_reps=False)
    st2.reps.copy_(st.reps)  # the running representatives, updated by the append
    out2 = st2.verify()
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0 and api.sv_read_status(st2.ws) == 0
    # the same two steps on the oracle
    ref1, _, _ = O.verify_layer(x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k, x.draft_v,
                                wl.parent_list(), wl.ctx, wl.blk, wl.budget)
    U.compare_out(out1, ref1, U.BF16_ATOL)
    kn, vn, _ = O.append_accepted(x.k_pool, x.v_pool, x.block_table, [wl.ctx] * wl.B, [n] * wl.B,
                                  accept.tolist(), x.draft_k, x.draft_v)
    assert torch.equal(xd.k_pool.cpu(), kn) and torch.equal(xd.v_pool.cpu(), vn)
    ref2, sel2, scores2 = O.verify_layer(q2, kn, vn, x.block_table, dk2, dv2, wl.parent_list(),
                                         wl2.ctx, wl.blk, wl.budget)
    if U.compare_selection(st2.sel.cpu(), scores2, st2.k):
        # a boundary-band difference: the oracle over the set the GPU used
        ref2, _, _ = O.verify_layer(q2, kn, vn, x.block_table, dk2, dv2, wl.parent_list(),
                                    wl2.ctx, wl.blk, wl.budget,
                                    reuse_sel=st2.sel.cpu()[:, :, :st2.k].long())
    U.compare_out(out2, ref2, U.BF16_ATOL)


# ------------------------------------------------------------------ reuse schedules, diagnostic
@pytest.mark.parametrize("every", [3, 4])
def test_stack_reuse_schedules(every):
    """Layers recompute the selection every `every`-th layer and reuse it in
    between (any schedule goes through the reuse flag); every layer against
    the oracle stack, with a partial last block."""
    from dataclasses import replace
    wl = replace(small_wl(ctx=64 * 30 + 20), name="stack", layers=6, compute_every=every, drift=2,
                 budget=W.Budget(W.BUDGET_FIXED, 9, 0, 0, 0, 0, 0))
    ps = W.planted_sets(wl)
    prev, sels, outs, cpu_layers = None, [], [], []
    for l in range(wl.layers):
        xd = W.make_layer(wl, l, device="cuda", planted=ps[l])
        st = api.LayerState(wl, xd)
        reuse = l % every != 0
        if reuse:
            st.slot = prev.slot.copy()
        st.verify(reuse=int(reuse))
        torch.cuda.synchronize()
        assert api.sv_read_status(st.ws) == 0
        sels.append(st.sel.cpu())
        outs.append(st.out.cpu())
        x = xd.to("cpu")
        cpu_layers.append((x.q, x.k_pool, x.v_pool, x.block_table, x.draft_k, x.draft_v))
        prev = st
    ref_outs, ref_sels = O.verify_stack(cpu_layers, wl.parent_list(), wl.ctx, wl.blk, wl.budget,
                                        every)
    for l in range(wl.layers):
        if l % every:
            assert torch.equal(sels[l], sels[l - l % every])
        else:
            reps = O.block_representatives(cpu_layers[l][1], cpu_layers[l][3], wl.NB, wl.blk)
            scores = O.block_scores(cpu_layers[l][0], reps, wl.G)
            assert not U.compare_selection(sels[l], scores, ref_sels[l].shape[-1])
        U.compare_out(outs[l], ref_outs[l], U.BF16_ATOL)


def test_draft_selection_overlap_vs_oracle():
    """The shared-set diagnostic on the device (the library's score and
    select per draft) equals the oracle's overlaps."""
    from sparse_verification_attention_gb300 import diagnostics
    wl = small_wl(B=2, ctx=64 * 40, T=8)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    k = 10
    got = diagnostics.draft_selection_overlap(st.shape, xd.q, st.reps, st.kv, k)
    reps = O.block_representatives(x.k_pool, x.block_table, wl.NB, wl.blk)
    want = O.draft_selection_overlap(x.q, reps, wl.G, k)
    assert got.shape == want.shape
    assert torch.all(got[:, :, 0] == 1.0)
    # selections match bit-exactly away from near-ties, so the overlaps agree
    # to within one block
    assert (got - want).abs().max().item() <= 1.0 / k + 1e-12
    assert (got - want).abs().mean().item() < 0.02


def test_reset_workspace_repairs_stale_words():
    """A call that gave up on a wait may leave a pair's count or claim words
    non-zero. sv_reset_workspace zeroes the status word and every
    per-(b, h) word, after which the same workspace gives the same result
    again (the garbage is written by the test, on the host's orders; no wait
    is made to run out)."""
    wl = small_wl(B=4, Hq=32, Hkv=8, ctx=64 * 60, budget=W.Budget(W.BUDGET_FIXED, 20, 0, 0, 0, 0, 0))
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    clean = st.verify().clone()
    torch.cuda.synchronize()
    pairs = wl.B * wl.Hkv
    header = 256 + 3 * pairs * 128  # status, then three arrays of one 128-byte line per pair
    st.ws[:header].fill_(0x5A)
    nb_max = st.x.block_table.shape[1]
    api.sv_reset_workspace(st.shape, nb_max, max(st.kmax, wl.NB, 1), st.ws)
    assert int(st.ws[:header].count_nonzero()) == 0
    again = st.verify()
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    assert torch.equal(again, clean)


def test_stale_merge_ticket_is_flagged():
    """A merge ticket word left non-zero by an earlier call (planted here by
    the host; nothing is made to fail on the device) gives no segment the
    pair's last ticket. The kernel flags it instead of leaving the pair's
    output silently unwritten, and sv_reset_workspace repairs the
    workspace."""
    wl = small_wl(B=4, Hq=32, Hkv=8, ctx=64 * 60, budget=W.Budget(W.BUDGET_FIXED, 20, 0, 0, 0, 0, 0))
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    plan = api.sv_attend_plan(st.shape, st.kv, st.k)
    assert plan.path == api.SV_PATH_TCGEN05 and plan.streamk == 1 and plan.cluster == 0
    clean = st.verify().clone()
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    pairs = wl.B * wl.Hkv
    ticket = 256 + pairs * 128 + 3 * 128 + 4  # pair 3's attention line, merge-ticket word
    st.ws[ticket:ticket + 4] = torch.tensor([0x5A, 0x5A, 0, 0], dtype=torch.uint8, device="cuda")
    st.verify()
    torch.cuda.synchronize()
    flags = int(st.ws[:4].view(torch.int32).item())
    assert flags & api.SV_FLAG_STALE_WORKSPACE, hex(flags)
    nb_max = st.x.block_table.shape[1]
    api.sv_reset_workspace(st.shape, nb_max, max(st.kmax, wl.NB, 1), st.ws)
    again = st.verify()
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    assert torch.equal(again, clean)


def test_reuse_guard_on_device():
    """A reuse layer may read a slot only after a computing layer wrote it for
    the same context and budget: the matching reuse attends over it, while a
    slot written for another context, or never written, is refused."""
    from dataclasses import replace
    wl = small_wl(ctx=64 * 30)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st0 = api.LayerState(wl, xd)
    st0.verify()
    st1 = api.LayerState(wl, xd, build_reps=False)
    out1 = st1.verify(reuse=api.VERIFY_REUSE, sel_from=st0)
    torch.cuda.synchronize()
    U.compare_out(out1, st0.out.cpu().double(), 0.0)  # same inputs, same set: same output
    st2 = api.LayerState(replace(wl, ctx=wl.ctx - 64), xd, build_reps=False)
    with pytest.raises(api.SvError) as e:
        st2.verify(reuse=api.VERIFY_REUSE, sel_from=st0)
    assert e.value.status == api.SV_ERR_INVALID_ARG
    fresh = api.LayerState(wl, xd, build_reps=False)
    with pytest.raises(api.SvError) as e:
        fresh.verify(reuse=api.VERIFY_REUSE)
    assert e.value.status == api.SV_ERR_INVALID_ARG


GUARD_CASES = [
    ("tc_streamk", dict(B=4, Hq=32, Hkv=8, ctx=64 * 200 + 21), 40),
    ("tc_cluster", dict(B=1, Hq=32, Hkv=8, ctx=64 * 100 + 7), 30),
    ("tc_cluster_tree_R128", dict(B=8, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                  ctx=64 * 40 + 9), 20),
    ("mma_blk32", dict(B=2, Hq=8, Hkv=2, blk=32, ctx=32 * 80 + 5), 15),
    ("generic_d96", dict(B=2, Hq=8, Hkv=2, d=96, blk=32, ctx=32 * 60 + 3), 11),
]


@pytest.mark.parametrize("name,over,k", GUARD_CASES, ids=[c[0] for c in GUARD_CASES])
def test_guard_pages_are_never_read(name, over, k):
    """Guard pages: the same layer with every page moved to an odd slot of a
    pool twice as large whose even slots hold NaN. Representatives, scores,
    selection and attention read only pages the block table names, so the
    result must equal the unguarded run bit for bit; a stray read of an
    unreferenced page would bring a NaN into it."""
    from dataclasses import replace
    wl = small_wl(budget=W.Budget(W.BUDGET_FIXED, k, 0, 0, 0, 0, 0), **over)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    ref = api.LayerState(wl, xd)
    out_ref = ref.verify().clone()
    sel_ref = ref.sel.clone()

    def guarded(pool):
        g = torch.full((2 * pool.shape[0],) + tuple(pool.shape[1:]), float("nan"),
                       dtype=pool.dtype, device=pool.device)
        g[1::2] = pool
        return g

    bt = xd.block_table
    xg = replace(xd, k_pool=guarded(xd.k_pool), v_pool=guarded(xd.v_pool),
                 block_table=torch.where(bt >= 0, 2 * bt + 1, bt).to(bt.dtype))
    st = api.LayerState(wl, xg)
    out = st.verify()
    torch.cuda.synchronize()
    assert api.sv_read_status(ref.ws) == 0 and api.sv_read_status(st.ws) == 0
    assert torch.equal(st.sel, sel_ref)
    assert not torch.isnan(out).any()
    assert torch.equal(out, out_ref)


@pytest.mark.parametrize("streams", [False, True], ids=["one_stream", "copy_streams"])
def test_verify_layer_host_buffers(streams):
    """sv_verify_layer_host takes the step's q and draft K/V from pinned host
    memory and returns the output there: it must give, bit for bit, what
    sv_verify_layer gives on device buffers, for a computing layer, a reuse
    layer after it and a full verification, on one stream and with separate
    copy streams."""
    wl = small_wl(B=2, Hq=32, Hkv=8, ctx=64 * 50 + 9)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    ref0 = api.LayerState(wl, xd)
    out0 = ref0.verify().clone()
    ref1 = api.LayerState(wl, xd, build_reps=False)
    out1 = ref1.verify(reuse=api.VERIFY_REUSE, sel_from=ref0).clone()
    torch.cuda.synchronize()
    hq, hk, hv = (t.contiguous().pin_memory() for t in (x.q, x.draft_k, x.draft_v))
    ci, co = (torch.cuda.Stream(), torch.cuda.Stream()) if streams else (None, None)
    st0 = api.LayerState(wl, xd)
    st1 = api.LayerState(wl, xd, build_reps=False)
    st1.slot = st0.slot
    st2 = api.LayerState(wl, xd, build_reps=False)
    ref2 = api.LayerState(wl, xd, build_reps=False)
    out2 = ref2.verify(reuse=api.VERIFY_FULL).clone()
    torch.cuda.synchronize()
    outs, ks = [], []
    for st, reuse in ((st0, api.VERIFY_COMPUTE), (st1, api.VERIFY_REUSE),
                      (st2, api.VERIFY_FULL)):
        q_dev, dk_dev, dv_dev = (torch.empty_like(t) for t in (xd.q, xd.draft_k, xd.draft_v))
        out_dev = torch.empty_like(st.out)
        out_h = torch.full(st.out.shape, float("nan"), dtype=st.out.dtype).pin_memory()
        ks.append(api.sv_verify_layer_host(st.shape, hq, q_dev, st.kv, st.reps, wl.budget, hk,
                                           hv, dk_dev, dv_dev, st.parents, reuse, st.slot,
                                           out_h, out_dev, st.ws, None, ci, co))
        outs.append(out_h)
    torch.cuda.synchronize()
    assert ks == [ref0.k, ref0.k, wl.NB]
    for st in (st0, st1, st2):
        assert api.sv_read_status(st.ws) == 0
    assert torch.equal(st0.sel, ref0.sel)
    assert torch.equal(outs[0], out0.cpu()) and torch.equal(outs[1], out1.cpu())
    assert torch.equal(outs[2], out2.cpu())


@pytest.mark.parametrize("tree", [False, True], ids=["chain", "tree16"])
def test_overlap_by_distance_vs_oracle(tree):
    """The overlap of draft pairs' own block sets by position distance (the
    figure after the Figure 1 caption), on the device: every draft's own
    selection against the oracle's (bit-exact outside a boundary band), and
    the per-distance means against the oracle's when the sets agree."""
    from sparse_verification_attention_gb300 import diagnostics
    over = dict(B=2, Hq=16, Hkv=2, T=16, parents=W.TREE16_PARENTS) if tree else dict(B=2, T=8)
    wl = small_wl(ctx=64 * 40, **over)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd)
    k = 10
    sels = diagnostics.draft_selections(st.shape, xd.q, st.reps, st.kv, k).cpu()
    reps = O.block_representatives(x.k_pool, x.block_table, wl.NB, wl.blk)
    differ = 0
    for t in range(wl.T):
        scores = O.block_scores(x.q[:, t:t + 1], reps, wl.G)
        differ += len(U.compare_selection(sels[t].view(wl.B, wl.Hkv, k), scores, k))
    ov0, byd = diagnostics.selection_overlaps(st.shape, xd.q, st.reps, st.kv, k, wl.parents)
    want = O.draft_overlap_by_distance(x.q, reps, wl.G, k, wl.parent_list())
    assert torch.equal(torch.isnan(byd), torch.isnan(want))
    assert torch.all(ov0[:, :, 0] == 1.0)
    if differ == 0:
        ok = ~torch.isnan(want)
        assert torch.allclose(byd[ok], want[ok], rtol=0, atol=1e-6)
        assert torch.allclose(ov0, O.draft_selection_overlap(x.q, reps, wl.G, k), rtol=0,
                              atol=1e-6)


def test_verify_full_mode_equals_dense():
    """sv_verify_layer(reuse = 2): full verification over every block and the
    partial one, against the oracle's dense attention; sel_cache untouched."""
    wl = small_wl(B=3, Hq=8, Hkv=2, ctx=64 * 22 + 30)
    x = W.make_layer(wl)
    xd = x.to("cuda")
    st = api.LayerState(wl, xd, kmax=wl.NB, build_reps=False)
    st.sel.fill_(-7)
    out = st.verify(reuse=api.VERIFY_FULL)
    torch.cuda.synchronize()
    assert api.sv_read_status(st.ws) == 0
    assert int((st.sel != -7).sum()) == 0
    ref = O.dense_verify_attention(x.q, O.logical_kv_tokens(x.k_pool, x.block_table, wl.ctx),
                                   O.logical_kv_tokens(x.v_pool, x.block_table, wl.ctx), x.draft_k,
                                   x.draft_v, wl.parent_list())
    U.compare_out(out, ref, U.BF16_ATOL)
