"""sv_sparse_attend_noalloc against sv_sparse_attend, through the C ABI.

The allocation-free entry serves callers that cannot allocate device memory
(an operation hosted by another runtime that hands it only its tensors after
that runtime's memory planner has claimed the device): its scratch is a
fixed array in the library's device code instead of a caller workspace. Each
case makes two calls in a row with different selections, so that anything
the shared array keeps from the previous call would show in the second
result. The file is named so that pytest collects it last.
"""
import pytest
import torch

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


def _wl(dtype="bf16", **kw):
    base = dict(name="noalloc", B=2, Hq=8, Hkv=2, d=128, blk=64, ctx=64 * 40, T=8, dtype=dtype,
                budget=W.Budget(W.BUDGET_FIXED, 13, 0, 0, 0, 0, 0), seed=33, n_planted=4,
                permute_pages=True)
    base.update(kw)
    return W.Workload(**base)


def _sel(B, H, NB, k, seed):
    g = torch.Generator().manual_seed(seed)
    sel = torch.full((B, H, max(k, 1)), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            if k:
                sel[b, h, :k] = torch.sort(torch.randperm(NB, generator=g)[:k]).values.to(torch.int32)
    return sel


CASES = [
    # name (expected path), workload overrides, selection sizes of the two calls
    ("tc", dict(), (13, 29)),
    ("tc_partial_last_block", dict(ctx=64 * 40 + 13), (13, 29)),
    ("tc_many_pairs_tree16", dict(B=8, Hq=32, Hkv=4, T=16, parents=W.TREE16_PARENTS,
                                  ctx=64 * 20), (11, 3)),
    ("mma", dict(Hq=4, Hkv=2, T=4, d=64, blk=32, ctx=32 * 50), (17, 40)),
    ("mma_cluster", dict(B=8, Hq=32, Hkv=8, blk=32, ctx=32 * 40), (9, 5)),
    ("generic_f32", dict(dtype="f32", d=64, blk=16, ctx=16 * 64, Hq=4, Hkv=2, T=4), (8, 21)),
    ("generic_R256", dict(T=32, Hq=16, Hkv=2, ctx=64 * 20), (6, 2)),
]
PATHS = {"tc": api.SV_PATH_TCGEN05, "mma": api.SV_PATH_MMA_SYNC,
         "generic": api.SV_PATH_CUDA_CORES}


@pytest.mark.parametrize("name,over,n_sels", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry(name, over, n_sels):
    over = dict(over)
    dtype = over.pop("dtype", "bf16")
    wl = _wl(dtype, **over)
    xd = W.make_layer(wl).to("cuda")
    st = api.LayerState(wl, xd, kmax=max(n_sels), build_reps=False)
    assert api.sv_attend_plan(st.shape, st.kv, n_sels[0]).path == PATHS[name.split("_")[0]]
    atol = U.out_atol(wl.torch_dtype)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, n_sel in enumerate(n_sels):
        sel = _sel(wl.B, wl.Hkv, wl.NB, n_sel, seed=100 * call + len(name)).cuda()
        want = torch.zeros_like(xd.q)
        api.sv_sparse_attend(st.shape, xd.q, st.kv, sel, n_sel, sel.shape[-1], xd.draft_k,
                             xd.draft_v, st.parents, want, st.ws)
        got = torch.full_like(xd.q, float("nan"))
        api.sv_sparse_attend_noalloc(st.shape, xd.q, st.kv, sel, n_sel, sel.shape[-1],
                                     xd.draft_k, xd.draft_v, st.parents, got, flags)
        torch.cuda.synchronize()
        assert api.sv_read_status(st.ws) == 0
        assert int(flags.item()) == 0, f"call {call}: flags {int(flags.item()):#x}"
        err = (got.double() - want.double()).abs().max().item()
        assert err <= atol, f"call {call} (n_sel={n_sel}): max abs diff {err}"


def test_noalloc_dense_twice():
    """sel == NULL attends to every block, on both calls."""
    wl = _wl(ctx=64 * 24)
    xd = W.make_layer(wl).to("cuda")
    st = api.LayerState(wl, xd, kmax=wl.NB, build_reps=False)
    want = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, None, 0, 0, xd.draft_k, xd.draft_v, None, want,
                         st.ws)
    for _ in range(2):
        got = torch.full_like(xd.q, float("nan"))
        api.sv_sparse_attend_noalloc(st.shape, xd.q, st.kv, None, 0, 0, xd.draft_k, xd.draft_v,
                                     None, got)
        torch.cuda.synchronize()
        assert (got.double() - want.double()).abs().max().item() <= U.BF16_ATOL


def test_noalloc_flags_are_per_call():
    """A bad selected block is reported in flags_out; the next call starts
    from a cleared status word and reports nothing."""
    wl = _wl(ctx=64 * 20)
    xd = W.make_layer(wl).to("cuda")
    st = api.LayerState(wl, xd, kmax=4, build_reps=False)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([[[0, 3, 5, wl.NB + 7]] * wl.Hkv] * wl.B, dtype=torch.int32).cuda()
    out = torch.zeros_like(xd.q)
    api.sv_sparse_attend_noalloc(st.shape, xd.q, st.kv, bad, 4, 4, xd.draft_k, xd.draft_v, None,
                                 out, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & api.SV_FLAG_BAD_BLOCK_INDEX
    good = torch.tensor([[[0, 3, 5, 6]] * wl.Hkv] * wl.B, dtype=torch.int32).cuda()
    api.sv_sparse_attend_noalloc(st.shape, xd.q, st.kv, good, 4, 4, xd.draft_k, xd.draft_v, None,
                                 out, flags)
    want = torch.zeros_like(xd.q)
    api.sv_sparse_attend(st.shape, xd.q, st.kv, good, 4, 4, xd.draft_k, xd.draft_v, None, want,
                         st.ws)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert (out.double() - want.double()).abs().max().item() <= U.BF16_ATOL


def test_noalloc_rejects_oversized_call():
    """256 (b, h) pairs of 256 stacked rows need about 32 MiB of partials even
    with one split each: more than the static scratch holds. The call is
    refused before anything is launched."""
    wl = _wl(B=64, Hq=16, Hkv=4, T=64, ctx=64 * 4, n_planted=0)
    xd = W.make_layer(wl).to("cuda")
    shape = api.make_shape(wl.B, wl.Hq, wl.Hkv, wl.d, wl.blk, wl.T, wl.torch_dtype)
    kv = api.make_kv(xd.k_pool, xd.v_pool, xd.block_table, wl.ctx)
    sel = _sel(wl.B, wl.Hkv, wl.NB, 2, seed=5).cuda()
    out = torch.zeros_like(xd.q)
    with pytest.raises(api.SvError) as ei:
        api.sv_sparse_attend_noalloc(shape, xd.q, kv, sel, 2, sel.shape[-1], xd.draft_k,
                                     xd.draft_v, None, out)
    assert ei.value.status == api.SV_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(out)) == 0
