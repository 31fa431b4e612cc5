"""Host-side checks of libsva.so that need no GPU: it loads, exports every
symbol include/sva.h declares, computes the piecewise budget exactly like the
oracle, sizes workspaces, and rejects bad arguments before launching."""
import ctypes as C
import os
import re

import pytest
import torch

from oracle import sva_oracle as O
from sparse_verification_attention_gb300 import api, build_lib
from sparse_verification_attention_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return api.lib()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "sva.h")).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\*]+\s+)+\**(sv_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(L):
    syms = header_symbols()
    assert len(syms) >= 12, syms
    for s in syms:
        assert hasattr(L, s), f"libsva.so does not export {s}"
    assert set(syms) == set(api.EXPORTED)


def test_abi_version(L):
    assert api.sv_abi_version() == api.ABI_VERSION == 4


def test_budget_matches_oracle_golden(L):
    path = os.path.join(ROOT, "tests", "golden", "budget_table.txt")
    n = 0
    for ln in open(path):
        ln = ln.split("#")[0].strip()
        if not ln:
            continue
        f = ln.split()
        ctx, nb, mode, fixed, short, floor = map(int, f[:6])
        b = W.Budget(mode, fixed, short, floor, float(f[6]), int(f[7]), float(f[8]))
        assert api.sv_budget_blocks(b, ctx, nb) == int(f[9]), ln
        n += 1
    assert n >= 10


def test_budget_matches_oracle_random(L):
    g = torch.Generator().manual_seed(1)
    fracs = [0.03125, 0.0625, 0.1, 0.125, 0.2, 0.25, 0.3, 0.5, 1.0]
    for _ in range(4500):
        mode = int(torch.randint(0, 3, (1,), generator=g))
        nb = int(torch.randint(0, 5000, (1,), generator=g))
        ctx = nb * int(torch.randint(1, 129, (1,), generator=g))
        b = W.Budget(mode, int(torch.randint(0, 300, (1,), generator=g)),
                     int(torch.randint(0, 70000, (1,), generator=g)),
                     int(torch.randint(0, 200, (1,), generator=g)),
                     fracs[int(torch.randint(0, len(fracs), (1,), generator=g))],
                     int(torch.randint(0, 300000, (1,), generator=g)),
                     fracs[int(torch.randint(0, len(fracs), (1,), generator=g))])
        if mode == W.BUDGET_SMOOTH and b.long_ctx < b.short_ctx:  # invalid for SMOOTH
            assert api.sv_budget_blocks(b, ctx, nb) == -1
            b = W.Budget(mode, b.fixed_blocks, b.long_ctx, b.floor_blocks, b.frac_mid,
                         b.short_ctx, b.frac_long)
        assert api.sv_budget_blocks(b, ctx, nb) == O.budget_from(b, ctx, nb), (b, ctx, nb)


def test_budget_rejects_invalid(L):
    assert L.sv_budget_blocks(None, 100, 10) == -1
    assert api.sv_budget_blocks(W.Budget(7), 100, 10) == -1
    assert api.sv_budget_blocks(W.Budget(1, 0, 0, 0, 1.5, 0, 0.1), 100, 10) == -1
    assert api.sv_budget_blocks(W.Budget(0, -1), 100, 10) == -1


def test_workspace_sizes(L):
    s = api.make_shape(4, 32, 8, 128, 64, 8, torch.bfloat16)
    n = api.sv_workspace_bytes(s, 2048, 128)
    # status + three arrays of per-(b,h) words, one 128-byte line per pair
    # (score and attend counts, a merge claim word) + the scores + the
    # kept blocks' pool rows (kmax per pair) + split partials o and (m, l);
    # 130 work units (128 blocks, a partial block, the draft tile) capped at
    # 64 slots
    pairs = 4 * 8
    ctrs = 3 * pairs * 128
    scores = pairs * 2048 * 4
    rows = pairs * 128 * 4
    part = pairs * 64 * 32 * 128 * 4
    ml = pairs * 64 * 32 * 2 * 4
    assert n == 256 + ctrs + scores + rows + part + ml
    # 8 selected blocks + a partial last block + the draft tile + one slot
    # for a run that leaves a pair mid-stream = 11 partial slots
    n8 = api.sv_workspace_bytes(s, 2048, 8)
    assert n8 == (256 + ctrs + scores + pairs * 8 * 4 + pairs * 11 * 32 * 128 * 4
                  + pairs * 11 * 32 * 2 * 4)
    bad = api.make_shape(4, 30, 8, 128, 64, 8, torch.bfloat16)  # Hq % Hkv != 0
    assert api.sv_workspace_bytes(bad, 2048, 128) == 0
    assert api.sv_workspace_bytes(api.make_shape(1, 4, 2, 12, 16, 4, 1), 64, 8) == 0  # d % 8


def _status(L, fn, *args):
    st = fn(*args)
    return st, L.sv_last_error().decode()


def test_invalid_arguments_rejected_before_launch(L):
    """Every call below must fail validation on the host (no GPU here: a
    launch attempt would come back as SV_ERR_CUDA instead)."""
    s = api.make_shape(1, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20  # never dereferenced: validation fails first
    kv = api.KV(fake, fake, fake, 64, 64, 1024)
    ws_n = api.sv_workspace_bytes(s, 64, 8)
    b = api.make_budget(W.Budget(W.BUDGET_FIXED, 8, 0, 0, 0, 0, 0))
    st, msg = _status(L, L.sv_sparse_attend, C.byref(s), None, C.byref(kv), None, 0, 0, None, None,
                      None, None, None, 0, None)
    assert st == api.SV_ERR_INVALID_ARG and "NULL" in msg
    # a partial last block (1000 = 62 * 16 + 8) needs its own block-table column
    tail_kv = api.KV(fake, fake, fake, 62, 64, 1000)
    st, msg = _status(L, L.sv_build_reps, C.byref(s), C.byref(tail_kv), 0, 1, fake, None)
    assert st == api.SV_ERR_INVALID_ARG and "nb_max" in msg
    # ... and gets no representative: only the 62 full blocks do
    tail_kv = api.KV(fake, fake, fake, 63, 64, 1000)
    st, msg = _status(L, L.sv_build_reps, C.byref(s), C.byref(tail_kv), 62, 1, fake, None)
    assert st == api.SV_ERR_INVALID_ARG, msg
    st, msg = _status(L, L.sv_build_reps, C.byref(s), C.byref(kv), 60, 10, fake, None)
    assert st == api.SV_ERR_INVALID_ARG, msg
    small = api.KV(fake, fake, fake, 10, 64, 1024)  # nb_max < NB
    st, msg = _status(L, L.sv_build_reps, C.byref(s), C.byref(small), 0, 1, fake, None)
    assert st == api.SV_ERR_INVALID_ARG and "nb_max" in msg
    k = C.c_int(0)
    st, msg = _status(L, L.sv_score_select, C.byref(s), fake, fake, C.byref(kv), C.byref(b),
                      fake, 4, C.byref(k), fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "kmax" in msg
    st, msg = _status(L, L.sv_score_select, C.byref(s), fake, fake, C.byref(kv), C.byref(b),
                      fake, 8, C.byref(k), fake, ws_n - 1, None)
    assert st == api.SV_ERR_WORKSPACE, msg
    bad_par = (C.c_int32 * 4)(-1, 0, 2, 1)  # parent[2] = 2 is not an earlier draft
    st, msg = _status(L, L.sv_sparse_attend, C.byref(s), fake, C.byref(kv), fake, 8, 8, fake, fake,
                      bad_par, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "draft_parent" in msg
    slot8 = api.SelSlotC(fake, 8, 0)
    st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), fake, C.byref(b), fake,
                      fake, None, 3, C.byref(slot8), None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "reuse" in msg
    big_t = api.make_shape(1, 4, 2, 64, 16, 65, torch.float32)
    st, msg = _status(L, L.sv_sparse_attend, C.byref(big_t), fake, C.byref(kv), fake, 8, 8, fake,
                      fake, None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_UNSUPPORTED, msg
    st, msg = _status(L, L.sv_clear_status, None, None)
    assert st == api.SV_ERR_INVALID_ARG
    # acceptance write-back: NULL index arrays, misaligned pools
    st, msg = _status(L, L.sv_append_kv, C.byref(s), fake, fake, fake, 64, 64, None, fake, fake,
                      fake, fake, None, None, None)
    assert st == api.SV_ERR_INVALID_ARG and "NULL" in msg
    st, msg = _status(L, L.sv_append_kv, C.byref(s), fake + 4, fake, fake, 64, 64, fake, fake, fake,
                      fake, fake, None, None, None)
    assert st == api.SV_ERR_INVALID_ARG and "aligned" in msg


def test_verify_schedule():
    s = api.VerifySchedule(full_period=4, compute_every=2)
    modes = [[s.mode(step, layer) for layer in range(4)] for step in range(8)]
    assert modes[3] == modes[7] == [api.VERIFY_FULL] * 4          # every 4th step is full
    assert modes[0] == [api.VERIFY_COMPUTE, api.VERIFY_REUSE] * 2  # otherwise compute / reuse
    assert api.VerifySchedule().mode(5, 3) == api.VERIFY_COMPUTE
    with pytest.raises(ValueError):
        api.VerifySchedule(compute_every=0)


def test_verify_full_mode_needs_no_selection_buffers(L):
    """reuse = 2 (full verification) validates without reps, budget or
    sel_cache; reuse = 3 is rejected."""
    s = api.make_shape(1, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20
    kv = api.KV(fake, fake, fake, 64, 64, 1024)
    ws_n = api.sv_workspace_bytes(s, 64, 8)
    st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), None, None, fake,
                      fake, None, 3, None, None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "reuse" in msg
    slot8 = api.SelSlotC(None, 8, 0)
    st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), None, None, fake,
                      fake, None, 2, C.byref(slot8), None, fake, fake, ws_n - 1, None)
    assert st == api.SV_ERR_WORKSPACE, msg  # got past every selection check


def test_reuse_of_unwritten_or_stale_slot_is_refused(L):
    """Inter-layer reuse may only read a selection that a computing call
    wrote for the same shape, context and budget: a slot whose stamp is 0
    (never written) or another call's digest is refused on the host, before
    anything is launched."""
    s = api.make_shape(1, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20
    kv = api.KV(fake, fake, fake, 64, 64, 1024)
    b = api.make_budget(W.Budget(W.BUDGET_FIXED, 8, 0, 0, 0, 0, 0))
    ws_n = api.sv_workspace_bytes(s, 64, 8)
    for stamp, words in ((0, "no computing call"), (0x1234, "another shape")):
        slot = api.SelSlotC(fake, 8, stamp)
        st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), None, C.byref(b),
                          fake, fake, None, 1, C.byref(slot), None, fake, fake, ws_n, None)
        assert st == api.SV_ERR_INVALID_ARG and words in msg, msg
    st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), None, C.byref(b),
                      fake, fake, None, 1, None, None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "slot" in msg


def test_verify_layer_host_validates_before_copying(L):
    """The host-buffer entry refuses NULL host buffers, and any argument
    sv_verify_layer refuses, before it enqueues a copy (no GPU is touched)."""
    s = api.make_shape(1, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20
    kv = api.KV(fake, fake, fake, 64, 64, 1024)
    b = api.make_budget(W.Budget(W.BUDGET_FIXED, 8, 0, 0, 0, 0, 0))
    ws_n = api.sv_workspace_bytes(s, 64, 8)
    slot = api.SelSlotC(fake, 8, 0)
    f = L.sv_verify_layer_host
    for hosts in ((None, fake, fake, fake), (fake, None, fake, fake), (fake, fake, None, fake),
                  (fake, fake, fake, None)):
        hq, hk, hv, ho = hosts
        st, msg = _status(L, f, C.byref(s), hq, fake, C.byref(kv), fake, C.byref(b), hk, hv, fake,
                          fake, None, 0, C.byref(slot), None, ho, fake, fake, ws_n, None, None,
                          None)
        assert st == api.SV_ERR_INVALID_ARG and "host" in msg, msg
    # a reuse of a slot no computing call wrote: refused like sv_verify_layer
    st, msg = _status(L, f, C.byref(s), fake, fake, C.byref(kv), None, C.byref(b), fake, fake,
                      fake, fake, None, 1, C.byref(slot), None, fake, fake, fake, ws_n, None, None,
                      None)
    assert st == api.SV_ERR_INVALID_ARG and "no computing call" in msg, msg


def test_per_sequence_context_validation(L):
    """seq_ctx is checked on the host: negative lengths, a block table too
    narrow for the longest sequence and more than 64 sequences are refused
    before anything is launched."""
    s = api.make_shape(3, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20
    ws_n = api.sv_workspace_bytes(s, 64, 8)

    def kv(ctxs, nb_max=64):
        k = api.KV(fake, fake, fake, nb_max, 64, 0)
        arr = (C.c_int32 * len(ctxs))(*ctxs)
        k.seq_ctx = C.cast(arr, C.POINTER(C.c_int32))
        return k, arr

    k1, _a1 = kv([100, -5, 16])
    st, msg = _status(L, L.sv_sparse_attend, C.byref(s), fake, C.byref(k1), None, 0, 0, fake, fake,
                      None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "seq_ctx[1]" in msg
    # the longest sequence (1000 tokens = 62 full blocks + 8) needs 63 columns
    k2, _a2 = kv([1000, 0, 17], nb_max=62)
    st, msg = _status(L, L.sv_sparse_attend, C.byref(s), fake, C.byref(k2), None, 0, 0, fake, fake,
                      None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "nb_max" in msg
    big = api.make_shape(65, 4, 2, 64, 16, 4, torch.float32)
    k3, _a3 = kv([16] * 65)
    st, msg = _status(L, L.sv_sparse_attend, C.byref(big), fake, C.byref(k3), None, 0, 0, fake,
                      fake, None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_UNSUPPORTED and "per-sequence" in msg
    # the uniform ctx is ignored when seq_ctx is given (here it is negative)
    k4, _a4 = kv([16, 32, 0])
    k4.ctx = -1
    st, msg = _status(L, L.sv_build_reps, C.byref(s), C.byref(k4), 0, 3, fake, None)
    assert st == api.SV_ERR_INVALID_ARG and "blocks [0, 3) outside [0, 2)" in msg


def test_make_kv_keeps_seq_ctx_alive():
    t = torch.zeros(4, 2, 16, 64)
    bt = torch.zeros(2, 8, dtype=torch.int32)
    kv = api.make_kv(t, t, bt, 0, [100, 7])
    assert [kv.seq_ctx[i] for i in range(2)] == [100, 7]
    assert not api.make_kv(t, t, bt, 50).seq_ctx  # NULL: the uniform ctx


def test_make_kv_rejects_short_seq_ctx():
    t = torch.zeros(4, 2, 16, 64)
    bt = torch.zeros(3, 8, dtype=torch.int32)
    with pytest.raises(ValueError):
        api.make_kv(t, t, bt, 0, [100, 7])  # 2 lengths for 3 sequences


def test_per_sequence_budget_checked_against_kmax(L):
    """With per-sequence lengths the largest per-sequence budget must fit
    kmax; it is checked before anything is launched."""
    s = api.make_shape(2, 4, 2, 64, 16, 4, torch.float32)
    fake = 1 << 20
    kv = api.KV(fake, fake, fake, 64, 64, 0)
    arr = (C.c_int32 * 2)(16 * 10, 16 * 40)  # 10 and 40 full blocks
    kv.seq_ctx = C.cast(arr, C.POINTER(C.c_int32))
    b = api.make_budget(W.Budget(W.BUDGET_FIXED, 30, 0, 0, 0, 0, 0))  # k_b = 10, 30
    k = C.c_int(-1)
    ws_n = api.sv_workspace_bytes(s, 64, 30)
    st, msg = _status(L, L.sv_score_select, C.byref(s), fake, fake, C.byref(kv), C.byref(b),
                      fake, 29, C.byref(k), fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "k=30 exceeds kmax=29" in msg
    slot29 = api.SelSlotC(fake, 29, 0)
    st, msg = _status(L, L.sv_verify_layer, C.byref(s), fake, C.byref(kv), fake, C.byref(b), fake,
                      fake, None, 0, C.byref(slot29), None, fake, fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "k=30 exceeds kmax=29" in msg
    # one sequence too long for the block table's width
    arr2 = (C.c_int32 * 2)(16, 16 * 64 + 1)  # needs 65 columns
    kv.seq_ctx = C.cast(arr2, C.POINTER(C.c_int32))
    st, msg = _status(L, L.sv_score_select, C.byref(s), fake, fake, C.byref(kv), C.byref(b),
                      fake, 30, C.byref(k), fake, ws_n, None)
    assert st == api.SV_ERR_INVALID_ARG and "nb_max" in msg
