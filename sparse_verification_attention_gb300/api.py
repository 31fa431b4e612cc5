"""Thin ctypes binding over libsva.so (include/sva.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. torch is used for device memory and streams; tensors are passed by
data_ptr(), streams by their cudaStream_t handle. Any non-OK status raises
SvError with the library's own message. There is no fallback: if libsva.so is
missing or was built for another machine, loading it raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

from . import workloads as W

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsva.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_WORKSPACE, SV_ERR_CUDA, \
    SV_ERR_DEVICE_FAULT = range(6)
SV_BF16, SV_F32 = 0, 1
SV_FLAG_BAD_BLOCK_INDEX, SV_FLAG_BAD_PAGE, SV_FLAG_WAIT_TIMEOUT, SV_FLAG_STALE_WORKSPACE = 1, 2, 4, 8

SV_PATH_CUDA_CORES, SV_PATH_MMA_SYNC, SV_PATH_TCGEN05 = 0, 1, 2
ABI_VERSION = 4  # SV_ABI_VERSION the structures below match

EXPORTED = ("sv_abi_version", "sv_last_error", "sv_budget_blocks", "sv_workspace_bytes",
            "sv_clear_status", "sv_read_status", "sv_build_reps", "sv_score_blocks",
            "sv_select_blocks", "sv_score_select", "sv_sparse_attend", "sv_attend_plan",
            "sv_verify_layer", "sv_sparse_attend_noalloc", "sv_append_kv",
            "sv_selection_overlap", "sv_reset_workspace", "sv_verify_layer_host")


class SvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"sva status {status}: {msg}")
        self.status = status


class Shape(C.Structure):
    _fields_ = [("B", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("d", C.c_int),
                ("blk", C.c_int), ("T", C.c_int), ("dtype", C.c_int)]


class BudgetC(C.Structure):
    _fields_ = [("mode", C.c_int), ("fixed_blocks", C.c_int), ("short_ctx", C.c_int),
                ("floor_blocks", C.c_int), ("frac_mid", C.c_double), ("long_ctx", C.c_int),
                ("frac_long", C.c_double)]


class KV(C.Structure):
    _fields_ = [("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("block_table", C.c_void_p),
                ("nb_max", C.c_int), ("num_pages", C.c_int), ("ctx", C.c_int),
                ("seq_ctx", C.POINTER(C.c_int32))]


class SelSlotC(C.Structure):
    _fields_ = [("sel", C.c_void_p), ("kmax", C.c_int), ("stamp", C.c_uint64)]


class SelSlot:
    """A selection cache slot (sv_sel_slot): the device selection [B, Hkv,
    kmax] int32 and the host-side stamp the library writes when a computing
    layer fills it and checks when a reuse layer reads it."""

    def __init__(self, B: int, Hkv: int, kmax: int, device="cuda"):
        self.tensor = torch.full((B, Hkv, max(kmax, 1)), -1, dtype=torch.int32, device=device)
        self.c = SelSlotC(self.tensor.data_ptr(), kmax, 0)

    def copy(self) -> "SelSlot":
        """A new slot holding a copy of this one's selection and stamp."""
        new = SelSlot.__new__(SelSlot)
        new.tensor = self.tensor.clone()
        new.c = SelSlotC(new.tensor.data_ptr(), self.c.kmax, self.c.stamp)
        return new

    @property
    def kmax(self) -> int:
        return self.c.kmax


class Plan(C.Structure):
    _fields_ = [("path", C.c_int), ("cluster", C.c_int), ("n_splits", C.c_int),
                ("blocks_per_split", C.c_int), ("ctas_per_sm", C.c_int),
                ("split_extra", C.c_int), ("streamk", C.c_int)]


_lib = None


def lib() -> C.CDLL:
    """Load libsva.so (once). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "sparse_verification_attention_gb300.build_lib.build()")
        L = C.CDLL(LIB_PATH)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "sv_abi_version": (i, []),
            "sv_last_error": (C.c_char_p, []),
            "sv_budget_blocks": (i, [C.POINTER(BudgetC), i, i]),
            "sv_workspace_bytes": (sz, [C.POINTER(Shape), i, i]),
            "sv_clear_status": (i, [vp, vp]),
            "sv_read_status": (i, [vp, C.POINTER(C.c_uint32), vp]),
            "sv_build_reps": (i, [C.POINTER(Shape), C.POINTER(KV), i, i, vp, vp]),
            "sv_score_blocks": (i, [C.POINTER(Shape), vp, vp, C.POINTER(KV), vp, vp]),
            "sv_select_blocks": (i, [C.POINTER(Shape), vp, i, i, vp, i, vp]),
            "sv_score_select": (i, [C.POINTER(Shape), vp, vp, C.POINTER(KV), C.POINTER(BudgetC),
                                    vp, i, C.POINTER(C.c_int), vp, sz, vp]),
            "sv_sparse_attend": (i, [C.POINTER(Shape), vp, C.POINTER(KV), vp, i, i, vp, vp,
                                     C.POINTER(C.c_int32), vp, vp, sz, vp]),
            "sv_attend_plan": (i, [C.POINTER(Shape), C.POINTER(KV), i, C.POINTER(Plan)]),
            "sv_verify_layer": (i, [C.POINTER(Shape), vp, C.POINTER(KV), vp, C.POINTER(BudgetC),
                                    vp, vp, C.POINTER(C.c_int32), i, C.POINTER(SelSlotC),
                                    C.POINTER(C.c_int), vp, vp, sz, vp]),
            "sv_sparse_attend_noalloc": (i, [C.POINTER(Shape), vp, C.POINTER(KV), vp, i, i, vp,
                                             vp, C.POINTER(C.c_int32), vp, vp, vp]),
            "sv_append_kv": (i, [C.POINTER(Shape), vp, vp, vp, i, i, vp, vp, vp, vp, vp, vp, vp,
                                 vp]),
            "sv_selection_overlap": (i, [vp, i, i, i, i, C.POINTER(C.c_int32), vp, vp, vp]),
            "sv_reset_workspace": (i, [C.POINTER(Shape), i, i, vp, sz, vp]),
            "sv_verify_layer_host": (i, [C.POINTER(Shape), vp, vp, C.POINTER(KV), vp,
                                         C.POINTER(BudgetC), vp, vp, vp, vp,
                                         C.POINTER(C.c_int32), i, C.POINTER(SelSlotC),
                                         C.POINTER(C.c_int), vp, vp, vp, sz, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        if L.sv_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{LIB_PATH} has ABI {L.sv_abi_version()}, the binding expects "
                               f"{ABI_VERSION}: rebuild it")
        _lib = L
    return _lib


def _check(status: int):
    if status != SV_OK:
        raise SvError(status, lib().sv_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return SV_BF16
    if t == torch.float32:
        return SV_F32
    raise ValueError(f"unsupported dtype {t}")


def make_shape(B, Hq, Hkv, d, blk, T, dtype) -> Shape:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return Shape(B, Hq, Hkv, d, blk, T, code)


def make_budget(b: W.Budget) -> BudgetC:
    return BudgetC(b.mode, b.fixed_blocks, b.short_ctx, b.floor_blocks, b.frac_mid, b.long_ctx,
                   b.frac_long)


def make_kv(k_pool: torch.Tensor, v_pool: Optional[torch.Tensor], block_table: torch.Tensor,
            ctx: int, seq_ctx: Optional[Sequence[int]] = None) -> KV:
    """The cache descriptor. seq_ctx (one prefix length per sequence, kept on
    the host) replaces the uniform ctx; the returned structure owns the
    array it points to. The library reads B entries of it, so it must have
    one per row of the block table."""
    kv = KV(k_pool.data_ptr(), None if v_pool is None else v_pool.data_ptr(),
            block_table.data_ptr(), block_table.shape[1], k_pool.shape[0], ctx)
    if seq_ctx is not None:
        if len(seq_ctx) != block_table.shape[0]:
            raise ValueError(f"seq_ctx has {len(seq_ctx)} entries for "
                             f"{block_table.shape[0]} sequences")
        arr = (C.c_int32 * len(seq_ctx))(*[int(c) for c in seq_ctx])
        kv._seq_ctx_keep = arr
        kv.seq_ctx = C.cast(arr, C.POINTER(C.c_int32))
    return kv


_parents_cache: dict = {}


def _parents(parents: Optional[Sequence[int]]):
    if parents is None:
        return None
    key = tuple(parents)
    arr = _parents_cache.get(key)
    if arr is None:  # the C array is only read during the call
        arr = (C.c_int32 * len(key))(*key)
        if len(_parents_cache) < 64:
            _parents_cache[key] = arr
    return arr


# ------------------------------------------------------------------ calls
def sv_abi_version() -> int:
    return lib().sv_abi_version()


def sv_budget_blocks(budget: W.Budget, ctx: int, nb: int) -> int:
    b = make_budget(budget)
    return lib().sv_budget_blocks(C.byref(b), ctx, nb)


def sv_workspace_bytes(shape: Shape, nb_max: int, kmax: int) -> int:
    return lib().sv_workspace_bytes(C.byref(shape), nb_max, kmax)


def alloc_workspace(shape: Shape, nb_max: int, kmax: int, device="cuda") -> torch.Tensor:
    n = sv_workspace_bytes(shape, nb_max, kmax)
    if n == 0:
        raise SvError(SV_ERR_INVALID_ARG, "invalid shape for a workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sv_clear_status(ws: torch.Tensor, stream=None):
    _check(lib().sv_clear_status(_ptr(ws), _stream(stream)))


def sv_reset_workspace(shape: Shape, nb_max: int, kmax: int, ws: torch.Tensor, stream=None):
    """Zero the workspace's status word and per-(b, h) counts and flags (what
    a workspace needs after a call that raised SV_FLAG_WAIT_TIMEOUT)."""
    _check(lib().sv_reset_workspace(C.byref(shape), nb_max, kmax, _ptr(ws), ws.numel(),
                                    _stream(stream)))


def sv_read_status(ws: torch.Tensor, stream=None) -> int:
    """Device status flags (0 = clean). Does not raise on set flags."""
    v = C.c_uint32(0)
    lib().sv_read_status(_ptr(ws), C.byref(v), _stream(stream))
    return int(v.value)


def sv_build_reps(shape: Shape, kv: KV, first_block: int, n_blocks: int, reps: torch.Tensor,
                  stream=None):
    _check(lib().sv_build_reps(C.byref(shape), C.byref(kv), first_block, n_blocks, _ptr(reps),
                               _stream(stream)))


def sv_score_blocks(shape: Shape, q, reps, kv: KV, scores, stream=None):
    _check(lib().sv_score_blocks(C.byref(shape), _ptr(q), _ptr(reps), C.byref(kv), _ptr(scores),
                                 _stream(stream)))


def sv_select_blocks(shape: Shape, scores, nb: int, k: int, sel, kmax: int, stream=None):
    _check(lib().sv_select_blocks(C.byref(shape), _ptr(scores), nb, k, _ptr(sel), kmax,
                                  _stream(stream)))


def sv_score_select(shape: Shape, q, reps, kv: KV, budget: W.Budget, sel, kmax: int, ws,
                    stream=None) -> int:
    b = make_budget(budget)
    k = C.c_int(-1)
    _check(lib().sv_score_select(C.byref(shape), _ptr(q), _ptr(reps), C.byref(kv), C.byref(b),
                                 _ptr(sel), kmax, C.byref(k), _ptr(ws),
                                 0 if ws is None else ws.numel(), _stream(stream)))
    return k.value


def sv_sparse_attend(shape: Shape, q, kv: KV, sel, n_sel: int, sel_stride: int, draft_k, draft_v,
                     parents, out, ws, stream=None):
    _check(lib().sv_sparse_attend(C.byref(shape), _ptr(q), C.byref(kv), _ptr(sel), n_sel,
                                  sel_stride, _ptr(draft_k), _ptr(draft_v), _parents(parents),
                                  _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(),
                                  _stream(stream)))


def sv_sparse_attend_noalloc(shape: Shape, q, kv: KV, sel, n_sel: int, sel_stride: int, draft_k,
                             draft_v, parents, out, flags_out=None, stream=None):
    """sv_sparse_attend with the library's static scratch instead of a
    workspace, for callers that cannot allocate device memory. flags_out: an
    optional device uint32/int32 tensor of one element that receives the
    call's status flags. Calls whose GPU work overlaps race on the scratch."""
    _check(lib().sv_sparse_attend_noalloc(C.byref(shape), _ptr(q), C.byref(kv), _ptr(sel), n_sel,
                                          sel_stride, _ptr(draft_k), _ptr(draft_v),
                                          _parents(parents), _ptr(out), _ptr(flags_out),
                                          _stream(stream)))


def sv_append_kv(shape: Shape, k_pool, v_pool, block_table, seq_ctx, n_accept, accept_idx,
                 draft_k, draft_v, reps=None, ws=None, stream=None):
    """Append each sequence's accepted drafts to its paged cache (and rebuild
    the representatives of blocks that fill). seq_ctx, n_accept: device int32
    [B]; accept_idx: device int32 [B, T]."""
    _check(lib().sv_append_kv(C.byref(shape), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                              block_table.shape[1], k_pool.shape[0], _ptr(seq_ctx),
                              _ptr(n_accept), _ptr(accept_idx), _ptr(draft_k), _ptr(draft_v),
                              _ptr(reps), _ptr(ws), _stream(stream)))


def sv_selection_overlap(sels, k: int, parents, overlap0, by_distance, stream=None):
    """Overlaps of T per-draft selections. sels: device int32 [T, pairs, kmax]
    (each row ascending in its first k entries); overlap0, by_distance:
    device float32 [pairs, T], written."""
    T, pairs, kmax = sels.shape
    _check(lib().sv_selection_overlap(_ptr(sels), T, pairs, kmax, k, _parents(parents),
                                      _ptr(overlap0), _ptr(by_distance), _stream(stream)))


def sv_attend_plan(shape: Shape, kv: KV, n_sel: int) -> Plan:
    p = Plan()
    _check(lib().sv_attend_plan(C.byref(shape), C.byref(kv), n_sel, C.byref(p)))
    return p


def sv_verify_layer(shape: Shape, q, kv: KV, reps, budget: Optional[W.Budget], draft_k, draft_v,
                    parents, reuse: int, slot: Optional[SelSlot], out, ws, stream=None) -> int:
    b = None if budget is None else C.byref(make_budget(budget))
    k = C.c_int(-1)
    _check(lib().sv_verify_layer(C.byref(shape), _ptr(q), C.byref(kv), _ptr(reps), b,
                                 _ptr(draft_k), _ptr(draft_v), _parents(parents), int(reuse),
                                 None if slot is None else C.byref(slot.c), C.byref(k), _ptr(out),
                                 _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return k.value


def sv_verify_layer_host(shape: Shape, q_host, q, kv: KV, reps, budget: Optional[W.Budget],
                         dk_host, dv_host, draft_k, draft_v, parents, reuse: int,
                         slot: Optional[SelSlot], out_host, out, ws, stream=None,
                         copy_in_stream=None, copy_out_stream=None) -> int:
    """sv_verify_layer with q, draft K/V and the output in host memory
    (pinned tensors for asynchronous copies); q, draft_k, draft_v and out are
    the device buffers the call stages them through."""
    b = None if budget is None else C.byref(make_budget(budget))
    k = C.c_int(-1)
    ci = None if copy_in_stream is None else _stream(copy_in_stream)
    co = None if copy_out_stream is None else _stream(copy_out_stream)
    _check(lib().sv_verify_layer_host(
        C.byref(shape), _ptr(q_host), _ptr(q), C.byref(kv), _ptr(reps), b, _ptr(dk_host),
        _ptr(dv_host), _ptr(draft_k), _ptr(draft_v), _parents(parents), int(reuse),
        None if slot is None else C.byref(slot.c), C.byref(k), _ptr(out_host), _ptr(out), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream), ci, co))
    return k.value


VERIFY_COMPUTE, VERIFY_REUSE, VERIFY_FULL = 0, 1, 2  # sv_verify_layer's reuse values


class VerifySchedule:
    """Which sv_verify_layer mode a (step, layer) runs: every `full_period`-th
    step is a full verification over every block (the periodic full steps that
    partial verification interleaves; 0 = never); in the other steps layer l
    recomputes its selection when l % compute_every == 0 and reuses the last
    one otherwise."""

    def __init__(self, full_period: int = 0, compute_every: int = 1):
        if full_period < 0 or compute_every < 1:
            raise ValueError("full_period >= 0 and compute_every >= 1")
        self.full_period = full_period
        self.compute_every = compute_every

    def mode(self, step: int, layer: int = 0) -> int:
        if self.full_period and step % self.full_period == self.full_period - 1:
            return VERIFY_FULL
        return VERIFY_COMPUTE if layer % self.compute_every == 0 else VERIFY_REUSE
class LayerState:
    """Device-resident state of one verification layer: the paged KV cache,
    its block representatives, a selection cache slot and a workspace.

    Built from workloads.LayerInputs already on the device. Only allocation
    and marshalling happen here; the computation is the library's.
    """

    def __init__(self, wl: W.Workload, x: W.LayerInputs, kmax: Optional[int] = None,
                 build_reps: bool = True, stream=None, seq_ctx: Optional[Sequence[int]] = None):
        """seq_ctx: one prefix length per sequence (each at most wl.ctx, the
        length the block table is laid out for); wl.ctx for all when None."""
        self.wl, self.x = wl, x
        self.shape = make_shape(wl.B, wl.Hq, wl.Hkv, wl.d, wl.blk, wl.T, wl.torch_dtype)
        self.kv = make_kv(x.k_pool, x.v_pool, x.block_table, wl.ctx, seq_ctx)
        nb = wl.NB
        ctxs = [wl.ctx] if seq_ctx is None else list(seq_ctx)
        # the largest per-sequence budget: the selection rows' valid prefix
        self.k = max(sv_budget_blocks(wl.budget, c, c // wl.blk) for c in ctxs) if ctxs else 0
        self.kmax = self.k if kmax is None else kmax
        dev = x.q.device
        # [B, Hkv, nb_max, d]: the calls index representatives with the block
        # table's width as stride (a partial last block gets a row, unused)
        nb_max = max(x.block_table.shape[1], 1)
        self.reps = torch.zeros(wl.B, wl.Hkv, nb_max, wl.d, dtype=torch.float32, device=dev)
        self.slot = SelSlot(wl.B, wl.Hkv, self.kmax, device=dev)
        self.out = torch.empty_like(x.q)
        # sized for the budgeted selection and for a dense (all-block) pass
        # sized for the block table's width (nb_max), as the calls check it
        self.ws = alloc_workspace(self.shape, nb_max, max(self.kmax, nb, 1), device=dev)
        self.parents = None if wl.parents is None else list(wl.parents)
        if build_reps and nb:
            sv_build_reps(self.shape, self.kv, 0, nb, self.reps, stream)

    @property
    def sel(self) -> torch.Tensor:
        """The layer's selection (its slot's device tensor)."""
        return self.slot.tensor

    def verify(self, reuse: int = 0, sel_from: Optional["LayerState"] = None, stream=None):
        """One sv_verify_layer call; sel_from shares that layer's selection
        slot (inter-layer reuse)."""
        if sel_from is not None:
            self.slot = sel_from.slot
        sv_verify_layer(self.shape, self.x.q, self.kv, self.reps, self.wl.budget, self.x.draft_k,
                        self.x.draft_v, self.parents, reuse, self.slot, self.out, self.ws, stream)
        return self.out
