"""The shared-set diagnostic, on the device.

"Accelerate Speculative Decoding with Sparse Computation in Verification"
(paper summary page, Figure 1 caption and the figure after it): every draft
token attends to the block set chosen with the first draft's query, on the
observation that the drafts' own choices overlap heavily, and more so for
drafts at nearby positions. This tool measures that for a given input: for
each draft t it scores the blocks with draft t's own query and keeps its
top-k (the library's scoring and selection calls, written straight into one
[T, pairs, k] tensor), then the library's overlap kernel counts, for every
pair of drafts, how many blocks their sets share:
  * overlap0[b, h, t]: |S_t ∩ S_0| / k, the overlap with the set every draft
    actually uses;
  * by_distance[b, h, delta]: the mean of |S_t ∩ S_u| / k over the draft pairs
    whose positions differ by delta (depth difference in a draft tree; |t - u|
    in a chain), NaN where no pair does.
Low overlap says the shared set is a poor fit for that workload. Python only
allocates tensors and reshapes the results.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import api


def draft_selections(shape: api.Shape, q: torch.Tensor, reps: torch.Tensor, kv: api.KV,
                     k: int, stream=None) -> torch.Tensor:
    """Every draft's own top-k: int32 [T, B*Hkv, kk] on the device (kk =
    min(k, NB)), rows ascending."""
    B, T, Hq, d = q.shape
    Hkv = shape.Hkv
    nb = kv.ctx // shape.blk
    kk = min(k, nb)
    sels = torch.empty(T, B * Hkv, max(kk, 1), dtype=torch.int32, device=q.device)
    if kk == 0:
        return sels[:, :, :0]
    one = api.make_shape(B, Hq, Hkv, d, shape.blk, 1, q.dtype)
    scores = torch.empty(B, Hkv, nb, dtype=torch.float32, device=q.device)
    for t in range(T):
        q_t = q[:, t:t + 1].contiguous()  # draft t's query in slot 0 of a T = 1 batch
        api.sv_score_blocks(one, q_t, reps, kv, scores, stream)
        api.sv_select_blocks(one, scores, nb, kk, sels[t], kk, stream)
    return sels


def selection_overlaps(shape: api.Shape, q: torch.Tensor, reps: torch.Tensor, kv: api.KV, k: int,
                       parents: Optional[Sequence[int]] = None, stream=None):
    """(overlap0 [B, Hkv, T], by_distance [B, Hkv, T]) as float64 host tensors."""
    B, T = q.shape[0], q.shape[1]
    Hkv = shape.Hkv
    sels = draft_selections(shape, q, reps, kv, k, stream)
    kk = sels.shape[-1]
    if kk == 0:
        ones = torch.ones(B, Hkv, T, dtype=torch.float64)
        return ones, ones.clone()
    ov0 = torch.empty(B * Hkv, T, dtype=torch.float32, device=q.device)
    byd = torch.empty(B * Hkv, T, dtype=torch.float32, device=q.device)
    api.sv_selection_overlap(sels, kk, parents, ov0, byd, stream)
    torch.cuda.synchronize()
    return (ov0.view(B, Hkv, T).double().cpu(), byd.view(B, Hkv, T).double().cpu())


def draft_selection_overlap(shape: api.Shape, q: torch.Tensor, reps: torch.Tensor, kv: api.KV,
                            k: int, stream=None) -> torch.Tensor:
    """overlap[b, h, t] = |S_t ∩ S_0| / k (float64, host)."""
    return selection_overlaps(shape, q, reps, kv, k, None, stream)[0]


def draft_overlap_by_distance(shape: api.Shape, q: torch.Tensor, reps: torch.Tensor, kv: api.KV,
                              k: int, parents: Optional[Sequence[int]] = None,
                              stream=None) -> torch.Tensor:
    """by_distance[b, h, delta] (float64, host; NaN where no draft pair is
    delta apart)."""
    return selection_overlaps(shape, q, reps, kv, k, parents, stream)[1]
