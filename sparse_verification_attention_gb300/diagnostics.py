"""The shared-set diagnostic, on the device.

"Accelerate Speculative Decoding with Sparse Computation in Verification"
(paper summary page, Figure 1 caption and the figure after it): every draft
token attends to the block set chosen with the first draft's query, on the
observation that the drafts' own choices overlap heavily. This tool measures
that overlap for a given input: for each draft t it scores the blocks with
draft t's own query and keeps its top-k (the library's scoring and
selection calls), then reports |S_t ∩ S_0| / k per (sequence, kv head,
draft). Low overlap at large t says the shared set is a poor fit for that
workload.
"""
from __future__ import annotations

import torch

from . import api


def draft_selection_overlap(shape: api.Shape, q: torch.Tensor, reps: torch.Tensor, kv: api.KV,
                            k: int, stream=None) -> torch.Tensor:
    """overlap[b, h, t] (float64, host) for q [B,T,Hq,d] and reps
    [B,Hkv,nb_max,d] on the device."""
    B, T, Hq, d = q.shape
    Hkv = shape.Hkv
    nb = kv.ctx // shape.blk
    kk = min(k, nb)
    if kk == 0:
        return torch.ones(B, Hkv, T, dtype=torch.float64)
    one = api.make_shape(B, Hq, Hkv, d, shape.blk, 1, q.dtype)
    scores = torch.empty(B, Hkv, nb, dtype=torch.float32, device=q.device)
    sels = []
    for t in range(T):
        q_t = q[:, t:t + 1].contiguous()  # draft t's query in slot 0 of a T = 1 batch
        api.sv_score_blocks(one, q_t, reps, kv, scores, stream)
        sel = torch.empty(B, Hkv, kk, dtype=torch.int32, device=q.device)
        api.sv_select_blocks(one, scores, nb, kk, sel, kk, stream)
        sels.append(sel)
    torch.cuda.synchronize()
    s0 = sels[0].cpu()
    out = torch.empty(B, Hkv, T, dtype=torch.float64)
    for t in range(T):
        st = sels[t].cpu()
        for b in range(B):
            for h in range(Hkv):
                out[b, h, t] = len(set(s0[b, h].tolist()) & set(st[b, h].tolist())) / kk
    return out
