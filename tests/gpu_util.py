"""Shared helpers for the GPU parity tests (CUDA path vs CPU oracle)."""
from __future__ import annotations

import torch

from oracle import sva_oracle as O

GAP_REL = 1e-4  # boundary-gap exemption for selection parity
BF16_ATOL = 1e-2  # max-abs on bf16 outputs (fp32 accumulate, unit-scale V)
F32_ATOL = 1e-4   # fp32 path: fp32 accumulate + fast exp2, far below this


def out_atol(dtype: torch.dtype) -> float:
    return BF16_ATOL if dtype == torch.bfloat16 else F32_ATOL


def band(scores_row, k: int, rel: float = GAP_REL) -> set:
    """Blocks whose oracle score lies within `rel` of the k-th or (k+1)-th
    highest score: either choice is correct for them when the boundary gap is
    below `rel`."""
    vals = sorted((float(x) for x in scores_row), reverse=True)
    if k <= 0 or k >= len(vals):
        return set()
    a, b = vals[k - 1], vals[k]
    if (a - b) / max(abs(a), 1e-30) >= rel:
        return set()
    ta, tb = rel * max(abs(a), 1e-30), rel * max(abs(b), 1e-30)
    return {j for j, s in enumerate(scores_row) if abs(s - a) <= ta or abs(s - b) <= tb}


def compare_selection(gpu_sel: torch.Tensor, oracle_scores: torch.Tensor, k: int):
    """Assert the GPU selection equals the oracle's, bit-exactly except for
    blocks inside a boundary band. Returns the set of (b, h) whose selection
    differed inside the band (their outputs are then compared elsewhere)."""
    B, H, NB = oracle_scores.shape
    differ = set()
    for b in range(B):
        for h in range(H):
            row = oracle_scores[b, h].tolist()
            want = O.select_blocks(row, k)
            got = [int(x) for x in gpu_sel[b, h, :k].tolist()]
            assert all(int(x) == -1 for x in gpu_sel[b, h, k:].tolist()), (b, h)
            assert got == sorted(got) and len(set(got)) == len(got), (b, h, got)
            if got == want:
                continue
            free = band(row, k)
            assert free, f"selection differs at (b={b}, h={h}) with a clear boundary gap"
            assert [j for j in got if j not in free] == [j for j in want if j not in free], (b, h)
            assert len(got) == len(want)
            differ.add((b, h))
    return differ


def check_topk_property(sel: torch.Tensor, scores: torch.Tensor, k: int):
    """The kept set is exactly the top-k of `scores` (as compared in their own
    precision), ties to the lower index, listed ascending."""
    B, H, NB = scores.shape
    kk = min(k, NB)
    for b in range(B):
        for h in range(H):
            s = scores[b, h].tolist()
            s = [0.0 if x == 0.0 else x for x in s]
            got = [int(x) for x in sel[b, h, :kk].tolist()]
            assert got == sorted(got) and len(set(got)) == kk
            gs = set(got)
            worst_in = min(((s[j], -j) for j in got), default=None)
            best_out = max(((s[j], -j) for j in range(NB) if j not in gs), default=None)
            if worst_in is not None and best_out is not None:
                assert worst_in > best_out, (b, h, worst_in, best_out)


def compare_out(gpu_out: torch.Tensor, ref: torch.Tensor, atol: float, skip_pairs=(), G=1):
    """Max-abs comparison of [B, T, Hq, d] outputs, skipping (b, kv head)
    pairs listed in skip_pairs. Returns the max abs error seen."""
    g = gpu_out.double().cpu()
    mask = torch.ones(g.shape[0], g.shape[2], dtype=torch.bool)
    for (b, h) in skip_pairs:
        mask[b, h * G:(h + 1) * G] = False
    err = (g - ref).abs().amax(dim=(1, 3))  # [B, Hq]
    worst = float(err[mask].max()) if mask.any() else 0.0
    assert worst <= atol, f"max abs err {worst} > {atol}"
    return worst
