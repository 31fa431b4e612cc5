"""Seeded synthetic workloads for sparse verification attention.

This module only *makes inputs*. It holds none of the method's arithmetic
(no representatives, scores, budgets, selection or attention); both the CUDA
path and the CPU oracle consume what it produces.

The shapes follow the models that "Accelerate Speculative Decoding with Sparse
Computation in Verification" evaluates on (tutorial page, section on the
experiments: Llama3.1-8B and Qwen3-30B-MoE) at 32K-128K contexts. The pages'
datasets are not available, so seeded Gaussian tensors with planted
high-affinity blocks stand in for real activations.

Recipe (per layer):
  * Q [B,T,Hq,d], K/V pools [P,Hkv,blk,d], draft K/V [B,T,Hkv,d] ~ N(0,1),
    drawn directly in the workload dtype from one seeded torch.Generator.
  * block_table[b, j] = physical page of logical block j (identity, or a seeded
    random permutation of all pages).
  * qbar0[b,h] = mean over the G query heads of group h of draft 0's query.
  * planted block j of (b,h): every key of that block += alpha * qbar0[b,h]
    (computed in fp32, rounded once to the workload dtype); the sink (block 0)
    gets sink_alpha instead.
  * multi-layer stacks: layer l uses seed + l; adjacent layers share at least
    n_planted - drift planted blocks (drift fresh indices replace old ones).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import torch

# Budget modes, mirrored from the C header (values are part of the ABI).
BUDGET_FIXED = 0
BUDGET_PIECEWISE = 1
BUDGET_SMOOTH = 2

# A 16-node draft tree: root -> 2 children -> 4 grandchildren -> chains, with
# node 15 a second child of node 3; maximum depth 4. Topology is plain data.
TREE16_PARENTS = (-1, 0, 0, 1, 1, 2, 2, 3, 4, 5, 6, 7, 8, 9, 10, 3)


@dataclass(frozen=True)
class Budget:
    mode: int = BUDGET_PIECEWISE
    fixed_blocks: int = 0
    short_ctx: int = 4096
    floor_blocks: int = 64
    frac_mid: float = 0.125
    long_ctx: int = 32768
    frac_long: float = 0.0625


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    blk: int
    ctx: int
    T: int
    dtype: str  # "bf16" or "f32"
    budget: Budget
    seed: int
    parents: Optional[Sequence[int]] = None  # None = linear chain
    n_planted: int = 16
    alpha: float = 0.5
    sink_alpha: Optional[float] = 1.0
    permute_pages: bool = False
    layers: int = 1
    compute_every: int = 1  # selection recomputed on layers l % compute_every == 0
    drift: int = 0
    description: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def NB(self) -> int:
        """Full blocks of the context (the candidates for selection)."""
        return self.ctx // self.blk

    @property
    def NBT(self) -> int:
        """Blocks holding the context, a partial last block included."""
        return (self.ctx + self.blk - 1) // self.blk

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elt(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def parent_list(self) -> list[int]:
        if self.parents is None:
            return [t - 1 for t in range(self.T)]
        return list(self.parents)


PIECEWISE_6P25_ABOVE_32K = Budget(BUDGET_PIECEWISE, 0, 4096, 64, 0.125, 32768, 0.0625)
PIECEWISE_12P5 = Budget(BUDGET_PIECEWISE, 0, 4096, 64, 0.125, 32768, 0.125)

WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", B=1, Hq=4, Hkv=2, d=64, blk=16, ctx=1024, T=4, dtype="f32",
        budget=Budget(BUDGET_FIXED, 8, 0, 0, 0.0, 0, 0.0), seed=0,
        n_planted=4, alpha=0.5, sink_alpha=None,
        description="tiny single layer, fp32, 4/2 heads, d64, ctx 1024 (64 blocks of 16), "
                    "T=4 chain, fixed budget 8, 4 planted blocks"),
    "llama8b_32k": Workload(
        "llama8b_32k", B=1, Hq=32, Hkv=8, d=128, blk=64, ctx=32768, T=8, dtype="bf16",
        budget=PIECEWISE_6P25_ABOVE_32K, seed=2,
        description="Llama-3.1-8B-shaped layer, bf16, B1, 32/8 heads, d128, ctx 32768 "
                    "(512 blocks of 64), T=8 chain"),
    "llama8b_128k_b4": Workload(
        "llama8b_128k_b4", B=4, Hq=32, Hkv=8, d=128, blk=64, ctx=131072, T=8, dtype="bf16",
        budget=PIECEWISE_6P25_ABOVE_32K, seed=3, permute_pages=True,
        description="Llama-3.1-8B-shaped layer, bf16, B4, 32/8 heads, d128, ctx 131072 "
                    "(2048 blocks of 64), T=8 chain, randomly permuted pages"),
    "qwen3moe_64k_b8_tree16": Workload(
        "qwen3moe_64k_b8_tree16", B=8, Hq=32, Hkv=4, d=128, blk=64, ctx=65536, T=16,
        dtype="bf16", budget=PIECEWISE_12P5, seed=4, parents=TREE16_PARENTS,
        description="Qwen3-30B-MoE-shaped attention, bf16, B8, 32/4 heads (G8), d128, "
                    "ctx 65536 (1024 blocks of 64), 16-node draft tree"),
    "llama8b_60k_32layer": Workload(
        "llama8b_60k_32layer", B=1, Hq=32, Hkv=8, d=128, blk=64, ctx=61440, T=8,
        dtype="bf16", budget=PIECEWISE_12P5, seed=5, layers=32, compute_every=2, drift=4,
        description="32-layer Llama-3.1-8B-shaped attention stack, bf16, B1, 32/8 heads, "
                    "d128, ctx 61440 (960 blocks of 64), T=8 chain, selection recomputed "
                    "every 2nd layer and reused by the next"),
}


def scaled(wl: Workload, **kw) -> Workload:
    """Same workload structure at other sizes (for oracle-sized parity cases)."""
    return replace(wl, **kw)


@dataclass
class LayerInputs:
    q: torch.Tensor            # [B, T, Hq, d]
    k_pool: torch.Tensor       # [P, Hkv, blk, d]
    v_pool: torch.Tensor       # [P, Hkv, blk, d]
    block_table: torch.Tensor  # [B, NB] int32
    draft_k: torch.Tensor      # [B, T, Hkv, d]
    draft_v: torch.Tensor      # [B, T, Hkv, d]
    planted: torch.Tensor      # [B, Hkv, n_planted] int64 (logical block indices)
    parents: list = field(default_factory=list)

    def to(self, device) -> "LayerInputs":
        return LayerInputs(*(getattr(self, n).to(device) for n in
                             ("q", "k_pool", "v_pool", "block_table", "draft_k",
                              "draft_v", "planted")), parents=list(self.parents))


def planted_sets(wl: Workload) -> list[torch.Tensor]:
    """Planted logical block indices per layer, [B, Hkv, n_planted] each.

    Layer 0 draws n_planted distinct blocks from [1, NB) per (b, h); each later
    layer keeps all but at most `drift` of the previous layer's blocks.
    """
    NB = wl.NB
    n = min(wl.n_planted, max(NB - 1, 0))
    g = torch.Generator().manual_seed(10_000 + wl.seed)
    out = []
    cur = torch.empty(wl.B, wl.Hkv, n, dtype=torch.int64)
    for b in range(wl.B):
        for h in range(wl.Hkv):
            if n:
                cur[b, h] = 1 + torch.randperm(NB - 1, generator=g)[:n]
    out.append(cur.clone())
    for _ in range(1, wl.layers):
        nxt = cur.clone()
        if wl.drift and n:
            for b in range(wl.B):
                for h in range(wl.Hkv):
                    r = int(torch.randint(0, wl.drift + 1, (1,), generator=g))
                    if r == 0:
                        continue
                    pos = torch.randperm(n, generator=g)[:r]
                    taken = set(nxt[b, h].tolist())
                    free = [j for j in range(1, NB) if j not in taken]
                    pick = torch.randperm(len(free), generator=g)[:r]
                    for p, f in zip(pos.tolist(), pick.tolist()):
                        nxt[b, h, p] = free[f]
        out.append(nxt.clone())
        cur = nxt
    return out


def make_layer(wl: Workload, layer: int = 0, device="cpu",
               planted: Optional[torch.Tensor] = None) -> LayerInputs:
    """Generate one layer's inputs, deterministic for (workload, layer, device)."""
    if planted is None:
        planted = planted_sets(wl)[layer] if wl.layers > 1 else planted_sets(wl)[0]
    dt = wl.torch_dtype
    NB, NBT = wl.NB, wl.NBT
    P = wl.B * NBT
    g = torch.Generator(device=device).manual_seed(wl.seed + layer)
    q = torch.randn(wl.B, wl.T, wl.Hq, wl.d, generator=g, device=device, dtype=dt)
    k_pool = torch.randn(P, wl.Hkv, wl.blk, wl.d, generator=g, device=device, dtype=dt)
    v_pool = torch.randn(P, wl.Hkv, wl.blk, wl.d, generator=g, device=device, dtype=dt)
    draft_k = torch.randn(wl.B, wl.T, wl.Hkv, wl.d, generator=g, device=device, dtype=dt)
    draft_v = torch.randn(wl.B, wl.T, wl.Hkv, wl.d, generator=g, device=device, dtype=dt)
    if wl.permute_pages and P > 0:
        perm = torch.randperm(P, generator=g, device=device)
    else:
        perm = torch.arange(P, device=device)
    block_table = perm.view(wl.B, NBT).to(torch.int32).contiguous()

    if NB > 0:
        qbar0 = q[:, 0].float().view(wl.B, wl.Hkv, wl.G, wl.d).mean(dim=2)  # [B,Hkv,d]
        planted_d = planted.to(device)
        for b in range(wl.B):
            bt = block_table[b].long()
            for h in range(wl.Hkv):
                shift = qbar0[b, h]
                if planted_d.shape[-1]:
                    pages = bt[planted_d[b, h]]
                    blocks = k_pool[pages, h].float() + wl.alpha * shift
                    k_pool[pages, h] = blocks.to(dt)
                if wl.sink_alpha is not None:
                    p0 = bt[0]
                    k_pool[p0, h] = (k_pool[p0, h].float() + wl.sink_alpha * shift).to(dt)
    return LayerInputs(q, k_pool, v_pool, block_table, draft_k, draft_v, planted,
                       parents=wl.parent_list())
