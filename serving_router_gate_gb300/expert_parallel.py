"""Expert parallelism across GPUs: each rank owns a contiguous range of expert
slots and a shard of the shared experts, computes a partial layer output, and
one SUM reduction over the ranks gives the layer output.

Method (vLLM EP-aware FusedMoE override, ep_fused_moe_patch.py):
  * module docstring "EP expert dispatch": top-k routing gives global expert
    ids, identical on every rank; each rank masks the experts outside its range
    (weight 0) and remaps its own to local ids -- moe_permute with a local range
    and MOE_NONLOCAL_SKIP;
  * the patched __init__: E_local = E / ep_size experts per rank, contiguous
    ranges, renormalisation over all k before the mask;
  * ep_reduce_output: the routed partial plus the shared experts' partial (a
    row-parallel shard: each rank holds a slice of their intermediate size),
    then one all-reduce -- DeepSpeed PR #6964 likewise forms the layer's
    reduction once, after the weighted sum of the selected experts' outputs.

Readings taken here: slot ranges split S as evenly as contiguous ranges allow
(rank r owns [r S / N, (r + 1) S / N)), which is E / N when N divides S; the
shared experts' intermediate is split the same way in units of 64 (the
library's row granularity); the reduction runs in fp32 (the pages do not fix
its precision) and the result is rounded to bf16 once.

Every rank calls the same three library calls as a one-GPU layer (moe_route,
moe_permute with its range, moe_forward with its shard); only the reduction is
a collective.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from .layer import MoELayer


def ep_slot_range(S: int, world: int, rank: int) -> Tuple[int, int]:
    """(first slot, slot count) of rank `rank` among `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if world > S:
        raise ValueError(f"{world} ranks for {S} slots")
    lo, hi = rank * S // world, (rank + 1) * S // world
    return lo, hi - lo


def ep_shared_range(I_shared: int, world: int, rank: int, unit: int = 64) -> Tuple[int, int]:
    """(first column, width) of rank `rank`'s slice of the shared experts' intermediate
    size, in whole units of `unit` columns (a rank may get none)."""
    if I_shared % unit:
        raise ValueError(f"shared intermediate {I_shared} is not a multiple of {unit}")
    n = I_shared // unit
    lo, hi = rank * n // world, (rank + 1) * n // world
    return lo * unit, (hi - lo) * unit


def ep_shared_shard(W1s: torch.Tensor, W2s: torch.Tensor, world: int, rank: int):
    """The row-parallel shard of the shared experts (as one concatenated MLP:
    W1s [2 I_sh, H] gate rows then up rows, W2s [H, I_sh]) that rank `rank` holds:
    gate rows [a, a + w), up rows [I_sh + a, I_sh + a + w), W2s columns [a, a + w).
    Returns (W1 shard [2 w, H], W2 shard [H, w]) or (None, None) for w = 0."""
    I_sh = W2s.shape[1]
    a, w = ep_shared_range(I_sh, world, rank)
    if w == 0:
        return None, None
    W1 = torch.cat([W1s[a:a + w], W1s[I_sh + a:I_sh + a + w]], 0).contiguous()
    W2 = W2s[:, a:a + w].contiguous()
    return W1, W2


def ep_reduce_output(partial: torch.Tensor, group=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Sum of the ranks' partial outputs [T, H] (routed + shared on each rank), in fp32,
    rounded once to the partial's dtype: the layer output on every rank."""
    import torch.distributed as dist
    acc = partial.float()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    res = acc.to(partial.dtype)
    if out is not None:
        out.copy_(res)
        return out
    return res


class EPMoELayer:
    """One rank's share of an expert-parallel MoE layer.

    Wg [E, H] (replicated), W1 [S, 2I, H], W2 [S, H, I] (all slots; only this
    rank's range is kept), optional shared experts W1s [2 I_sh, H], W2s [H, I_sh]
    (concatenated; only this rank's shard is kept) and their gate vector; further
    keyword options (routing variant, weight format) go to MoELayer as they are.
    forward(x) returns the full layer output [T, H] after the reduction."""

    def __init__(self, Wg, W1, W2, k, renorm, max_T, world: int, rank: int, logit_bias=None, rep_offset=None,
                 rep_slots=None, W1s=None, W2s=None, shared_gate_w=None, group=None, **layer_options):
        S = W1.shape[0]
        self.world, self.rank, self.group = world, rank, group
        self.start, self.count = ep_slot_range(S, world, rank)
        W1l = W1[self.start:self.start + self.count].contiguous()
        W2l = W2[self.start:self.start + self.count].contiguous()
        W1sh = W2sh = None
        gate = None
        if W1s is not None:
            W1sh, W2sh = ep_shared_shard(W1s, W2s, world, rank)
            gate = shared_gate_w if W1sh is not None else None
        self.layer = MoELayer(Wg, W1l, W2l, k, renorm, max_T, logit_bias=logit_bias, rep_offset=rep_offset,
                              rep_slots=rep_slots, S=S, local_start=self.start, local_count=self.count,
                              W1s=W1sh, W2s=W2sh, shared_gate_w=gate, **layer_options)

    def partial(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        """This rank's partial output (its slots' experts and its shared shard), bf16 [T, H]."""
        return self.layer.forward(x, stream)

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        return ep_reduce_output(self.partial(x, stream), self.group)
