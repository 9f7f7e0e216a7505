"""The one exchange step of the scaled FP8 linear when a tensor is sharded.

"Mixed Precision LLM Training: The Complete Guide", section "FP8 with FSDP,
TP, and pipeline parallelism" > "FP8 + tensor parallelism (TP)": the
per-tensor scale of a weight split across tensor-parallel ranks must be the
same on every rank, computed from the global max over all ranks.  amax is a
max of magnitudes, so reducing the per-rank amaxes with MAX gives exactly the
amax of the whole tensor, independent of the order of the reduction.

Usage with the C-ABI calls (delayed scaling): fp8_quantize(..., amax_out=a)
on each rank's shard -> sync_amax(a) -> fp8_update_scale(a, ...).  Data-
parallel replicas need no exchange: each keeps its own scaling state.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def sync_amax(amax: torch.Tensor, group=None) -> torch.Tensor:
    """In-place all-reduce (MAX) of an amax tensor across `group`."""
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def max_over_ranks(value: float, device=None, group=None) -> float:
    """Largest `value` over the ranks of `group` (step-time reduction)."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
