"""Data-parallel reduction of the chain loss across ranks.

Each rank runs ``mtp_chain_loss`` on its own packed rows and obtains per-term
(loss sum, supervised-row count) pairs.  The global loss is assembled from the
*reduced* numerators and denominators -- never from per-rank normalised losses
-- as "M7.6 - DeepSeek MTP" §0x06A prescribes for distributed training.  This
module only moves those 2(D+1) fp64 values between ranks; the assembly itself
runs in the library (``lib.loss_assemble``)."""
from __future__ import annotations

import torch
import torch.distributed as dist


def allreduce_sums_counts(sums_counts: torch.Tensor, group=None) -> torch.Tensor:
    """In-place SUM all-reduce of a [2*(D+1)] fp64 (sum, count) tensor."""
    if sums_counts.dtype != torch.float64:
        raise TypeError("sums_counts must be float64")
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(sums_counts, op=dist.ReduceOp.SUM, group=group)
    return sums_counts


def global_positions(B: int, T: int, group=None) -> int:
    """B*T summed over ranks: the fixed-denominator policy's global B*T."""
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    return world * B * T


def deepseek_v3_lambda(tokens_seen: float) -> float:
    """MTP loss weight of the DeepSeek-V3 schedule ("M7.6 - DeepSeek MTP"
    §0x05): 0.3 for the first 10T training tokens, 0.1 afterwards."""
    return 0.3 if tokens_seen < 10e12 else 0.1
