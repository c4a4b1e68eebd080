"""Data-parallel replicas of the layer: each rank routes its own tokens with
identical weights and bias; the one exchange is the sum of the per-expert
loads before the bias update (the batch-wise load of the method counts all
tokens of the step: qwbw.cn essay on the report, "统计整批样本各个专家的负载情况").
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def allreduce_loads(load: torch.Tensor, group=None) -> int:
    """Sums the int32 per-expert loads over the ranks of `group` in place and
    returns the number of ranks (the global batch is world * local T).

    Raises ValueError, on every rank, if the ranks disagree on the number of
    experts, so no replica applies a bias update built from mismatched loads."""
    E = load.numel()
    probe = torch.tensor([E, -E], dtype=torch.int64, device=load.device)
    dist.all_reduce(probe, op=dist.ReduceOp.MAX, group=group)
    if int(probe[0]) != E or int(-probe[1]) != E:
        raise ValueError(f"ranks disagree on the number of experts "
                         f"({int(-probe[1])}..{int(probe[0])}, this rank {E})")
    dist.all_reduce(load, op=dist.ReduceOp.SUM, group=group)
    return dist.get_world_size(group)
