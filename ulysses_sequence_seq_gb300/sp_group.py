"""Loss of a sequence-parallel group: gather every rank's (loss, good tokens) and take
the good-token weighted mean on the device (``usp_sp_weighted_loss``).

jianying88 article on DeepSpeed Ulysses in Transformers, section
"3. 跨 rank 的加权 loss 聚合": each SP rank computes its loss over its own shard; the
ranks' losses and their counts of tokens whose shifted label is not -100 are
all-gathered over the SP group, and the group's loss is their weighted mean, leaving out
ranks without good tokens (a shard made only of prompt tokens).
"""
from __future__ import annotations

from ._lib import sp_weighted_loss


def gather_loss_and_good(loss, good_tokens, group=None):
    """All-gather this rank's scalar loss and good-token count over ``group``.

    One collective of a float64 pair per rank (counts stay exact below 2^53). Returns
    (float32[sp], int64[sp]) on the device of ``loss``, ordered by rank in the group.
    """
    import torch
    import torch.distributed as dist
    sp = dist.get_world_size(group)
    mine = torch.stack([loss.detach().reshape(()).to(torch.float64),
                        good_tokens.detach().reshape(()).to(torch.float64)])
    parts = [torch.empty_like(mine) for _ in range(sp)]
    dist.all_gather(parts, mine, group=group)
    both = torch.stack(parts)
    return both[:, 0].to(torch.float32).contiguous(), both[:, 1].to(torch.int64).contiguous()


def sp_group_loss(loss, good_tokens, group=None, out=None, stream=None):
    """The SP group's loss (a float32 device scalar): the gathered ranks' losses weighted
    by their good-token counts, ranks with none left out, 0 if no rank has any."""
    import torch
    losses, goods = gather_loss_and_good(loss, good_tokens, group)
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=losses.device)
    sp_weighted_loss(losses, goods, losses.numel(), out, stream)
    return out
