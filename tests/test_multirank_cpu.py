"""The N > 1 bench path on CPU: gloo, world size 2. Every rank runs its own replica of
the per-GPU step with no data-path collective; the only exchange is the max over
ranks of the timed duration, which rank 0 reports."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(10.0 + 3.5 * rank, dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 13.5, 1: 13.5}


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(4.25) == 4.25


# ------------------------------------------------------- SP loss over a real process group
def _loss_worker(rank, world, port, out):
    """Each rank holds its shard of one packed batch, computes its own loss over its good
    tokens and gathers (loss, good) over the group (the device-side weighted mean is
    covered by the GPU tests; here the oracle takes the gathered values)."""
    import numpy as np

    from oracle import sp_loss
    from ulysses_sequence_seq_gb300.sp_group import gather_loss_and_good
    from ulysses_sequence_seq_gb300.synth import packed_labels, token_losses

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cu = np.array([0, 40, 52, 128], dtype=np.int32)
        lab = packed_labels(cu, vocab=100, seed=21)
        lab[:64] = -100                                  # rank 0's shard: prompt only
        sh = sp_loss.shift_labels(lab, cu)
        tok = token_losses(128, seed=22)
        S = 128 // world
        keep = sh[rank * S:(rank + 1) * S] != -100
        n = int(keep.sum())
        mine = float(tok[rank * S:(rank + 1) * S][keep].astype(np.float64).mean()) if n else float("nan")
        losses, goods = gather_loss_and_good(torch.tensor(mine, dtype=torch.float32), torch.tensor(n))
        out[rank] = (losses.tolist(), goods.tolist(), float(tok[sh != -100].astype(np.float64).mean()))
    finally:
        dist.destroy_process_group()


def test_gather_loss_and_good_gloo_world2():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_loss_worker, args=(world, port, out), nprocs=world, join=True)
    from oracle import sp_loss
    (l0, g0, want), (l1, g1, _) = out[0], out[1]
    assert l0[1:] == l1[1:] and g0 == g1 and g0[0] == 0 and g0[1] > 0
    assert l0[0] != l0[0]                                # rank 0's own loss is NaN (no good token)
    assert abs(sp_loss.sp_weighted_loss(l0, g0) - want) <= 1e-6 * want
