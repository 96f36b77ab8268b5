"""The exchange over a real process group, on CPU ranks (gloo, world size 2 and 4).

Each rank holds its shard of one seeded global tensor and runs SPExchange: the
collective (all_to_all_single on raw bytes) and its host-side bookkeeping -- which block
goes to which rank, chunking of the heads, the asynchronous handles, replicated
key/value heads -- are the library's; the rank-local pack/unpack steps, which are CUDA
kernels in the library (checked against the same oracle functions on the GPU), are
replaced here by the oracle's index formulas. The results are compared bit for bit with
the oracle's single-buffer layout swap.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import relayout


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _from_bits(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def oracle_pack(x, out, sp, head0, nheads):
    out.copy_(_from_bits(relayout.a2a_pack(_bits(x), sp, head0, nheads), x.dtype))


def oracle_unpack(recv, out, sp, head0, nheads):
    if out.dtype == torch.float32:    # replicas' gradients: summed (float64 in the oracle)
        got = relayout.a2a_unpack(recv.numpy(), sp, out.shape[1], head0, nheads)
        out.copy_(torch.from_numpy(got).to(torch.float32))
    else:
        cur = _bits(out).copy()
        relayout.a2a_unpack(_bits(recv), sp, out.shape[1], head0, nheads, out=cur)
        out.copy_(_from_bits(cur, out.dtype))


def _global(T, H, D, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=(T, H, D), dtype=np.uint32).astype(np.uint16)


def _worker(rank, world, port, out):
    from ulysses_sequence_seq_gb300.sp_exchange import SPExchange
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ex = SPExchange(pack=oracle_pack, unpack=oracle_unpack)
        T, H, D = 8 * world, 2 * world, 8
        S, Hl = T // world, H // world
        xg = _global(T, H, D, 5)
        x = _from_bits(xg[rank * S:(rank + 1) * S], torch.bfloat16)
        want = np.ascontiguousarray(relayout.seq_to_head(xg.reshape(world, S, H, D), world)[rank].transpose(1, 0, 2))
        res = {}
        heads = ex.to_heads(x)
        res["to_heads"] = np.array_equal(_bits(heads), want)
        parts = [ex.to_heads(x, c, 1, async_op=True) for c in range(Hl)]
        res["to_heads_chunks"] = np.array_equal(np.concatenate([_bits(p.wait()) for p in parts], axis=1), want)
        back = torch.zeros(S, H, D, dtype=torch.bfloat16)
        ex.to_seq(heads, back)
        res["round_trip"] = np.array_equal(_bits(back), xg[rank * S:(rank + 1) * S])
        back2 = torch.zeros(S, H, D, dtype=torch.bfloat16)
        pend = [ex.to_seq(heads[:, c:c + 1].contiguous(), back2, c, 1, async_op=True) for c in range(Hl)]
        for p in pend:
            p.wait()
        res["round_trip_chunks"] = np.array_equal(_bits(back2), xg[rank * S:(rank + 1) * S])
        if world >= 4:
            # two key/value heads over four ranks: each rank receives the head its query
            # heads read, and the gradients of the replicas are summed on the way back
            hkv = 2
            kg = _global(T, hkv, D, 6)
            k = _from_bits(kg[rank * S:(rank + 1) * S], torch.bfloat16)
            kh = ex.to_heads(k)
            res["kv_replica"] = np.array_equal(_bits(kh)[:, 0], kg[:, rank * hkv // world])
            rng = np.random.default_rng(7)
            grads = rng.standard_normal((world, T, 1, D)).astype(np.float32)
            dk = torch.zeros(S, hkv, D, dtype=torch.float32)
            ex.to_seq(torch.from_numpy(grads[rank]), dk)
            ref = relayout.head_to_seq_kv_grad(grads[:, :, 0, :], world, hkv)[rank * S:(rank + 1) * S]
            res["kv_grad_sum"] = bool(np.allclose(dk.numpy(), ref, rtol=0, atol=1e-6))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def _run(world):
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    return dict(out)


def test_exchange_gloo_world2():
    got = _run(2)
    assert set(got) == {0, 1}
    for rank, res in got.items():
        assert res and all(res.values()), (rank, res)


def test_exchange_gloo_world4_with_replicated_kv_heads():
    got = _run(4)
    assert set(got) == {0, 1, 2, 3}
    for rank, res in got.items():
        assert res and all(res.values()) and "kv_grad_sum" in res, (rank, res)
