"""Layout swap of Ulysses sequence parallelism, written as its index formula.

TEST INFRASTRUCTURE ONLY.

Before attention every rank holds a contiguous chunk of S = T/sp tokens with
all H heads; after the first all-to-all it holds all T tokens for H/sp heads,
and the second all-to-all undoes that (HF Transformers "Ulysses sequence
parallelism" guide, opening paragraph and its layout figure; congresoia365
article, "Cómo Funciona Ulysses", steps 1, 3 and 5). With the sp simulated
ranks stored as shards of one buffer:

    seq-sharded  x[r_s][s][h][d]     token t = r_s*S + s, all heads
    head-sharded y[r][hl][t][d]      head  h = r*Hl + hl, all tokens

    y[r][hl][t][d] = x[t // S][t % S][r*Hl + hl][d]

Arrays hold raw 16-bit patterns: the swap moves bits and never does arithmetic
on them.
"""
from __future__ import annotations

import numpy as np


def _check(T: int, H: int, sp: int):
    if sp <= 0 or T % sp != 0:
        raise ValueError("total tokens must be a multiple of sp_size")
    if H % sp != 0:
        raise ValueError("head count must be divisible by sp_size")


def seq_to_head(x: np.ndarray, sp: int) -> np.ndarray:
    """x: [sp][S][H][D] (or [T][H][D]) -> y: [sp][H/sp][T][D]."""
    H, D = x.shape[-2], x.shape[-1]
    T = x.size // (H * D)
    _check(T, H, sp)
    S, Hl = T // sp, H // sp
    xs = x.reshape(sp, S, H, D)
    y = np.empty((sp, Hl, T, D), dtype=x.dtype)
    t = np.arange(T)
    for r in range(sp):
        for hl in range(Hl):
            y[r, hl, t, :] = xs[t // S, t % S, r * Hl + hl, :]
    return y


def head_to_seq(y: np.ndarray, sp: int) -> np.ndarray:
    """y: [sp][H/sp][T][D] (or [H][T][D]) -> x: [sp][S][H][D]."""
    T, D = y.shape[-2], y.shape[-1]
    H = y.size // (T * D)
    _check(T, H, sp)
    S, Hl = T // sp, H // sp
    ys = y.reshape(sp, Hl, T, D)
    x = np.empty((sp, S, H, D), dtype=y.dtype)
    t = np.arange(T)
    for r in range(sp):
        for hl in range(Hl):
            x[t // S, t % S, r * Hl + hl, :] = ys[r, hl, t, :]
    return x


def seq_to_head_elem(x: np.ndarray, sp: int, r: int, hl: int, t: int, d: int):
    """One element of the head-sharded view, straight from the formula (for sampled checks)."""
    H, D = x.shape[-2], x.shape[-1]
    T = x.size // (H * D)
    S, Hl = T // sp, H // sp
    return x.reshape(sp, S, H, D)[t // S, t % S, r * Hl + hl, d]


def kv_replication(sp: int, hkv: int) -> int:
    """Ranks sharing one key/value head: 1 when the heads split over the ranks, sp / hkv
    when there are fewer heads than ranks (each rank then needs the head its query heads
    read: query head h of rank r reads kv head h // (hq / hkv), which for every h of rank
    r is r * hkv // sp)."""
    if hkv % sp == 0:
        return 1
    if sp % hkv == 0:
        return sp // hkv
    raise ValueError("key/value heads must divide over sp_size or divide it")


def seq_to_head_kv(x: np.ndarray, sp: int) -> np.ndarray:
    """[T][hkv][D] bits -> [max(sp, hkv)][T][D]: rank r's heads; with fewer heads than
    ranks, out[r] = x[:, r * hkv // sp]."""
    T, hkv, D = x.shape
    rep = kv_replication(sp, hkv)
    if rep == 1:
        return np.ascontiguousarray(x.transpose(1, 0, 2))
    out = np.empty((sp, T, D), dtype=x.dtype)
    for r in range(sp):
        out[r] = x[:, r * hkv // sp, :]
    return out


def head_to_seq_kv_grad(y: np.ndarray, sp: int, hkv: int) -> np.ndarray:
    """[max(sp, hkv)][T][D] float gradients -> [T][hkv][D]: the gradient of a replicated
    head is the sum of its replicas' gradients (float64 here)."""
    rep = kv_replication(sp, hkv)
    _, T, D = y.shape
    out = np.zeros((T, hkv, D), dtype=np.float64)
    for r in range(y.shape[0]):
        out[:, r // rep, :] += y[r].astype(np.float64)
    return out


# ------------------------------------------------------------------ the exchange between real ranks
def _rank_heads(H: int, sp: int, head0: int, nheads):
    """(per-rank heads Hl, chunk size nh, replication) of a rank-local exchange step."""
    if H % sp == 0:
        Hl = H // sp
        nh = Hl - head0 if nheads is None else nheads
        if head0 < 0 or nh < 1 or head0 + nh > Hl:
            raise ValueError("head chunk outside the rank's heads")
        return Hl, nh, 1
    rep = kv_replication(sp, H)
    if head0 != 0 or (nheads not in (None, 1)):
        raise ValueError("replicated heads move whole")
    return 1, 1, rep


def a2a_pack(x_shard: np.ndarray, sp: int, head0: int = 0, nheads=None) -> np.ndarray:
    """What one rank sends in the sequence -> heads all-to-all, one block per destination.

    x_shard: [S][H][D] bits, this rank's S tokens with all heads. Returns [sp][S][nh][D]
    whose block r goes to rank r: the rank's tokens of rank r's heads r*Hl + head0 + j
    (j < nh); with fewer heads than ranks, the one head rank r reads, r*H // sp.
    """
    S, H, D = x_shard.shape
    Hl, nh, rep = _rank_heads(H, sp, head0, nheads)
    out = np.empty((sp, S, nh, D), dtype=x_shard.dtype)
    for r in range(sp):
        for j in range(nh):
            h = r * H // sp if rep > 1 else r * Hl + head0 + j
            out[r, :, j, :] = x_shard[:, h, :]
    return out


def exchange_blocks(sends):
    """The all-to-all itself over ranks given as a list: rank r receives, in rank order,
    block r of every rank's send buffer (recv_r[r'] = send_{r'}[r])."""
    sp = len(sends)
    return [np.stack([sends[src][r] for src in range(sp)]) for r in range(sp)]


def a2a_unpack(recv: np.ndarray, sp: int, H: int, head0: int = 0, nheads=None, out=None) -> np.ndarray:
    """What one rank does with what it receives in the heads -> sequence all-to-all.

    recv: [sp][S][nh][D], block r from rank r: this rank's tokens of rank r's heads.
    Writes out[s][r*Hl + head0 + j] = recv[r][s][j] into `out` ([S][H][D], created when
    None). With fewer heads than ranks the blocks are gradients of replicas of one head
    (rank r's is head r*H // sp) and are summed (float64 result).
    """
    _, S, nh_in, D = recv.shape
    Hl, nh, rep = _rank_heads(H, sp, head0, nheads)
    if nh_in != nh:
        raise ValueError("received blocks do not match the head chunk")
    if rep > 1:
        if out is None:
            out = np.zeros((S, H, D), dtype=np.float64)
        for r in range(sp):
            out[:, r * H // sp, :] += recv[r, :, 0, :].astype(np.float64)
        return out
    if out is None:
        out = np.zeros((S, H, D), dtype=recv.dtype)
    for r in range(sp):
        for j in range(nh):
            out[:, r * Hl + head0 + j, :] = recv[r, :, j, :]
    return out
