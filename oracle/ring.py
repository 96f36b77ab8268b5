"""Ring-attention steps: attention of one query chunk against one key/value chunk of the
same sequence, and the merge of such partial results.

TEST INFRASTRUCTURE ONLY.

In ring attention every rank keeps a chunk of the queries and the key/value chunks travel
around the ring; each step attends the local queries to the visiting keys and the partial
results are combined through their log-sum-exp (ColossalAI sequence parallelism tutorial,
the ring-attention plugin set-up and its closing comparison of Ulysses and ring
attention). The causal mask is the ordinary one on global positions: a query at global
position q_off + i may see a key at k_off + j iff k_off + j <= q_off + i. Everything here
is float64 numpy, one head at a time, with the mask predicate evaluated for every pair.
"""
from __future__ import annotations

import math

import numpy as np


def _decode(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def chunk_attn_fwd(q, k, v, q_off: int, k_off: int, causal: bool = True, scale=None):
    """q: [hq][Lq][D], k, v: [hkv][Lk][D] bf16 bits. Returns the partial output O
    [hq][Lq][D] and log-sum-exp [hq][Lq] of the queries over this key chunk alone; rows
    that see no key of the chunk get O = 0 and lse = -inf."""
    qf, kf, vf = _decode(q), _decode(k), _decode(v)
    hq, Lq, D = qf.shape
    hkv, Lk, _ = kf.shape
    G = hq // hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o = np.zeros((hq, Lq, D))
    lse = np.full((hq, Lq), -np.inf)
    allowed = np.array([[(not causal) or (k_off + j <= q_off + i) for j in range(Lk)] for i in range(Lq)])
    for h in range(hq):
        s = scale * qf[h] @ kf[h // G].T
        for i in range(Lq):
            idx = np.nonzero(allowed[i])[0]
            if idx.size == 0:
                continue
            m = s[i, idx].max()
            e = np.exp(s[i, idx] - m)
            lse[h, i] = m + math.log(e.sum())
            o[h, i] = (e / e.sum()) @ vf[h // G][idx]
    return o, lse


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Softmax over the union of two disjoint key sets from each set's normalised output
    and log-sum-exp: lse = log(e^lse_a + e^lse_b), O = e^(lse_a - lse) O_a + e^(lse_b - lse) O_b
    (a side with lse = -inf contributes nothing; both -inf stays O = 0, lse = -inf)."""
    lse = np.logaddexp(lse_a, lse_b)
    with np.errstate(invalid="ignore"):
        wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - lse))
        wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - lse))
    return wa[..., None] * o_a + wb[..., None] * o_b, lse


def chunk_attn_bwd(q, k, v, do, o, lse, q_off: int, k_off: int, causal: bool = True, scale=None):
    """One step's share of the gradients: with P_ij = exp(s_ij - lse_i) taken from the
    FINAL log-sum-exp of each query row and Delta_i = sum over the step's keys j of
    P_ij dP_ij plus the other steps' share -- i.e. dO_i . O_i for the final output O --
    returns dQ (this chunk's keys' contribution), dK and dV of this key chunk (summed
    over the query heads of each key/value head). o: [hq][Lq][D] final output (float),
    lse: [hq][Lq] final log-sum-exp, do: [hq][Lq][D] bits."""
    qf, kf, vf, dof = _decode(q), _decode(k), _decode(v), _decode(do)
    hq, Lq, D = qf.shape
    hkv, Lk, _ = kf.shape
    G = hq // hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    allowed = np.array([[(not causal) or (k_off + j <= q_off + i) for j in range(Lk)] for i in range(Lq)])
    dq = np.zeros((hq, Lq, D))
    dk = np.zeros((hkv, Lk, D))
    dv = np.zeros((hkv, Lk, D))
    for h in range(hq):
        g = h // G
        s = scale * qf[h] @ kf[g].T
        with np.errstate(invalid="ignore", over="ignore"):
            p = np.where(allowed & np.isfinite(lse[h])[:, None], np.exp(s - lse[h][:, None]), 0.0)
        dp = dof[h] @ vf[g].T
        delta = (dof[h] * o[h]).sum(axis=1)
        ds = p * (dp - delta[:, None])
        dq[h] = scale * ds @ kf[g]
        dk[g] += scale * ds.T @ qf[h]
        dv[g] += p.T @ dof[h]
    return dq, dk, dv
