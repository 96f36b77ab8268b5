"""Pure-Python attention for tiny inputs, and finite-difference gradients.

TEST INFRASTRUCTURE ONLY. Nested Python loops over the full T x T score
matrix with ``math.exp``; meant for T <= 24 and D <= 8, where it is an
independent cross-check of the C oracle. Definitions as in ``attn_ref.c``:
softmax attention per head, masked to pairs in the same sample and, when
causal, to keys at or before the query.
"""
from __future__ import annotations

import math


def _seg(cu, T):
    seg = [0] * T
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1]):
            seg[t] = b
    return seg


def attention(q, k, v, cu, causal=True, scale=None):
    """q, k, v: nested lists [T][D] of floats (one head). Returns (O [T][D], lse [T])."""
    T, D = len(q), len(q[0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    seg = _seg(cu, T)
    O, L = [], []
    for i in range(T):
        s = []
        for j in range(T):
            ok = seg[i] == seg[j] and (not causal or j <= i)
            s.append(scale * sum(q[i][d] * k[j][d] for d in range(D)) if ok else None)
        m = max(x for x in s if x is not None)
        z = sum(math.exp(x - m) for x in s if x is not None)
        lse = m + math.log(z)
        row = [0.0] * D
        for j in range(T):
            if s[j] is None:
                continue
            p = math.exp(s[j] - lse)
            for d in range(D):
                row[d] += p * v[j][d]
        O.append(row)
        L.append(lse)
    return O, L


def loss(q, k, v, do, cu, causal=True, scale=None):
    """L = sum_{i,d} O_id * dO_id, whose gradients are dQ, dK, dV."""
    O, _ = attention(q, k, v, cu, causal, scale)
    return sum(O[i][d] * do[i][d] for i in range(len(O)) for d in range(len(O[0])))


def finite_diff_grads(q, k, v, do, cu, causal=True, scale=None, eps=1e-5):
    """Central differences of :func:`loss` with respect to every element of q, k and v."""
    grads = []
    for which in range(3):
        base = [q, k, v][which]
        g = [[0.0] * len(base[0]) for _ in base]
        for t in range(len(base)):
            for d in range(len(base[0])):
                args_p = [[row[:] for row in a] for a in (q, k, v)]
                args_m = [[row[:] for row in a] for a in (q, k, v)]
                args_p[which][t][d] += eps
                args_m[which][t][d] -= eps
                lp = loss(*args_p, do, cu, causal, scale)
                lm = loss(*args_m, do, cu, causal, scale)
                g[t][d] = (lp - lm) / (2 * eps)
        grads.append(g)
    return grads
