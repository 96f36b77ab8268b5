"""Pins for the CPU oracle: checks against facts the pages and the mathematics fix,
never against the oracle's own formulas retyped (CPU only)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute, relayout
from ulysses_sequence_seq_gb300.synth import (bf16_bits_to_f32, f32_to_bf16_bits,
                                              index_pattern_bits)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_bits(rng, shape, std=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


# ============================================================================ re-layout
def test_layout_figure_worked_example():
    """The two-GPU layout figure: which (token, head) pairs each rank holds."""
    T, H, D, sp = 8, 4, 1, 2
    x = index_pattern_bits(T, H, D)              # value = t*H + h (D = 1)
    xs = x.reshape(sp, T // sp, H, D)
    y = relayout.seq_to_head(xs, sp)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "layout_figure_2gpu.txt"))
            if l.strip() and not l.startswith("#")]
    for phase, r, t0, t1, h0, h1 in rows:
        r, t0, t1, h0, h1 = map(int, (r, t0, t1, h0, h1))
        want = {(t, h) for t in range(t0, t1) for h in range(h0, h1)}
        if phase == "seq":
            got = {(int(v) // H, int(v) % H) for v in xs[r].ravel()}
        else:
            got = {(int(v) // H, int(v) % H) for v in y[r].ravel()}
        assert got == want, (phase, r)
    back = relayout.head_to_seq(y, sp)
    assert np.array_equal(back, xs)


def test_head_divisibility_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "head_divisibility_32.txt"))
            if l.strip() and not l.startswith("#")]
    for row in rows:
        H, ok = int(row[0]), {int(s) for s in row[1:]}
        x = np.zeros((64, H, 2), dtype=np.uint16)
        for sp in range(1, H + 1):
            if 64 % sp:
                continue
            if sp in ok:
                relayout.seq_to_head(x, sp)
            else:
                with pytest.raises(ValueError):
                    relayout.seq_to_head(x, sp)


@pytest.mark.parametrize("sp", [1, 2, 4, 8])
def test_relayout_round_trip_and_transpose(sp):
    rng = np.random.default_rng(7)
    T, H, D = 64, 8, 6
    x = rng.integers(0, 65536, size=(T, H, D), dtype=np.uint16)
    y = relayout.seq_to_head(x, sp)
    # round trip is the identity ("back to seq-sharded")
    assert np.array_equal(relayout.head_to_seq(y, sp).reshape(T, H, D), x)
    # on one device the swap is the (token, head) transpose (library routine)
    assert np.array_equal(y.reshape(H, T, D), np.transpose(x, (1, 0, 2)))


def test_relayout_pure_python_loops():
    """Four nested loops on a tiny case, written from the figure's description."""
    T, H, D, sp = 12, 6, 2, 3
    x = index_pattern_bits(T, H, D).reshape(sp, T // sp, H, D)
    y = relayout.seq_to_head(x, sp)
    S, Hl = T // sp, H // sp
    for r in range(sp):              # destination rank owns heads r*Hl .. r*Hl+Hl-1
        for hl in range(Hl):
            for src_rank in range(sp):   # gathers every rank's token chunk in order
                for s in range(S):
                    for d in range(D):
                        assert y[r, hl, src_rank * S + s, d] == x[src_rank, s, r * Hl + hl, d]


def test_relayout_rejects_ragged():
    x = np.zeros((10, 4, 2), dtype=np.uint16)
    with pytest.raises(ValueError):
        relayout.seq_to_head(x, 4)     # 10 tokens not a multiple of 4
    x = np.zeros((12, 6, 2), dtype=np.uint16)
    with pytest.raises(ValueError):
        relayout.seq_to_head(x, 4)     # 6 heads not divisible by 4


# ============================================================================ forward
def sdpa_reference(q, k, v, cu, causal, scale=None):
    """torch float64 scaled_dot_product_attention, one sample at a time."""
    hq, T, D = q.shape
    G = hq // k.shape[0]
    qt, kt, vt = (torch.from_numpy(f64(a)) for a in (q, k, v))
    kt = kt.repeat_interleave(G, dim=0)
    vt = vt.repeat_interleave(G, dim=0)
    out = torch.zeros(hq, T, D, dtype=torch.float64)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        out[:, a:e] = torch.nn.functional.scaled_dot_product_attention(
            qt[:, a:e], kt[:, a:e], vt[:, a:e], is_causal=bool(causal), scale=scale)
    return out.numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_fwd_matches_library_sdpa_per_sample(causal):
    rng = np.random.default_rng(1)
    cu = np.array([0, 37, 40, 100], dtype=np.int32)
    q = rand_bits(rng, (4, 100, 16))
    k = rand_bits(rng, (2, 100, 16))
    v = rand_bits(rng, (2, 100, 16))
    o, lse = oracle.attn_fwd(q, k, v, cu, causal=causal)
    ref = sdpa_reference(q, k, v, cu, causal)
    assert np.abs(o - ref).max() < 1e-12


def test_fwd_lse_library_logsumexp():
    rng = np.random.default_rng(2)
    cu = np.array([0, 30, 64], dtype=np.int32)
    q, k, v = (rand_bits(rng, (2, 64, 8)) for _ in range(3))
    _, lse = oracle.attn_fwd(q, k, v, cu)
    for h in range(2):
        for b in range(2):
            a, e = cu[b], cu[b + 1]
            s = torch.from_numpy(f64(q[h, a:e]) @ f64(k[h, a:e]).T) / math.sqrt(8)
            s = s.masked_fill(torch.ones_like(s, dtype=torch.bool).triu(1), -math.inf)
            assert np.abs(torch.logsumexp(s, dim=1).numpy() - lse[h, a:e]).max() < 1e-12


def test_fwd_closed_form_zero_queries():
    """q = 0: uniform weights, O_i = mean of v over [start, i], lse_i = ln(i - start + 1)."""
    rng = np.random.default_rng(3)
    cu = np.array([0, 5, 21, 48], dtype=np.int32)
    T, D = 48, 8
    q = np.zeros((1, T, D), dtype=np.uint16)
    k = rand_bits(rng, (1, T, D))
    v = rand_bits(rng, (1, T, D))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    vf = f64(v[0])
    for b in range(3):
        for i in range(cu[b], cu[b + 1]):
            n = i - cu[b] + 1
            assert abs(lse[0, i] - math.log(n)) < 1e-12
            assert np.abs(o[0, i] - vf[cu[b]:i + 1].mean(axis=0)).max() < 1e-12


def test_fwd_closed_form_equal_keys():
    """All keys equal: uniform weights again, lse_i = ln(n) + scale * q_i.k."""
    rng = np.random.default_rng(4)
    T, D = 40, 16
    cu = np.array([0, 40], dtype=np.int32)
    q = rand_bits(rng, (1, T, D))
    k = np.repeat(rand_bits(rng, (1, 1, D)), T, axis=1)
    v = rand_bits(rng, (1, T, D))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    qf, kf, vf = f64(q[0]), f64(k[0, 0]), f64(v[0])
    for i in range(T):
        assert abs(lse[0, i] - (math.log(i + 1) + qf[i] @ kf / math.sqrt(D))) < 1e-12
        assert np.abs(o[0, i] - vf[:i + 1].mean(axis=0)).max() < 1e-12


def test_fwd_constant_values_and_singletons():
    """v = c gives O = c (weights sum to 1); a one-token sample gives O = v."""
    rng = np.random.default_rng(5)
    cu = np.array([0, 1, 2, 30, 31], dtype=np.int32)
    T, D = 31, 8
    q, k = rand_bits(rng, (1, T, D), 3.0), rand_bits(rng, (1, T, D), 3.0)
    c = f32_to_bf16_bits(np.float32([1.5]))[0]
    v = np.full((1, T, D), c, dtype=np.uint16)
    o, _ = oracle.attn_fwd(q, k, v, cu)
    assert np.abs(o - 1.5).max() < 1e-13
    v = rand_bits(rng, (1, T, D))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    for i in (0, 1, 30):   # singleton samples
        assert np.abs(o[0, i] - f64(v[0, i])).max() == 0.0


def test_fwd_matches_pure_python_brute_force():
    rng = np.random.default_rng(6)
    cu = [0, 7, 12]
    T, D = 12, 4
    q, k, v = (rand_bits(rng, (1, T, D)) for _ in range(3))
    for causal in (True, False):
        o, lse = oracle.attn_fwd(q, k, v, np.array(cu, np.int32), causal=causal)
        ob, lb = brute.attention(f64(q[0]).tolist(), f64(k[0]).tolist(), f64(v[0]).tolist(), cu,
                                 causal)
        assert np.abs(o[0] - np.array(ob)).max() < 1e-12
        assert np.abs(lse[0] - np.array(lb)).max() < 1e-12


def test_fwd_no_leakage_across_samples():
    """Packed attention equals each sample attended on its own, and changing one
    sample's keys/values leaves every other sample's output bit-identical."""
    rng = np.random.default_rng(8)
    cu = np.array([0, 24, 25, 60, 96], dtype=np.int32)
    T, D = 96, 8
    q, k, v = (rand_bits(rng, (2, T, D)) for _ in range(3))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    for b in range(4):
        a, e = cu[b], cu[b + 1]
        ob, lb = oracle.attn_fwd(q[:, a:e], k[:, a:e], v[:, a:e], np.array([0, e - a], np.int32))
        assert np.array_equal(ob, o[:, a:e]) and np.array_equal(lb, lse[:, a:e])
    k2, v2 = k.copy(), v.copy()
    k2[:, 25:60] = rand_bits(rng, (2, 35, D))
    v2[:, 25:60] = rand_bits(rng, (2, 35, D))
    o2, _ = oracle.attn_fwd(q, k2, v2, cu)
    assert np.array_equal(o2[:, :25], o[:, :25]) and np.array_equal(o2[:, 60:], o[:, 60:])
    assert not np.array_equal(o2[:, 25:60], o[:, 25:60])


def test_fwd_head_sharding_invariance():
    """Heads are independent: attention on each rank's head shard after the layout
    swap, swapped back, equals unsharded attention for every sp dividing H."""
    rng = np.random.default_rng(9)
    T, H, D = 32, 8, 4
    cu = np.array([0, 12, 32], dtype=np.int32)
    xq, xk, xv = (rand_bits(rng, (T, H, D)) for _ in range(3))
    full, _ = oracle.attn_fwd(np.transpose(xq, (1, 0, 2)), np.transpose(xk, (1, 0, 2)),
                              np.transpose(xv, (1, 0, 2)), cu)
    full_seq = np.transpose(full, (1, 0, 2))            # [T][H][D]
    for sp in (1, 2, 4, 8):
        yq, yk, yv = (relayout.seq_to_head(a, sp) for a in (xq, xk, xv))
        outs = []
        for r in range(sp):                             # each simulated rank on its own
            o_r, _ = oracle.attn_fwd(yq[r], yk[r], yv[r], cu)
            outs.append(o_r)
        o_head = np.stack(outs)                         # [sp][Hl][T][D]
        # head_to_seq on float64 data: the same index map as for bits
        back = np.empty((sp, T // sp, H, D))
        S, Hl = T // sp, H // sp
        for r in range(sp):
            for hl in range(Hl):
                for t in range(T):
                    back[t // S, t % S, r * Hl + hl] = o_head[r, hl, t]
        assert np.array_equal(back.reshape(T, H, D), full_seq)


def test_fwd_row_subset_equals_full():
    rng = np.random.default_rng(10)
    cu = np.array([0, 50, 77], dtype=np.int32)
    q = rand_bits(rng, (4, 77, 8))
    k, v = rand_bits(rng, (2, 77, 8)), rand_bits(rng, (2, 77, 8))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    rows, heads = [76, 0, 49, 50, 13], [3, 1]
    os_, ls = oracle.attn_fwd(q, k, v, cu, heads=heads, rows=rows)
    assert np.array_equal(os_, o[heads][:, rows]) and np.array_equal(ls, lse[heads][:, rows])


def test_fwd_rejects_malformed_cu():
    q = np.zeros((1, 8, 4), dtype=np.uint16)
    for cu in ([0, 4, 7], [1, 8], [0, 6, 4, 8]):
        with pytest.raises(ValueError):
            oracle.attn_fwd(q, q, q, np.array(cu, np.int32))


# ============================================================================ backward
def autograd_reference(q, k, v, do, cu, causal):
    """torch float64 autograd through per-sample SDPA (GQA by repeating kv heads)."""
    hq, T, D = q.shape
    G = hq // k.shape[0]
    qt, kt, vt = (torch.from_numpy(f64(a)).requires_grad_(True) for a in (q, k, v))
    out = torch.zeros(hq, T, D, dtype=torch.float64)
    ke, ve = kt.repeat_interleave(G, 0), vt.repeat_interleave(G, 0)
    pieces = []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        pieces.append(torch.nn.functional.scaled_dot_product_attention(
            qt[:, a:e], ke[:, a:e], ve[:, a:e], is_causal=bool(causal)))
    out = torch.cat(pieces, dim=1)
    (out * torch.from_numpy(f64(do))).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy(), out.detach().numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_matches_library_autograd(causal):
    rng = np.random.default_rng(11)
    cu = np.array([0, 19, 20, 64], dtype=np.int32)
    q, do = rand_bits(rng, (4, 64, 16)), rand_bits(rng, (4, 64, 16))
    k, v = rand_bits(rng, (2, 64, 16)), rand_bits(rng, (2, 64, 16))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, cu, causal=causal)
    rq, rk, rv, _ = autograd_reference(q, k, v, do, cu, causal)
    assert np.abs(dq - rq).max() < 1e-11
    assert np.abs(dk - rk).max() < 1e-11
    assert np.abs(dv - rv).max() < 1e-11


def test_bwd_matches_finite_differences():
    rng = np.random.default_rng(12)
    cu = [0, 6, 10]
    T, D = 10, 3
    q, k, v, do = (rand_bits(rng, (1, T, D)) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, np.array(cu, np.int32))
    fq, fk, fv = brute.finite_diff_grads(f64(q[0]).tolist(), f64(k[0]).tolist(),
                                         f64(v[0]).tolist(), f64(do[0]).tolist(), cu)
    for got, fd in ((dq[0], fq), (dk[0], fk), (dv[0], fv)):
        fd = np.array(fd)
        assert np.abs(got - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max())


def test_bwd_delta_identity_and_key_gradient_sums():
    """sum_j P_ij dP_ij = dO_i . O_i, and since every row of dS sums to zero the
    key gradients of each sample sum to zero."""
    rng = np.random.default_rng(13)
    cu = np.array([0, 33, 34, 80], dtype=np.int32)
    q, do = rand_bits(rng, (2, 80, 8)), rand_bits(rng, (2, 80, 8))
    k, v = rand_bits(rng, (1, 80, 8)), rand_bits(rng, (1, 80, 8))
    o, lse = oracle.attn_fwd(q, k, v, cu)
    dq, dk, dv, lse_b, delta = oracle.attn_bwd(q, k, v, do, cu, want_stats=True)
    assert np.abs(lse_b - lse).max() < 1e-12
    assert np.abs(delta - (o * f64(do)).sum(-1)).max() < 1e-11
    for b in range(3):
        assert np.abs(dk[:, cu[b]:cu[b + 1]].sum(axis=1)).max() < 1e-11


def test_bwd_subsets_equal_full():
    rng = np.random.default_rng(14)
    cu = np.array([0, 40, 72], dtype=np.int32)
    q, do = rand_bits(rng, (4, 72, 8)), rand_bits(rng, (4, 72, 8))
    k, v = rand_bits(rng, (2, 72, 8)), rand_bits(rng, (2, 72, 8))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, cu)
    rows, keys = [71, 3, 40, 39], [0, 39, 40, 70, 71]
    sq, sk, sv = oracle.attn_bwd(q, k, v, do, cu, q_heads=[2, 0], q_rows=rows,
                                 kv_heads=[1], k_rows=keys)
    assert np.array_equal(sq, dq[[2, 0]][:, rows])
    assert np.allclose(sk, dk[[1]][:, keys], rtol=0, atol=1e-13)
    assert np.allclose(sv, dv[[1]][:, keys], rtol=0, atol=1e-13)


# ======================================================== key/value heads over the ranks
@pytest.mark.parametrize("hq,hkv,sp", [(32, 8, 8), (32, 8, 16), (32, 2, 8), (8, 1, 4), (32, 32, 4), (8, 8, 8)])
def test_kv_replica_is_the_head_each_rank_reads(hq, hkv, sp):
    """Rank r's query heads [r*Hl, (r+1)*Hl) read kv heads h // G; the head the rank
    receives must be exactly that head (so there is only one)."""
    G, Hl = hq // hkv, hq // sp
    T, D = 8 * sp, 1
    x = index_pattern_bits(T, hkv, D)          # value = t * hkv + h
    y = relayout.seq_to_head_kv(x.reshape(T, hkv, D), sp)
    rep = relayout.kv_replication(sp, hkv)
    per_rank = y.shape[0] // sp                # key/value heads held by each rank
    for r in range(sp):
        needed = sorted({h // G for h in range(r * Hl, (r + 1) * Hl)})
        held = sorted({int(v) % hkv for v in y[r * per_rank:(r + 1) * per_rank].ravel()})
        assert held == needed
        assert all(int(v) // hkv == t for i in range(per_rank) for t, v in enumerate(y[r * per_rank + i, :, 0]))
    assert (rep == 1) == (hkv % sp == 0)


def test_kv_swap_without_replication_is_the_plain_swap():
    rng = np.random.default_rng(41)
    T, H, D, sp = 16, 8, 4, 4
    x = rand_bits(rng, (T, H, D))
    plain = relayout.seq_to_head(x.reshape(sp, T // sp, H, D), sp).reshape(H, T, D)
    assert np.array_equal(relayout.seq_to_head_kv(x, sp), plain)


@pytest.mark.parametrize("hkv,sp", [(2, 8), (1, 4), (4, 4), (8, 2)])
def test_kv_grad_is_the_adjoint_of_the_replication(hkv, sp):
    """<R x, y> = <x, R^T y>: the gradient of a replication is the sum over replicas."""
    rng = np.random.default_rng(hkv * 10 + sp)
    T, D = 12, 3
    x = rng.standard_normal((T, hkv, D))
    y = rng.standard_normal((max(sp, hkv), T, D))
    xb = f32_to_bf16_bits(x.astype(np.float32))
    rx = f64(relayout.seq_to_head_kv(xb, sp))
    lhs = float((rx * y).sum())
    rhs = float((f64(xb) * relayout.head_to_seq_kv_grad(y, sp, hkv)).sum())
    assert abs(lhs - rhs) <= 1e-9 * max(1.0, abs(lhs))


def test_kv_grad_of_identical_replicas_scales():
    y1 = np.arange(24, dtype=np.float64).reshape(1, 6, 4)
    y = np.concatenate([y1] * 4)               # four ranks sharing one head
    assert np.array_equal(relayout.head_to_seq_kv_grad(y, 4, 1), 4 * y1.transpose(1, 0, 2))


def test_kv_replication_rejects_indivisible():
    with pytest.raises(ValueError):
        relayout.kv_replication(4, 3)


# ================================================================ fp16 inputs
def test_decoders_exhaustive():
    """Every 16-bit pattern decodes as numpy's own float16 / the bf16 bit layout says."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got16 = oracle.decode16(allbits, "f16")
    want16 = allbits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got16), np.isnan(want16))
    ok = ~np.isnan(want16)
    assert np.array_equal(got16[ok], want16[ok])
    gotb = oracle.decode16(allbits, "bf16")
    wantb = (allbits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    ok = ~np.isnan(wantb)
    assert np.array_equal(gotb[ok], wantb[ok]) and np.array_equal(np.isnan(gotb), np.isnan(wantb))


def test_f16_attention_equals_bf16_attention_on_shared_values():
    """Inputs exactly representable in both types give the same float64 attention."""
    rng = np.random.default_rng(52)
    H, T, D = 2, 40, 16
    cu = np.array([0, 17, 40], dtype=np.int32)
    xs = []
    for _ in range(4):
        b = rand_bits(rng, (H, T, D))
        x = f64(b)
        x[np.abs(x) < 2.0 ** -14] = 0.0            # outside fp16's normal range: drop
        xs.append(x.astype(np.float32))
    bf = [f32_to_bf16_bits(x) for x in xs]
    hf = [x.astype(np.float16).view(np.uint16) for x in xs]
    assert all(np.array_equal(f64(b), oracle.decode16(h, "f16")) for b, h in zip(bf, hf))
    o1, l1 = oracle.attn_fwd(bf[0], bf[1], bf[2], cu)
    o2, l2 = oracle.attn_fwd(hf[0], hf[1], hf[2], cu, dtype="f16")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    g1 = oracle.attn_bwd(bf[0], bf[1], bf[2], bf[3], cu)
    g2 = oracle.attn_bwd(hf[0], hf[1], hf[2], hf[3], cu, dtype="f16")
    assert all(np.array_equal(a, b) for a, b in zip(g1, g2))


# ====================================================== the exchange between real ranks
def _exchange_to_heads(x, sp, head0=0, nheads=None):
    """Every rank packs its shard, the blocks are exchanged; returns each rank's receive
    buffer as a token-major [T][nh][D] array."""
    T, H, D = x.shape
    S = T // sp
    sends = [relayout.a2a_pack(x[r * S:(r + 1) * S], sp, head0, nheads) for r in range(sp)]
    return [recv.reshape(T, recv.shape[2], D) for recv in relayout.exchange_blocks(sends)]


def test_exchange_layout_figure_worked_example():
    """The two-GPU layout figure, now as what each rank holds after packing and the
    all-to-all: rank r's receive buffer is every token of its heads, in token order."""
    T, H, D, sp = 8, 4, 1, 2
    x = index_pattern_bits(T, H, D)              # value = t*H + h
    got_heads = _exchange_to_heads(x, sp)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "layout_figure_2gpu.txt"))
            if l.strip() and not l.startswith("#")]
    for phase, r, t0, t1, h0, h1 in rows:
        r, t0, t1, h0, h1 = map(int, (r, t0, t1, h0, h1))
        if phase != "head":
            continue
        recv = got_heads[r]
        assert [int(v) // H for v in recv[:, 0, 0]] == list(range(t0, t1))       # token order
        assert {int(v) % H for v in recv.ravel()} == set(range(h0, h1))
    # back: every rank sends its token-major result in sp blocks of S tokens and unpacks
    S = T // sp
    back = relayout.exchange_blocks([g.reshape(sp, S, -1, D) for g in got_heads])
    for r in range(sp):
        assert np.array_equal(relayout.a2a_unpack(back[r], sp, H), x[r * S:(r + 1) * S])


def test_exchange_pure_python_loops():
    """From the step description: rank r receives, from each source rank in order, the
    source's tokens of rank r's heads."""
    T, H, D, sp = 12, 6, 2, 3
    S, Hl = T // sp, H // sp
    x = index_pattern_bits(T, H, D)
    got = _exchange_to_heads(x, sp)
    for r in range(sp):
        for src in range(sp):
            for s in range(S):
                for hl in range(Hl):
                    for d in range(D):
                        assert got[r][src * S + s, hl, d] == x[src * S + s, r * Hl + hl, d]


def test_exchange_head_chunks_reassemble():
    """Exchanging each rank's heads in chunks (to overlap the exchange with attention)
    gives the same heads as one exchange."""
    rng = np.random.default_rng(43)
    T, H, D, sp = 16, 8, 4, 2
    x = rand_bits(rng, (T, H, D))
    whole = _exchange_to_heads(x, sp)
    parts = [_exchange_to_heads(x, sp, head0, 2) for head0 in (0, 2)]
    for r in range(sp):
        assert np.array_equal(np.concatenate([p[r] for p in parts], axis=1), whole[r])


@pytest.mark.parametrize("hkv,sp", [(2, 4), (1, 2), (2, 8)])
def test_exchange_replication_adjoint(hkv, sp):
    """With fewer key/value heads than ranks the exchange replicates; its adjoint -- the
    gradient's way back -- must sum the replicas: <E x, y> = <x, E^T y>."""
    rng = np.random.default_rng(hkv * 100 + sp)
    T, D = 4 * sp, 3
    S = T // sp
    xb = f32_to_bf16_bits(rng.standard_normal((T, hkv, D)).astype(np.float32))
    ex = _exchange_to_heads(xb, sp)                              # rank r: [T][1][D]
    y = [rng.standard_normal((T, 1, D)) for _ in range(sp)]
    lhs = sum(float((f64(ex[r]) * y[r]).sum()) for r in range(sp))
    back = relayout.exchange_blocks([yr.reshape(sp, S, 1, D) for yr in y])
    grads = [relayout.a2a_unpack(back[r], sp, hkv) for r in range(sp)]
    rhs = sum(float((f64(xb[r * S:(r + 1) * S]) * grads[r]).sum()) for r in range(sp))
    assert abs(lhs - rhs) <= 1e-9 * max(1.0, abs(lhs))
    # and each rank received the head its query heads read (kv_replication's rule)
    for r in range(sp):
        assert np.array_equal(ex[r][:, 0], xb[:, r * hkv // sp])


# ======================================================= ring-attention steps and merges
from oracle import ring  # noqa: E402


def _ring_inputs(seed, T=96, hq=4, hkv=2, D=16):
    rng = np.random.default_rng(seed)
    return (rand_bits(rng, (hq, T, D)), rand_bits(rng, (hkv, T, D)), rand_bits(rng, (hkv, T, D)),
            rand_bits(rng, (hq, T, D)))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("order", ["forward", "reverse"])
def test_ring_merged_chunks_equal_full_attention(causal, order):
    """Attending one query chunk to each key chunk of the sequence and merging the partial
    results through their log-sum-exp gives full attention (softmax over a disjoint union),
    checked against the C oracle (itself pinned to torch SDPA), in either ring order."""
    q, k, v, _ = _ring_inputs(51)
    T, nc = q.shape[1], 4
    L = T // nc
    ro, rl = oracle.attn_fwd(q, k, v, np.array([0, T], dtype=np.int32), causal=causal)
    for qc in range(nc):
        o = np.zeros((q.shape[0], L, q.shape[2]))
        lse = np.full((q.shape[0], L), -np.inf)
        chunks = range(nc) if order == "forward" else reversed(range(nc))
        for kc in chunks:
            po, pl = ring.chunk_attn_fwd(q[:, qc * L:(qc + 1) * L], k[:, kc * L:(kc + 1) * L],
                                         v[:, kc * L:(kc + 1) * L], qc * L, kc * L, causal)
            o, lse = ring.lse_merge(o, lse, po, pl)
        assert np.allclose(o, ro[:, qc * L:(qc + 1) * L], rtol=0, atol=1e-12)
        assert np.allclose(lse, rl[:, qc * L:(qc + 1) * L], rtol=0, atol=1e-12)


def test_ring_step_mask_on_global_positions():
    """A key chunk wholly after the query chunk contributes nothing (lse -inf, O 0); one
    wholly before it is unmasked attention; the diagonal chunk is causal attention."""
    q, k, v, _ = _ring_inputs(52, T=32)
    a, b = slice(0, 16), slice(16, 32)
    o, lse = ring.chunk_attn_fwd(q[:, a], k[:, b], v[:, b], 0, 16, True)
    assert np.isneginf(lse).all() and (o == 0).all()
    o1, l1 = ring.chunk_attn_fwd(q[:, b], k[:, a], v[:, a], 16, 0, True)
    o2, l2 = ring.chunk_attn_fwd(q[:, b], k[:, a], v[:, a], 16, 0, False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o3, l3 = ring.chunk_attn_fwd(q[:, b], k[:, b], v[:, b], 16, 16, True)
    r3, rl3 = oracle.attn_fwd(q[:, b], k[:, b], v[:, b], np.array([0, 16], dtype=np.int32), causal=True)
    assert np.allclose(o3, r3, rtol=0, atol=1e-12) and np.allclose(l3, rl3, rtol=0, atol=1e-12)


def test_ring_lse_merge_identities():
    rng = np.random.default_rng(53)
    o, lse = rng.standard_normal((2, 5, 3)), rng.standard_normal((2, 5))
    z, zl = np.zeros_like(o), np.full_like(lse, -np.inf)
    mo, ml = ring.lse_merge(o, lse, z, zl)
    assert np.array_equal(mo, o) and np.array_equal(ml, lse)
    o2, l2 = rng.standard_normal((2, 5, 3)), rng.standard_normal((2, 5))
    a, al = ring.lse_merge(o, lse, o2, l2)
    b, bl = ring.lse_merge(o2, l2, o, lse)
    assert np.allclose(a, b, rtol=0, atol=1e-14) and np.allclose(al, bl, rtol=0, atol=1e-14)
    eo, el = ring.lse_merge(z, zl, z, zl)
    assert (eo == 0).all() and np.isneginf(el).all()


@pytest.mark.parametrize("causal", [True, False])
def test_ring_step_gradients_sum_to_full_gradients(causal):
    """Each step's gradient share, taken with the final output and log-sum-exp, summed over
    the ring equals the full gradient of the C oracle (itself pinned to torch autograd)."""
    q, k, v, do = _ring_inputs(54)
    T, nc = q.shape[1], 3 if q.shape[1] % 3 == 0 else 4
    L = T // nc
    cu = np.array([0, T], dtype=np.int32)
    ro, rl = oracle.attn_fwd(q, k, v, cu, causal=causal)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, cu, causal=causal)
    dq, dk, dv = np.zeros(rq.shape), np.zeros(rk.shape), np.zeros(rv.shape)
    for qc in range(nc):
        qs = slice(qc * L, (qc + 1) * L)
        for kc in range(nc):
            ks = slice(kc * L, (kc + 1) * L)
            a, b, c = ring.chunk_attn_bwd(q[:, qs], k[:, ks], v[:, ks], do[:, qs], ro[:, qs], rl[:, qs],
                                          qc * L, kc * L, causal)
            dq[:, qs] += a
            dk[:, ks] += b
            dv[:, ks] += c
    for got, want in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.allclose(got, want, rtol=0, atol=1e-10)
