"""GPU parity of the ring-attention steps: the merge kernel against the oracle's merge, and
a whole ring (sp equal chunks of one sequence, or of evenly split packed samples, every
query chunk against every key chunk in ring order) against the oracle's full attention:
the merged output within 1e-2 (output plus residual), LSE within 1e-3, fp32 gradients
summed over the ring within 2e-2."""
import numpy as np
import pytest
import torch

import oracle
from oracle import ring as oring
from tests.gpu_util import dev_bf16, f64, needs_gpu
from ulysses_sequence_seq_gb300 import _lib
from ulysses_sequence_seq_gb300.ring import RingAttention
from ulysses_sequence_seq_gb300.synth import bf16_bits_to_f32, custom_workload, f32_to_bf16_bits, head_sharded_bits

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, G_TOL = 1e-2, 1e-3, 2e-2


@pytest.mark.parametrize("init", [False, True])
def test_lse_merge_kernel_matches_oracle(init):
    needs_gpu()
    rng = np.random.default_rng(61)
    T, H, D = 300, 4, 128
    o_acc = rng.standard_normal((T, H, D)).astype(np.float32)
    lse_acc = rng.standard_normal((H, T)).astype(np.float32) * 3
    o_part = f32_to_bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32))
    o_res = f32_to_bf16_bits((rng.standard_normal((T, H, D)) * 1e-3).astype(np.float32))
    lse_part = rng.standard_normal((H, T)).astype(np.float32) * 3
    lse_acc[0, :7] = -np.inf                       # rows the merged keys had not reached yet
    lse_part[1, 5:9] = -np.inf                     # rows the new chunk does not reach
    lse_acc[2, 3] = lse_part[2, 3] = -np.inf       # neither
    d_acc, d_lse = torch.from_numpy(o_acc).cuda(), torch.from_numpy(lse_acc).cuda()
    _lib.lse_merge(d_acc, d_lse, dev_bf16(o_part), torch.from_numpy(lse_part).cuda(), o_part_res=dev_bf16(o_res),
                   init=init)
    part = bf16_bits_to_f32(o_part).astype(np.float64) + bf16_bits_to_f32(o_res).astype(np.float64)
    if init:   # the part alone; a row whose part saw no key has output 0 by definition
        want_o = np.where(np.isneginf(lse_part)[:, :, None], 0.0, part.transpose(1, 0, 2))
        want_l = lse_part.astype(np.float64)
    else:
        want_o, want_l = oring.lse_merge(o_acc.astype(np.float64).transpose(1, 0, 2), lse_acc.astype(np.float64),
                                         part.transpose(1, 0, 2), lse_part.astype(np.float64))
    got_o = d_acc.cpu().numpy().astype(np.float64).transpose(1, 0, 2)
    got_l = d_lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got_l), np.isneginf(want_l))
    fin = np.isfinite(want_l)
    assert np.abs(got_l[fin] - want_l[fin]).max() <= 1e-5
    assert np.abs(got_o - want_o).max() <= 1e-5


def _ring(w, sp, grad=True, chunk_cu=None, bits=None):
    """Run the ring for every query chunk of `w` split into sp chunks (token-major), in ring
    order (own chunk first, then the chunk arriving from each earlier rank). Returns the
    per-chunk outputs (o + o_res), LSE and the gradients summed over the ring. chunk_cu:
    the chunk-local cu_seqlens shared by every chunk (default: one sample); bits: head-major
    q, k, v, do to use instead of the workload's draws."""
    T, hq, hkv, D = w.total_tokens, w.hq, w.hkv, w.head_dim
    L = T // sp
    src = bits if bits is not None else {t: head_sharded_bits(w, t) for t in ("q", "k", "v", "do")}
    tm = {t: src[t].transpose(1, 0, 2) for t in ("q", "k", "v", "do")}   # [T][H][D] bits
    chunk = {t: [dev_bf16(np.ascontiguousarray(tm[t][r * L:(r + 1) * L])) for r in range(sp)] for t in tm}
    ccu = np.array([0, L] if chunk_cu is None else chunk_cu, dtype=np.int32)
    cu = torch.from_numpy(ccu).cuda()
    nseq = len(ccu) - 1
    outs, lses, dq = [], [], []
    dk = [torch.zeros(L, hkv, D, device="cuda") for _ in range(sp)]
    dv = [torch.zeros(L, hkv, D, device="cuda") for _ in range(sp)]
    for r in range(sp):
        ra = RingAttention(L, nseq, hq, hkv, D)
        ra.forward_begin()
        order = [(r - s) % sp for s in range(sp)]
        for kr in order:
            ra.forward_step(chunk["q"][r], chunk["k"][kr], chunk["v"][kr], cu, r, kr)
        o = ra.forward_end()
        outs.append(f64(o) + f64(ra.o_res))
        lses.append(f64(ra.lse))
        if grad:
            ra.backward_begin()
            for kr in order:
                sh = ra.backward_step(chunk["q"][r], chunk["k"][kr], chunk["v"][kr], chunk["do"][r], cu, r, kr)
                if sh is not None:
                    dk[kr] += sh[0]
                    dv[kr] += sh[1]
            dq.append(f64(ra.backward_end().clone()))
    torch.cuda.synchronize()
    return outs, lses, dq, [f64(x) for x in dk], [f64(x) for x in dv]


@pytest.mark.parametrize("causal_ring", [True])
def test_ring_equals_full_attention(causal_ring):
    """One 2560-token sequence over 4 chunks of 640 (ragged 128-row tiles), GQA 2:1."""
    needs_gpu()
    w = custom_workload("ring", [2560], sp=4, hq=4, hkv=2, head_dim=128, index=26)
    sp, L = 4, 640
    outs, lses, dq, dk, dv = _ring(w, sp)
    q, k, v, do = (head_sharded_bits(w, t) for t in ("q", "k", "v", "do"))
    cu = w.cu_seqlens()
    ro, rl = oracle.attn_fwd(q, k, v, cu)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, cu)
    for r in range(sp):
        sl = slice(r * L, (r + 1) * L)
        assert np.abs(outs[r].transpose(1, 0, 2) - ro[:, sl]).max() <= O_TOL
        assert np.abs(lses[r] - rl[:, sl]).max() <= LSE_TOL
        assert np.abs(dq[r].transpose(1, 0, 2) - rq[:, sl]).max() <= G_TOL
        assert np.abs(dk[r].transpose(1, 0, 2) - rk[:, sl]).max() <= G_TOL
        assert np.abs(dv[r].transpose(1, 0, 2) - rv[:, sl]).max() <= G_TOL


def test_ring_growing_scores():
    """Peaked rows whose maxima grow along the sequence (every query's first component 4, key
    t's 0.03 t): the later chunks' LSEs exceed the earlier ones' by up to ~20, so the merge
    must weight the chunks' partial outputs by exp(LSE differences) of that size. Forward at
    1e-2 / 1e-3, dK and dV at 2e-2, dQ at 2e-2 plus the large-key allowance
    (gpu_util.dq_key_amplified_bound)."""
    needs_gpu()
    from tests.gpu_util import dq_key_amplified_bound
    w = custom_workload("ringgrow", [2560], sp=4, hq=2, hkv=2, head_dim=128, index=29)
    sp, L = 4, 640
    b = {t: head_sharded_bits(w, t) for t in ("q", "k", "v", "do")}
    qf, kf = bf16_bits_to_f32(b["q"]), bf16_bits_to_f32(b["k"])
    qf[:, :, 0] = 4.0
    kf[:, :, 0] = 0.03 * np.arange(2560, dtype=np.float32)
    b["q"], b["k"] = f32_to_bf16_bits(qf), f32_to_bf16_bits(kf)
    outs, lses, dq, dk, dv = _ring(w, sp, bits=b)
    cu = w.cu_seqlens()
    ro, rl = oracle.attn_fwd(b["q"], b["k"], b["v"], cu)
    rq, rk, rv = oracle.attn_bwd(b["q"], b["k"], b["v"], b["do"], cu)
    o_kernel = np.concatenate(outs, axis=0).transpose(1, 0, 2)
    bound = G_TOL + dq_key_amplified_bound(b["q"], b["k"], b["v"], b["do"], cu, o_kernel)
    for r in range(sp):
        sl = slice(r * L, (r + 1) * L)
        assert np.abs(outs[r].transpose(1, 0, 2) - ro[:, sl]).max() <= O_TOL
        assert np.abs(lses[r] - rl[:, sl]).max() <= LSE_TOL
        assert (np.abs(dq[r].transpose(1, 0, 2) - rq[:, sl]) <= bound[:, sl]).all()
        assert np.abs(dk[r].transpose(1, 0, 2) - rk[:, sl]).max() <= G_TOL
        assert np.abs(dv[r].transpose(1, 0, 2) - rv[:, sl]).max() <= G_TOL


def test_ring_packed_samples_split_evenly():
    """Three packed samples, each split evenly over 4 chunks (every chunk holds the r-th
    quarter of each sample, chunk-local cu_seqlens {0, 100, 400, 640}); the oracle attends
    each whole sample, reassembled from its quarters in rank order."""
    needs_gpu()
    sp, L = 4, 640
    ccu = [0, 100, 400, 640]
    w = custom_workload("ringpk", [sp * L], sp=sp, hq=4, hkv=2, head_dim=128, index=28)
    outs, lses, dq, dk, dv = _ring(w, sp, chunk_cu=ccu)
    bits = {t: head_sharded_bits(w, t) for t in ("q", "k", "v", "do")}   # chunk r = tokens [r*L, (r+1)*L)
    for b in range(3):
        a, e = ccu[b], ccu[b + 1]
        n = e - a
        whole = {t: np.concatenate([x[:, r * L + a:r * L + e] for r in range(sp)], axis=1) for t, x in bits.items()}
        cu = np.array([0, sp * n], dtype=np.int32)
        ro, rl = oracle.attn_fwd(whole["q"], whole["k"], whole["v"], cu)
        rq, rk, rv = oracle.attn_bwd(whole["q"], whole["k"], whole["v"], whole["do"], cu)
        for r in range(sp):
            sl = slice(r * n, (r + 1) * n)
            assert np.abs(outs[r][a:e].transpose(1, 0, 2) - ro[:, sl]).max() <= O_TOL
            assert np.abs(lses[r][:, a:e] - rl[:, sl]).max() <= LSE_TOL
            assert np.abs(dq[r][a:e].transpose(1, 0, 2) - rq[:, sl]).max() <= G_TOL
            assert np.abs(dk[r][a:e].transpose(1, 0, 2) - rk[:, sl]).max() <= G_TOL
            assert np.abs(dv[r][a:e].transpose(1, 0, 2) - rv[:, sl]).max() <= G_TOL


def test_ring_step_matches_oracle_step():
    """A single non-diagonal step (query chunk 2 against key chunk 0) and the diagonal one,
    against the oracle's chunk attention with the mask on global positions."""
    needs_gpu()
    w = custom_workload("ringstep", [1536], sp=3, hq=2, hkv=2, head_dim=64, index=27)
    L = 512
    tm = {t: head_sharded_bits(w, t) for t in ("q", "k", "v")}
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    for qr, kr in ((2, 0), (1, 1)):
        ra = RingAttention(L, 1, 2, 2, 64)
        ra.forward_begin()
        dev = {t: dev_bf16(np.ascontiguousarray(tm[t][:, (qr if t == "q" else kr) * L:((qr if t == "q" else kr) + 1) * L]
                                                .transpose(1, 0, 2))) for t in tm}
        ra.forward_step(dev["q"], dev["k"], dev["v"], cu, qr, kr)
        ra.forward_end()
        po, pl = oring.chunk_attn_fwd(tm["q"][:, qr * L:(qr + 1) * L], tm["k"][:, kr * L:(kr + 1) * L],
                                      tm["v"][:, kr * L:(kr + 1) * L], qr * L, kr * L, True)
        got = (f64(ra.o) + f64(ra.o_res)).transpose(1, 0, 2)
        assert np.abs(got - po).max() <= O_TOL
        assert np.abs(f64(ra.lse) - pl).max() <= LSE_TOL
