"""GPU parity of the fused Ulysses steps (layout swaps inside the attention kernels):
seq-sharded q, k, v, dO in; seq-sharded o, dq, dk, dv out.

Checked against the float64 oracle (the computed O -- output plus rounding residual --
within 1e-2 and the bf16 output within 1e-2 plus its half-ulp, LSE within 1e-3, fp32
gradients within 2e-2, as the unfused tests) and against the unfused path: the forward
output must be bit-identical, since only the rows the kernel reads and writes differ.
The packed, long and gqa workloads run here in the configuration the benchmark times:
one rank's slice of heads, token-major buffers.
"""
import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import dev_bf16, f64, host_bits, needs_gpu, sample_rows
from ulysses_sequence_seq_gb300.synth import (WORKLOADS, custom_workload, head_sharded_bits, rank_slice,
                                              seq_sharded_bits)

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, G_TOL = 1e-2, 1e-3, 2e-2


def heads_of(x_seq):
    """[sp][S][H][D] bits -> [H][T][D] bits (for the oracle)."""
    sp, S, H, D = x_seq.shape
    return np.ascontiguousarray(x_seq.reshape(sp * S, H, D).transpose(1, 0, 2))


class Fused:
    def __init__(self, w, grad_dtype=torch.float32):
        self.w = w
        self.xq, self.xk, self.xv, self.xdo = (seq_sharded_bits(w, t) for t in ("q", "k", "v", "do"))
        self.cu_host = w.cu_seqlens()
        self.layer = usp.UlyssesAttention(w.total_tokens, w.num_seqs, w.hq, w.hkv, w.head_dim, w.sp,
                                          causal=w.causal, grad_dtype=grad_dtype, fused=True)
        self.dq, self.dk, self.dv, self.ddo = (dev_bf16(a) for a in (self.xq, self.xk, self.xv, self.xdo))
        self.cu = torch.from_numpy(self.cu_host).cuda()

    def run(self):
        o = self.layer.forward(self.dq, self.dk, self.dv, self.cu).clone()
        self.o_res = self.layer.o_res_seq.clone()
        lse = self.layer.lse.clone()
        g = [t.clone() for t in self.layer.backward(self.ddo, self.cu)]
        torch.cuda.synchronize()
        assert self.layer.device_status() == 0
        return o, lse, g


def check(w, q_heads=None, rows=None, kv_heads=None, k_rows=None, grad_dtype=torch.float32):
    f = Fused(w, grad_dtype)
    o, lse, (gq, gk, gv) = f.run()
    q, k, v, do = (heads_of(a) for a in (f.xq, f.xk, f.xv, f.xdo))
    T = w.total_tokens
    ro, rl = oracle.attn_fwd(q, k, v, f.cu_host, causal=w.causal, heads=q_heads, rows=rows)
    hs = list(range(w.hq)) if q_heads is None else list(q_heads)
    rs = np.arange(T) if rows is None else np.asarray(rows)
    o_h = f64(o).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)        # [H][T][D]
    r_h = f64(f.o_res).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)
    assert np.abs(o_h[hs][:, rs] + r_h[hs][:, rs] - ro).max() <= O_TOL
    assert (np.abs(o_h[hs][:, rs] - ro) <= O_TOL + np.abs(ro) * 2.0 ** -8).all()
    assert np.abs(f64(lse)[hs][:, rs] - rl).max() <= LSE_TOL
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, f.cu_host, causal=w.causal, q_heads=q_heads, q_rows=rows,
                                 kv_heads=kv_heads, k_rows=k_rows)
    kh = list(range(w.hkv)) if kv_heads is None else list(kv_heads)
    kr = np.arange(T) if k_rows is None else np.asarray(k_rows)
    gq_h = f64(gq).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)
    gk_h = f64(gk).reshape(T, w.hkv, w.head_dim).transpose(1, 0, 2)
    gv_h = f64(gv).reshape(T, w.hkv, w.head_dim).transpose(1, 0, 2)
    for name, g, r in (("dQ", gq_h[hs][:, rs], rq), ("dK", gk_h[kh][:, kr], rk), ("dV", gv_h[kh][:, kr], rv)):
        tol = G_TOL if grad_dtype == torch.float32 else G_TOL + np.abs(r) * 2.0 ** -8
        assert (np.abs(g - r) <= tol).all(), f"{name} max-abs error {np.abs(g - r).max()}"
    return f, o


def test_fused_tiny_full():
    needs_gpu()
    check(WORKLOADS["tiny"])


def test_fused_tiny_bf16_grads():
    needs_gpu()
    check(WORKLOADS["tiny"], grad_dtype=torch.bfloat16)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_fused_ragged_gqa(causal, D):
    needs_gpu()
    w = custom_workload("fused_ragged", [1, 7, 129, 163, 1, 255], sp=2, hq=4, hkv=2, head_dim=D, causal=causal,
                        index=18)
    check(w)


def test_fused_llama_matches_unfused_and_oracle():
    """All 32 heads of the 2 x 4096 batch (the benchmark's launch); two heads checked
    against the oracle, the whole output bitwise against the unfused path."""
    needs_gpu()
    w = WORKLOADS["llama"]
    f, o = check(w, q_heads=[0, 31], kv_heads=[0, 31])
    layer = usp.UlyssesAttention(w.total_tokens, w.num_seqs, w.hq, w.hkv, w.head_dim, w.sp, fused=False,
                                 grad_dtype=torch.float32)
    o2 = layer.forward(f.dq, f.dk, f.dv, f.cu)
    g2 = layer.backward(f.ddo, f.cu)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(o), host_bits(o2))
    gq, gk, gv = f.layer.backward(f.ddo, f.cu)
    for a, b in zip((gq, gk, gv), g2):
        assert (a - b).abs().max().item() <= 1e-3     # atomics add dQ in a different order


def test_fused_gqa_sampled():
    needs_gpu()
    w = WORKLOADS["gqa"]
    cu = w.cu_seqlens()
    ends = [int(x) for x in cu[1:]]
    check(w, q_heads=[0, 13], rows=sample_rows(cu, 24, seed=19), kv_heads=[3],
          k_rows=sorted({r for e in ends for r in (e - 1, e - 129)}))


def test_fused_packed_rank_slice_sampled():
    """The packed workload as the benchmark runs it: one rank's 4 heads over all 65536
    tokens in the token-major layout, sampled rows and key rows at every sample end."""
    needs_gpu()
    w = rank_slice(WORKLOADS["packed"])
    cu = w.cu_seqlens()
    ends = [int(x) for x in cu[1:]]
    check(w, q_heads=[1, 3], rows=sample_rows(cu, 48, seed=21), kv_heads=[2],
          k_rows=sorted({r for e in ends for r in (e - 1, e - 2, e - 129)} | {0, 127, 128}))


def test_fused_long_rank_slice_sampled():
    """The headline workload as the benchmark runs it: one rank's 4 heads over the
    262144-token sequence, token-major."""
    needs_gpu()
    w = rank_slice(WORKLOADS["long"])
    T = w.total_tokens
    rows = np.array([0, 1, 127, 128, 4095, 65536, 200003, T - 129, T - 1], dtype=np.int64)
    k_rows = np.array([T - 300, T - 129, T - 128, T - 2, T - 1], dtype=np.int64)
    check(w, q_heads=[0], rows=rows, kv_heads=[0], k_rows=k_rows)


def test_fused_shortest_samples_gqa():
    """Packed samples of 128 to 300 tokens, GQA 4:1, N(0, 1), sp = 2, all heads in full."""
    needs_gpu()
    rng = np.random.default_rng(33)
    lengths = [int(x) for x in rng.integers(16, 38, size=16) * 8]
    w = custom_workload("fused_short", lengths, sp=2, hq=8, hkv=2, head_dim=128, index=20)
    check(w)


def test_fused_rejects_sp_violations():
    needs_gpu()
    z = torch.zeros(64, 4, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(4, 64, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for sp, hq, hkv, T in ((3, 4, 4, 64), (2, 6, 3, 64), (8, 4, 4, 64)):
        with pytest.raises(usp.UspError):
            usp.ulysses_attn_fwd(z, z, z, z, lse, cu, 1, T, sp, hq, hkv, 64, 0.0, True, ws, ws.numel())
