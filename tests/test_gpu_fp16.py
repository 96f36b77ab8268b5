"""GPU parity of the fused Ulysses steps with fp16 activations (same tolerances as bf16:
O within 1e-2, LSE within 1e-3, fp32 gradients within 2e-2, fp16 gradients with an extra
fp16 half-ulp, 2^-11 |ref|), against the float64 oracle decoding the same fp16 bits."""
import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import dev_16, f64, needs_gpu, sample_rows
from ulysses_sequence_seq_gb300.synth import WORKLOADS, custom_workload, seq_sharded_bits

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, G_TOL = 1e-2, 1e-3, 2e-2


def heads_of(x_seq):
    sp, S, H, D = x_seq.shape
    return np.ascontiguousarray(x_seq.reshape(sp * S, H, D).transpose(1, 0, 2))


def growing_scores(w, xq, xk):
    """A large first component in every query and keys whose first component grows with their
    position in the sample: causal rows whose block maxima rise by about 8 (log2 units) per
    key block, so the forward's running max is overtaken by more than 2^8 every block or two."""
    from ulysses_sequence_seq_gb300.synth import f32_to_f16_bits
    T, D = w.total_tokens, w.head_dim
    qf = xq.view(np.float16).astype(np.float32).reshape(T, -1, D)
    kf = xk.view(np.float16).astype(np.float32).reshape(T, -1, D)
    qf[:, :, 0] = 4.0
    cu = w.cu_seqlens()
    for b in range(len(cu) - 1):
        kf[cu[b]:cu[b + 1], :, 0] = (0.12 * np.sqrt(D / 128.0) * np.arange(cu[b + 1] - cu[b]))[:, None]
    return f32_to_f16_bits(qf).reshape(xq.shape), f32_to_f16_bits(kf).reshape(xk.shape)


def run_check(w, grad_dtype, q_heads=None, rows=None, kv_heads=None, k_rows=None, grow=False):
    """grow: the growing-score inputs; dQ is then checked against 2e-2 plus the allowance of
    gpu_util.dq_key_amplified_bound (what 16-bit dS and Delta leave, scaled by the large keys),
    the rest at the gates."""
    xs = [seq_sharded_bits(w, t, dtype="f16") for t in ("q", "k", "v", "do")]
    if grow:
        xs[0], xs[1] = growing_scores(w, xs[0], xs[1])
    cu_host = w.cu_seqlens()
    layer = usp.UlyssesAttention(w.total_tokens, w.num_seqs, w.hq, w.hkv, w.head_dim, w.sp, causal=w.causal,
                                 grad_dtype=grad_dtype, dtype=torch.float16)
    dq_, dk_, dv_, ddo = (dev_16(x, torch.float16) for x in xs)
    cu = torch.from_numpy(cu_host).cuda()
    o = layer.forward(dq_, dk_, dv_, cu).clone()
    o_res = layer.o_res_seq.clone()
    lse = layer.lse.clone()
    gq, gk, gv = (t.clone() for t in layer.backward(ddo, cu))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert o.dtype == torch.float16 and gq.dtype == grad_dtype
    q, k, v, do = (heads_of(x) for x in xs)
    T = w.total_tokens
    ro, rl = oracle.attn_fwd(q, k, v, cu_host, causal=w.causal, heads=q_heads, rows=rows, dtype="f16")
    hs = list(range(w.hq)) if q_heads is None else list(q_heads)
    rs = np.arange(T) if rows is None else np.asarray(rows)
    o_h = f64(o).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)
    assert np.abs(o_h[hs][:, rs] - ro).max() <= O_TOL
    assert np.abs(f64(lse)[hs][:, rs] - rl).max() <= LSE_TOL
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, cu_host, causal=w.causal, q_heads=q_heads, q_rows=rows,
                                 kv_heads=kv_heads, k_rows=k_rows, dtype="f16")
    kh = list(range(w.hkv)) if kv_heads is None else list(kv_heads)
    kr = np.arange(T) if k_rows is None else np.asarray(k_rows)
    got = [f64(gq).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)[hs][:, rs],
           f64(gk).reshape(T, w.hkv, w.head_dim).transpose(1, 0, 2)[kh][:, kr],
           f64(gv).reshape(T, w.hkv, w.head_dim).transpose(1, 0, 2)[kh][:, kr]]
    for name, g, r in zip(("dQ", "dK", "dV"), got, (rq, rk, rv)):
        tol = G_TOL if grad_dtype == torch.float32 else G_TOL + np.abs(r) * 2.0 ** -11
        if grow and name == "dQ":
            from tests.gpu_util import dq_key_amplified_bound
            assert q_heads is None and rows is None and w.hq == w.hkv
            o_kernel = (f64(o) + f64(o_res)).reshape(T, w.hq, w.head_dim).transpose(1, 0, 2)
            tol = tol + dq_key_amplified_bound(q, k, v, do, cu_host, o_kernel, dtype="f16")
        assert (np.abs(g - r) <= tol).all(), f"{name} max-abs error {np.abs(g - r).max()}"


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.float16])
def test_fp16_tiny(grad_dtype):
    needs_gpu()
    run_check(WORKLOADS["tiny"], grad_dtype)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_fp16_ragged_gqa(causal, D):
    needs_gpu()
    w = custom_workload("f16_ragged", [1, 7, 129, 163, 1, 255], sp=2, hq=4, hkv=2, head_dim=D, causal=causal,
                        index=36)
    run_check(w, torch.float16)


def test_fp16_llama_sampled():
    needs_gpu()
    w = WORKLOADS["llama"]
    run_check(w, torch.float32, q_heads=[0, 31], rows=sample_rows(w.cu_seqlens(), 24, seed=5), kv_heads=[7],
              k_rows=[0, 1, 127, 128, 4095, 4096, 8191])


def test_fp16_rejects_mixed_types():
    needs_gpu()
    z = torch.zeros(64, 4, 64, dtype=torch.float16, device="cuda")
    lse = torch.zeros(4, 64, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    zb = torch.zeros(64, 4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(usp.UspError):    # fp16 activations, bf16 gradients
        usp.ulysses_attn_bwd(z, z, z, z, lse, z, zb, zb, zb, usp.USP_BF16, cu, 1, 64, 2, 4, 4, 64, 0.0, True, ws,
                             ws.numel())
    zf = torch.zeros(64, 4, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(usp.UspError):    # fp32 activations
        usp.ulysses_attn_fwd(zf, zf, zf, zf, lse, cu, 1, 64, 2, 4, 4, 64, 0.0, True, ws, ws.numel())


@pytest.mark.parametrize("D", [64, 128])
def test_fp16_growing_scores(D):
    """Peaked rows whose running max moves often (the forward's rescale path) in fp16, through
    the forward and the backward (dQ with the large-key allowance)."""
    needs_gpu()
    w = custom_workload("grow16", [700, 300, 130], sp=2, hq=2, hkv=2, head_dim=D, index=21)
    run_check(w, torch.float32, grow=True)
