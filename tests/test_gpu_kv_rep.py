"""GPU parity for models with fewer key/value heads than ranks: the replicating swap of
K/V, the summing swap of their gradients, and attention with hkv < sp through the fused
and the separate-call paths."""
import numpy as np
import pytest
import torch

from oracle import relayout as ref
import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import dev_bf16, f64, host_bits, needs_gpu
from tests.test_gpu_fused import check
from ulysses_sequence_seq_gb300.synth import bf16_bits_to_f32, custom_workload, f32_to_bf16_bits, seq_sharded_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,hkv,sp,D", [(256, 2, 8, 128), (96, 1, 4, 64), (64, 8, 4, 128), (4104, 4, 8, 128)])
def test_seq_to_head_kv_bit_exact(T, hkv, sp, D):
    needs_gpu()
    rng = np.random.default_rng(T + hkv)
    x = f32_to_bf16_bits(rng.standard_normal((T, hkv, D)).astype(np.float32))
    out = torch.empty(max(sp, hkv), T, D, dtype=torch.bfloat16, device="cuda")
    usp.seq_to_head_kv(dev_bf16(x), out, sp)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), ref.seq_to_head_kv(x, sp))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("hkv,sp", [(2, 8), (1, 4), (8, 4)])
def test_head_to_seq_kv_grad(dtype, hkv, sp):
    needs_gpu()
    T, D = 1032, 128
    rng = np.random.default_rng(hkv * 100 + sp)
    y32 = rng.standard_normal((max(sp, hkv), T, D)).astype(np.float32)
    if dtype == torch.bfloat16:
        y32 = bf16_bits_to_f32(f32_to_bf16_bits(y32))
    y = torch.from_numpy(y32).to(dtype).cuda()
    out = torch.empty(T, hkv, D, dtype=dtype, device="cuda")
    usp.head_to_seq_kv_grad(y, out, sp, hkv)
    want = ref.head_to_seq_kv_grad(y32.astype(np.float64), sp, hkv)
    got = f64(out)
    rep = ref.kv_replication(sp, hkv)
    if dtype == torch.float32:
        tol = rep * 2.0 ** -23 * np.abs(y32).max() * rep
    else:   # one rounding of an fp32 sum to bf16
        tol = 2.0 ** -8 * np.abs(want) + rep * 2.0 ** -23 * np.abs(y32).max() * rep
    assert (np.abs(got - want) <= tol).all()


@pytest.mark.parametrize("causal", [True, False])
def test_fused_attention_with_replicated_kv(causal):
    """hq = 8, hkv = 2 over sp = 4 ranks: each kv head is shared by two ranks."""
    needs_gpu()
    w = custom_workload("kv_rep", [1, 7, 129, 163, 1, 255, 60], sp=4, hq=8, hkv=2, head_dim=128, causal=causal,
                        index=33)
    check(w)


def test_separate_path_with_replication_matches_fused():
    needs_gpu()
    w = custom_workload("kv_rep2", [300, 213, 511], sp=8, hq=16, hkv=2, head_dim=128, index=34)
    xs = [dev_bf16(seq_sharded_bits(w, t)) for t in ("q", "k", "v", "do")]
    cu = torch.from_numpy(w.cu_seqlens()).cuda()
    outs = []
    for fused in (True, False):
        layer = usp.UlyssesAttention(w.total_tokens, w.num_seqs, w.hq, w.hkv, w.head_dim, w.sp, fused=fused,
                                     grad_dtype=torch.float32)
        o = layer.forward(xs[0], xs[1], xs[2], cu).clone()
        g = [t.clone() for t in layer.backward(xs[3], cu)]
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        outs.append((o, g))
    assert np.array_equal(host_bits(outs[0][0]), host_bits(outs[1][0]))
    for a, b in zip(outs[0][1], outs[1][1]):
        assert (a - b).abs().max().item() <= 1e-3
