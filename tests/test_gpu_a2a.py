"""GPU checks of the exchange's rank-local kernels (usp_a2a_pack / usp_a2a_unpack) and of
the whole Ulysses step built on them.

The kernels are compared bit for bit with the oracle's index formulas. The step is run
for sp simulated ranks on one GPU -- pack, the block exchange done as host-side copies
(the collective's data movement), attention on each rank's received heads, the way back
and unpack -- and compared with the single-launch fused step, which the oracle checks
elsewhere. Last, the layer over a real NCCL group (world size 1) runs end to end.
"""
import os
import socket

import numpy as np
import pytest
import torch

import ulysses_sequence_seq_gb300 as usp
from oracle import relayout
from tests.gpu_util import dev_bf16, f64, host_bits, needs_gpu
from ulysses_sequence_seq_gb300 import _lib
from ulysses_sequence_seq_gb300.synth import (bf16_bits_to_f32, custom_workload, f32_to_bf16_bits,
                                              seq_sharded_bits)

pytestmark = pytest.mark.gpu


def rand_bits(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("sp,S,H,D,head0,nh", [(4, 300, 8, 128, 0, 2), (4, 300, 8, 128, 1, 1), (2, 129, 4, 64, 0, 2),
                                               (8, 16, 32, 128, 2, 2), (8, 40, 2, 128, 0, 1), (4, 33, 1, 64, 0, 1)])
def test_pack_matches_oracle(sp, S, H, D, head0, nh):
    needs_gpu()
    x = rand_bits((S, H, D), seed=S + H)
    out = torch.full((sp, S, nh, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    _lib.a2a_pack(dev_bf16(x), out, sp, head0, nh)
    assert np.array_equal(host_bits(out), relayout.a2a_pack(x, sp, head0, nh))


@pytest.mark.parametrize("sp,S,H,D,head0,nh", [(4, 300, 8, 128, 0, 2), (4, 300, 8, 128, 1, 1), (8, 16, 32, 128, 2, 2)])
def test_unpack_matches_oracle_and_leaves_other_heads(sp, S, H, D, head0, nh):
    needs_gpu()
    recv = rand_bits((sp, S, nh, D), seed=7 * S)
    base = rand_bits((S, H, D), seed=11 * S)
    out = dev_bf16(base)
    _lib.a2a_unpack(dev_bf16(recv), out, sp, head0, nh)
    assert np.array_equal(host_bits(out), relayout.a2a_unpack(recv, sp, H, head0, nh, out=base.copy()))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("sp,H", [(8, 2), (4, 1), (8, 4)])
def test_unpack_sums_replicas(dtype, sp, H):
    """Fewer heads than ranks: the replicas' gradients are summed (fp32 in rank order,
    rounded once; exact here, so bit for bit with the float64 sum rounded the same way)."""
    needs_gpu()
    S, D = 96, 128
    rng = np.random.default_rng(sp * 10 + H)
    g = rng.standard_normal((sp, S, 1, D)).astype(np.float32)
    if dtype == torch.bfloat16:
        gb = f32_to_bf16_bits(g)
        recv = dev_bf16(gb)
        want = f32_to_bf16_bits(relayout.a2a_unpack(bf16_bits_to_f32(gb), sp, H).astype(np.float32))
    else:
        recv = torch.from_numpy(g).cuda()
        want = relayout.a2a_unpack(g, sp, H)
    out = torch.full((S, H, D), float("nan"), dtype=dtype, device="cuda")
    _lib.a2a_unpack(recv, out, sp)
    if dtype == torch.bfloat16:
        assert np.array_equal(host_bits(out), want)
    else:
        assert np.allclose(out.cpu().numpy(), want, rtol=0, atol=1e-6)


def test_a2a_validation():
    needs_gpu()
    z = torch.zeros(16, 6, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(usp.UspError):
        _lib.a2a_pack(z, o, 4, 0, 1)            # 6 heads neither divide over 4 ranks nor divide 4
    z8 = torch.zeros(16, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(usp.UspError):
        _lib.a2a_pack(z8, o, 4, 2, 1)           # chunk past the rank's 2 heads
    with pytest.raises(usp.UspError):
        _lib.a2a_unpack(o.half(), torch.zeros(16, 2, 64, dtype=torch.float16, device="cuda"), 4)   # fp16 sum


def _simulated_exchange(sends):
    """The collective's data movement for sp simulated ranks: recv_r[r'] = send_{r'}[r]."""
    sp = len(sends)
    return [torch.stack([sends[src][r] for src in range(sp)]) for r in range(sp)]


def test_step_through_the_exchange_equals_the_fused_step():
    """Per simulated rank: pack Q, K, V, exchange, fused attention on the received
    token-major heads (sp = 1, one rank's heads), exchange back, unpack. The output must
    be bit-identical to the all-ranks fused forward; the gradients match it within the
    dQ reduction-order tolerance."""
    needs_gpu()
    w = custom_workload("exch", [700, 1, 300, 1047], sp=4, hq=8, hkv=4, head_dim=128, index=24)
    T, S, sp, D = w.total_tokens, w.total_tokens // 4, 4, 128
    xs = {t: dev_bf16(seq_sharded_bits(w, t)).view(T, -1, D) for t in ("q", "k", "v", "do")}
    cu = torch.from_numpy(w.cu_seqlens()).cuda()
    ref = usp.UlyssesAttention(T, w.num_seqs, w.hq, w.hkv, D, sp, grad_dtype=torch.float32)
    o_ref = ref.forward(xs["q"], xs["k"], xs["v"], cu).clone()
    g_ref = [g.clone() for g in ref.backward(xs["do"], cu)]

    def to_heads(x):
        H = x.shape[1]
        sends = []
        for r in range(sp):
            buf = torch.empty(sp, S, H // sp, D, dtype=x.dtype, device="cuda")
            _lib.a2a_pack(x[r * S:(r + 1) * S].contiguous(), buf, sp)
            sends.append(buf)
        return [recv.view(T, H // sp, D) for recv in _simulated_exchange(sends)]

    def to_seq(ys, H, dtype):
        back = _simulated_exchange([y.view(sp, S, -1, D) for y in ys])
        out = torch.empty(T, H, D, dtype=dtype, device="cuda")
        for r in range(sp):
            shard = torch.empty(S, H, D, dtype=dtype, device="cuda")
            _lib.a2a_unpack(back[r].contiguous(), shard, sp)
            out[r * S:(r + 1) * S] = shard
        return out

    q, k, v, do = (to_heads(xs[t]) for t in ("q", "k", "v", "do"))
    hl, hkvl = w.hq // sp, w.hkv // sp
    os_, gq, gk, gv = [], [], [], []
    for r in range(sp):
        layer = usp.UlyssesAttention(T, w.num_seqs, hl, hkvl, D, 1, grad_dtype=torch.float32)
        os_.append(layer.forward(q[r], k[r], v[r], cu).clone())
        a, b, c = layer.backward(do[r], cu)
        gq.append(a.clone())
        gk.append(b.clone())
        gv.append(c.clone())
    o = to_seq(os_, w.hq, torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(o), host_bits(o_ref))
    for got, want in zip((to_seq(gq, w.hq, torch.float32), to_seq(gk, w.hkv, torch.float32),
                          to_seq(gv, w.hkv, torch.float32)), g_ref):
        assert (got - want).abs().max().item() <= 1e-3


def test_sp_layer_over_a_real_process_group():
    """UlyssesSPAttention on an NCCL group of one rank, its heads in two chunks (the
    overlap path): equals the single-device fused layer."""
    needs_gpu()
    import torch.distributed as dist
    from ulysses_sequence_seq_gb300.sp_exchange import UlyssesSPAttention
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        w = custom_workload("splayer", [500, 268], sp=1, hq=4, hkv=2, head_dim=128, index=25)
        T, D = w.total_tokens, 128
        xs = {t: dev_bf16(seq_sharded_bits(w, t)).view(T, -1, D) for t in ("q", "k", "v", "do")}
        cu = torch.from_numpy(w.cu_seqlens()).cuda()
        layer = UlyssesSPAttention(T, w.num_seqs, w.hq, w.hkv, D, chunks=2, grad_dtype=torch.float32)
        o = layer.forward(xs["q"], xs["k"], xs["v"], cu)
        g = layer.backward(xs["do"])
        ref = usp.UlyssesAttention(T, w.num_seqs, w.hq, w.hkv, D, 1, grad_dtype=torch.float32)
        o_ref = ref.forward(xs["q"], xs["k"], xs["v"], cu)
        g_ref = ref.backward(xs["do"], cu)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(o), host_bits(o_ref))
        for a, b in zip(g, g_ref):
            assert (a - b).abs().max().item() <= 1e-3
    finally:
        dist.destroy_process_group()
