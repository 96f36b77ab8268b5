"""Out-of-bounds writes, checked without a sanitizer: every output of the forward and the
backward (o, its rounding residual, LSE, dQ, dK, dV) lives inside a larger allocation with
4 KB canary regions in front of and behind it. After the calls the canaries must be intact
and the outputs must match the oracle. Ragged samples (a one-token one, tiles ending
mid-box) make the kernels' stores reach the tensors' ends, where TMA stores clip and
row-by-row stores check their rows."""
import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_seq_gb300 as usp
from ulysses_sequence_seq_gb300 import _lib
from tests.gpu_util import dev_bf16, f64, needs_gpu
from ulysses_sequence_seq_gb300.synth import custom_workload, head_sharded_bits

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096


def guarded(shape, dtype):
    """A tensor of `shape` inside a buffer with GUARD_BYTES of canary on both sides."""
    n = int(np.prod(shape))
    esz = torch.empty((), dtype=dtype).element_size()
    g = GUARD_BYTES // esz
    buf = torch.empty(n + 2 * g, dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(0xA5)
    return buf, buf[g:g + n].view(shape), g


def canaries_intact(buf, g):
    b = buf.view(torch.uint8)
    esz = buf.element_size()
    front, back = b[:g * esz], b[b.numel() - g * esz:]
    return bool((front == 0xA5).all()) and bool((back == 0xA5).all())


@pytest.mark.parametrize("D,grad_dtype", [(128, torch.float32), (128, torch.bfloat16), (64, torch.float32)])
def test_outputs_stay_inside_their_tensors(D, grad_dtype):
    needs_gpu()
    w = custom_workload("guard", [300, 129, 1, 270], sp=1, hq=4, hkv=2, head_dim=D, index=80)
    q, k, v, do = (head_sharded_bits(w, t) for t in ("q", "k", "v", "do"))
    T, hq, hkv = w.total_tokens, w.hq, w.hkv
    cu_host = w.cu_seqlens()
    cu = torch.from_numpy(cu_host).cuda()
    ws_bytes = max(usp.attn_workspace_size(T, w.num_seqs, hq, hkv, D, b) for b in (False, True))
    ws_buf, ws, wg = guarded((ws_bytes,), torch.uint8)
    o_buf, o, og = guarded((hq, T, D), torch.bfloat16)
    r_buf, ores, rg = guarded((hq, T, D), torch.bfloat16)
    l_buf, lse, lg = guarded((hq, T), torch.float32)
    dq_buf, dq, qg = guarded((hq, T, D), grad_dtype)
    dk_buf, dk, kg = guarded((hkv, T, D), grad_dtype)
    dv_buf, dv, vg = guarded((hkv, T, D), grad_dtype)
    dq_, dk_, dv_, ddo = (dev_bf16(x) for x in (q, k, v, do))
    usp.attn_fwd_varlen(dq_, dk_, dv_, o, lse, cu, w.num_seqs, T, hq, hkv, D, 0.0, True, ws, ws_bytes, o_res=ores)
    assert usp.get_device_status(ws) == usp.USP_OK
    gcode = usp.USP_FP32 if grad_dtype == torch.float32 else usp.USP_BF16
    usp.attn_bwd_varlen(dq_, dk_, dv_, o, lse, ddo, dq, dk, dv, gcode, cu, w.num_seqs, T, hq, hkv, D, 0.0, True, ws,
                        ws_bytes, o_res=ores)
    assert usp.get_device_status(ws) == usp.USP_OK
    torch.cuda.synchronize()
    for name, buf, g in (("workspace", ws_buf, wg), ("o", o_buf, og), ("o_res", r_buf, rg), ("lse", l_buf, lg),
                         ("dq", dq_buf, qg), ("dk", dk_buf, kg), ("dv", dv_buf, vg)):
        assert canaries_intact(buf, g), f"a write left {name}"
    ro, rl = oracle.attn_fwd(q, k, v, cu_host)
    assert np.abs(f64(o) + f64(ores) - ro).max() <= 1e-2
    assert np.abs(f64(lse) - rl).max() <= 1e-3
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, cu_host)
    for g_, r in ((dq, rq), (dk, rk), (dv, rv)):
        tol = 2e-2 if grad_dtype == torch.float32 else 2e-2 + np.abs(r) * 2.0 ** -8
        assert (np.abs(f64(g_) - r) <= tol).all()


@pytest.mark.parametrize("D", [128, 64])
def test_fused_outputs_stay_inside_their_tensors(D):
    """The same on the fused calls, whose stores go to the token-major [sp][T/sp][H][D] layout."""
    needs_gpu()
    from ulysses_sequence_seq_gb300.synth import seq_sharded_bits
    w = custom_workload("guardf", [300, 129, 1, 270], sp=2, hq=4, hkv=2, head_dim=D, index=81)
    T, hq, hkv, sp = w.total_tokens, w.hq, w.hkv, w.sp
    xs = [seq_sharded_bits(w, t) for t in ("q", "k", "v", "do")]
    cu_host = w.cu_seqlens()
    cu = torch.from_numpy(cu_host).cuda()
    ws_bytes = max(usp.attn_workspace_size(T, w.num_seqs, hq, hkv, D, b) for b in (False, True))
    ws_buf, ws, wg = guarded((ws_bytes,), torch.uint8)
    o_buf, o, og = guarded((sp, T // sp, hq, D), torch.bfloat16)
    r_buf, ores, rg = guarded((sp, T // sp, hq, D), torch.bfloat16)
    l_buf, lse, lg = guarded((hq, T), torch.float32)
    dq_buf, dq, qg = guarded((sp, T // sp, hq, D), torch.float32)
    dk_buf, dk, kg = guarded((sp, T // sp, hkv, D), torch.float32)
    dv_buf, dv, vg = guarded((sp, T // sp, hkv, D), torch.float32)
    xq, xk, xv, xdo = (dev_bf16(x) for x in xs)
    usp.ulysses_attn_fwd(xq, xk, xv, o, lse, cu, w.num_seqs, T, sp, hq, hkv, D, 0.0, True, ws, ws_bytes, o_res=ores)
    assert usp.get_device_status(ws) == usp.USP_OK
    usp.ulysses_attn_bwd(xq, xk, xv, o, lse, xdo, dq, dk, dv, usp.USP_FP32, cu, w.num_seqs, T, sp, hq, hkv, D, 0.0,
                         True, ws, ws_bytes, o_res=ores)
    assert usp.get_device_status(ws) == usp.USP_OK
    torch.cuda.synchronize()
    for name, buf, g in (("workspace", ws_buf, wg), ("o", o_buf, og), ("o_res", r_buf, rg), ("lse", l_buf, lg),
                         ("dq", dq_buf, qg), ("dk", dk_buf, kg), ("dv", dv_buf, vg)):
        assert canaries_intact(buf, g), f"a write left {name}"

    def heads(x):   # [sp][S][H][D] -> [H][T][D]
        return np.ascontiguousarray(np.asarray(x).reshape(T, -1, D).transpose(1, 0, 2))

    q, k, v, do = (heads(x) for x in xs)
    ro, _ = oracle.attn_fwd(q, k, v, cu_host)
    assert np.abs(heads(f64(o) + f64(ores)) - ro).max() <= 1e-2
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, cu_host)
    for g_, r in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(heads(f64(g_)) - r).max() <= 2e-2


def test_relayout_and_merge_outputs_stay_inside_their_tensors():
    """The stand-alone layout swaps (including the replicating key/value swap and its summing
    gradient), the rank-local halves of the exchange, and the ring-merge kernels, on sizes
    whose last rows end mid-warp: canaries intact, results as their inverses or oracles give."""
    needs_gpu()
    sp, T, H, HKV, D = 4, 4 * 37, 8, 2, 128
    rng = np.random.default_rng(83)
    x = torch.from_numpy(rng.integers(-30000, 30000, size=(sp, T // sp, H, D), dtype=np.int16)).cuda().view(torch.bfloat16)
    bh, h, gh = guarded((sp, H // sp, T, D), torch.bfloat16)
    usp.seq_to_head(x, h, sp)
    bs, back, gs = guarded((sp, T // sp, H, D), torch.bfloat16)
    usp.head_to_seq(h, back, sp)
    xk = torch.from_numpy(rng.integers(-30000, 30000, size=(sp, T // sp, HKV, D), dtype=np.int16)).cuda().view(torch.bfloat16)
    bk, hk, gk = guarded((max(sp, HKV), T, D), torch.bfloat16)
    usp.seq_to_head_kv(xk, hk, sp)
    bg, gsum, gg = guarded((sp, T // sp, HKV, D), torch.float32)
    usp.head_to_seq_kv_grad(hk.float(), gsum, sp, HKV)
    S = T // sp
    shard = x[0].contiguous()                                           # one rank's [S][H][D]
    bp, packed, gp = guarded((sp, S, H // sp, D), torch.bfloat16)
    _lib.a2a_pack(shard, packed, sp)
    bu, unpacked, gu = guarded((S, H, D), torch.bfloat16)
    _lib.a2a_unpack(packed, unpacked, sp)
    o_acc = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)).cuda()
    lse_acc = torch.from_numpy(rng.standard_normal((H, T)).astype(np.float32)).cuda()
    o_part = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    lse_part = torch.from_numpy(rng.standard_normal((H, T)).astype(np.float32)).cuda()
    _lib.lse_merge(o_acc, lse_acc, o_part, lse_part)
    bo, o16, go = guarded((T, H, D), torch.bfloat16)
    br, ores, gr = guarded((T, H, D), torch.bfloat16)
    _lib.o_finalize(o_acc, o16, ores)
    ba, acc, ga = guarded((T, H, D), torch.float32)
    acc.zero_()
    _lib.accumulate_f32(acc, o_acc)
    torch.cuda.synchronize()
    for name, buf, g in (("seq_to_head", bh, gh), ("head_to_seq", bs, gs), ("seq_to_head_kv", bk, gk),
                         ("head_to_seq_kv_grad", bg, gg), ("a2a_pack", bp, gp), ("a2a_unpack", bu, gu),
                         ("o_finalize o", bo, go), ("o_finalize residual", br, gr), ("accumulate_f32", ba, ga)):
        assert canaries_intact(buf, g), f"a write left {name}'s output"
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))   # the swaps are inverse permutations
    assert torch.equal(acc, o_acc)                                      # 0 + o_acc
    assert float((o16.float() + ores.float() - o_acc).abs().max()) <= 2.0 ** -14 * float(o_acc.abs().max()) + 1e-30
