"""A whole fused Ulysses attention step (forward and backward through UlyssesAttention) captured
once into a CUDA graph and replayed with new inputs copied into the same buffers. Every call
rewrites its workspace header on the device and launches on the caller's stream with no host
synchronisation, so the calls are capturable, including the programmatic-dependent launches
between a call's kernels and the forward's cluster launch. Each replay must give what direct
calls give on the same inputs: O and LSE, dK and dV bitwise, dQ within 1e-6 of its largest
magnitude (its partial sums arrive in any order)."""
import numpy as np
import pytest
import torch

import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import dev_bf16, needs_gpu
from ulysses_sequence_seq_gb300.synth import custom_workload, seq_sharded_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_graph_replay_matches_direct_calls(D):
    needs_gpu()
    base = custom_workload("graph", [700, 300, 56], sp=2, hq=4, hkv=2, head_dim=D, index=70)
    T = base.total_tokens
    cu = torch.from_numpy(base.cu_seqlens()).cuda()
    layer = usp.UlyssesAttention(T, base.num_seqs, 4, 2, D, 2, causal=True, grad_dtype=torch.float32)
    inputs = []
    for n in range(3):   # three draws of the same shapes
        w = custom_workload("graph", [700, 300, 56], sp=2, hq=4, hkv=2, head_dim=D, index=71 + n)
        inputs.append([dev_bf16(seq_sharded_bits(w, t)) for t in ("q", "k", "v", "do")])
    static = [x.clone() for x in inputs[0]]

    def step():
        o = layer.forward(static[0], static[1], static[2], cu)
        dq, dk, dv = layer.backward(static[3], cu)
        return o, layer.lse, dq, dk, dv

    # direct calls (also the warm-up that sets up the kernels before the capture)
    want = []
    for x in inputs:
        for s, src in zip(static, x):
            s.copy_(src)
        want.append([t.clone() for t in step()])
    torch.cuda.synchronize()
    assert layer.device_status() == usp.USP_OK

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                 # one more warm-up on the capture's stream
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(g):
        outs = step()
    for n in (2, 0, 1):
        for s, src in zip(static, inputs[n]):
            s.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert layer.device_status() == usp.USP_OK
        o, lse, dq, dk, dv = outs
        wo, wl, wq, wk, wv = want[n]
        assert torch.equal(o.view(torch.int16), wo.view(torch.int16)) and torch.equal(lse, wl)
        assert torch.equal(dk.view(torch.int32), wk.view(torch.int32))
        assert torch.equal(dv.view(torch.int32), wv.view(torch.int32))
        assert float((dq - wq).abs().max()) <= 1e-6 * float(wq.abs().max())
