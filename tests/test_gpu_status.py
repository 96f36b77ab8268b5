"""Device-side error reporting: a bounded wait that runs out is reported through the
status word and leaves the CUDA context usable (no trap, no hang)."""
import numpy as np
import pytest
import torch

import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import Problem, needs_gpu
from ulysses_sequence_seq_gb300.synth import custom_workload, head_sharded_bits

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    needs_gpu()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    usp.debug_wait_timeout(ws, ws.numel(), 50_000_000)          # 50 ms limit
    assert usp.get_device_status(ws) == 5                       # USP_ERR_TIMEOUT
    # the context still works: a small forward succeeds afterwards
    w = custom_workload("after", [256], sp=1, hq=2, hkv=2, head_dim=64, index=17)
    p = Problem(head_sharded_bits(w, "q"), head_sharded_bits(w, "k"), head_sharded_bits(w, "v"),
                w.cu_seqlens(), True)
    o, lse, status = p.forward()
    assert status == 0 and torch.isfinite(o.float()).all()


def test_workspace_header_is_rewritten_by_every_call():
    """The scheduler writes the call's status, item count and item counter itself: a
    workspace full of stale bytes, one left with a device-check error and one left with a
    timeout all give USP_OK and the results of a clean workspace on the next good call
    (bit for bit, except dQ, whose fp32 additions from different CTAs may come in another
    order)."""
    needs_gpu()
    w = custom_workload("reuse", [300, 129, 40], sp=1, hq=4, hkv=2, head_dim=128, index=18)
    q, k, v, do = (head_sharded_bits(w, t) for t in ("q", "k", "v", "do"))
    p = Problem(q, k, v, w.cu_seqlens(), True, do_bits=do)
    p.ws.zero_()
    o0, l0, st = p.forward()
    assert st == 0
    dq0, dk0, dv0, st = p.backward(o0, l0)
    assert st == 0

    def check():
        o, lse, st = p.forward()
        assert st == 0 and torch.equal(o.view(torch.int16), o0.view(torch.int16)) and torch.equal(lse, l0)
        dq, dk, dv, st = p.backward(o, lse)
        assert st == 0 and torch.equal(dk, dk0) and torch.equal(dv, dv0)
        assert (dq - dq0).abs().max().item() <= 1e-4

    p.ws.fill_(0xFF)                                    # stale counters and status
    check()
    good_cu = p.cu
    p.cu = torch.tensor([0, 200, 100, 469], dtype=torch.int32, device="cuda")   # decreasing offsets
    _, _, st = p.forward()
    assert st == 6                                      # USP_ERR_DEVICE_CHECK
    p.cu = good_cu
    check()
    usp.debug_wait_timeout(p.ws, p.ws.numel(), 20_000_000)
    assert usp.get_device_status(p.ws) == 5             # USP_ERR_TIMEOUT left in the header
    check()
