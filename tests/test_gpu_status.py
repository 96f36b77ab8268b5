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
