"""usp_attn_fwd_varlen_noalloc: the forward for callers that cannot allocate device
memory (code under a framework-owned allocator, fixed-budget real-time hosts,
plug-in code with no allocator handle).

Its scratch is a static array inside the library, so it takes no workspace. Each
call is compared with the workspace-taking entry point on the same inputs, within
the forward tolerances of the other tests, for two different problems called one
after the other (the second call finds the first call's leftovers in the array).
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import ulysses_sequence_seq_gb300 as usp
from tests.gpu_util import Problem, f64, needs_gpu
from ulysses_sequence_seq_gb300 import _lib
from ulysses_sequence_seq_gb300.synth import custom_workload, head_sharded_bits

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


def problem(lengths, hq, hkv, D, index):
    w = custom_workload("noalloc", lengths, sp=1, hq=hq, hkv=hkv, head_dim=D, index=index)
    return Problem(head_sharded_bits(w, "q"), head_sharded_bits(w, "k"), head_sharded_bits(w, "v"),
                   w.cu_seqlens(), True)


def run_noalloc(p):
    o = torch.full((p.hq, p.T, p.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.hq, p.T), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = _lib.load().usp_attn_fwd_varlen_noalloc(
        p.q.data_ptr(), p.k.data_ptr(), p.v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), p.cu.data_ptr(), p.B, p.T, p.hq, p.hkv, p.D, 0.0, 1, status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.USP_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    return o, lse, int(status.item())


def test_noalloc_matches_workspace_entry_point_twice():
    needs_gpu()
    first = problem([700, 1, 300, 1047], hq=8, hkv=2, D=128, index=21)
    second = problem([129, 64], hq=4, hkv=4, D=64, index=22)
    for p in (first, second):
        o_ref, lse_ref, st_ref = p.forward()
        o, lse, st = run_noalloc(p)
        assert st_ref == 0 and st == 0
        assert np.abs(f64(o) - f64(o_ref)).max() <= O_TOL
        assert np.abs(f64(lse) - f64(lse_ref)).max() <= LSE_TOL


def test_noalloc_reports_bad_cu_seqlens_and_rejects_oversize():
    needs_gpu()
    p = problem([256, 256], hq=2, hkv=2, D=128, index=23)
    p.cu = torch.tensor([0, 300, 200], dtype=torch.int32, device="cuda")   # decreasing offsets
    o, lse, st = run_noalloc(p)
    assert st == _lib.USP_ERR_DEVICE_CHECK
    assert torch.isnan(o.float()).all()
    # a work list larger than the static array is refused on the host, before any launch
    with pytest.raises(usp.UspError) as e:
        _lib.attn_fwd_varlen_noalloc(p.q, p.k, p.v, o, lse, p.cu, 1, 1 << 22, 512, 512, 128, 0.0, True)
    assert e.value.code == _lib.USP_ERR_WORKSPACE


def test_noalloc_host_checks_match_the_workspace_entry_point():
    """Sizes the workspace entry point refuses on the host are refused here too, before any
    launch (no scheduler run with a truncated work-list size), and more than 2^30 tokens is
    a scratch-size refusal. Only host checks run: every pointer is a dummy aligned address."""
    needs_gpu()
    fake = 1 << 20
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    # hq * (T / 128 + num_seqs + 1) beyond what the work list can index
    rc = lib.usp_attn_fwd_varlen_noalloc(fake, fake, fake, fake, fake, fake, 1, 1 << 28, 1 << 14, 1, 128, 0.0, 1,
                                         None, stream)
    assert rc == _lib.USP_ERR_UNSUPPORTED
    rc_ws = lib.usp_attn_fwd_varlen(fake, fake, fake, fake, None, fake, fake, 1, 1 << 28, 1 << 14, 1, 128, 0.0, 1,
                                    fake, 1 << 40, stream)
    assert rc_ws == rc
    # more than 2^30 tokens: beyond the static array whatever the heads
    rc = lib.usp_attn_fwd_varlen_noalloc(fake, fake, fake, fake, fake, fake, 1, (1 << 30) + 8, 1, 1, 128, 0.0, 1,
                                         None, stream)
    assert rc == _lib.USP_ERR_WORKSPACE
