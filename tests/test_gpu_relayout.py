"""GPU parity of the layout swap: bit-exact against the oracle's index formula."""
import numpy as np
import pytest
import torch

import ulysses_sequence_seq_gb300 as usp
from oracle import relayout
from tests.gpu_util import dev_bf16, host_bits, needs_gpu
from ulysses_sequence_seq_gb300.synth import WORKLOADS, seq_sharded_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,tensor", [("tiny", "q"), ("llama", "q"), ("packed", "k"), ("gqa", "q"),
                                         ("gqa", "v")])
def test_relayout_bit_exact(name, tensor):
    needs_gpu()
    w = WORKLOADS[name]
    x = seq_sharded_bits(w, tensor)                  # [sp][S][H][D]
    sp, H, D = w.sp, x.shape[2], x.shape[3]
    xd = dev_bf16(x)
    y = torch.empty(sp, H // sp, w.total_tokens, D, dtype=torch.bfloat16, device="cuda")
    usp.seq_to_head(xd, y, sp)
    want = relayout.seq_to_head(x, sp)
    assert np.array_equal(host_bits(y), want)
    back = torch.empty_like(xd)
    usp.head_to_seq(y, back, sp)
    assert np.array_equal(host_bits(back), x)


def test_relayout_long_sampled_and_round_trip():
    """262144 tokens x 32 heads x 128 (2 GiB per tensor): every element carries its own
    index; sampled outputs are checked against the formula, the round trip in full."""
    needs_gpu()
    w = WORKLOADS["long"]
    T, H, D, sp = w.total_tokens, w.hq, w.head_dim, w.sp
    x = (torch.arange(T * H * D, device="cuda", dtype=torch.int64) % 65521).to(torch.int16)
    x = x.view(torch.bfloat16).view(sp, T // sp, H, D)
    y = torch.empty(sp, H // sp, T, D, dtype=torch.bfloat16, device="cuda")
    usp.seq_to_head(x, y, sp)
    rng = np.random.default_rng(0)
    S, Hl = T // sp, H // sp
    idx = rng.integers(0, [sp, Hl, T, D], size=(4096, 4))
    ti = [torch.from_numpy(idx[:, c]).cuda() for c in range(4)]
    got = host_bits(y[ti[0], ti[1], ti[2], ti[3]])
    r, hl, t, d = idx.T
    want = ((t * H + (r * Hl + hl)) * D + d) % 65521   # the value stored at x[t//S][t%S][r*Hl+hl][d]
    assert np.array_equal(got.astype(np.int64), want.astype(np.int16).view(np.uint16).astype(np.int64))
    back = torch.empty_like(x)
    usp.head_to_seq(y, back, sp)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("sp", [1, 2, 4, 8, 16])
def test_relayout_fp32_and_every_sp(sp):
    needs_gpu()
    T, H, D = 160, 16, 64
    x = torch.randn(T, H, D, device="cuda", dtype=torch.float32)
    y = torch.empty(H, T, D, device="cuda", dtype=torch.float32)
    usp.seq_to_head(x, y, sp)
    # on one device the swap is the (token, head) transpose, whatever sp is
    assert torch.equal(y, x.transpose(0, 1))
    z = torch.empty_like(x)
    usp.head_to_seq(y, z, sp)
    assert torch.equal(z, x)


def test_relayout_rejects_on_host():
    needs_gpu()
    x = torch.zeros(64, 6, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(6, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(usp.UspError):
        usp.seq_to_head(x, y, 4)          # 6 heads, sp 4
    with pytest.raises(usp.UspError):
        usp.seq_to_head(x, x, 2)          # in == out
