"""GPU parity of the sample and loss bookkeeping (position_ids <-> cu_seqlens, label shift
with good-token counts, weighted SP loss) against oracle/sp_loss.py. Integer results are
compared bit for bit; the loss within one float32 rounding of the float64 oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import sp_loss as ref
import ulysses_sequence_seq_gb300 as usp
from ulysses_sequence_seq_gb300._lib import USP_ERR_DEVICE_CHECK
from tests.gpu_util import dev_bf16, host_bits, needs_gpu
from ulysses_sequence_seq_gb300.synth import (WORKLOADS, custom_workload, head_sharded_bits, packed_labels,
                                              token_losses)

pytestmark = pytest.mark.gpu

SENTINEL = -7


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def pos_to_cu(pos, max_seqs):
    T = len(pos)
    ws_bytes = usp.position_ids_workspace_size(T)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    cu = torch.full((max_seqs + 1,), SENTINEL, dtype=torch.int32, device="cuda")
    n = torch.full((1,), SENTINEL, dtype=torch.int32, device="cuda")
    usp.position_ids_to_cu_seqlens(_dev(pos, torch.int64) if T else torch.empty(0, dtype=torch.int64, device="cuda"),
                                   T, cu, max_seqs, n, ws, ws_bytes)
    status = usp.get_device_status(ws)
    return cu.cpu().numpy(), int(n.item()), status


CASES = {
    "one": [300],
    "chunk_edges": [2047, 1, 1, 2049, 2048, 4096],      # starts right at 2048-token chunk edges
    "singles": [1] * 700,
    "ragged": [1, 7, 129, 163, 1, 255, 3000],
}


@pytest.mark.parametrize("name", list(CASES) + ["tiny", "llama", "packed", "gqa", "long"])
def test_position_ids_to_cu_seqlens(name):
    needs_gpu()
    if name in CASES:
        lengths = CASES[name]
        cu_true = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    else:
        cu_true = WORKLOADS[name].cu_seqlens()
    T = int(cu_true[-1])
    pos = ref.position_ids_from_cu_seqlens(cu_true, T)
    want = ref.cu_seqlens_from_position_ids(pos)
    n_true = len(want) - 1
    for max_seqs in (n_true, n_true + 5):
        cu, n, status = pos_to_cu(pos, max_seqs)
        assert status == usp.USP_OK and n == n_true
        assert np.array_equal(cu[:n_true + 1], want)
        assert (cu[n_true + 1:] == T).all()


def test_position_ids_empty_samples_vanish():
    needs_gpu()
    cu_true = np.array([0, 5, 5, 9, 9, 9, 20], dtype=np.int32)
    pos = ref.position_ids_from_cu_seqlens(cu_true, 20)
    cu, n, status = pos_to_cu(pos, 8)
    assert status == 0 and n == 3
    assert cu.tolist() == [0, 5, 9, 20, 20, 20, 20, 20, 20]


@pytest.mark.parametrize("bad_at", [0, 1, 2047, 2048, 5000])
def test_position_ids_malformed(bad_at):
    needs_gpu()
    pos = ref.position_ids_from_cu_seqlens([0, 3000, 6000], 6000)
    pos[bad_at] += 5
    with pytest.raises(ValueError):
        ref.cu_seqlens_from_position_ids(pos)
    cu, n, status = pos_to_cu(pos, 4)
    assert status == USP_ERR_DEVICE_CHECK
    assert (cu == SENTINEL).all() and n == SENTINEL


def test_position_ids_too_many_samples():
    needs_gpu()
    pos = ref.position_ids_from_cu_seqlens(np.arange(0, 101, dtype=np.int32), 100)   # 100 one-token samples
    cu, n, status = pos_to_cu(pos, 64)
    assert status == USP_ERR_DEVICE_CHECK and n == 100 and (cu == SENTINEL).all()


def test_position_ids_zero_tokens():
    needs_gpu()
    cu, n, status = pos_to_cu(np.zeros(0, dtype=np.int64), 3)
    assert status == 0 and n == 0 and cu.tolist() == [0, 0, 0, 0]


def test_position_ids_rejects_bad_args():
    needs_gpu()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pos = torch.zeros(16, dtype=torch.int64, device="cuda")
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(usp.UspError):
        usp.position_ids_to_cu_seqlens(pos, 16, cu, 0, None, ws, 4096)        # max_seqs < 1
    with pytest.raises(usp.UspError):
        usp.position_ids_to_cu_seqlens(pos, 16, cu, 3, None, ws, 16)          # workspace too small
    with pytest.raises(usp.UspError):
        usp.position_ids_to_cu_seqlens(pos.data_ptr() + 4, 16, cu, 3, None, ws, 4096)  # misaligned


def test_padded_cu_feeds_attention_without_host_sync():
    """cu_seqlens built on the device (padded with empty samples up to max_seqs) drives the
    forward to the same bits as the exact cu_seqlens."""
    needs_gpu()
    w = custom_workload("pos_pad", [1, 7, 129, 163, 1, 255], sp=2, hq=4, hkv=2, head_dim=128, index=31)
    T, cu_true = w.total_tokens, w.cu_seqlens()
    pos = _dev(ref.position_ids_from_cu_seqlens(cu_true, T), torch.int64)
    max_seqs = 16
    ws_p = torch.zeros(usp.position_ids_workspace_size(T), dtype=torch.uint8, device="cuda")
    cu_dev = torch.empty(max_seqs + 1, dtype=torch.int32, device="cuda")
    usp.position_ids_to_cu_seqlens(pos, T, cu_dev, max_seqs, None, ws_p, ws_p.numel())
    q, k, v = (dev_bf16(head_sharded_bits(w, t)) for t in ("q", "k", "v"))
    outs = []
    for cu, B in ((cu_dev, max_seqs), (torch.from_numpy(cu_true).cuda(), w.num_seqs)):
        o = torch.empty(w.hq, T, w.head_dim, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.hq, T, dtype=torch.float32, device="cuda")
        wsb = usp.attn_workspace_size(T, B, w.hq, w.hkv, w.head_dim, False)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        usp.attn_fwd_varlen(q, k, v, o, lse, cu, B, T, w.hq, w.hkv, w.head_dim, 0.0, True, ws, wsb)
        assert usp.get_device_status(ws) == 0
        outs.append((host_bits(o), lse.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert usp.get_device_status(ws_p) == 0


@pytest.mark.parametrize("name", ["ragged", "singles", "tiny", "packed", "long"])
def test_cu_seqlens_to_position_ids(name):
    needs_gpu()
    if name in CASES:
        cu = np.concatenate([[0], np.cumsum(CASES[name])]).astype(np.int32)
    else:
        cu = WORKLOADS[name].cu_seqlens()
    cu = np.concatenate([cu[:2], cu[1:2], cu[1:], cu[-1:]]).astype(np.int32)   # empty samples too
    T = int(cu[-1])
    out = torch.full((T,), SENTINEL, dtype=torch.int64, device="cuda")
    usp.cu_seqlens_to_position_ids(_dev(cu, torch.int32), len(cu) - 1, T, out)
    assert np.array_equal(out.cpu().numpy(), ref.position_ids_from_cu_seqlens(cu, T))


@pytest.mark.parametrize("name,sp", [("tiny", 2), ("llama", 4), ("packed", 8), ("gqa", 8), ("odd", 6)])
def test_shift_labels_and_good_tokens(name, sp):
    needs_gpu()
    if name == "odd":   # shards of 37 tokens: warps straddle rank boundaries
        cu = np.array([0, 50, 51, 130, 222], dtype=np.int32)
    else:
        cu = WORKLOADS[name].cu_seqlens()
    T = int(cu[-1])
    lab = packed_labels(cu, vocab=32000, seed=40 + sp)
    shifted = torch.full((T,), SENTINEL, dtype=torch.int64, device="cuda")
    good = torch.full((sp,), SENTINEL, dtype=torch.int64, device="cuda")
    usp.shift_labels(_dev(lab, torch.int64), _dev(cu, torch.int32), len(cu) - 1, T, sp, shifted, good)
    want = ref.shift_labels(lab, cu)
    assert np.array_equal(shifted.cpu().numpy(), want)
    assert np.array_equal(good.cpu().numpy(), ref.good_tokens(want, sp))


def test_shift_labels_rejects_in_place_and_bad_sp():
    needs_gpu()
    lab = torch.zeros(64, dtype=torch.int64, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    good = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(usp.UspError):
        usp.shift_labels(lab, cu, 1, 64, 4, lab, good)
    with pytest.raises(usp.UspError):
        usp.shift_labels(lab, cu, 1, 64, 3, torch.empty_like(lab), good)


def _f32_close(got, want):
    return got == np.float32(want) or abs(got - want) <= 2.0 ** -23 * abs(want)


@pytest.mark.parametrize("sp", [1, 2, 8, 33, 1000])
def test_sp_weighted_loss(sp):
    needs_gpu()
    rng = np.random.default_rng(sp)
    good = rng.integers(0, 5000, size=sp).astype(np.int64)
    good[rng.random(sp) < 0.3] = 0
    loss = (rng.random(sp) * 8).astype(np.float32)
    loss[good == 0] = np.nan                     # a mean over no token
    out = torch.full((), float(SENTINEL), dtype=torch.float32, device="cuda")
    usp.sp_weighted_loss(_dev(loss, torch.float32), _dev(good, torch.int64), sp, out)
    got = float(out.item())
    want = ref.sp_weighted_loss(loss.astype(np.float64), good)
    assert math.isfinite(got) and _f32_close(got, want)


def test_sp_weighted_loss_no_good_tokens():
    needs_gpu()
    out = torch.full((), 1.0, dtype=torch.float32, device="cuda")
    usp.sp_weighted_loss(torch.full((4,), float("nan"), device="cuda"), torch.zeros(4, dtype=torch.int64,
                                                                                   device="cuda"), 4, out)
    assert out.item() == 0.0


def test_group_loss_equals_global_token_mean():
    """Labels -> shifted labels and good counts (device) -> each simulated rank's own mean
    loss -> weighted loss (device) equals the mean over every good token of the batch."""
    needs_gpu()
    w = WORKLOADS["packed"]
    cu, T, sp = w.cu_seqlens(), w.total_tokens, w.sp
    lab = packed_labels(cu, vocab=32000, seed=77)
    lab[: T // sp + 5] = -100                                # rank 0 prompt only
    tok = token_losses(T, seed=78)
    shifted = torch.empty(T, dtype=torch.int64, device="cuda")
    good = torch.empty(sp, dtype=torch.int64, device="cuda")
    usp.shift_labels(_dev(lab, torch.int64), _dev(cu, torch.int32), len(cu) - 1, T, sp, shifted, good)
    sh_ref = ref.shift_labels(lab, cu)
    rank_loss = ref.rank_mean_loss(tok, sh_ref, sp).astype(np.float32)   # each rank's own loss (input)
    out = torch.empty((), dtype=torch.float32, device="cuda")
    usp.sp_weighted_loss(_dev(rank_loss, torch.float32), good, sp, out)
    g = good.cpu().numpy()
    assert g[0] == 0
    want = tok.astype(np.float64)[sh_ref != -100].mean()
    assert abs(out.item() - want) <= 1e-6 * want
