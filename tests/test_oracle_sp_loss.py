"""Pins for oracle/sp_loss.py (CPU only): each check comes from the definition or from a
property the pages state, computed another way than the oracle computes it."""
import math

import numpy as np
import pytest

from oracle import sp_loss
from ulysses_sequence_seq_gb300.synth import packed_labels, packed_lengths


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


@pytest.mark.parametrize("lengths", [[6], [3, 1, 2], [1, 1, 1, 1], [5, 0, 4, 0], [129, 7, 300]])
def test_position_ids_are_offsets_in_sample(lengths):
    cu = _cu(lengths)
    T = int(cu[-1])
    want = np.arange(T) - np.repeat(cu[:-1], lengths)
    got = sp_loss.position_ids_from_cu_seqlens(cu, T)
    assert np.array_equal(got, want)


def test_position_ids_worked_example():
    # three packed samples of 3, 1 and 2 tokens
    pos = sp_loss.position_ids_from_cu_seqlens([0, 3, 4, 6], 6)
    assert pos.tolist() == [0, 1, 2, 0, 0, 1]
    assert sp_loss.cu_seqlens_from_position_ids(pos).tolist() == [0, 3, 4, 6]


def test_cu_round_trip_drops_only_empty_samples():
    rng = np.random.default_rng(5)
    for _ in range(20):
        lengths = rng.integers(0, 40, size=rng.integers(1, 12))
        if lengths.sum() == 0:
            continue
        cu = _cu(lengths)
        back = sp_loss.cu_seqlens_from_position_ids(sp_loss.position_ids_from_cu_seqlens(cu, int(cu[-1])))
        assert back.tolist() == sorted(set(cu.tolist()))
        starts = np.flatnonzero(sp_loss.position_ids_from_cu_seqlens(cu, int(cu[-1])) == 0)
        assert back[:-1].tolist() == starts.tolist()


@pytest.mark.parametrize("bad", [[1, 2, 3], [0, 1, 3], [0, 1, 1], [0, 2], [0, -1]])
def test_malformed_position_ids_raise(bad):
    with pytest.raises(ValueError):
        sp_loss.cu_seqlens_from_position_ids(bad)


def test_empty_row():
    assert sp_loss.cu_seqlens_from_position_ids([]).tolist() == [0]


def test_shift_labels_by_row_shift_and_boundary_mask():
    rng = np.random.default_rng(7)
    lengths = [5, 1, 9, 3]
    cu = _cu(lengths)
    labels = rng.integers(0, 32000, size=int(cu[-1]))
    labels[rng.random(len(labels)) < 0.3] = -100
    # whole-row shift, then the last token of every sample cannot predict anything
    want = np.concatenate([labels[1:], [-100]])
    want[cu[1:] - 1] = -100
    assert np.array_equal(sp_loss.shift_labels(labels, cu), want)


def test_shift_matches_row_shift_when_first_labels_are_ignored():
    """With the first label of every sample already -100 (the usual packed-sample collator),
    the per-sample shift and a plain shift of the whole row agree."""
    rng = np.random.default_rng(8)
    lengths = [4, 7, 2, 6]
    cu = _cu(lengths)
    labels = rng.integers(0, 100, size=int(cu[-1]))
    labels[cu[:-1]] = -100
    row = np.concatenate([labels[1:], [-100]])
    assert np.array_equal(sp_loss.shift_labels(labels, cu), row)


def test_good_tokens_count_by_sample():
    rng = np.random.default_rng(9)
    lengths = [10, 3, 19]
    cu = _cu(lengths)
    labels = rng.integers(0, 50, size=int(cu[-1]))
    labels[rng.random(len(labels)) < 0.5] = -100
    sh = sp_loss.shift_labels(labels, cu)
    good = sp_loss.good_tokens(sh, 4)
    # total: per sample, the labels at positions 1..L-1 that are not ignored
    total = sum(int(np.count_nonzero(labels[cu[b] + 1:cu[b + 1]] != -100)) for b in range(len(lengths)))
    assert int(good.sum()) == total
    per = [sum(1 for t in range(r * 8, r * 8 + 8) if sh[t] != -100) for r in range(4)]
    assert good.tolist() == per


def test_weighted_loss_is_global_mean():
    """The weighted aggregation equals the mean over all good tokens of the whole batch."""
    rng = np.random.default_rng(11)
    T, sp = 64, 4
    cu = _cu([20, 30, 14])
    labels = rng.integers(0, 10, size=T)
    labels[:24] = -100                                  # rank 0 all prompt, rank 1 half
    sh = sp_loss.shift_labels(labels, cu)
    tok = rng.random(T) * 5
    good = sp_loss.good_tokens(sh, sp)
    assert good[0] == 0 and len(set(good.tolist())) > 2
    rl = sp_loss.rank_mean_loss(tok, sh, sp)
    assert math.isnan(rl[0])
    got = sp_loss.sp_weighted_loss(rl, good)
    want = tok[sh != -100].mean()
    assert abs(got - want) <= 1e-12 * abs(want)
    # the plain mean of the ranks' losses differs once good counts differ
    assert abs(np.nanmean(rl) - want) > 1e-3


def test_weighted_loss_no_good_tokens():
    assert sp_loss.sp_weighted_loss([float("nan")] * 3, [0, 0, 0]) == 0.0


def test_weighted_loss_single_rank_is_its_loss():
    assert sp_loss.sp_weighted_loss([2.5], [7]) == 2.5


def test_synthetic_labels_recipe():
    """The seeded label generator: prompt spans at the start of samples, vocab range."""
    lengths = packed_lengths(4096, 3, lambda r: int(r.integers(64, 2048)))
    cu = _cu(lengths)
    lab = packed_labels(cu, vocab=32000, seed=4)
    assert lab.dtype == np.int64 and len(lab) == 4096
    assert ((lab == -100) | ((lab >= 0) & (lab < 32000))).all()
    assert all(lab[c] == -100 for c in cu[:-1])
