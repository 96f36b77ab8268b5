"""Sample boundaries, label shift and the weighted loss across sequence-parallel ranks.

TEST INFRASTRUCTURE ONLY.

These are the bookkeeping steps around the attention of Ulysses sequence parallelism
that the HF Transformers "Ulysses sequence parallelism" guide (Portuguese mirror,
section on the Accelerate configuration file) lists: position_ids generation, the
label shift, and the aggregation of the loss over the SP ranks. The jianying88
article on DeepSpeed Ulysses in Transformers (section "3. 跨 rank 的加权 loss 聚合")
defines the aggregation: every rank gathers each rank's loss and its count of tokens
whose shifted label is not -100 ("good tokens"), the loss is the good-token weighted
mean of the rank losses, and ranks with no good token are left out.

Readings taken where the pages leave a step open:

* position_ids of packed samples count up from 0 inside each sample; a sample starts
  wherever the position id is 0. Any other step than +1 inside a sample is malformed.
* The shifted label of token t is the label of token t+1 when t+1 is in the same
  sample, else -100 (the last token of a sample has nothing to predict).
* The weighted mean over zero good tokens is 0 (a sum over an empty set), so a batch
  whose labels are all -100 gives a finite loss.

Plain Python loops over numpy arrays: a reader can check each line against the text.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def position_ids_from_cu_seqlens(cu_seqlens, total_tokens: int) -> np.ndarray:
    """position id of every token: its offset inside its own sample."""
    cu = [int(x) for x in cu_seqlens]
    pos = np.zeros(total_tokens, dtype=np.int64)
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1]):
            pos[t] = t - cu[b]
    return pos


def cu_seqlens_from_position_ids(position_ids) -> np.ndarray:
    """Sample boundaries [0, starts..., T] of a packed row; ValueError when malformed."""
    pos = [int(x) for x in position_ids]
    T = len(pos)
    starts = []
    for t in range(T):
        if pos[t] == 0:
            starts.append(t)
        elif t == 0 or pos[t] != pos[t - 1] + 1:
            raise ValueError(f"position id {pos[t]} at token {t} neither starts a sample nor follows "
                             f"{pos[t - 1] if t else 'nothing'}")
    return np.array(starts + [T] if T else [0], dtype=np.int32)


def shift_labels(labels, cu_seqlens) -> np.ndarray:
    """Label each token with the next token of its own sample; -100 at a sample's end."""
    lab = np.asarray(labels, dtype=np.int64)
    out = np.full(lab.shape, IGNORE_INDEX, dtype=np.int64)
    cu = [int(x) for x in cu_seqlens]
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1] - 1):
            out[t] = lab[t + 1]
    return out


def good_tokens(shifted, sp: int) -> np.ndarray:
    """Per SP rank (contiguous shards of T/sp tokens): tokens whose shifted label is not -100."""
    s = np.asarray(shifted)
    S = len(s) // sp
    return np.array([int(np.count_nonzero(s[r * S:(r + 1) * S] != IGNORE_INDEX)) for r in range(sp)],
                    dtype=np.int64)


def rank_mean_loss(token_loss, shifted, sp: int) -> np.ndarray:
    """Each rank's own loss: the mean of its tokens' losses over its good tokens (NaN if none)."""
    tl = np.asarray(token_loss, dtype=np.float64)
    s = np.asarray(shifted)
    S = len(s) // sp
    out = np.empty(sp, dtype=np.float64)
    for r in range(sp):
        keep = s[r * S:(r + 1) * S] != IGNORE_INDEX
        n = int(np.count_nonzero(keep))
        out[r] = tl[r * S:(r + 1) * S][keep].sum() / n if n else float("nan")
    return out


def sp_weighted_loss(rank_loss, good) -> float:
    """sum over ranks with good > 0 of loss_r * good_r, divided by the sum of good_r."""
    num = 0.0
    den = 0
    for loss_r, good_r in zip(rank_loss, good):
        if int(good_r) > 0:
            num += float(loss_r) * int(good_r)
            den += int(good_r)
    return num / den if den else 0.0
