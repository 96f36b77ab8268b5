"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and packs them; it holds none of the
attention or re-layout arithmetic, so the CUDA path and the CPU oracle can both
consume its output without sharing any of the method's code.

Workloads (shapes follow the pages' Llama-style layers: 32 heads, head dim 128,
4k-256k tokens, sp_size 2-8; DeepSpeed-Ulysses / ColossalAI "sequence
parallelism" pages, sections "Configurar" and "choose"):

* ``tiny``   one causal sequence of 256 tokens, sp=2, H=4, D=64.
* ``llama``  a random-token batch of 2 x 4096 tokens treated as one packed
  stream (cu_seqlens = {0, 4096, 8192}), sp=4, H=32, D=128.
* ``packed`` 65536 tokens of samples with lognormal(ln 4096, 1) lengths clipped
  to [128, 32768] and rounded up to a multiple of 8, sp=8, H=32, D=128.
* ``long``   one causal sequence of 262144 tokens, sp=8, H=32, D=128.
* ``gqa``    131072 tokens of samples with uniform[1024, 32768] lengths rounded
  up to a multiple of 8, sp=8, 32 query heads / 8 KV heads, D=128.

Activations are N(0, 1) float32 draws rounded to bf16 (round to nearest even)
and carried as raw uint16 bit patterns. Every head of every tensor has its own
generator, so one head can be drawn without drawing the others.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np

TENSORS = {"q": 0, "k": 1, "v": 2, "do": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # position in the workload list; seeds derive from it
    total_tokens: int     # T
    sp: int               # sp_size (simulated ranks)
    hq: int               # query heads (all ranks)
    hkv: int              # key/value heads (all ranks)
    head_dim: int         # D
    causal: bool = True
    lengths: tuple = field(default=())  # per-sample lengths, sum == T

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(len(self.lengths) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(np.asarray(self.lengths, dtype=np.int64))
        return cu

    def allowed_pairs(self) -> int:
        """Number of (query, key) pairs one head attends to (causal within a sample)."""
        if self.causal:
            return int(sum(L * (L + 1) // 2 for L in self.lengths))
        return int(sum(L * L for L in self.lengths))


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def packed_lengths(total: int, seed: int, draw, multiple: int = 8) -> List[int]:
    """Draw sample lengths until they cover ``total``; the last one is shortened.

    ``draw(rng)`` returns one raw length. Each is rounded up to ``multiple``;
    once the running sum reaches ``total`` the last sample is cut so the sum is
    exactly ``total`` (it stays a multiple of ``multiple`` when ``total`` is).
    """
    rng = np.random.default_rng(seed)
    out: List[int] = []
    acc = 0
    while acc < total:
        L = _round_up(int(draw(rng)), multiple)
        if acc + L >= total:
            L = total - acc
        out.append(L)
        acc += L
    return out


def _lognormal_len(rng) -> int:
    x = int(np.floor(rng.lognormal(mean=np.log(4096.0), sigma=1.0)))
    return min(max(x, 128), 32768)


def _uniform_len(rng) -> int:
    return int(rng.integers(1024, 32769))


def make_workloads() -> Dict[str, Workload]:
    w = {}
    w["tiny"] = Workload("tiny", 1, 256, 2, 4, 4, 64, True, (256,))
    w["llama"] = Workload("llama", 2, 8192, 4, 32, 32, 128, True, (4096, 4096))
    w["packed"] = Workload("packed", 3, 65536, 8, 32, 32, 128, True,
                           tuple(packed_lengths(65536, 1000 * 3 + 99, _lognormal_len)))
    w["long"] = Workload("long", 4, 262144, 8, 32, 32, 128, True, (262144,))
    w["gqa"] = Workload("gqa", 5, 131072, 8, 32, 8, 128, True,
                        tuple(packed_lengths(131072, 1000 * 5 + 99, _uniform_len)))
    return w


WORKLOADS = make_workloads()


def custom_workload(name: str, lengths, sp: int, hq: int, hkv: int, head_dim: int,
                    causal: bool = True, index: int = 9) -> Workload:
    lengths = tuple(int(x) for x in lengths)
    return Workload(name, index, int(sum(lengths)), sp, hq, hkv, head_dim, causal, lengths)


# ----------------------------------------------------------------------------- labels
def packed_labels(cu_seqlens, vocab: int = 32000, seed: int = 0, max_prompt_frac: float = 0.5) -> np.ndarray:
    """int64 labels of packed fine-tuning samples: each sample opens with a prompt span of
    -100 (at least its first token, up to ``max_prompt_frac`` of it), the rest are token ids
    drawn uniformly from [0, vocab)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = int(cu[-1])
    rng = np.random.default_rng(seed)
    lab = rng.integers(0, vocab, size=T, dtype=np.int64)
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        if L:
            prompt = 1 + int(rng.integers(0, max(1, int(L * max_prompt_frac))))
            lab[cu[b]:cu[b] + prompt] = -100
    return lab


def token_losses(T: int, seed: int = 0) -> np.ndarray:
    """float32 per-token losses (exponential, mean 2) standing in for a model's cross entropy."""
    return np.random.default_rng(seed).exponential(2.0, size=T).astype(np.float32)


# ----------------------------------------------------------------------------- bf16 packing
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE fp16 (numpy's conversion: nearest, ties to even) as uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_f16_bits(x) if dtype == "f16" else f32_to_bf16_bits(x)


# ----------------------------------------------------------------------------- activations
def head_bits(w: Workload, tensor: str, head: int, std: float = 1.0, dtype: str = "bf16") -> np.ndarray:
    """One head of one activation tensor: uint16 bits (bf16, or fp16 for dtype "f16") of
    the same N(0, std^2) float32 draws, shape [T][D]."""
    seed = 1000 * w.index + TENSORS[tensor]
    rng = np.random.default_rng([seed, head])
    x = rng.standard_normal((w.total_tokens, w.head_dim), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bits(x, dtype)


def num_heads(w: Workload, tensor: str) -> int:
    return w.hkv if tensor in ("k", "v") else w.hq


def head_sharded_bits(w: Workload, tensor: str, heads=None, dtype: str = "bf16") -> np.ndarray:
    """Head-sharded activation [H][T][D] (uint16 bits) for the listed heads."""
    if heads is None:
        heads = range(num_heads(w, tensor))
    heads = list(heads)
    out = np.empty((len(heads), w.total_tokens, w.head_dim), dtype=np.uint16)
    for i, h in enumerate(heads):
        out[i] = head_bits(w, tensor, h, dtype=dtype)
    return out


def seq_sharded_bits(w: Workload, tensor: str, dtype: str = "bf16") -> np.ndarray:
    """Seq-sharded activation [sp][T/sp][H][D] (uint16 bits): the same draws as
    :func:`head_sharded_bits`, stored token-major."""
    H = num_heads(w, tensor)
    out = np.empty((w.total_tokens, H, w.head_dim), dtype=np.uint16)
    for h in range(H):
        out[:, h, :] = head_bits(w, tensor, h, dtype=dtype)
    return out.reshape(w.sp, w.total_tokens // w.sp, H, w.head_dim)


def index_pattern_bits(T: int, H: int, D: int) -> np.ndarray:
    """A seq-sharded [T][H][D] uint16 array whose values encode their own position
    (used to check permutations exhaustively). Values are ((t*H + h)*D + d) mod 2^16."""
    return (np.arange(T * H * D, dtype=np.int64) % 65536).astype(np.uint16).reshape(T, H, D)


# ----------------------------------------------------------------------------- one rank's slice
def rank_slice(w: Workload) -> Workload:
    """Rank 0's share of ``w`` after the sequence -> heads exchange: all T tokens of its
    hq/sp query heads and max(1, hkv/sp) key/value heads (heads 0.. of ``w``, so the same
    draws), as a one-rank workload. Stacking what every peer sends it, in rank order, gives
    the token-major [T][hq/sp][D] buffer the fused attention reads."""
    from dataclasses import replace
    return replace(w, hq=w.hq // w.sp, hkv=max(1, w.hkv // w.sp), sp=1)
