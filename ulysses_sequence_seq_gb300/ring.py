"""Ring-attention steps on top of the library's attention calls.

In ring attention every rank keeps one chunk of the queries while the key/value chunks
travel around the ring; at each step the rank attends its queries to the visiting chunk
and combines the partial result with what it has through the log-sum-exp; the backward
walks the ring again with the final output and log-sum-exp (ColossalAI sequence
parallelism tutorial, the ring-attention plugin set-up and its closing comparison of
Ulysses and ring attention).

Chunks are equal slices of one sequence in rank order (packed samples are split evenly,
so every chunk has the same chunk-local cu_seqlens). The causal mask on global positions
-- a query at q_rank*L + i sees a key at k_rank*L + j iff k_rank*L + j <= q_rank*L + i --
then makes a step unmasked for an earlier key chunk, causal for the query chunk's own
keys and empty for a later one (:func:`step_kind`). Each non-empty step is one fused
attention call on the token-major chunk; usp_lse_merge, usp_o_finalize and
usp_accumulate_f32 do the rest.
"""
from __future__ import annotations

import math

from . import _lib


def step_kind(q_rank: int, k_rank: int, causal: bool = True) -> str:
    """"full", "causal" or "none": what the causal mask on global positions leaves of the
    (query chunk q_rank, key chunk k_rank) block when both chunks have the same length."""
    if not causal or k_rank < q_rank:
        return "full"
    return "causal" if k_rank == q_rank else "none"


class RingAttention:
    """The steps of one rank: its query chunk of L tokens against visiting key/value chunks.

    Tensors are token-major chunks: q, dO [L][hq][D]; k, v [L][hkv][D] (bf16).
    ``forward_step`` / ``forward_end`` accumulate the output over the ring;
    ``backward_step`` returns this step's dK, dV shares (fp32, to travel back with the
    chunk) and accumulates dQ; ``backward_end`` returns dQ.
    """

    def __init__(self, chunk_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int, causal: bool = True,
                 softmax_scale: float = 0.0, device=None, dtype=None):
        import torch
        self.L, self.B, self.hq, self.hkv, self.D = chunk_tokens, num_seqs, hq, hkv, head_dim
        self.causal = causal
        self.scale = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(head_dim)
        self.dtype = dtype or torch.bfloat16
        dev = device or torch.device("cuda", torch.cuda.current_device())
        L, D = chunk_tokens, head_dim
        self.ws_bytes = max(_lib.attn_workspace_size(L, num_seqs, hq, hkv, D, b) for b in (False, True))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.o_part = torch.empty(L, hq, D, dtype=self.dtype, device=dev)
        self.o_part_res = torch.empty_like(self.o_part)
        self.lse_part = torch.empty(hq, L, dtype=torch.float32, device=dev)
        self.o_acc = torch.empty(L, hq, D, dtype=torch.float32, device=dev)
        self.lse = torch.empty(hq, L, dtype=torch.float32, device=dev)
        self.o = torch.empty(L, hq, D, dtype=self.dtype, device=dev)
        self.o_res = torch.empty_like(self.o)
        self.dq_acc = torch.empty(L, hq, D, dtype=torch.float32, device=dev)
        self.dq_part = torch.empty_like(self.dq_acc)
        self._steps = 0

    def forward_begin(self):
        self._steps = 0

    def forward_step(self, q, k, v, cu_seqlens, q_rank: int, k_rank: int):
        kind = step_kind(q_rank, k_rank, self.causal)
        if kind == "none":
            return kind
        _lib.ulysses_attn_fwd(q, k, v, self.o_part, self.lse_part, cu_seqlens, self.B, self.L, 1, self.hq, self.hkv,
                              self.D, self.scale, kind == "causal", self.ws, self.ws_bytes, o_res=self.o_part_res)
        _lib.lse_merge(self.o_acc, self.lse, self.o_part, self.lse_part, o_part_res=self.o_part_res,
                       init=self._steps == 0)
        self._steps += 1
        return kind

    def forward_end(self):
        """The merged output of the query chunk (o, and o_res its rounding residual)."""
        if self._steps == 0:
            raise RuntimeError("no step of the ring saw a key (a chunk always sees its own)")
        _lib.o_finalize(self.o_acc, self.o, self.o_res)
        return self.o

    def backward_begin(self):
        self.dq_acc.zero_()

    def backward_step(self, q, k, v, d_out, cu_seqlens, q_rank: int, k_rank: int):
        """This step's dK, dV shares (fp32 [L][hkv][D]) for the visiting chunk, or None for
        an empty step; dQ's share is added to the rank's accumulator."""
        import torch
        kind = step_kind(q_rank, k_rank, self.causal)
        if kind == "none":
            return None
        dk = torch.empty(self.L, self.hkv, self.D, dtype=torch.float32, device=self.o.device)
        dv = torch.empty_like(dk)
        _lib.ulysses_attn_bwd(q, k, v, self.o, self.lse, d_out, self.dq_part, dk, dv, _lib.USP_FP32, cu_seqlens,
                              self.B, self.L, 1, self.hq, self.hkv, self.D, self.scale, kind == "causal", self.ws,
                              self.ws_bytes, o_res=self.o_res)
        _lib.accumulate_f32(self.dq_acc, self.dq_part)
        return dk, dv

    def backward_end(self):
        return self.dq_acc
