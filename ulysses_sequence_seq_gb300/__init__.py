"""GB300-native hot path of Ulysses sequence parallelism.

The library (``libusp.so``, C ABI in ``include/usp.h``) implements the per-rank
step of Ulysses sequence parallelism with sp ranks simulated as shards of one
device buffer:

* :func:`seq_to_head` / :func:`head_to_seq` -- the two all-to-alls as
  device-local permutations [sp][T/sp][H][D] <-> [sp][H/sp][T][D];
* :func:`attn_fwd_varlen` / :func:`attn_bwd_varlen` -- causal, packed-sample
  (cu_seqlens) softmax attention forward and backward on tcgen05 tensor cores;
* :func:`ulysses_attn_fwd` / :func:`ulysses_attn_bwd` -- the same with both layout
  swaps fused into the attention kernels (seq-sharded tensors in and out);
* :func:`position_ids_to_cu_seqlens`, :func:`cu_seqlens_to_position_ids`,
  :func:`shift_labels`, :func:`sp_weighted_loss` -- the sample and loss bookkeeping
  around the attention, on the device; :mod:`.sp_group` gathers each rank's loss
  and good-token count over a real SP process group.

:class:`UlyssesAttention` chains them into the layer-level step: the seq-sharded
Q, K, V of all ranks in, the seq-sharded attention output out, and the same in
reverse for the gradients. PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import math

from ._lib import (USP_BF16, USP_FP16, USP_FP32, USP_OK, UspError, attn_bwd_varlen, attn_fwd_varlen,  # noqa: F401
                   attn_workspace_size, cu_seqlens_to_position_ids, debug_wait_timeout, get_device_status,
                   head_to_seq, head_to_seq_kv_grad, load, position_ids_to_cu_seqlens, seq_to_head_kv, position_ids_workspace_size, seq_to_head,
                   shift_labels, sp_weighted_loss, status_string, ulysses_attn_bwd, ulysses_attn_fwd)
from .sp_group import gather_loss_and_good, sp_group_loss  # noqa: F401

__all__ = [
    "seq_to_head", "head_to_seq", "attn_fwd_varlen", "attn_bwd_varlen", "ulysses_attn_fwd", "ulysses_attn_bwd",
    "attn_workspace_size", "get_device_status", "status_string", "UspError", "UlyssesAttention", "load",
    "position_ids_to_cu_seqlens", "position_ids_workspace_size", "cu_seqlens_to_position_ids", "shift_labels",
    "sp_weighted_loss", "gather_loss_and_good", "sp_group_loss", "seq_to_head_kv", "head_to_seq_kv_grad",
]


class UlyssesAttention:
    """The attention step of one Ulysses layer for all sp simulated ranks of one GPU.

    Buffers are allocated once for a fixed (T, num_seqs, hq, hkv, D, sp) and reused.
    ``forward`` takes seq-sharded bf16 tensors ([sp][T/sp][H][D] or [T][H][D]) and
    returns the seq-sharded output (it also keeps the output's rounding residual, from
    which the backward takes Delta = dO . O); ``backward`` takes the seq-sharded output
    gradient and returns seq-sharded dQ, dK, dV. With ``fused=True`` (the default)
    the layout swaps happen inside the attention kernels; with ``fused=False`` they
    run as separate re-layout kernels around head-sharded attention.
    """

    def __init__(self, total_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int, sp: int,
                 causal: bool = True, softmax_scale: float = 0.0, device="cuda", grad_dtype=None,
                 fused: bool = True, dtype=None):
        import torch
        self.T, self.B, self.hq, self.hkv, self.D, self.sp = total_tokens, num_seqs, hq, hkv, head_dim, sp
        self.causal = causal
        self.fused = fused
        self.scale = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(head_dim)
        self.dtype = dtype or torch.bfloat16
        if self.dtype not in (torch.bfloat16, torch.float16):
            raise TypeError("activations must be bf16 or fp16")
        if self.dtype == torch.float16 and not fused:
            raise ValueError("fp16 activations run on the fused path")
        self.grad_dtype = grad_dtype or self.dtype
        bf = self.dtype
        T, D = total_tokens, head_dim
        # key/value heads of the head-sharded layout: split over the ranks, or with fewer
        # heads than ranks one replicated head per rank
        self.hkv_h = max(hkv, sp)
        if not fused:
            hk = self.hkv_h
            self.q_h = torch.empty(hq, T, D, dtype=bf, device=device)
            self.k_h = torch.empty(hk, T, D, dtype=bf, device=device)
            self.v_h = torch.empty(hk, T, D, dtype=bf, device=device)
            self.o_h = torch.empty(hq, T, D, dtype=bf, device=device)
            self.o_res_h = torch.empty(hq, T, D, dtype=bf, device=device)
            self.do_h = torch.empty(hq, T, D, dtype=bf, device=device)
            gd = self.grad_dtype
            self.dq_h = torch.empty(hq, T, D, dtype=gd, device=device)
            self.dk_h = torch.empty(hk, T, D, dtype=gd, device=device)
            self.dv_h = torch.empty(hk, T, D, dtype=gd, device=device)
        self.lse = torch.empty(hq, T, dtype=torch.float32, device=device)
        self.o_seq = torch.empty(T, hq, D, dtype=bf, device=device)
        # the rounding residual of the output, kept for the backward's Delta = dO . O
        self.o_res_seq = torch.empty(T, hq, D, dtype=bf, device=device) if fused else None
        gd = self.grad_dtype
        self.dq_seq = torch.empty(T, hq, D, dtype=gd, device=device)
        self.dk_seq = torch.empty(T, hkv, D, dtype=gd, device=device)
        self.dv_seq = torch.empty(T, hkv, D, dtype=gd, device=device)
        self.ws_bytes = max(attn_workspace_size(T, num_seqs, hq, h, D, b) for h in (hkv, self.hkv_h)
                            for b in (False, True))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self._saved = None

    def forward(self, xq, xk, xv, cu_seqlens, stream=None):
        sp = self.sp
        if self.fused:
            ulysses_attn_fwd(xq, xk, xv, self.o_seq, self.lse, cu_seqlens, self.B, self.T, sp, self.hq, self.hkv,
                             self.D, self.scale, self.causal, self.ws, self.ws_bytes, stream, o_res=self.o_res_seq)
            self._saved = (xq, xk, xv)
            return self.o_seq
        seq_to_head(xq, self.q_h, sp, stream)
        seq_to_head_kv(xk, self.k_h, sp, stream)
        seq_to_head_kv(xv, self.v_h, sp, stream)
        attn_fwd_varlen(self.q_h, self.k_h, self.v_h, self.o_h, self.lse, cu_seqlens, self.B, self.T, self.hq,
                        self.hkv_h, self.D, self.scale, self.causal, self.ws, self.ws_bytes, stream,
                        o_res=self.o_res_h)
        head_to_seq(self.o_h, self.o_seq, sp, stream)
        return self.o_seq

    def backward(self, d_out, cu_seqlens, stream=None):
        import torch
        sp = self.sp
        gdt = {torch.float32: USP_FP32, torch.bfloat16: USP_BF16, torch.float16: USP_FP16}[self.grad_dtype]
        if self.fused:
            if self._saved is None:
                raise RuntimeError("backward() needs a forward() first")
            xq, xk, xv = self._saved
            ulysses_attn_bwd(xq, xk, xv, self.o_seq, self.lse, d_out, self.dq_seq, self.dk_seq, self.dv_seq, gdt,
                             cu_seqlens, self.B, self.T, sp, self.hq, self.hkv, self.D, self.scale, self.causal,
                             self.ws, self.ws_bytes, stream, o_res=self.o_res_seq)
            return self.dq_seq, self.dk_seq, self.dv_seq
        seq_to_head(d_out, self.do_h, sp, stream)
        attn_bwd_varlen(self.q_h, self.k_h, self.v_h, self.o_h, self.lse, self.do_h, self.dq_h, self.dk_h,
                        self.dv_h, gdt, cu_seqlens, self.B, self.T, self.hq, self.hkv_h, self.D, self.scale,
                        self.causal, self.ws, self.ws_bytes, stream, o_res=self.o_res_h)
        head_to_seq(self.dq_h, self.dq_seq, sp, stream)
        head_to_seq_kv_grad(self.dk_h, self.dk_seq, sp, self.hkv, stream)
        head_to_seq_kv_grad(self.dv_h, self.dv_seq, sp, self.hkv, stream)
        return self.dq_seq, self.dk_seq, self.dv_seq

    def device_status(self, stream=None) -> int:
        return get_device_status(self.ws, stream)
