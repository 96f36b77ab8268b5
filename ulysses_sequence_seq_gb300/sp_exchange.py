"""Ulysses' two all-to-alls over a real sequence-parallel process group.

Before attention each of the sp ranks holds S = T/sp consecutive tokens with all H
heads; the first all-to-all gives each rank all T tokens of its H/sp heads, attention
runs on them, and the second all-to-all returns the output to the sequence-sharded
layout (HF Transformers "Ulysses sequence parallelism" guide, opening paragraph and
layout figure; congresoia365 article, "Cómo Funciona Ulysses", steps 3 to 5). The
backward runs the same exchanges for dO and for dQ, dK, dV.

Each exchange is one collective that moves equal contiguous blocks
(``torch.distributed.all_to_all_single``, NCCL between GPUs) plus a rank-local step in
the library's kernels: ``usp_a2a_pack`` lays out one block per destination before the
sequence -> heads exchange, and ``usp_a2a_unpack`` scatters (or, for replicated
key/value heads, sums) the received blocks after the heads -> sequence exchange. The
receive buffer of the first exchange is the token-major [T][nh][D] layout the fused
attention calls read, and their token-major outputs go back as they are, so nothing
else is copied. Blocks move as bytes, so the collective never converts values.

Overlap: every rank's heads can be exchanged in chunks. All chunks' exchanges are issued
at once (asynchronous collectives on the process group's own stream), and the attention
on a chunk starts as soon as that chunk has arrived, while the next chunks are still in
flight; each chunk's output leaves as soon as its attention is done.

The rank-local steps are the library's CUDA kernels. Tests that run the exchange on CPU
process groups (gloo) pass their own ``pack``/``unpack`` callables; this module has no
host implementation of them.
"""
from __future__ import annotations

import math

from . import _lib


def _all_to_all_bytes(recv, send, group, async_op):
    """recv[r] = block r of every rank's send, in rank order: equal blocks along dim 0,
    moved as raw bytes (any 16- or 32-bit element type, bit for bit)."""
    import torch
    import torch.distributed as dist
    return dist.all_to_all_single(recv.view(torch.uint8).reshape(-1), send.view(torch.uint8).reshape(-1),
                                  group=group, async_op=async_op)


class _PendingUnpack:
    """A heads -> sequence exchange in flight: wait() orders the unpack after it."""

    def __init__(self, work, unpack, recv, out, sp, head0, nheads):
        self.work, self.unpack, self.args = work, unpack, (recv, out, sp, head0, nheads)

    def wait(self):
        if self.work is not None:
            self.work.wait()
            self.work = None
            recv, out, sp, head0, nheads = self.args
            self.unpack(recv, out, sp, head0, nheads)
        return self.args[1]


class _Ready:
    def __init__(self, work, value):
        self.work, self.value = work, value

    def wait(self):
        if self.work is not None:
            self.work.wait()
            self.work = None
        return self.value


class SPExchange:
    """The two all-to-alls of one SP group, for tensors of this rank.

    ``pack(x, out, sp, head0, nheads)`` and ``unpack(recv, out, sp, head0, nheads)``
    default to the library's kernels (usp_a2a_pack / usp_a2a_unpack)."""

    def __init__(self, group=None, pack=None, unpack=None):
        import torch.distributed as dist
        self.group = group
        self.sp = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self._pack = pack or (lambda x, out, sp, h0, nh: _lib.a2a_pack(x, out, sp, h0, nh))
        self._unpack = unpack or (lambda recv, out, sp, h0, nh: _lib.a2a_unpack(recv, out, sp, h0, nh))

    def chunk(self, heads: int, head0: int = 0, nheads: int = 0):
        """(head0, nheads) of a chunk of each rank's heads; a replicated head moves whole."""
        if heads % self.sp == 0:
            hl = heads // self.sp
            nh = nheads or hl - head0
            if head0 < 0 or nh < 1 or head0 + nh > hl:
                raise ValueError("head chunk outside each rank's heads")
            return head0, nh
        if self.sp % heads != 0:
            raise ValueError("heads must divide over the SP group or divide its size")
        if head0 != 0 or nheads not in (0, 1):
            raise ValueError("a replicated head moves whole")
        return 0, 1

    def to_heads(self, x, head0: int = 0, nheads: int = 0, async_op: bool = False):
        """x: [S][H][D] this rank's tokens -> [T][nh][D] (token-major): every rank's tokens
        of this rank's heads r*H/sp + head0 .. (+nh), or with H < sp of the one head this
        rank's query heads read. With async_op, returns a handle whose wait() gives it."""
        import torch
        S, H, D = x.shape
        head0, nh = self.chunk(H, head0, nheads)
        send = torch.empty(self.sp, S, nh, D, dtype=x.dtype, device=x.device)
        self._pack(x, send, self.sp, head0, nh)
        recv = torch.empty_like(send)
        work = _all_to_all_bytes(recv, send, self.group, async_op)
        out = recv.view(self.sp * S, nh, D)
        return _Ready(work, out) if async_op else out

    def to_seq(self, y, out, head0: int = 0, nheads: int = 0, async_op: bool = False):
        """y: [T][nh][D] (token-major, this rank's heads) -> written into out: [S][H][D],
        this rank's tokens; heads outside the chunk are untouched. With H < sp the
        received blocks are the replicas' gradients of each head and are summed."""
        import torch
        S, H, D = out.shape
        head0, nh = self.chunk(H, head0, nheads)
        if y.shape[0] != self.sp * S or y.shape[1] != nh:
            raise ValueError("y must be [sp * S][nheads][D]")
        recv = torch.empty(self.sp, S, nh, D, dtype=y.dtype, device=y.device)
        work = _all_to_all_bytes(recv, y.contiguous().view(self.sp, S, nh, D), self.group, async_op)
        pending = _PendingUnpack(work, self._unpack, recv, out, self.sp, head0, nh)
        if async_op:
            return pending
        if work is not None:
            work.wait()
        pending.work = None
        self._unpack(recv, out, self.sp, head0, nh)
        return out


class UlyssesSPAttention:
    """One Ulysses attention layer over a real SP group, one GPU per rank.

    ``forward`` takes this rank's shard of Q, K, V ([S][H][D], bf16) and the global
    cu_seqlens of the packed sequence; it returns this rank's shard of the output.
    ``backward`` takes this rank's shard of dO and returns its shards of dQ, dK, dV.
    Between the exchanges each rank runs the fused attention calls on the token-major
    heads it received. ``chunks`` splits every rank's heads for overlap (see the module
    notes); with fewer key/value heads than ranks the key/value head is exchanged once.
    """

    def __init__(self, total_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int, group=None,
                 chunks: int = 1, causal: bool = True, softmax_scale: float = 0.0, device=None, dtype=None,
                 grad_dtype=None, exchange: SPExchange | None = None):
        import torch
        self.ex = exchange or SPExchange(group)
        sp = self.ex.sp
        if total_tokens % sp or hq % sp:
            raise ValueError("tokens and query heads must divide over the SP group")
        if hq % hkv:
            raise ValueError("query heads must be a multiple of key/value heads")
        self.T, self.S, self.B = total_tokens, total_tokens // sp, num_seqs
        self.hq, self.hkv, self.D, self.sp = hq, hkv, head_dim, sp
        self.hl = hq // sp
        self.kv_rep = hkv < sp
        if not self.kv_rep and hkv % sp:
            raise ValueError("key/value heads must divide over the SP group or divide its size")
        self.hkvl = 1 if self.kv_rep else hkv // sp
        self.chunks = 1 if self.kv_rep else chunks
        if self.hl % self.chunks or self.hkvl % self.chunks:
            raise ValueError("chunks must divide every rank's query and key/value heads")
        self.hc, self.hkvc = self.hl // self.chunks, self.hkvl // self.chunks
        self.causal = causal
        self.scale = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(head_dim)
        self.dtype = dtype or torch.bfloat16
        self.grad_dtype = grad_dtype or self.dtype
        self.device = device or torch.device("cuda", torch.cuda.current_device())
        self.ws_bytes = max(_lib.attn_workspace_size(self.T, num_seqs, self.hc, self.hkvc, head_dim, b)
                            for b in (False, True))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self._saved = None

    def _kv_chunk(self, c):
        return (0, 1) if self.kv_rep else (c * self.hkvc, self.hkvc)

    def forward(self, xq, xk, xv, cu_seqlens):
        import torch
        ex, T, D = self.ex, self.T, self.D
        q_in = [ex.to_heads(xq, c * self.hc, self.hc, async_op=True) for c in range(self.chunks)]
        k_in = [ex.to_heads(xk, *self._kv_chunk(c), async_op=True) for c in range(self.chunks)]
        v_in = [ex.to_heads(xv, *self._kv_chunk(c), async_op=True) for c in range(self.chunks)]
        out = torch.empty(self.S, self.hq, D, dtype=self.dtype, device=self.device)
        saved, pending = [], []
        for c in range(self.chunks):
            q, k, v = q_in[c].wait(), k_in[c].wait(), v_in[c].wait()
            o = torch.empty(T, self.hc, D, dtype=self.dtype, device=self.device)
            o_res = torch.empty_like(o)
            lse = torch.empty(self.hc, T, dtype=torch.float32, device=self.device)
            _lib.ulysses_attn_fwd(q, k, v, o, lse, cu_seqlens, self.B, T, 1, self.hc, k.shape[1], D, self.scale,
                                  self.causal, self.ws, self.ws_bytes, o_res=o_res)
            pending.append(ex.to_seq(o, out, c * self.hc, self.hc, async_op=True))
            saved.append((q, k, v, o, o_res, lse))
        for p in pending:
            p.wait()
        self._saved = (saved, cu_seqlens)
        return out

    def backward(self, d_out):
        import torch
        if self._saved is None:
            raise RuntimeError("backward() needs a forward() first")
        saved, cu = self._saved
        ex, T, D = self.ex, self.T, self.D
        gdt = {torch.float32: _lib.USP_FP32, torch.bfloat16: _lib.USP_BF16, torch.float16: _lib.USP_FP16}
        do_in = [ex.to_heads(d_out, c * self.hc, self.hc, async_op=True) for c in range(self.chunks)]
        dq = torch.empty(self.S, self.hq, D, dtype=self.grad_dtype, device=self.device)
        dk = torch.empty(self.S, self.hkv, D, dtype=self.grad_dtype, device=self.device)
        dv = torch.empty_like(dk)
        pending = []
        for c in range(self.chunks):
            q, k, v, o, o_res, lse = saved[c]
            do = do_in[c].wait()
            gq = torch.empty(T, self.hc, D, dtype=self.grad_dtype, device=self.device)
            gk = torch.empty(T, k.shape[1], D, dtype=self.grad_dtype, device=self.device)
            gv = torch.empty_like(gk)
            _lib.ulysses_attn_bwd(q, k, v, o, lse, do, gq, gk, gv, gdt[self.grad_dtype], cu, self.B, T, 1, self.hc,
                                  k.shape[1], D, self.scale, self.causal, self.ws, self.ws_bytes, o_res=o_res)
            pending.append(ex.to_seq(gq, dq, c * self.hc, self.hc, async_op=True))
            h0, nh = self._kv_chunk(c)
            pending.append(ex.to_seq(gk, dk, h0, nh, async_op=True))
            pending.append(ex.to_seq(gv, dv, h0, nh, async_op=True))
        for p in pending:
            p.wait()
        return dq, dk, dv
