"""ctypes binding of ``libusp.so`` (argument marshalling only).

Every function takes torch CUDA tensors (or raw integer device pointers), passes
their addresses, sizes and the current CUDA stream to the C ABI declared in
``include/usp.h``, and raises :class:`UspError` on a non-OK status. All work
runs in the library's CUDA kernels; there is no fallback of any kind: if the
library is missing or cannot be loaded, import-time loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from . import build_lib

USP_OK = 0
USP_ERR_INVALID_ARG = 1
USP_ERR_UNSUPPORTED = 2
USP_ERR_CUDA = 3
USP_ERR_WORKSPACE = 4
USP_ERR_TIMEOUT = 5
USP_ERR_DEVICE_CHECK = 6

USP_BF16 = 0
USP_FP16 = 1
USP_FP32 = 2

EXPORTED = (
    "usp_seq_to_head",
    "usp_head_to_seq",
    "usp_attn_workspace_size",
    "usp_attn_fwd_varlen",
    "usp_attn_bwd_varlen",
    "usp_get_device_status",
    "usp_status_string",
    "usp_debug_wait_timeout",
    "usp_attn_fwd_varlen_noalloc",
    "usp_ulysses_attn_fwd",
    "usp_ulysses_attn_bwd",
    "usp_seq_to_head_kv",
    "usp_head_to_seq_kv_grad",
    "usp_position_ids_workspace_size",
    "usp_position_ids_to_cu_seqlens",
    "usp_cu_seqlens_to_position_ids",
    "usp_shift_labels",
    "usp_sp_weighted_loss",
    "usp_a2a_pack",
    "usp_a2a_unpack",
    "usp_lse_merge",
    "usp_o_finalize",
    "usp_accumulate_f32",
)


class UspError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = int(code)
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


_lib = None


def lib_path() -> str:
    return build_lib.LIB


def load(build_if_missing: bool = True):
    """Load libusp.so (building it first when absent or stale and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB
    if build_if_missing and not build_lib.up_to_date():
        build_lib.build()
    if not os.path.exists(path):
        raise ImportError(f"libusp.so not found at {path}; run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    P, I, I64, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.usp_seq_to_head.argtypes = [P, P, I, I64, I, I, I, P]
    L.usp_head_to_seq.argtypes = [P, P, I, I64, I, I, I, P]
    L.usp_attn_workspace_size.argtypes = [I64, I, I, I, I, I]
    L.usp_attn_workspace_size.restype = Z
    L.usp_attn_fwd_varlen.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, F, I, P, Z, P]
    L.usp_attn_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, P, I, P, I, I64, I, I, I, F, I, P, Z, P]
    L.usp_get_device_status.argtypes = [P, P]
    L.usp_status_string.argtypes = [I]
    L.usp_status_string.restype = ctypes.c_char_p
    L.usp_debug_wait_timeout.argtypes = [P, Z, ctypes.c_uint64, P]
    L.usp_attn_fwd_varlen_noalloc.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, I, P, P]
    L.usp_ulysses_attn_fwd.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I, I, P, Z, P]
    L.usp_ulysses_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, P, I, I64, I, I, I, I, F, I, I, P, Z, P]
    L.usp_seq_to_head_kv.argtypes = [P, P, I, I64, I, I, I, P]
    L.usp_head_to_seq_kv_grad.argtypes = [P, P, I, I64, I, I, I, P]
    L.usp_position_ids_workspace_size.argtypes = [I64]
    L.usp_position_ids_workspace_size.restype = Z
    L.usp_position_ids_to_cu_seqlens.argtypes = [P, I64, P, I, P, P, Z, P]
    L.usp_cu_seqlens_to_position_ids.argtypes = [P, I, I64, P, P]
    L.usp_shift_labels.argtypes = [P, P, I, I64, I, P, P, P]
    L.usp_sp_weighted_loss.argtypes = [P, P, I, P, P]
    L.usp_a2a_pack.argtypes = [P, P, I, I64, I, I, I, I, I, P]
    L.usp_a2a_unpack.argtypes = [P, P, I, I64, I, I, I, I, I, P]
    L.usp_lse_merge.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, P]
    L.usp_o_finalize.argtypes = [P, P, P, I64, I, P]
    L.usp_accumulate_f32.argtypes = [P, P, I64, P]
    for name in ("usp_seq_to_head", "usp_head_to_seq", "usp_attn_fwd_varlen", "usp_attn_bwd_varlen",
                 "usp_get_device_status", "usp_debug_wait_timeout", "usp_attn_fwd_varlen_noalloc",
                 "usp_ulysses_attn_fwd", "usp_ulysses_attn_bwd", "usp_position_ids_to_cu_seqlens",
                 "usp_cu_seqlens_to_position_ids", "usp_shift_labels", "usp_sp_weighted_loss",
                 "usp_seq_to_head_kv", "usp_head_to_seq_kv_grad", "usp_a2a_pack", "usp_a2a_unpack", "usp_lse_merge", "usp_o_finalize",
                 "usp_accumulate_f32"):
        getattr(L, name).restype = I
    _lib = L
    return _lib


def status_string(code: int) -> str:
    return load().usp_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != USP_OK:
        raise UspError(fn, code)


def _ptr(x):
    """Device address of a tensor (or an integer address as given). The kernels index
    every buffer as the dense layout the call documents, so a strided view or a host
    tensor is refused here rather than handed over."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("usp: expected a contiguous tensor (the kernels assume the dense layout)")
    if not x.is_cuda:
        raise ValueError("usp: expected a CUDA tensor")
    import torch
    cur = torch.cuda.current_device()
    if x.device.index != cur:   # the call launches on the current device and its stream
        raise ValueError(f"usp: tensor on cuda:{x.device.index}, but the current device is cuda:{cur}")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return USP_BF16
    if t.dtype == torch.float16:
        return USP_FP16
    if t.dtype == torch.float32:
        return USP_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _input_dtype(x) -> int:
    return _dtype_code(x) if hasattr(x, "dtype") else USP_BF16


def seq_to_head(x, out, sp: int, stream=None):
    """x: [sp][T/sp][H][D] (any view with those bytes) -> out: [sp][H/sp][T][D]."""
    H, D = x.shape[-2], x.shape[-1]
    T = x.numel() // (H * D)
    _check("usp_seq_to_head", load().usp_seq_to_head(_ptr(x), _ptr(out), int(sp), int(T), int(H), int(D),
                                                     _dtype_code(x), _stream(stream)))
    return out


def head_to_seq(y, out, sp: int, stream=None):
    """y: [sp][H/sp][T][D] -> out: [sp][T/sp][H][D]."""
    T, D = y.shape[-2], y.shape[-1]
    H = y.numel() // (T * D)
    _check("usp_head_to_seq", load().usp_head_to_seq(_ptr(y), _ptr(out), int(sp), int(T), int(H), int(D),
                                                     _dtype_code(y), _stream(stream)))
    return out


def seq_to_head_kv(x, out, sp: int, stream=None):
    """x: [sp][T/sp][hkv][D] -> out: [max(sp, hkv)][T][D] grouped per rank; with fewer
    heads than ranks each head is replicated to sp / hkv consecutive ranks."""
    H, D = x.shape[-2], x.shape[-1]
    T = x.numel() // (H * D)
    _check("usp_seq_to_head_kv", load().usp_seq_to_head_kv(_ptr(x), _ptr(out), int(sp), int(T), int(H), int(D),
                                                            _dtype_code(x), _stream(stream)))
    return out


def head_to_seq_kv_grad(y, out, sp: int, hkv: int, stream=None):
    """y: [max(sp, hkv)][T][D] per-rank key/value gradients -> out: [sp][T/sp][hkv][D];
    the gradients of a replicated head are summed."""
    D = y.shape[-1]
    T = y.numel() // (D * max(sp, hkv))
    _check("usp_head_to_seq_kv_grad", load().usp_head_to_seq_kv_grad(_ptr(y), _ptr(out), int(sp), int(T), int(hkv),
                                                                      int(D), _dtype_code(y), _stream(stream)))
    return out


def a2a_pack(x, out, sp: int, head0: int = 0, nheads: int = 0, stream=None):
    """x: [S][H][D] this rank's shard -> out: [sp][S][nheads][D], block r for rank r
    (heads r*H/sp + head0 ..; with H < sp the one head rank r reads). nheads 0: all the
    rank's heads from head0 (1 when replicated)."""
    S, H, D = x.shape[-3], x.shape[-2], x.shape[-1]
    nh = nheads or (H // sp - head0 if H % sp == 0 else 1)
    _check("usp_a2a_pack", load().usp_a2a_pack(_ptr(x), _ptr(out), int(sp), int(S), int(H), int(D), int(head0),
                                               int(nh), _dtype_code(x), _stream(stream)))
    return out


def a2a_unpack(recv, out, sp: int, head0: int = 0, nheads: int = 0, stream=None):
    """recv: [sp][S][nheads][D] (block r from rank r) -> out: [S][H][D], the chunk's heads
    of every rank written (with H < sp: the replicas' gradients summed)."""
    S, H, D = out.shape[-3], out.shape[-2], out.shape[-1]
    nh = nheads or (H // sp - head0 if H % sp == 0 else 1)
    _check("usp_a2a_unpack", load().usp_a2a_unpack(_ptr(recv), _ptr(out), int(sp), int(S), int(H), int(D),
                                                   int(head0), int(nh), _dtype_code(out), _stream(stream)))
    return out


def lse_merge(o_acc, lse_acc, o_part, lse_part, o_part_res=None, token_major=True, init=False, stream=None):
    """o_acc (fp32), lse_acc <- merged with a partial result over disjoint keys (usp_lse_merge).
    o_*: [T][H][D] (token_major) or [H][T][D]; lse_*: [H][T]."""
    H, T = lse_acc.shape
    _check("usp_lse_merge", load().usp_lse_merge(
        _ptr(o_acc), _ptr(lse_acc), _ptr(o_part), _ptr(o_part_res), _ptr(lse_part), int(T), int(H),
        int(o_part.shape[-1]), int(bool(token_major)), _dtype_code(o_part), int(bool(init)), _stream(stream)))


def o_finalize(o_acc, o, o_res=None, stream=None):
    """o (16-bit) = round(o_acc), o_res = round(o_acc - o)."""
    _check("usp_o_finalize", load().usp_o_finalize(_ptr(o_acc), _ptr(o), _ptr(o_res), int(o_acc.numel()),
                                                   _dtype_code(o), _stream(stream)))


def accumulate_f32(acc, part, stream=None):
    """acc += part (fp32)."""
    _check("usp_accumulate_f32", load().usp_accumulate_f32(_ptr(acc), _ptr(part), int(acc.numel()),
                                                           _stream(stream)))


def attn_workspace_size(total_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int, bwd: bool) -> int:
    return int(load().usp_attn_workspace_size(int(total_tokens), int(num_seqs), int(hq), int(hkv),
                                              int(head_dim), int(bool(bwd))))


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, num_seqs: int, total_tokens: int, hq: int, hkv: int,
                    head_dim: int, softmax_scale: float, causal: bool, workspace, ws_bytes: int, stream=None,
                    o_res=None):
    """Head-major forward; `o_res` (optional, like `o`) receives the rounding residual of o."""
    _check("usp_attn_fwd_varlen", load().usp_attn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(cu_seqlens), int(num_seqs),
        int(total_tokens), int(hq), int(hkv), int(head_dim), float(softmax_scale), int(bool(causal)),
        _ptr(workspace), int(ws_bytes), _stream(stream)))


def attn_bwd_varlen(q, k, v, o, lse, d_o, dq, dk, dv, grad_dt: int, cu_seqlens, num_seqs: int,
                    total_tokens: int, hq: int, hkv: int, head_dim: int, softmax_scale: float, causal: bool,
                    workspace, ws_bytes: int, stream=None, o_res=None):
    """Head-major backward; pass the forward's `o_res` to take Delta from o + o_res."""
    _check("usp_attn_bwd_varlen", load().usp_attn_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv),
        int(grad_dt), _ptr(cu_seqlens), int(num_seqs), int(total_tokens), int(hq), int(hkv), int(head_dim),
        float(softmax_scale), int(bool(causal)), _ptr(workspace), int(ws_bytes), _stream(stream)))


def ulysses_attn_fwd(q, k, v, o, lse, cu_seqlens, num_seqs: int, total_tokens: int, sp: int, hq: int, hkv: int,
                     head_dim: int, softmax_scale: float, causal: bool, workspace, ws_bytes: int, stream=None,
                     o_res=None):
    """Fused forward on the seq-sharded layout: q, k, v, o (and o_res) are [sp][T/sp][H][D],
    bf16 or fp16 (taken from q)."""
    _check("usp_ulysses_attn_fwd", load().usp_ulysses_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(cu_seqlens), int(num_seqs),
        int(total_tokens), int(sp), int(hq), int(hkv), int(head_dim), float(softmax_scale), int(bool(causal)),
        _input_dtype(q), _ptr(workspace), int(ws_bytes), _stream(stream)))


def ulysses_attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, grad_dt: int, cu_seqlens, num_seqs: int, total_tokens: int,
                     sp: int, hq: int, hkv: int, head_dim: int, softmax_scale: float, causal: bool, workspace,
                     ws_bytes: int, stream=None, o_res=None):
    """Fused backward on the seq-sharded layout: every activation and gradient is [sp][T/sp][H][D];
    activations bf16 or fp16 (taken from q), gradients of grad_dt (that type or fp32)."""
    _check("usp_ulysses_attn_bwd", load().usp_ulysses_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv),
        int(grad_dt), _ptr(cu_seqlens), int(num_seqs), int(total_tokens), int(sp), int(hq), int(hkv),
        int(head_dim), float(softmax_scale), int(bool(causal)), _input_dtype(q), _ptr(workspace), int(ws_bytes),
        _stream(stream)))


def attn_fwd_varlen_noalloc(q, k, v, o, lse, cu_seqlens, num_seqs: int, total_tokens: int, hq: int, hkv: int,
                            head_dim: int, softmax_scale: float, causal: bool, status=None, stream=None):
    """The forward without a workspace: scratch lives in the library's static device
    array (for callers that cannot allocate; calls must not overlap on the GPU)."""
    _check("usp_attn_fwd_varlen_noalloc", load().usp_attn_fwd_varlen_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), int(num_seqs), int(total_tokens),
        int(hq), int(hkv), int(head_dim), float(softmax_scale), int(bool(causal)), _ptr(status),
        _stream(stream)))


def position_ids_workspace_size(total_tokens: int) -> int:
    return int(load().usp_position_ids_workspace_size(int(total_tokens)))


def position_ids_to_cu_seqlens(position_ids, total_tokens: int, cu_seqlens, max_seqs: int, num_seqs, workspace,
                               ws_bytes: int, stream=None):
    _check("usp_position_ids_to_cu_seqlens", load().usp_position_ids_to_cu_seqlens(
        _ptr(position_ids), int(total_tokens), _ptr(cu_seqlens), int(max_seqs), _ptr(num_seqs), _ptr(workspace),
        int(ws_bytes), _stream(stream)))


def cu_seqlens_to_position_ids(cu_seqlens, num_seqs: int, total_tokens: int, position_ids, stream=None):
    _check("usp_cu_seqlens_to_position_ids", load().usp_cu_seqlens_to_position_ids(
        _ptr(cu_seqlens), int(num_seqs), int(total_tokens), _ptr(position_ids), _stream(stream)))


def shift_labels(labels, cu_seqlens, num_seqs: int, total_tokens: int, sp: int, shifted, good_tokens, stream=None):
    _check("usp_shift_labels", load().usp_shift_labels(
        _ptr(labels), _ptr(cu_seqlens), int(num_seqs), int(total_tokens), int(sp), _ptr(shifted),
        _ptr(good_tokens), _stream(stream)))


def sp_weighted_loss(rank_loss, good_tokens, sp: int, loss, stream=None):
    _check("usp_sp_weighted_loss", load().usp_sp_weighted_loss(
        _ptr(rank_loss), _ptr(good_tokens), int(sp), _ptr(loss), _stream(stream)))


def get_device_status(workspace, stream=None) -> int:
    return int(load().usp_get_device_status(_ptr(workspace), _stream(stream)))


def debug_wait_timeout(workspace, ws_bytes: int, limit_ns: int, stream=None):
    _check("usp_debug_wait_timeout", load().usp_debug_wait_timeout(_ptr(workspace), int(ws_bytes),
                                                                   int(limit_ns), _stream(stream)))
