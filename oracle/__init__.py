"""CPU oracle for the Ulysses sequence-parallel hot path.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package; the library
(``ulysses_sequence_seq_gb300``) never does, and shares no code with it.

* :mod:`oracle.relayout` -- the seq-sharded <-> head-sharded layout swap as a
  literal index formula on raw bits.
* :func:`attn_fwd` / :func:`attn_bwd` -- float64 softmax attention with an
  explicit mask predicate (C, ``attn_ref.c``), for all or for listed rows.
* :mod:`oracle.brute` -- pure-Python attention and finite differences for tiny
  inputs.
* :mod:`oracle.sp_loss` -- position_ids <-> cu_seqlens, the label shift, good-token
  counts per SP rank and the good-token weighted loss over the ranks.

Every function is pinned by ``tests/test_oracle_pins.py`` and ``tests/test_oracle_sp_loss.py``.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .build import build_oracle
from . import relayout, sp_loss  # noqa: F401

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        p = ctypes.c_void_p
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_fwd.argtypes = [p, p, p, p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                        p, ctypes.c_int, p, ctypes.c_int64, p, p, ctypes.c_int]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [p, p, p, p, p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                        p, ctypes.c_int, p, ctypes.c_int64,
                                        p, ctypes.c_int, p, ctypes.c_int64,
                                        p, p, p, p, p, ctypes.c_int]
        lib.oracle_decode16.restype = None
        lib.oracle_decode16.argtypes = [p, ctypes.c_int64, ctypes.c_int, p]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "oracle inputs are 16-bit patterns (uint16)"
    return a


def _f16_flag(dtype: str) -> int:
    if dtype not in ("bf16", "f16"):
        raise ValueError("dtype is 'bf16' or 'f16'")
    return 1 if dtype == "f16" else 0


def decode16(bits, dtype: str = "bf16") -> np.ndarray:
    """The oracle's exact 16-bit -> float64 decoding (bf16 or IEEE fp16)."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode16(_ptr(b), int(b.size), _f16_flag(dtype), _ptr(out))
    return out


def _opt_list(x, dtype):
    if x is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(x, dtype=dtype))
    return arr, int(arr.size)


def attn_fwd(q, k, v, cu_seqlens, causal=True, scale=None, heads=None, rows=None, dtype="bf16"):
    """float64 O [nheads][nrows][D] and LSE [nheads][nrows].

    q: uint16 [hq][T][D]; k, v: uint16 [hkv][T][D] (bf16 or fp16 bits per `dtype`);
    cu_seqlens: int32 [B+1].
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    hq, T, D = q.shape
    hkv = k.shape[0]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    h_arr, nh = _opt_list(heads, np.int32)
    r_arr, nr = _opt_list(rows, np.int64)
    nh_out = nh if heads is not None else hq
    nr_out = nr if rows is not None else T
    o = np.zeros((nh_out, nr_out, D), dtype=np.float64)
    lse = np.zeros((nh_out, nr_out), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, T, hq, hkv, D,
                                 float(scale), int(bool(causal)), _ptr(h_arr), nh, _ptr(r_arr), nr,
                                 _ptr(o), _ptr(lse), _f16_flag(dtype))
    if rc != 0:
        raise ValueError("oracle_attn_fwd: invalid arguments or cu_seqlens")
    return o, lse


def attn_bwd(q, k, v, do, cu_seqlens, causal=True, scale=None, q_heads=None, q_rows=None,
             kv_heads=None, k_rows=None, want_stats=False, dtype="bf16"):
    """float64 dQ [nqh][nqr][D], dK/dV [nkvh][nkr][D] (and lse, Delta of the dQ rows)."""
    q, k, v, do = _bits(q), _bits(k), _bits(v), _bits(do)
    hq, T, D = q.shape
    hkv = k.shape[0]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qh, nqh = _opt_list(q_heads, np.int32)
    qr, nqr = _opt_list(q_rows, np.int64)
    kh, nkh = _opt_list(kv_heads, np.int32)
    kr, nkr = _opt_list(k_rows, np.int64)
    nqh_o = nqh if q_heads is not None else hq
    nqr_o = nqr if q_rows is not None else T
    nkh_o = nkh if kv_heads is not None else hkv
    nkr_o = nkr if k_rows is not None else T
    dq = np.zeros((nqh_o, nqr_o, D))
    dk = np.zeros((nkh_o, nkr_o, D))
    dv = np.zeros((nkh_o, nkr_o, D))
    lse = np.zeros((nqh_o, nqr_o))
    dl = np.zeros((nqh_o, nqr_o))
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, T, hq,
                                 hkv, D, float(scale), int(bool(causal)),
                                 _ptr(qh), nqh, _ptr(qr), nqr, _ptr(kh), nkh, _ptr(kr), nkr,
                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(lse), _ptr(dl), _f16_flag(dtype))
    if rc != 0:
        raise ValueError("oracle_attn_bwd: invalid arguments or cu_seqlens")
    if want_stats:
        return dq, dk, dv, lse, dl
    return dq, dk, dv
