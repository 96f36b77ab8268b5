"""Helpers shared by the GPU tests: moving seeded bf16 bit patterns to the device,
reading results back, and choosing sampled rows for large-size parity checks."""
from __future__ import annotations

import numpy as np
import torch

import ulysses_sequence_seq_gb300 as usp


def needs_gpu():
    if not torch.cuda.is_available():
        import pytest
        pytest.skip("no CUDA device")


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bf16 tensor with exactly those bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_rows(cu, n_random: int, seed: int = 0, T: int | None = None):
    """Rows worth checking: the first and last rows of every sample, rows around
    128-row tile edges, plus random rows (sorted, unique)."""
    cu = [int(x) for x in cu]
    T = cu[-1] if T is None else T
    rows = set()
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        for r in (s, s + 1, s + 127, s + 128, s + 129, s + 255, s + 256, e - 129, e - 128, e - 2, e - 1):
            if s <= r < e:
                rows.add(r)
    rng = np.random.default_rng(seed)
    if T > 0:
        rows.update(int(x) for x in rng.integers(0, T, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


class Problem:
    """Device buffers for one attention problem in the head-major layout."""

    def __init__(self, q_bits, k_bits, v_bits, cu, causal=True, do_bits=None, scale=0.0):
        self.q, self.k, self.v = dev_bf16(q_bits), dev_bf16(k_bits), dev_bf16(v_bits)
        self.do = dev_bf16(do_bits) if do_bits is not None else None
        self.cu_host = np.asarray(cu, dtype=np.int32)
        self.cu = torch.from_numpy(self.cu_host).cuda()
        self.hq, self.T, self.D = q_bits.shape
        self.hkv = k_bits.shape[0]
        self.B = len(cu) - 1
        self.causal = causal
        self.scale = scale   # <= 0: 1/sqrt(D)
        self.ws_bytes = max(usp.attn_workspace_size(self.T, self.B, self.hq, self.hkv, self.D, False),
                            usp.attn_workspace_size(self.T, self.B, self.hq, self.hkv, self.D, True))
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device="cuda")

    def forward(self, residual=True):
        """O, LSE and the device status; the rounding residual of O is kept in self.o_res
        (None with residual=False) and handed to the next backward."""
        o = torch.full((self.hq, self.T, self.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((self.hq, self.T), float("nan"), dtype=torch.float32, device="cuda")
        self.o_res = torch.full_like(o, float("nan")) if residual else None
        usp.attn_fwd_varlen(self.q, self.k, self.v, o, lse, self.cu, self.B, self.T, self.hq, self.hkv, self.D,
                            self.scale, self.causal, self.ws, self.ws_bytes, o_res=self.o_res)
        status = usp.get_device_status(self.ws)
        return o, lse, status

    def backward(self, o, lse, grad_dtype=torch.float32):
        gd = usp.USP_FP32 if grad_dtype == torch.float32 else usp.USP_BF16
        dq = torch.full((self.hq, self.T, self.D), float("nan"), dtype=grad_dtype, device="cuda")
        dk = torch.full((self.hkv, self.T, self.D), float("nan"), dtype=grad_dtype, device="cuda")
        dv = torch.full((self.hkv, self.T, self.D), float("nan"), dtype=grad_dtype, device="cuda")
        usp.attn_bwd_varlen(self.q, self.k, self.v, o, lse, self.do, dq, dk, dv, gd, self.cu, self.B, self.T,
                            self.hq, self.hkv, self.D, self.scale, self.causal, self.ws, self.ws_bytes,
                            o_res=getattr(self, "o_res", None))
        status = usp.get_device_status(self.ws)
        return dq, dk, dv, status


def dev_16(bits: np.ndarray, dtype) -> torch.Tensor:
    """uint16 bit patterns -> CUDA tensor of the 16-bit `dtype` (bf16 or fp16) with those bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(dtype).cuda()


def dq_key_amplified_bound(q, k, v, do, cu, o_kernel, dtype="bf16", causal=True):
    """Per element of dQ [hq][T][D], what the 16-bit arithmetic of the backward can add beyond
    plain rounding when keys are large, both terms scaled by max_j |K_j| (over the row's
    sample, per column) and the softmax scale:
      * the bias of Delta = dO . O: the forward's O multiplies P rounded to 16 bits, so Delta
        exceeds sum_j P_j dP_j by eps = dO . (O_kernel - O), dS sums to -eps over the row
        instead of 0 and dQ gains -scale * eps * sum_j P_j K_j;
      * dS's own three roundings to fp16 (P, the bracket dP - Delta, their product), each at
        most 2^-11 relative: 3 * 2^-11 * sum_j |dS_j| for the row.
    The float64 P, dP and dS come from the oracle's LSE and the same inputs; query head h
    reads key/value head h // (hq / hkv)."""
    import oracle
    dec = (lambda x: np.asarray(x, dtype=np.uint16).view(np.float16).astype(np.float64)) if dtype == "f16" else \
        (lambda x: (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    Q, K, V, dO = dec(q), dec(k), dec(v), dec(do)
    group = Q.shape[0] // K.shape[0]
    ro, rl = oracle.attn_fwd(q, k, v, cu, causal=causal, dtype=dtype)
    eps = np.einsum("htd,htd->ht", dO, o_kernel - ro)
    sc = 1.0 / np.sqrt(Q.shape[2])
    bound = np.zeros_like(Q)
    for h in range(Q.shape[0]):
        for b in range(len(cu) - 1):
            s0, s1 = int(cu[b]), int(cu[b + 1])
            if s1 == s0:
                continue
            kh = h // group
            S = Q[h, s0:s1] @ K[kh, s0:s1].T * sc
            if causal:
                S = S + np.triu(np.full((s1 - s0, s1 - s0), -np.inf), 1)
            P = np.exp(S - rl[h, s0:s1, None])
            dP = dO[h, s0:s1] @ V[kh, s0:s1].T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            kmax = np.abs(K[kh, s0:s1]).max(axis=0)
            per_row = np.abs(eps[h, s0:s1]) + 3 * 2.0 ** -11 * np.abs(dS).sum(axis=1)
            bound[h, s0:s1] = sc * per_row[:, None] * kmax[None, :]
    return bound
