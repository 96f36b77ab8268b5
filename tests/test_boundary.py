"""The C-ABI library: it builds, loads, exports every declared symbol, and rejects
invalid arguments on the host (CPU only: no call here reaches a CUDA API)."""
import os
import re

import pytest

from ulysses_sequence_seq_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "usp.h")

A = 1 << 20          # fake, 16-byte aligned "device" addresses: never dereferenced
B = 1 << 30
MIS = A + 8          # misaligned


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(usp_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = _lib.load()
    syms = declared_symbols()
    assert set(syms) == set(_lib.EXPORTED)
    for s in syms:
        assert hasattr(L, s), s


def test_status_strings():
    assert _lib.status_string(0) == "USP_OK"
    assert _lib.status_string(5) == "USP_ERR_TIMEOUT"
    assert _lib.status_string(6) == "USP_ERR_DEVICE_CHECK"
    assert _lib.status_string(99) == "USP_ERR_UNKNOWN"


def relayout(fn, inp, out, sp, T, H, D, dt=_lib.USP_BF16):
    return getattr(_lib.load(), fn)(inp, out, sp, T, H, D, dt, None)


@pytest.mark.parametrize("fn", ["usp_seq_to_head", "usp_head_to_seq"])
def test_relayout_validation(fn):
    ok = relayout(fn, A, B, 4, 0, 32, 128)            # T == 0: a valid no-op
    assert ok == _lib.USP_OK
    assert relayout(fn, 0, B, 4, 64, 32, 128) == _lib.USP_ERR_INVALID_ARG       # NULL
    assert relayout(fn, MIS, B, 4, 64, 32, 128) == _lib.USP_ERR_INVALID_ARG     # misaligned
    assert relayout(fn, A, B, 4, 64, 30, 128) == _lib.USP_ERR_INVALID_ARG       # heads % sp
    assert relayout(fn, A, B, 4, 66, 32, 128) == _lib.USP_ERR_INVALID_ARG       # tokens % sp
    assert relayout(fn, A, A + 4096, 4, 64, 32, 128) == _lib.USP_ERR_INVALID_ARG  # overlap
    assert relayout(fn, A, B, 0, 64, 32, 128) == _lib.USP_ERR_INVALID_ARG       # sp < 1
    assert relayout(fn, A, B, 4, 64, 32, 4) == _lib.USP_ERR_UNSUPPORTED         # 8-byte rows


def test_head_divisibility_matches_worked_example():
    """32 heads: exactly sp = 1, 2, 4, 8, 16, 32 pass validation (HF guide, "Configurar")."""
    L = _lib.load()
    accepted = []
    for sp in range(1, 33):
        # T == 0 is a valid no-op, so only the head-count rule decides (nothing is launched)
        if L.usp_seq_to_head(A, B, sp, 0, 32, 128, _lib.USP_BF16, None) == _lib.USP_OK:
            accepted.append(sp)
    assert accepted == [1, 2, 4, 8, 16, 32]


def fwd(q=A, k=A, v=A, o=B, o_res=None, lse=B, cu=A, nseq=1, T=256, hq=4, hkv=4, D=128, ws=A, wsb=1 << 40):
    return _lib.load().usp_attn_fwd_varlen(q, k, v, o, o_res, lse, cu, nseq, T, hq, hkv, D, 0.0, 1, ws, wsb, None)


def test_attn_fwd_validation():
    assert fwd(q=0) == _lib.USP_ERR_INVALID_ARG
    assert fwd(o=MIS) == _lib.USP_ERR_INVALID_ARG
    assert fwd(o_res=MIS) == _lib.USP_ERR_INVALID_ARG
    assert fwd(hq=6, hkv=4) == _lib.USP_ERR_INVALID_ARG
    assert fwd(nseq=0) == _lib.USP_ERR_INVALID_ARG
    assert fwd(cu=0) == _lib.USP_ERR_INVALID_ARG
    assert fwd(T=-1) == _lib.USP_ERR_INVALID_ARG
    assert fwd(D=96) == _lib.USP_ERR_UNSUPPORTED
    assert fwd(wsb=16) == _lib.USP_ERR_WORKSPACE


def test_attn_bwd_validation():
    L = _lib.load()

    def bwd(gdt=_lib.USP_FP32, dq=B, D=128, wsb=1 << 40, hq=4, hkv=2, o_res=None):
        return L.usp_attn_bwd_varlen(A, A, A, A, o_res, A, A, dq, B, B, gdt, A, 1, 256, hq, hkv, D, 0.0, 1, A, wsb,
                                     None)

    assert bwd(gdt=_lib.USP_FP16) == _lib.USP_ERR_UNSUPPORTED
    assert bwd(gdt=7) == _lib.USP_ERR_INVALID_ARG
    assert bwd(dq=0) == _lib.USP_ERR_INVALID_ARG
    assert bwd(dq=MIS) == _lib.USP_ERR_INVALID_ARG
    assert bwd(o_res=MIS) == _lib.USP_ERR_INVALID_ARG
    assert bwd(D=32) == _lib.USP_ERR_UNSUPPORTED
    assert bwd(hq=3) == _lib.USP_ERR_INVALID_ARG
    assert bwd(wsb=100) == _lib.USP_ERR_WORKSPACE


def test_workspace_sizes_grow_with_problem():
    ws = _lib.attn_workspace_size
    a = ws(8192, 2, 32, 32, 128, False)
    b = ws(8192, 2, 32, 32, 128, True)
    c = ws(65536, 9, 32, 32, 128, True)
    assert 0 < a < b < c
    # the backward holds Delta and an fp32 dQ accumulator: at least 4*hq*T*(D+1) bytes
    assert b >= 4 * 32 * 8192 * 129
    assert ws(-1, 1, 4, 4, 128, False) == 0


def test_kv_swap_validation():
    L = _lib.load()
    f, g = L.usp_seq_to_head_kv, L.usp_head_to_seq_kv_grad
    assert f(A, B, 8, 0, 2, 128, _lib.USP_BF16, None) == _lib.USP_OK            # empty, replicated
    assert f(A, B, 4, 64, 3, 128, _lib.USP_BF16, None) == _lib.USP_ERR_INVALID_ARG  # 3 heads over 4 ranks
    assert f(A, B, 8, 63, 2, 128, _lib.USP_BF16, None) == _lib.USP_ERR_INVALID_ARG  # tokens % sp
    assert f(A, A + 4096, 8, 64, 2, 128, _lib.USP_BF16, None) == _lib.USP_ERR_INVALID_ARG  # overlap
    assert g(A, B, 4, 64, 3, 128, _lib.USP_FP32, None) == _lib.USP_ERR_INVALID_ARG
    assert g(A, B, 8, 64, 2, 128, _lib.USP_FP16, None) == _lib.USP_ERR_UNSUPPORTED   # fp16 sums
    assert g(0, B, 8, 64, 2, 128, _lib.USP_FP32, None) == _lib.USP_ERR_INVALID_ARG


def test_binding_refuses_host_and_strided_tensors():
    """The Python binding hands only dense device buffers to the C ABI."""
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="contiguous"):
        _lib._ptr(torch.zeros(8, 8).t())
    with pytest.raises(ValueError, match="CUDA"):
        _lib._ptr(torch.zeros(8))
    assert _lib._ptr(A) == A and _lib._ptr(None) is None


def _declarations():
    """Return type and parameter count of every usp_* declaration in the public header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"(usp_status|size_t|const char\*)\s+(usp_\w+)\s*\(([^)]*)\)\s*;", text):
        args = m.group(3).strip()
        out[m.group(2)] = (m.group(1), 0 if args in ("", "void") else len(args.split(",")))
    return out


def test_binding_argument_lists_match_the_header():
    """Each ctypes argument list has as many entries as the C declaration has parameters,
    and each return type is the declared one."""
    import ctypes
    L = _lib.load()
    decl = _declarations()
    assert set(decl) == set(_lib.EXPORTED)
    restypes = {"usp_status": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p}
    for name, (ret, n) in decl.items():
        fn = getattr(L, name)
        assert fn.argtypes is not None and len(fn.argtypes) == n, (name, n, fn.argtypes and len(fn.argtypes))
        assert fn.restype is restypes[ret], (name, ret, fn.restype)
