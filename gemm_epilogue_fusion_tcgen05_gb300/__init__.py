"""Python binding of libcoda (ctypes): the same entry points as include/coda.h,
taking torch CUDA tensors and marshalling them to device pointers on the
current torch stream. No arithmetic happens here: every step runs in the CUDA
library, and a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "CodaError", "lib", "LIB_PATH", "EXPORTS", "col_tiles", "row_tiles32", "set_timeout_ms",
    "get_device_error", "coda_gemm", "coda_gemm_resid_norm_stats", "coda_row_rms",
    "coda_gemm_rowscale_swiglu", "coda_gemm_rope", "coda_rope_table", "coda_lmhead_ce",
    "coda_lmhead_ce_workspace_size", "coda_gemm_rowscale_swiglu_bwd", "coda_row_rms_bwd",
    "coda_gemm_resid_norm_stats_bwd", "coda_col_reduce", "coda_gemm_rope_bwd",
    "coda_selftest_bounded_wait", "coda_lmhead_ce_noalloc", "coda_lmhead_ce_bwd",
    "coda_lmhead_ce_bwd_workspace_size", "coda_gemm_resid_ln_stats", "coda_row_ln",
    "coda_gemm_ln_rowscale_swiglu", "coda_gemm_ln_rowscale_swiglu_bwd", "coda_row_ln_bwd",
    "coda_gemm_resid_ln_stats_bwd",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcoda.so")

(CODA_OK, CODA_ERR_INVALID_VALUE, CODA_ERR_UNSUPPORTED, CODA_ERR_LAUNCH, CODA_ERR_TIMEOUT,
 CODA_ERR_RANGE) = range(6)
_STATUS = {0: "CODA_OK", 1: "CODA_ERR_INVALID_VALUE", 2: "CODA_ERR_UNSUPPORTED",
           3: "CODA_ERR_LAUNCH", 4: "CODA_ERR_TIMEOUT", 5: "CODA_ERR_RANGE"}

_P, _I, _F, _D, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t

# name -> (restype, argtypes); the full list of symbols the header declares
EXPORTS = {
    "coda_version": (_I, []),
    "coda_col_tiles": (_I, [_I]),
    "coda_row_tiles32": (_I, [_I]),
    "coda_set_timeout_ms": (None, [_I]),
    "coda_debug_skip_kblock": (None, [_I]),
    "coda_get_device_error": (_I, [_P]),
    "coda_last_error_string": (ctypes.c_char_p, []),
    "coda_gemm": (_I, [_P, _I, _I, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "coda_gemm_resid_norm_stats": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_row_rms": (_I, [_P, _I, _I, _I, _F, _P, _P]),
    "coda_gemm_rowscale_swiglu": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_gemm_rope": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _P]),
    "coda_rope_table": (_I, [_P, _I, _I, _D, _P]),
    "coda_lmhead_ce_workspace_size": (_Z, [_I, _I]),
    "coda_lmhead_ce": (_I, [_P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _P]),
    "coda_gemm_rowscale_swiglu_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_row_rms_bwd": (_I, [_P, _I, _I, _I, _P, _P]),
    "coda_gemm_resid_norm_stats_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_col_reduce": (_I, [_P, _I, _I, _P, _P]),
    "coda_gemm_rope_bwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _P]),
    "coda_selftest_bounded_wait": (_I, [_I, _P]),
    "coda_lmhead_ce_bwd_workspace_size": (_Z, [_I, _I]),
    "coda_lmhead_ce_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _P]),
    "coda_gemm_resid_ln_stats": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_row_ln": (_I, [_P, _P, _I, _I, _I, _F, _P, _P, _P]),
    "coda_gemm_ln_rowscale_swiglu": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "coda_gemm_ln_rowscale_swiglu_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                              _P]),
    "coda_row_ln_bwd": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "coda_gemm_resid_ln_stats_bwd": (_I, [_P] * 14 + [_I, _I, _I, _P]),
    "coda_lmhead_ce_noalloc_capacity": (_Z, []),
    "coda_lmhead_ce_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
}


class CodaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib():
    """The loaded libcoda.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcoda.so is missing ({LIB_PATH}); build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != CODA_OK:
        raise CodaError(status, lib().coda_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _req(t: torch.Tensor, dtype, name: str, ndim: int = 2):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim}-D tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


bf16, f16, f32, i32 = torch.bfloat16, torch.float16, torch.float32, torch.int32


def col_tiles(N: int) -> int:
    return lib().coda_col_tiles(N)


def row_tiles32(M: int) -> int:
    return lib().coda_row_tiles32(M)


def set_timeout_ms(ms: int) -> None:
    lib().coda_set_timeout_ms(ms)


def get_device_error(stream=None) -> int:
    """Synchronises the stream; returns the device status (0 = OK) and clears it."""
    return lib().coda_get_device_error(_stream(stream))


# ---------------------------------------------------------------- forward

def coda_gemm(A, B, C, *, transA=False, transB=False, resid=None, rowsq_part=None, stream=None):
    """C = op(A) op(B) (+ resid); see coda.h. A, B bf16 (row strides taken from
    the tensors), C bf16 or fp32."""
    if A.dtype != bf16 or B.dtype != bf16:
        raise TypeError("A and B must be bf16")
    if C.dtype not in (bf16, f32):
        raise TypeError("C must be bf16 or fp32")
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{n}: 2-D with unit column stride required")
    M, N = C.shape
    K = A.shape[0] if transA else A.shape[1]
    if (A.shape[1] if transA else A.shape[0]) != M:
        raise ValueError("A / C row mismatch")
    if (B.shape[1] if transB else B.shape[0]) != K or (B.shape[0] if transB else B.shape[1]) != N:
        raise ValueError("B shape mismatch")
    if resid is not None and (resid.shape != C.shape or resid.stride() != C.stride()
                              or resid.dtype != C.dtype):
        raise ValueError("resid must have C's shape, strides and dtype")
    _check(lib().coda_gemm(_ptr(A), A.stride(0), int(transA), _ptr(B), B.stride(0), int(transB),
                           _ptr(resid), _ptr(rowsq_part), _ptr(C), C.stride(0),
                           int(C.dtype == f32), M, N, K, _stream(stream)))
    return C


def coda_gemm_resid_norm_stats(x, W0, z, gamma, h, hg, part, stream=None):
    M, K = x.shape
    N = W0.shape[1]
    for t, n in ((x, "x"), (W0, "W0"), (z, "z"), (h, "h"), (hg, "hg")):
        _req(t, bf16, n)
    _req(gamma, bf16, "gamma", 1)
    _req(part, f32, "part")
    if part.shape != (col_tiles(N), M):
        raise ValueError("part must be [col_tiles(N), M]")
    _check(lib().coda_gemm_resid_norm_stats(_ptr(x), _ptr(W0), _ptr(z), _ptr(gamma), _ptr(h),
                                            _ptr(hg), _ptr(part), M, N, K, _stream(stream)))


def coda_row_rms(part, r, d: int, eps: float = 1e-6, stream=None):
    _req(part, f32, "part")
    _req(r, f32, "r", 1)
    nparts, M = part.shape
    _check(lib().coda_row_rms(_ptr(part), nparts, M, d, eps, _ptr(r), _stream(stream)))


def coda_gemm_rowscale_swiglu(hg, W1, r, a, y_save=None, stream=None):
    M, K = hg.shape
    two_f = W1.shape[1]
    _req(hg, bf16, "hg")
    _req(W1, bf16, "W1")
    _req(a, bf16, "a")
    _req(r, f32, "r", 1)
    if y_save is not None:
        _req(y_save, f16, "y_save")
    _check(lib().coda_gemm_rowscale_swiglu(_ptr(hg), _ptr(W1), _ptr(r), _ptr(a), _ptr(y_save),
                                           M, two_f, K, _stream(stream)))


def coda_rope_table(cos_sin, seq_len: int, head_dim: int, theta: float, stream=None):
    _req(cos_sin, f32, "cos_sin", 3)
    _check(lib().coda_rope_table(_ptr(cos_sin), seq_len, head_dim, float(theta), _stream(stream)))


def coda_gemm_rope(A, W, r, cos_sin, seq_len: int, head_dim: int, n_rope_cols: int, out,
                   out_f16=None, stream=None):
    M, K = A.shape
    N = W.shape[1]
    _req(A, bf16, "A")
    _req(W, bf16, "W")
    _req(out, bf16, "out")
    if out_f16 is not None:
        _req(out_f16, f16, "out_f16")
    _check(lib().coda_gemm_rope(_ptr(A), _ptr(W), _ptr(r), _ptr(cos_sin), seq_len, head_dim,
                                n_rope_cols, _ptr(out), _ptr(out_f16), M, N, K, _stream(stream)))


def coda_lmhead_ce_workspace_size(M: int, V: int) -> int:
    return lib().coda_lmhead_ce_workspace_size(M, V)


def coda_lmhead_ce(hidden, W, targets, lse, loss, ws, stream=None):
    M, d = hidden.shape
    V = W.shape[1]
    _req(hidden, bf16, "hidden")
    _req(W, bf16, "W")
    _req(targets, i32, "targets", 1)
    _req(lse, f32, "lse", 1)
    _req(loss, f32, "loss", 1)
    _check(lib().coda_lmhead_ce(_ptr(hidden), _ptr(W), _ptr(targets), _ptr(lse), _ptr(loss),
                                _ptr(ws), ws.numel() * ws.element_size(), M, V, d,
                                _stream(stream)))


def coda_lmhead_ce_bwd_workspace_size(M: int, V: int) -> int:
    return lib().coda_lmhead_ce_bwd_workspace_size(M, V)


def coda_lmhead_ce_bwd(hidden, W, targets, lse, dloss, dhidden, dW, ws, stream=None):
    """dhidden (fp32 [M, d]) and dW (fp32 [d, V]) of sum(dloss * loss)."""
    M, d = hidden.shape
    V = W.shape[1]
    _req(hidden, bf16, "hidden")
    _req(W, bf16, "W")
    _req(targets, i32, "targets", 1)
    _req(lse, f32, "lse", 1)
    _req(dloss, f32, "dloss", 1)
    _req(dhidden, f32, "dhidden")
    _req(dW, f32, "dW")
    _check(lib().coda_lmhead_ce_bwd(_ptr(hidden), _ptr(W), _ptr(targets), _ptr(lse), _ptr(dloss),
                                    _ptr(dhidden), _ptr(dW), _ptr(ws), ws.numel() * ws.element_size(),
                                    M, V, d, _stream(stream)))


# ---------------------------------------------------------------- LayerNorm variant

def coda_gemm_resid_ln_stats(x, W0, z, gamma, h, hg, part_sq, part_sum, stream=None):
    M, K = x.shape
    N = W0.shape[1]
    for t, n in ((x, "x"), (W0, "W0"), (z, "z"), (h, "h"), (hg, "hg")):
        _req(t, bf16, n)
    _req(part_sq, f32, "part_sq")
    _req(part_sum, f32, "part_sum")
    _check(lib().coda_gemm_resid_ln_stats(_ptr(x), _ptr(W0), _ptr(z), _ptr(gamma), _ptr(h),
                                          _ptr(hg), _ptr(part_sq), _ptr(part_sum), M, N, K,
                                          _stream(stream)))


def coda_row_ln(part_sq, part_sum, r, mu, d: int, eps: float = 1e-6, stream=None):
    nparts, M = part_sq.shape
    _check(lib().coda_row_ln(_ptr(part_sq), _ptr(part_sum), nparts, M, d, eps, _ptr(r), _ptr(mu),
                             _stream(stream)))


def coda_gemm_ln_rowscale_swiglu(hg, W1, r, mu, w1, b1, a, y_save=None, stream=None):
    M, K = hg.shape
    two_f = W1.shape[1]
    _req(hg, bf16, "hg")
    _req(W1, bf16, "W1")
    _req(a, bf16, "a")
    for t, n in ((r, "r"), (mu, "mu"), (w1, "w1"), (b1, "b1")):
        _req(t, f32, n, 1)
    if y_save is not None:
        _req(y_save, f16, "y_save")
    _check(lib().coda_gemm_ln_rowscale_swiglu(_ptr(hg), _ptr(W1), _ptr(r), _ptr(mu), _ptr(w1),
                                              _ptr(b1), _ptr(a), _ptr(y_save), M, two_f, K,
                                              _stream(stream)))


def coda_gemm_ln_rowscale_swiglu_bwd(dout, W2, y, r, w1, b1, dyhat, spart, spart_w, spart_b,
                                     stream=None):
    M, d = dout.shape
    f = W2.shape[0]
    _req(y, f16, "y")
    _check(lib().coda_gemm_ln_rowscale_swiglu_bwd(_ptr(dout), _ptr(W2), _ptr(y), _ptr(r),
                                                  _ptr(w1), _ptr(b1), _ptr(dyhat), _ptr(spart),
                                                  _ptr(spart_w), _ptr(spart_b), M, f, d,
                                                  _stream(stream)))


def coda_row_ln_bwd(spart, spart_w, spart_b, s_a, s_b, d: int, stream=None):
    nparts, M = spart.shape
    _check(lib().coda_row_ln_bwd(_ptr(spart), _ptr(spart_w), _ptr(spart_b), nparts, M, d,
                                 _ptr(s_a), _ptr(s_b), _stream(stream)))


def coda_gemm_resid_ln_stats_bwd(dyhat, W1, h, gamma, beta, r, mu, s_a, s_b, dh, dgamma_part,
                                 dbeta_part, hhat=None, dresid=None, stream=None):
    M, two_f = dyhat.shape
    d = W1.shape[0]
    _check(lib().coda_gemm_resid_ln_stats_bwd(_ptr(dyhat), _ptr(W1), _ptr(h), _ptr(gamma),
                                              _ptr(beta), _ptr(r), _ptr(mu), _ptr(s_a), _ptr(s_b),
                                              _ptr(dresid), _ptr(dh), _ptr(hhat), _ptr(dgamma_part),
                                              _ptr(dbeta_part), M, d, two_f, _stream(stream)))


def coda_lmhead_ce_noalloc(hidden, W, targets, lse, loss, stream=None):
    """coda_lmhead_ce with the library's own fixed scratch array instead of a
    caller workspace, for callers that may not allocate device memory (see
    include/coda.h for the row limit and the sharing rules)."""
    M, d = hidden.shape
    V = W.shape[1]
    _req(hidden, bf16, "hidden")
    _req(W, bf16, "W")
    _req(targets, i32, "targets", 1)
    _req(lse, f32, "lse", 1)
    _req(loss, f32, "loss", 1)
    _check(lib().coda_lmhead_ce_noalloc(_ptr(hidden), _ptr(W), _ptr(targets), _ptr(lse),
                                        _ptr(loss), M, V, d, _stream(stream)))


# ---------------------------------------------------------------- backward

def coda_gemm_rowscale_swiglu_bwd(dout, W2, y, r, dyhat, spart, stream=None):
    M, d = dout.shape
    f = W2.shape[0]
    for t, n in ((dout, "dout"), (W2, "W2"), (dyhat, "dyhat")):
        _req(t, bf16, n)
    _req(y, f16, "y")
    _req(spart, f32, "spart")
    _check(lib().coda_gemm_rowscale_swiglu_bwd(_ptr(dout), _ptr(W2), _ptr(y), _ptr(r), _ptr(dyhat),
                                               _ptr(spart), M, f, d, _stream(stream)))


def coda_row_rms_bwd(spart, s, d: int, stream=None):
    nparts, M = spart.shape
    _check(lib().coda_row_rms_bwd(_ptr(spart), nparts, M, d, _ptr(s), _stream(stream)))


def coda_gemm_resid_norm_stats_bwd(dyhat, W1, h, gamma, r, s, dh, dgamma_part, dresid=None,
                                   stream=None):
    M, two_f = dyhat.shape
    d = W1.shape[0]
    for t, n in ((dyhat, "dyhat"), (W1, "W1"), (h, "h"), (dh, "dh")):
        _req(t, bf16, n)
    _check(lib().coda_gemm_resid_norm_stats_bwd(_ptr(dyhat), _ptr(W1), _ptr(h), _ptr(gamma),
                                                _ptr(r), _ptr(s), _ptr(dresid), _ptr(dh),
                                                _ptr(dgamma_part), M, d, two_f, _stream(stream)))


def coda_col_reduce(part, out, stream=None):
    nparts, N = part.shape
    _check(lib().coda_col_reduce(_ptr(part), nparts, N, _ptr(out), _stream(stream)))


def coda_gemm_rope_bwd(dqkv_rot, qkv_rot, r, cos_sin, seq_len: int, head_dim: int,
                       n_rope_cols: int, dqkv_hat, s, d: int, stream=None):
    M, N = dqkv_rot.shape
    _req(dqkv_rot, bf16, "dqkv_rot")
    _req(qkv_rot, f16, "qkv_rot")
    _check(lib().coda_gemm_rope_bwd(_ptr(dqkv_rot), _ptr(qkv_rot), _ptr(r), _ptr(cos_sin), seq_len,
                                    head_dim, n_rope_cols, _ptr(dqkv_hat), _ptr(s), M, N, d,
                                    _stream(stream)))


def coda_selftest_bounded_wait(timeout_ms: int = 20, stream=None) -> int:
    """Runs the bounded-wait probe; returns the status (CODA_ERR_TIMEOUT expected)."""
    return lib().coda_selftest_bounded_wait(timeout_ms, _stream(stream))
