"""CPU oracle for the CODA GEMM-plus-epilogue block: plain, slow, fp64.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run this module. The CUDA
library never calls it, and it shares no code with the CUDA library: it
computes everything from the plain definitions, with numpy matmul as the only
library step.

Sources (the pages' titles and sections):
  [pith]   "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
           (pith.science summary of arXiv 2605.19269): Fig. 4 and Fig. 5
           captions (GEMM-RMSNorm-GEMM, r = 1/sqrt(reduce(r_hat) + eps)),
           Fig. 7 caption (pairwise maps), Appendix A.1 "Tile-wise Epilogue",
           Listing 2 "Kernel Example" (residual + mean-of-squares + RMSNorm
           weight epilogue).
  [notes]  "Reading notes on CODA" (jianyuh.github.io): section 2
           "Forward-Pass Reparameterizations" (GEMM -> Residual -> RMSNorm ->
           GEMM; pairwise activations; cross-entropy loss), section 3 "The
           Backward Pass: Reverse Fusion" (including "Eliminating the RMSNorm
           backward kernel").
  [thread] digg thread on CODA: Patterns 1-3 and the commutation identity.

Two forms are kept:
  * canonical  -- the block as frameworks write it (RMSNorm applied before the
                  second GEMM, autograd-by-hand backward). This is the
                  reference every GPU result is compared with.
  * reparam    -- the pages' rewritten form (delayed row scale r, statistic s
                  from (grad y, y)). It must equal the canonical form in exact
                  arithmetic; with ``store_bf16=True`` it also rounds, to bf16,
                  the tensors that the rewritten kernels write to memory, which
                  models the storage precision of the fused path.

Parity status: every function here is pinned by the CPU tests in
tests/test_oracle_*.py (closed forms, invariants, finite differences, torch
library special cases, brute force on tiny inputs). The relative-error study
of the pages' Fig. 6 prints no values; the GPU test checks only its
qualitative claim (the rewritten path's error is below the PyTorch path's),
so that one comparison has no value pin.

The rewritten forms also run in an fp32 mode (``fp32=True``: GEMMs through
the tensor-core model ``tc_matmul``, elementwise work in fp32). It is not a
reference for the GPU: it measures how far fp32 arithmetic by itself moves
the chained backward statistics from their fp64 values, which is where the
tests take their bound for those statistics from
(tests/golden/make_stat_spread.py). ``tc_matmul`` is pinned by closed forms
(exact sums, the truncation point, the truncation bound) in
tests/test_oracle_pins.py.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

EPS = 1e-6          # RMSNorm epsilon, inside the square root
ROPE_THETA = 500000.0

f64 = np.float64


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------

def bf16_round(a) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned
    as fp64. bf16 keeps 8 significant bits; fp64 has 53, so the low 45 bits
    of the fp64 significand are rounded away. Below 2^-126 bf16 is
    subnormal with a fixed spacing of 2^-133."""
    a = np.ascontiguousarray(np.asarray(a, dtype=f64))
    u = a.view(np.uint64)
    lsb = (u >> np.uint64(45)) & np.uint64(1)
    bias = np.uint64((1 << 44) - 1) + lsb
    mask = np.uint64(~((1 << 45) - 1) & 0xFFFFFFFFFFFFFFFF)
    r = ((u + bias) & mask).view(f64)
    tiny = np.abs(a) < 2.0 ** -126
    if np.any(tiny):
        r = np.where(tiny, np.round(a * 2.0 ** 133) * 2.0 ** -133, r)
    return r


def f16_round(a) -> np.ndarray:
    """Round fp64 values to the nearest IEEE binary16 value (ties to even),
    returned as fp64: numpy's float16 conversion, which rounds correctly
    from fp64. 11 significant bits; magnitudes from 65520 up become inf."""
    with np.errstate(over="ignore"):
        return np.asarray(a, dtype=f64).astype(np.float16).astype(f64)


def _store(store_bf16: bool):
    return bf16_round if store_bf16 else (lambda t: t)


def _store_saved(store_bf16: bool):
    """The storage point of the copies the rewritten forward keeps only for
    the backward's relocated statistics (y, qkv_save): fp16, whose 11-bit
    significand keeps those statistics within 1e-3 where bf16 would not."""
    return f16_round if store_bf16 else (lambda t: t)


def tc_matmul(a, b, group: int = 16) -> np.ndarray:
    """A model of a tensor-core GEMM with an fp32 accumulator, for operands
    that are exact in fp32 (bf16 / fp16 values): along K, each group of
    `group` products is summed in fp64 (exact up to rounding far below
    fp32's for the value ranges of these workloads) and added to the fp32
    accumulator, and that addition rounds toward zero (drops the bits below
    fp32's 24-bit significand). Truncating accumulation is what the fp32
    results of a GB300 GEMM show: their error is biased toward zero and some
    twenty times a round-to-nearest fp32 GEMM's; this model errs slightly
    more than the GB300 does (a GPU test checks both). Returns fp32 values."""
    a = np.asarray(a, dtype=f64)
    b = np.asarray(b, dtype=f64)
    keep = np.uint64(0xFFFFFFFFE0000000)  # sign, exponent, top 23 fraction bits
    acc = np.zeros((a.shape[0], b.shape[1]), dtype=f64)
    for k0 in range(0, a.shape[1], group):
        acc += a[:, k0:k0 + group] @ b[k0:k0 + group, :]
        acc = (acc.view(np.uint64) & keep).view(f64)
    return acc.astype(np.float32)


def _precision(fp32: bool):
    """Arithmetic of the rewritten forms: fp64 by default. fp32=True runs the
    same steps as an fp32 tensor-core implementation would: GEMMs through
    tc_matmul, elementwise maps and row sums in fp32. It serves only to
    measure how far that arithmetic by itself moves a result from the fp64
    one; it is meant for store_bf16=True, where the stored tensors are bf16
    / fp16 values and so exact in fp32. Returns (dtype, matmul)."""
    if fp32:
        return np.float32, tc_matmul
    return f64, (lambda x, y: x @ y)


def _stored(rounder, dt):
    """A storage point that rounds (bf16 / fp16, or not at all) and hands the
    value on in the arithmetic type dt."""
    return lambda t: np.asarray(rounder(t), dtype=dt)


# --------------------------------------------------------------------------
# elementwise maps
# --------------------------------------------------------------------------

def sigmoid(t, dtype=f64):
    t = np.asarray(t, dtype=dtype)
    return 1.0 / (1.0 + np.exp(-t))


def silu(t, dtype=f64):
    """silu(t) = t * sigmoid(t) (the SwiGLU gate activation)."""
    t = np.asarray(t, dtype=dtype)
    return t * sigmoid(t, dtype)


def silu_grad(t, dtype=f64):
    """d silu / dt = sigmoid(t) * (1 + t * (1 - sigmoid(t)))."""
    t = np.asarray(t, dtype=dtype)
    s = sigmoid(t, dtype)
    return s * (1.0 + t * (1.0 - s))


def rms_factor(h, eps: float = EPS, dtype=f64):
    """Row-wise inverse RMS: r = 1 / sqrt(mean_j h_j^2 + eps)  [notes s2;
    pith Fig. 5 caption: eps inside the square root]."""
    h = np.asarray(h, dtype=dtype)
    return 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)


def swiglu(y, dtype=f64):
    """Pairwise SwiGLU on gate/up-interleaved columns: column 2k is gate g_k,
    column 2k+1 is up u_k, output a_k = silu(g_k) * u_k  [pith Fig. 7
    caption; notes s2 "Pairwise activations"]."""
    g = y[:, 0::2]
    u = y[:, 1::2]
    return silu(g, dtype) * u


# --------------------------------------------------------------------------
# MLP block: GEMM -> residual -> RMSNorm -> GEMM -> SwiGLU -> GEMM
# --------------------------------------------------------------------------

def mlp_fwd(x, z, W0, W1, W2, gamma, eps: float = EPS) -> Dict[str, np.ndarray]:
    """Canonical forward [notes s2 "GEMM -> Residual -> RMSNorm -> GEMM"]:
        h  = x W0 + z
        r  = 1/sqrt(mean(h^2) + eps)
        n  = r h ;  h2 = n * gamma
        y  = h2 W1 ;  a = silu(y[:,0::2]) * y[:,1::2]
        out = a W2
    """
    x, z, W0, W1, W2, gamma = (np.asarray(t, dtype=f64) for t in (x, z, W0, W1, W2, gamma))
    h = x @ W0 + z
    r = rms_factor(h, eps)
    n = r[:, None] * h
    h2 = n * gamma[None, :]
    y = h2 @ W1
    a = swiglu(y)
    out = a @ W2
    return {"h": h, "r": r, "n": n, "h2": h2, "y": y, "a": a, "out": out}


def mlp_fwd_reparam(x, z, W0, W1, W2, gamma, eps: float = EPS,
                    store_bf16: bool = False, fp32: bool = False) -> Dict[str, np.ndarray]:
    """The pages' rewritten forward [notes s2; pith Fig. 4; thread Pattern 1]:
        GEMM 1 epilogue: h = x W0 + z (stored), hg = h * gamma (stored),
                         row statistic from the unscaled h (Listing 2: the
                         mean of squares is taken on D before the RMSNorm
                         weight multiplies it)
        auxiliary:       r = 1/sqrt(mean(h^2) + eps)
        GEMM 2 epilogue: y = r * (hg W1)  (delayed row scale, saved for the
                         backward in fp16), a = silu(y_gate) * y_up (stored)
        GEMM 3:          out = a W2
    With store_bf16, each tensor the rewritten kernels store in bf16 (h, hg,
    a, out) is rounded to bf16 where it is written; its consumers read the
    rounded value, the statistics are taken before rounding. The saved y is
    rounded to fp16 (a is computed from the unrounded y). fp32: the same
    steps in fp32 arithmetic (see _precision)."""
    dt, mm = _precision(fp32)
    st = _stored(_store(store_bf16), dt)
    sv = _stored(_store_saved(store_bf16), dt)
    x, z, W0, W1, W2, gamma = (np.asarray(t, dtype=dt) for t in (x, z, W0, W1, W2, gamma))
    h_acc = mm(x, W0) + z
    r = rms_factor(h_acc, eps, dt)
    h = st(h_acc)
    hg = st(h_acc * gamma[None, :])
    y_acc = r[:, None] * mm(hg, W1)
    a = st(swiglu(y_acc, dt))
    y = sv(y_acc)
    out = st(mm(a, W2))
    return {"h": h, "r": r, "hg": hg, "y": y, "a": a, "out": out}


def mlp_bwd(fwd: Dict[str, np.ndarray], x, W0, W1, W2, gamma, dout) -> Dict[str, np.ndarray]:
    """Canonical backward of ``mlp_fwd`` for the scalar L = sum(dout * out),
    written out by hand (chain rule through each op in turn):
        da  = dout W2^T ;          dW2 = a^T dout
        dg  = da * u * silu'(g) ;  du = da * silu(g) ;  dy = interleave(dg, du)
        dW1 = h2^T dy ;            dh2 = dy W1^T
        dgamma = sum_rows dh2 * n ;  dn = gamma * dh2
        s   = mean_j(dn * n)      (equals (1/d) sumcols(dh2 * h2), notes s3)
        dh  = r (dn - s n)        (RMSNorm backward)
        dz  = dh ;  dx = dh W0^T ;  dW0 = x^T dh
    """
    x, W0, W1, W2, gamma, dout = (np.asarray(t, dtype=f64) for t in (x, W0, W1, W2, gamma, dout))
    h, r, n, h2, y, a = (fwd[k] for k in ("h", "r", "n", "h2", "y", "a"))
    d = h.shape[1]
    da = dout @ W2.T
    dW2 = a.T @ dout
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g)
    dy[:, 1::2] = da * silu(g)
    dW1 = h2.T @ dy
    dh2 = dy @ W1.T
    dgamma = np.sum(dh2 * n, axis=0)
    dn = gamma[None, :] * dh2
    s = np.sum(dn * n, axis=1) / d
    dh = r[:, None] * (dn - s[:, None] * n)
    dx = dh @ W0.T
    dW0 = x.T @ dh
    return {"da": da, "dy": dy, "dh2": dh2, "s": s, "dh": dh, "dz": dh, "dx": dx,
            "dW0": dW0, "dW1": dW1, "dW2": dW2, "dgamma": dgamma}


def mlp_bwd_reparam(fwd: Dict[str, np.ndarray], x, W0, W1, W2, gamma, dout,
                    store_bf16: bool = False, stat_only: bool = False,
                    fp32: bool = False) -> Dict[str, np.ndarray]:
    """The pages' reverse-fused backward [notes s3 "Reverse Fusion" and
    "Eliminating the RMSNorm backward kernel"], on the tensors saved by
    ``mlp_fwd_reparam`` (h, hg, r, y, a):
        GEMM (dout W2^T) epilogue: f'(h) multiplies into the gradient GEMM:
            dg = da * u * silu'(g), du = da * silu(g)  (one incoming gradient,
            two outgoing: the SwiGLU backward pairwise map, pith Fig. 7),
            s-partial = sum_j dy_j * y_j, stored dyhat = r * dy
        auxiliary: s = (1/d) sumcols(dy * y)
        GEMM (dyhat W1^T) epilogue: P = r dh2;  dh = gamma * P - r^2 s h ;
            dgamma = sum_rows P * h
        dW1 = hg^T dyhat ; dW2 = a^T dout ; dx = dh W0^T ; dW0 = x^T dh
    ``stat_only`` stops after s (and dy, dyhat). fp32: the same steps in
    fp32 arithmetic (see _precision)."""
    dt, mm = _precision(fp32)
    st = _stored(_store(store_bf16), dt)
    x, W0, W1, W2, gamma, dout = (np.asarray(t, dtype=dt) for t in (x, W0, W1, W2, gamma, dout))
    h, hg, r, y, a = (np.asarray(fwd[k], dtype=dt) for k in ("h", "hg", "r", "y", "a"))
    d = h.shape[1]
    da = mm(dout, W2.T)
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g, dt)
    dy[:, 1::2] = da * silu(g, dt)
    s = np.sum(dy * y, axis=1) / d
    dyhat = st(r[:, None] * dy)
    if stat_only:
        return {"dy": dy, "dyhat": dyhat, "s": s}
    P = mm(dyhat, W1.T)
    dh = st(gamma[None, :] * P - (r * r * s)[:, None] * h)
    dgamma = np.sum(P * h, axis=0)
    dW1 = hg.T @ dyhat
    dW2 = a.T @ dout
    dx = st(mm(dh, W0.T))
    dW0 = x.T @ dh
    return {"dy": dy, "dyhat": dyhat, "s": s, "P": P, "dh": dh, "dz": dh, "dx": dx,
            "dW0": dW0, "dW1": dW1, "dW2": dW2, "dgamma": dgamma}


# --------------------------------------------------------------------------
# LayerNorm variant of the block (the pages promise it, they do not work it)
# --------------------------------------------------------------------------

def ln_mlp_fwd(x, z, W0, W1, W2, gamma, beta, eps: float = EPS) -> Dict[str, np.ndarray]:
    """Canonical forward with LayerNorm in place of RMSNorm:
        h = x W0 + z ; mu = mean(h) ; r = 1/sqrt(mean((h - mu)^2) + eps)
        nh = (h - mu) r ; h2 = nh * gamma + beta ; y = h2 W1
        a = silu(y_gate) * y_up ; out = a W2
    """
    x, z, W0, W1, W2, gamma, beta = (np.asarray(t, dtype=f64) for t in (x, z, W0, W1, W2, gamma, beta))
    h = x @ W0 + z
    mu = np.mean(h, axis=1)
    hc = h - mu[:, None]
    r = 1.0 / np.sqrt(np.mean(hc * hc, axis=1) + eps)
    nh = hc * r[:, None]
    h2 = nh * gamma[None, :] + beta[None, :]
    y = h2 @ W1
    a = swiglu(y)
    out = a @ W2
    return {"h": h, "mu": mu, "r": r, "nh": nh, "h2": h2, "y": y, "a": a, "out": out}


def ln_mlp_bwd(fwd, x, W0, W1, W2, gamma, beta, dout) -> Dict[str, np.ndarray]:
    """Canonical backward of ``ln_mlp_fwd`` for L = sum(dout * out); the
    LayerNorm backward is dh = r (dnh - mean(dnh) - nh mean(dnh * nh)),
    dnh = gamma * dh2."""
    x, W0, W1, W2, gamma, beta, dout = (np.asarray(t, dtype=f64) for t in
                                        (x, W0, W1, W2, gamma, beta, dout))
    h, r, nh, h2, y, a = (fwd[k] for k in ("h", "r", "nh", "h2", "y", "a"))
    da = dout @ W2.T
    dW2 = a.T @ dout
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g)
    dy[:, 1::2] = da * silu(g)
    dW1 = h2.T @ dy
    dh2 = dy @ W1.T
    dgamma = np.sum(dh2 * nh, axis=0)
    dbeta = np.sum(dh2, axis=0)
    dnh = gamma[None, :] * dh2
    sa = np.mean(dnh, axis=1)
    sb = np.mean(dnh * nh, axis=1)
    dh = r[:, None] * (dnh - sa[:, None] - nh * sb[:, None])
    return {"dy": dy, "sa": sa, "sb": sb, "dh": dh, "dz": dh, "dx": dh @ W0.T,
            "dW0": x.T @ dh, "dW1": dW1, "dW2": dW2, "dgamma": dgamma, "dbeta": dbeta}


def ln_mlp_fwd_reparam(x, z, W0, W1, W2, gamma, beta, eps: float = EPS,
                       store_bf16: bool = False) -> Dict[str, np.ndarray]:
    """Rewritten LayerNorm forward (this library's reading, following the
    pages' RMSNorm rewrite [notes s2]): GEMM 1's epilogue stores h and
    hg = h * gamma and emits per-row sums of h and h^2; the auxiliary step
    gives mu and r; with the n-vectors w1 = gamma W1 and b1 = beta W1,
        y = r (hg W1) - (r mu) w1 + b1
    which equals (r (h - mu) gamma + beta) W1. With store_bf16 the storage
    points are those of the RMSNorm form (y saved in fp16)."""
    st = _store(store_bf16)
    sv = _store_saved(store_bf16)
    x, z, W0, W1, W2, gamma, beta = (np.asarray(t, dtype=f64) for t in (x, z, W0, W1, W2, gamma, beta))
    h_acc = x @ W0 + z
    d = h_acc.shape[1]
    s1 = np.sum(h_acc, axis=1)
    s2 = np.sum(h_acc * h_acc, axis=1)
    mu = s1 / d
    r = 1.0 / np.sqrt(np.maximum(s2 / d - mu * mu, 0.0) + eps)
    h = st(h_acc)
    hg = st(h_acc * gamma[None, :])
    w1 = gamma @ W1
    b1 = beta @ W1
    y = r[:, None] * (hg @ W1) - (r * mu)[:, None] * w1[None, :] + b1[None, :]
    a = st(swiglu(y))
    out = st(a @ W2)
    return {"h": h, "hg": hg, "mu": mu, "r": r, "w1": w1, "b1": b1, "y": sv(y), "a": a,
            "out": out}


def ln_mlp_bwd_reparam(fwd, x, W0, W1, W2, gamma, beta, dout,
                       store_bf16: bool = False) -> Dict[str, np.ndarray]:
    """Rewritten LayerNorm backward: both statistics move into the epilogue
    of the GEMM that produces dy (as s does in [notes s3]):
        s_a = (1/d) sum_k dy_k w1_k ,  s_b = (1/d) (sum_k dy_k y_k - sum_k dy_k b1_k)
    and with dyhat = r dy, P = dyhat W1^T (= r dh2):
        dh = gamma P - r s_a - r^2 (h - mu) s_b
        dgamma = sum_rows P (h - mu) ,  dbeta = sum_rows P / r
        dW1 = hhat^T dyhat with hhat = (h - mu) gamma + beta / r (= h2 / r)
    """
    st = _store(store_bf16)
    x, W0, W1, W2, gamma, beta, dout = (np.asarray(t, dtype=f64) for t in
                                        (x, W0, W1, W2, gamma, beta, dout))
    h, hg, mu, r, w1, b1, y, a = (fwd[k] for k in ("h", "hg", "mu", "r", "w1", "b1", "y", "a"))
    d = h.shape[1]
    da = dout @ W2.T
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g)
    dy[:, 1::2] = da * silu(g)
    sa = (dy @ w1) / d
    sb = (np.sum(dy * y, axis=1) - dy @ b1) / d
    dyhat = st(r[:, None] * dy)
    nb = ln_norm_bwd_stage(dyhat, W1, h, gamma, beta, r, mu, sa, sb, store_bf16)
    dh = nb["dh"]
    return {"dy": dy, "sa": sa, "sb": sb, "dyhat": dyhat, "P": nb["P"], "dh": dh, "dz": dh,
            "hhat": nb["hhat"], "dgamma": np.sum(nb["dgamma_rows"], axis=0),
            "dbeta": np.sum(nb["dbeta_rows"], axis=0), "dW1": nb["hhat"].T @ dyhat,
            "dW2": a.T @ dout, "dx": st(dh @ W0.T), "dW0": x.T @ dh}


def ln_norm_bwd_stage(dyhat, W1, h, gamma, beta, r, mu, sa, sb, store_bf16: bool = False):
    """The LayerNorm backward as the epilogue of P = dyhat W1^T (the last
    step of ``ln_mlp_bwd_reparam``), on any subset of rows:
        dh = gamma P - r s_a - r^2 s_b (h - mu)
        hhat = (h - mu) gamma + beta / r
    with the per-row terms of the weight gradients, dgamma_rows = P (h - mu)
    and dbeta_rows = P / r (their column sums are dgamma, dbeta)."""
    st = _store(store_bf16)
    dyhat, W1, h, gamma, beta, r, mu, sa, sb = (np.asarray(t, dtype=f64) for t in
                                                (dyhat, W1, h, gamma, beta, r, mu, sa, sb))
    P = dyhat @ W1.T
    hc = h - mu[:, None]
    dh = st(gamma[None, :] * P - (r * sa)[:, None] - (r * r * sb)[:, None] * hc)
    hhat = st(hc * gamma[None, :] + beta[None, :] / r[:, None])
    return {"P": P, "dh": dh, "hhat": hhat, "dgamma_rows": P * hc, "dbeta_rows": P / r[:, None]}


# --------------------------------------------------------------------------
# RoPE on adjacent pairs
# --------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, theta: float = ROPE_THETA) -> np.ndarray:
    """theta_i = theta^(-2i/head_dim), i = 0 .. head_dim/2 - 1."""
    i = np.arange(head_dim // 2, dtype=f64)
    return np.power(f64(theta), -2.0 * i / head_dim)


def rope_cos_sin(pos, head_dim: int, theta: float = ROPE_THETA):
    """cos and sin of angle[p, i] = pos[p] * theta_i, in fp64."""
    ang = np.asarray(pos, dtype=f64)[:, None] * rope_inv_freq(head_dim, theta)[None, :]
    return np.cos(ang), np.sin(ang)


def rope_apply(v, pos, n_rope_cols: int, head_dim: int, theta: float = ROPE_THETA,
               inverse: bool = False, dtype=f64) -> np.ndarray:
    """Rotate each adjacent feature pair (2i, 2i+1) inside every head_dim-wide
    head of the first n_rope_cols columns by angle pos * theta_i (pith Fig. 7:
    RoPE rotates each feature pair and returns two outputs):
        v'_{2i}   = v_{2i} cos - v_{2i+1} sin
        v'_{2i+1} = v_{2i} sin + v_{2i+1} cos
    Columns from n_rope_cols on are returned unchanged. ``inverse`` rotates by
    the negative angle (the transpose of the rotation). dtype: arithmetic
    type (the cos / sin values are computed in fp64 and rounded to it)."""
    v = np.array(v, dtype=dtype, copy=True)
    c, s = (np.asarray(t, dtype=dtype) for t in rope_cos_sin(pos, head_dim, theta))
    if inverse:
        s = -s
    nh = n_rope_cols // head_dim
    for hidx in range(nh):
        base = hidx * head_dim
        e = v[:, base:base + head_dim:2].copy()
        o = v[:, base + 1:base + head_dim:2].copy()
        v[:, base:base + head_dim:2] = e * c - o * s
        v[:, base + 1:base + head_dim:2] = e * s + o * c
    return v


# --------------------------------------------------------------------------
# LM head + cross-entropy
# --------------------------------------------------------------------------

def lmhead_ce(hidden, W, targets) -> Dict[str, np.ndarray]:
    """Per-token loss l_i = -h_{i,y_i} + log sum_k exp(h_{i,k}) on logits
    h = hidden W [notes s2 "Cross-entropy loss"]; natural log, no reduction.
    The log-sum-exp is taken with the row maximum factored out."""
    hidden = np.asarray(hidden, dtype=f64)
    W = np.asarray(W, dtype=f64)
    t = np.asarray(targets, dtype=np.int64)
    logits = hidden @ W
    m = np.max(logits, axis=1)
    lse = m + np.log(np.sum(np.exp(logits - m[:, None]), axis=1))
    tl = logits[np.arange(logits.shape[0]), t]
    return {"lse": lse, "loss": lse - tl, "target_logit": tl}


def lse_two_level(logits, tile: int) -> np.ndarray:
    """The pages' two-level log-sum-exp [notes s2 "Cross-entropy loss";
    thread Pattern 3]: each column tile j keeps its own (max m_j, sum-exp
    s_j = sum exp(l - m_j)); an auxiliary step combines them as
    M = max_j m_j, LSE = M + log sum_j s_j exp(m_j - M)."""
    logits = np.asarray(logits, dtype=f64)
    V = logits.shape[1]
    ms, ss = [], []
    for c0 in range(0, V, tile):
        blk = logits[:, c0:c0 + tile]
        mj = np.max(blk, axis=1)
        ms.append(mj)
        ss.append(np.sum(np.exp(blk - mj[:, None]), axis=1))
    ms = np.stack(ms, axis=1)
    ss = np.stack(ss, axis=1)
    Mx = np.max(ms, axis=1)
    return Mx + np.log(np.sum(ss * np.exp(ms - Mx[:, None]), axis=1))


def lmhead_ce_bwd(hidden, W, targets, dloss) -> Dict[str, np.ndarray]:
    """Backward of the per-token loss for L = sum_i dloss_i * loss_i [notes s2
    "Cross-entropy loss"; thread Pattern 3, which computes it "as in Cut
    Cross Entropy"]: with p = softmax(hidden W) per row and e_t the one-hot
    target row,
        G       = dloss[:, None] * (p - e_t)
        dhidden = G W^T ,  dW = hidden^T G
    """
    hidden = np.asarray(hidden, dtype=f64)
    W = np.asarray(W, dtype=f64)
    t = np.asarray(targets, dtype=np.int64)
    dloss = np.asarray(dloss, dtype=f64)
    logits = hidden @ W
    m = np.max(logits, axis=1)
    p = np.exp(logits - m[:, None])
    p /= np.sum(p, axis=1)[:, None]
    G = p
    G[np.arange(G.shape[0]), t] -= 1.0
    G *= dloss[:, None]
    return {"G": G, "dhidden": G @ W.T, "dW": hidden.T @ G}


def lmhead_ce_dW_columns(hidden, W, targets, dloss, cols, chunk: int = 8192) -> np.ndarray:
    """Columns ``cols`` of dW = hidden^T G for inputs too large to hold all
    logits: the per-row log-sum-exp over the whole vocabulary is taken chunk
    by chunk (per-chunk max and sum-exp, combined as in ``lse_two_level``),
    then G[:, cols] = dloss * (exp(logits[:, cols] - LSE) - onehot)."""
    hidden = np.asarray(hidden, dtype=f64)
    W = np.asarray(W, dtype=f64)
    t = np.asarray(targets, dtype=np.int64)
    dloss = np.asarray(dloss, dtype=f64)
    V = W.shape[1]
    ms, ss = [], []
    for c0 in range(0, V, chunk):
        blk = hidden @ W[:, c0:c0 + chunk]
        mj = np.max(blk, axis=1)
        ms.append(mj)
        ss.append(np.sum(np.exp(blk - mj[:, None]), axis=1))
    ms = np.stack(ms, axis=1)
    ss = np.stack(ss, axis=1)
    Mx = np.max(ms, axis=1)
    lse = Mx + np.log(np.sum(ss * np.exp(ms - Mx[:, None]), axis=1))
    cols = np.asarray(cols, dtype=np.int64)
    Gc = np.exp(hidden @ W[:, cols] - lse[:, None])
    Gc -= (t[:, None] == cols[None, :])
    Gc *= dloss[:, None]
    return hidden.T @ Gc


# --------------------------------------------------------------------------
# Llama-3-8B-shaped non-attention block (output projection .. QKV + RoPE)
# --------------------------------------------------------------------------

def block8b_fwd(o, z, Wo, W1, W2, gamma2, gamma1, Wqkv, pos, n_rope_cols: int,
                head_dim: int, theta: float = ROPE_THETA, eps: float = EPS):
    """Canonical forward of the non-attention part of a layer, with the
    attention output o given:
        h   = o Wo + z                       (output projection + residual)
        n   = rmsnorm(h) ; h2 = n * gamma2
        y   = h2 W1 ; a = silu(g) * u        (SwiGLU MLP)
        out = a W2 + h                       (down projection + residual)
        n'  = rmsnorm(out) ; q_in = n' * gamma1
        qkv = RoPE(q_in Wqkv) on the q and k columns
    """
    o, z, Wo, W1, W2, gamma2, gamma1, Wqkv = (np.asarray(t, dtype=f64) for t in
                                               (o, z, Wo, W1, W2, gamma2, gamma1, Wqkv))
    h = o @ Wo + z
    r = rms_factor(h, eps)
    n = r[:, None] * h
    h2 = n * gamma2[None, :]
    y = h2 @ W1
    a = swiglu(y)
    out = a @ W2 + h
    r1 = rms_factor(out, eps)
    n1 = r1[:, None] * out
    q_in = n1 * gamma1[None, :]
    qkv_pre = q_in @ Wqkv
    qkv = rope_apply(qkv_pre, pos, n_rope_cols, head_dim, theta)
    return {"h": h, "r": r, "n": n, "h2": h2, "y": y, "a": a, "out": out, "r1": r1,
            "n1": n1, "q_in": q_in, "qkv_pre": qkv_pre, "qkv": qkv}


def block8b_bwd(fwd, o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres, pos,
                n_rope_cols: int, head_dim: int, theta: float = ROPE_THETA):
    """Canonical backward of ``block8b_fwd`` for L = sum(dqkv * qkv) +
    sum(dres * out), written out by hand."""
    o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres = (
        np.asarray(t, dtype=f64) for t in (o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres))
    d = fwd["h"].shape[1]
    dqkv_pre = rope_apply(dqkv, pos, n_rope_cols, head_dim, theta, inverse=True)
    dWqkv = fwd["q_in"].T @ dqkv_pre
    dq_in = dqkv_pre @ Wqkv.T
    dgamma1 = np.sum(dq_in * fwd["n1"], axis=0)
    dn1 = gamma1[None, :] * dq_in
    s1 = np.sum(dn1 * fwd["n1"], axis=1) / d
    dout = fwd["r1"][:, None] * (dn1 - s1[:, None] * fwd["n1"]) + dres
    da = dout @ W2.T
    dW2 = fwd["a"].T @ dout
    y = fwd["y"]
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g)
    dy[:, 1::2] = da * silu(g)
    dW1 = fwd["h2"].T @ dy
    dh2 = dy @ W1.T
    dgamma2 = np.sum(dh2 * fwd["n"], axis=0)
    dn = gamma2[None, :] * dh2
    s = np.sum(dn * fwd["n"], axis=1) / d
    dh = fwd["r"][:, None] * (dn - s[:, None] * fwd["n"]) + dout
    do = dh @ Wo.T
    dWo = o.T @ dh
    return {"dqkv_pre": dqkv_pre, "dWqkv": dWqkv, "dgamma1": dgamma1, "s1": s1,
            "dout": dout, "da": da, "dW2": dW2, "dy": dy, "dW1": dW1, "dgamma2": dgamma2,
            "s": s, "dh": dh, "dz": dh, "do": do, "dWo": dWo}


def block8b_fwd_reparam(o, z, Wo, W1, W2, gamma2, gamma1, Wqkv, pos, n_rope_cols: int,
                        head_dim: int, theta: float = ROPE_THETA, eps: float = EPS,
                        store_bf16: bool = False, fp32: bool = False):
    """The pages' rewritten form of ``block8b_fwd`` [notes s2; pith Fig. 4 and
    Fig. 7]: each RMSNorm is split into a GEMM-epilogue statistic on the
    unscaled residual sum and a delayed row scale in the next GEMM's epilogue:
        h = o Wo + z ; hg = h * gamma2 ; r = rms factor of h
        y = r (hg W1) ; a = silu(g) u
        out = a W2 + h ; outg = out * gamma1 ; r1 = rms factor of out
        qkv = RoPE(r1 (outg Wqkv))
    With store_bf16, the tensors the rewritten kernels store in bf16 (h, hg,
    a, out, outg, qkv) are rounded where they are written and read back
    rounded; y and the copy of qkv kept for the backward's statistic
    (``qkv_save``) are rounded to fp16 (the bf16 outputs come from the
    unrounded values). fp32: the same steps in fp32 arithmetic (see
    _precision)."""
    dt, mm = _precision(fp32)
    st = _stored(_store(store_bf16), dt)
    sv = _stored(_store_saved(store_bf16), dt)
    o, z, Wo, W1, W2, gamma2, gamma1, Wqkv = (np.asarray(t, dtype=dt) for t in
                                               (o, z, Wo, W1, W2, gamma2, gamma1, Wqkv))
    h_acc = mm(o, Wo) + z
    r = rms_factor(h_acc, eps, dt)
    h = st(h_acc)
    hg = st(h_acc * gamma2[None, :])
    y = r[:, None] * mm(hg, W1)
    a = st(swiglu(y, dt))
    out_acc = mm(a, W2) + h
    r1 = rms_factor(out_acc, eps, dt)
    out = st(out_acc)
    outg = st(out_acc * gamma1[None, :])
    qkv_acc = rope_apply(r1[:, None] * mm(outg, Wqkv), pos, n_rope_cols, head_dim, theta, dtype=dt)
    return {"h": h, "hg": hg, "r": r, "y": sv(y), "a": a, "out": out, "outg": outg, "r1": r1,
            "qkv": st(qkv_acc), "qkv_save": sv(qkv_acc)}


def block8b_bwd_reparam(fwd, o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres, pos,
                        n_rope_cols: int, head_dim: int, theta: float = ROPE_THETA,
                        store_bf16: bool = False, stat_only: bool = False,
                        fp32: bool = False):
    """Reverse-fused backward of ``block8b_fwd_reparam`` [notes s3]:
        dqh = r1 R^T dqkv (stored) ; s1 = (1/d) sumcols(dqkv * qkv_save)
        P1 = dqh Wqkv^T ; dout = gamma1 P1 - r1^2 s1 out + dres (stored)
        dgamma1 = sum_rows P1 * out ; dWqkv = outg^T dqh
        da = dout W2^T ; dy from the SwiGLU pair rule ; s = (1/d) sumcols(dy * y)
        dyhat = r dy (stored) ; P = dyhat W1^T
        dh = gamma2 P - r^2 s h + dout (stored) ; dgamma2 = sum_rows P * h
        dW2 = a^T dout ; dW1 = hg^T dyhat ; dWo = o^T dh ; do = dh Wo^T
    ``stat_only`` stops after s1 and s (and the tensors they need). fp32:
    the same steps in fp32 arithmetic (see _precision)."""
    dt, mm = _precision(fp32)
    st = _stored(_store(store_bf16), dt)
    o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres = (
        np.asarray(t, dtype=dt) for t in (o, Wo, W1, W2, gamma2, gamma1, Wqkv, dqkv, dres))
    fwd = {k: np.asarray(v, dtype=dt) for k, v in fwd.items()}
    d = fwd["h"].shape[1]
    r, r1 = fwd["r"], fwd["r1"]
    dqh = st(r1[:, None] * rope_apply(dqkv, pos, n_rope_cols, head_dim, theta, inverse=True,
                                      dtype=dt))
    s1 = np.sum(dqkv * fwd["qkv_save"], axis=1) / d
    P1 = mm(dqh, Wqkv.T)
    dout = st(gamma1[None, :] * P1 - (r1 * r1 * s1)[:, None] * fwd["out"] + dres)
    da = mm(dout, W2.T)
    y = fwd["y"]
    g = y[:, 0::2]
    u = y[:, 1::2]
    dy = np.empty_like(y)
    dy[:, 0::2] = da * u * silu_grad(g, dt)
    dy[:, 1::2] = da * silu(g, dt)
    s = np.sum(dy * y, axis=1) / d
    dyhat = st(r[:, None] * dy)
    res = {"dqkv_hat": dqh, "s1": s1, "dout": dout, "dy": dy, "s": s, "dyhat": dyhat}
    if stat_only:
        return res
    P = mm(dyhat, W1.T)
    dh = st(gamma2[None, :] * P - (r * r * s)[:, None] * fwd["h"] + dout)
    res.update({"dgamma1": np.sum(P1 * fwd["out"], axis=0), "dWqkv": fwd["outg"].T @ dqh,
                "dW2": fwd["a"].T @ dout, "dh": dh, "dz": dh,
                "dgamma2": np.sum(P * fwd["h"], axis=0), "dW1": fwd["hg"].T @ dyhat,
                "dWo": o.T @ dh, "do": st(mm(dh, Wo.T))})
    return res


def to64(t) -> np.ndarray:
    """Convert a torch tensor or array-like (e.g. bf16 inputs) to fp64 numpy."""
    if hasattr(t, "detach"):
        import torch  # local: only for the dtype conversion of inputs
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, dtype=f64)

