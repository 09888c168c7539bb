"""Block-level sequences of libcoda calls (host orchestration only).

Each function enqueues the GEMM-plus-epilogue kernels and auxiliary
reductions of one Transformer-block piece on the current stream, with output
buffers allocated through torch (the caller's allocator). No arithmetic runs
here.

  mlp_block_fwd  -- h = xW0 + z ; r ; y = r (h gamma) W1 ; a = SwiGLU(y) ; out = a W2
  mlp_block_bwd  -- reverse-fused backward: dyhat, s, dh, dgamma, dW0..dW2, dx
  lmhead_ce      -- per-token LSE and loss without logits
  block8b_fwd / block8b_bwd -- output projection .. QKV + RoPE (Llama-3-8B shape)
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import (coda_col_reduce, coda_gemm, coda_gemm_resid_norm_stats,
               coda_gemm_resid_norm_stats_bwd, coda_gemm_rope, coda_gemm_rope_bwd,
               coda_gemm_rowscale_swiglu, coda_gemm_rowscale_swiglu_bwd, coda_lmhead_ce,
               coda_lmhead_ce_workspace_size, coda_lmhead_ce_bwd, coda_lmhead_ce_bwd_workspace_size,
               coda_rope_table, coda_row_rms, coda_row_rms_bwd,
               col_tiles, row_tiles32)

bf16, f16, f32 = torch.bfloat16, torch.float16, torch.float32


def _e(shape, dtype, dev):
    return torch.empty(shape, dtype=dtype, device=dev)


def mlp_block_fwd(x, z, W0, W1, W2, gamma, eps: float = 1e-6, save_y: bool = True,
                  buf: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """GEMM 1 (+ residual, RMSNorm weight, row partials) -> r -> GEMM 2
    (delayed r, SwiGLU) -> GEMM 3 (down projection). Four launches."""
    M, d = x.shape
    two_f = W1.shape[1]
    dev = x.device
    b = buf if buf is not None else {}
    h = b.get("h") if "h" in b else _e((M, d), bf16, dev)
    hg = b.get("hg") if "hg" in b else _e((M, d), bf16, dev)
    part = b.get("part") if "part" in b else _e((col_tiles(d), M), f32, dev)
    r = b.get("r") if "r" in b else _e((M,), f32, dev)
    a = b.get("a") if "a" in b else _e((M, two_f // 2), bf16, dev)
    y = (b.get("y") if "y" in b else _e((M, two_f), f16, dev)) if save_y else None
    out = b.get("out") if "out" in b else _e((M, d), bf16, dev)
    coda_gemm_resid_norm_stats(x, W0, z, gamma, h, hg, part)
    coda_row_rms(part, r, d, eps)
    coda_gemm_rowscale_swiglu(hg, W1, r, a, y)
    coda_gemm(a, W2, out)
    return {"h": h, "hg": hg, "part": part, "r": r, "a": a, "y": y, "out": out}


def mlp_block_bwd(fwd: Dict[str, torch.Tensor], x, W0, W1, W2, gamma, dout,
                  buf: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """Reverse-fused backward of mlp_block_fwd. Launches: SwiGLU-bwd GEMM
    (dyhat, s partials), s, RMSNorm-bwd GEMM (dh, dgamma partials), dgamma,
    dW2, dW1, dW0 (weight gradients, fp32), dx."""
    M, d = x.shape
    two_f = W1.shape[1]
    f = two_f // 2
    dev = x.device
    b = buf if buf is not None else {}
    g = lambda k, shape, dt: b[k] if k in b else _e(shape, dt, dev)
    dyhat = g("dyhat", (M, two_f), bf16)
    spart = g("spart", (col_tiles(f), M), f32)
    s = g("s", (M,), f32)
    dh = g("dh", (M, d), bf16)
    dgp = g("dgpart", (row_tiles32(M), d), f32)
    dgamma = g("dgamma", (d,), f32)
    dW0 = g("dW0", (d, d), f32)
    dW1 = g("dW1", (d, two_f), f32)
    dW2 = g("dW2", (f, d), f32)
    dx = g("dx", (M, d), bf16)
    coda_gemm_rowscale_swiglu_bwd(dout, W2, fwd["y"], fwd["r"], dyhat, spart)
    coda_row_rms_bwd(spart, s, d)
    coda_gemm_resid_norm_stats_bwd(dyhat, W1, fwd["h"], gamma, fwd["r"], s, dh, dgp)
    coda_col_reduce(dgp, dgamma)
    coda_gemm(fwd["a"], dout, dW2, transA=True)
    coda_gemm(fwd["hg"], dyhat, dW1, transA=True)
    coda_gemm(x, dh, dW0, transA=True)
    coda_gemm(dh, W0, dx, transB=True)
    return {"dyhat": dyhat, "s": s, "dh": dh, "dz": dh, "dgamma": dgamma, "dW0": dW0,
            "dW1": dW1, "dW2": dW2, "dx": dx}


def ln_mlp_block_fwd(x, z, W0, W1, W2, gamma, beta, eps: float = 1e-6) -> Dict[str, torch.Tensor]:
    """LayerNorm variant of mlp_block_fwd: GEMM 1 (+ residual, gamma side
    output, sum and sum-of-squares partials) -> mu, r -> GEMM 2 (delayed
    normalisation r (hg W1) - (r mu) w1 + b1, SwiGLU) -> GEMM 3. The
    n-vectors w1 = gamma W1 and b1 = beta W1 come from two one-row GEMMs
    (they change only when the weights do)."""
    from . import (coda_gemm_ln_rowscale_swiglu, coda_gemm_resid_ln_stats, coda_row_ln)
    M, d = x.shape
    two_f = W1.shape[1]
    dev = x.device
    h, hg = _e((M, d), bf16, dev), _e((M, d), bf16, dev)
    psq, psum = _e((col_tiles(d), M), f32, dev), _e((col_tiles(d), M), f32, dev)
    r, mu = _e((M,), f32, dev), _e((M,), f32, dev)
    w1, b1 = _e((1, two_f), f32, dev), _e((1, two_f), f32, dev)
    a, y = _e((M, two_f // 2), bf16, dev), _e((M, two_f), f16, dev)
    out = _e((M, d), bf16, dev)
    coda_gemm(gamma.view(1, d), W1, w1)
    coda_gemm(beta.view(1, d), W1, b1)
    coda_gemm_resid_ln_stats(x, W0, z, gamma, h, hg, psq, psum)
    coda_row_ln(psq, psum, r, mu, d, eps)
    coda_gemm_ln_rowscale_swiglu(hg, W1, r, mu, w1.view(-1), b1.view(-1), a, y)
    coda_gemm(a, W2, out)
    return {"h": h, "hg": hg, "r": r, "mu": mu, "w1": w1.view(-1), "b1": b1.view(-1), "a": a,
            "y": y, "out": out}


def ln_mlp_block_bwd(fwd: Dict[str, torch.Tensor], x, W0, W1, W2, gamma, beta,
                     dout) -> Dict[str, torch.Tensor]:
    """Reverse-fused backward of ln_mlp_block_fwd."""
    from . import (coda_gemm_ln_rowscale_swiglu_bwd, coda_gemm_resid_ln_stats_bwd,
                   coda_row_ln_bwd)
    M, d = x.shape
    two_f = W1.shape[1]
    f = two_f // 2
    dev = x.device
    dyhat = _e((M, two_f), bf16, dev)
    sp, spw, spb = (_e((col_tiles(f), M), f32, dev) for _ in range(3))
    sa, sb = _e((M,), f32, dev), _e((M,), f32, dev)
    dh, hhat = _e((M, d), bf16, dev), _e((M, d), bf16, dev)
    dgp, dbp = _e((row_tiles32(M), d), f32, dev), _e((row_tiles32(M), d), f32, dev)
    dgamma, dbeta = _e((d,), f32, dev), _e((d,), f32, dev)
    dW0, dW1, dW2 = _e((d, d), f32, dev), _e((d, two_f), f32, dev), _e((f, d), f32, dev)
    dx = _e((M, d), bf16, dev)
    coda_gemm_ln_rowscale_swiglu_bwd(dout, W2, fwd["y"], fwd["r"], fwd["w1"], fwd["b1"], dyhat,
                                     sp, spw, spb)
    coda_row_ln_bwd(sp, spw, spb, sa, sb, d)
    coda_gemm_resid_ln_stats_bwd(dyhat, W1, fwd["h"], gamma, beta, fwd["r"], fwd["mu"], sa, sb,
                                 dh, dgp, dbp, hhat=hhat)
    coda_col_reduce(dgp, dgamma)
    coda_col_reduce(dbp, dbeta)
    coda_gemm(fwd["a"], dout, dW2, transA=True)
    coda_gemm(hhat, dyhat, dW1, transA=True)
    coda_gemm(x, dh, dW0, transA=True)
    coda_gemm(dh, W0, dx, transB=True)
    return {"dyhat": dyhat, "sa": sa, "sb": sb, "dh": dh, "dz": dh, "hhat": hhat,
            "dgamma": dgamma, "dbeta": dbeta, "dW0": dW0, "dW1": dW1, "dW2": dW2, "dx": dx}


def lmhead_ce(hidden, W, targets, ws: Optional[torch.Tensor] = None,
              out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """Per-token LSE and CE loss; the logits never reach memory."""
    M = hidden.shape[0]
    V = W.shape[1]
    dev = hidden.device
    if ws is None:
        ws = torch.empty(coda_lmhead_ce_workspace_size(M, V), dtype=torch.uint8, device=dev)
    lse = out["lse"] if out else _e((M,), f32, dev)
    loss = out["loss"] if out else _e((M,), f32, dev)
    coda_lmhead_ce(hidden, W, targets, lse, loss, ws)
    return {"lse": lse, "loss": loss}


def lmhead_ce_bwd(hidden, W, targets, lse, dloss, ws: Optional[torch.Tensor] = None,
                  out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """dhidden and dW of sum(dloss * loss), the logits recomputed chunk by
    chunk and never stored."""
    M, d = hidden.shape
    V = W.shape[1]
    dev = hidden.device
    if ws is None:
        ws = torch.empty(coda_lmhead_ce_bwd_workspace_size(M, V), dtype=torch.uint8, device=dev)
    dh = out["dhidden"] if out else _e((M, d), f32, dev)
    dW = out["dW"] if out else _e((d, V), f32, dev)
    coda_lmhead_ce_bwd(hidden, W, targets, lse, dloss, dh, dW, ws)
    return {"dhidden": dh, "dW": dW}


def rope_table(seq_len: int, head_dim: int, theta: float, device) -> torch.Tensor:
    cs = torch.empty((seq_len, head_dim // 2, 2), dtype=f32, device=device)
    coda_rope_table(cs, seq_len, head_dim, theta)
    return cs


def block8b_fwd(inp: Dict[str, torch.Tensor], seq_len: int, head_dim: int, n_rope_cols: int,
                cos_sin: torch.Tensor, eps: float = 1e-6) -> Dict[str, torch.Tensor]:
    """Output projection + residual + RMSNorm stats -> r -> SwiGLU MLP with
    delayed r -> down projection + residual + RMSNorm stats -> r1 -> QKV with
    delayed r1 and RoPE. Seven launches."""
    o, z = inp["o"], inp["z"]
    M, d = o.shape
    two_f = inp["W1"].shape[1]
    nq = inp["Wqkv"].shape[1]
    dev = o.device
    h, hg = _e((M, d), bf16, dev), _e((M, d), bf16, dev)
    part = _e((col_tiles(d), M), f32, dev)
    r = _e((M,), f32, dev)
    a = _e((M, two_f // 2), bf16, dev)
    y = _e((M, two_f), f16, dev)
    out, outg = _e((M, d), bf16, dev), _e((M, d), bf16, dev)
    part1 = _e((col_tiles(d), M), f32, dev)
    r1 = _e((M,), f32, dev)
    qkv = _e((M, nq), bf16, dev)
    qkv_save = _e((M, nq), f16, dev)
    coda_gemm_resid_norm_stats(o, inp["Wo"], z, inp["gamma2"], h, hg, part)
    coda_row_rms(part, r, d, eps)
    coda_gemm_rowscale_swiglu(hg, inp["W1"], r, a, y)
    coda_gemm_resid_norm_stats(a, inp["W2"], h, inp["gamma1"], out, outg, part1)
    coda_row_rms(part1, r1, d, eps)
    coda_gemm_rope(outg, inp["Wqkv"], r1, cos_sin, seq_len, head_dim, n_rope_cols, qkv, qkv_save)
    return {"h": h, "hg": hg, "r": r, "a": a, "y": y, "out": out, "outg": outg, "r1": r1,
            "qkv": qkv, "qkv_save": qkv_save}


def block8b_bwd(fwd: Dict[str, torch.Tensor], inp: Dict[str, torch.Tensor], seq_len: int,
                head_dim: int, n_rope_cols: int, cos_sin: torch.Tensor) -> Dict[str, torch.Tensor]:
    """Backward for upstream gradients dqkv (of the rotated qkv) and dres (of
    the residual stream leaving the block)."""
    o = inp["o"]
    M, d = o.shape
    two_f = inp["W1"].shape[1]
    f = two_f // 2
    nq = inp["Wqkv"].shape[1]
    dev = o.device
    dqh = _e((M, nq), bf16, dev)
    s1 = _e((M,), f32, dev)
    coda_gemm_rope_bwd(inp["dqkv"], fwd["qkv_save"], fwd["r1"], cos_sin, seq_len, head_dim,
                       n_rope_cols, dqh, s1, d)
    dout = _e((M, d), bf16, dev)
    dgp1 = _e((row_tiles32(M), d), f32, dev)
    coda_gemm_resid_norm_stats_bwd(dqh, inp["Wqkv"], fwd["out"], inp["gamma1"], fwd["r1"], s1,
                                   dout, dgp1, dresid=inp["dres"])
    dgamma1 = _e((d,), f32, dev)
    coda_col_reduce(dgp1, dgamma1)
    dWqkv = _e((d, nq), f32, dev)
    coda_gemm(fwd["outg"], dqh, dWqkv, transA=True)
    dyhat = _e((M, two_f), bf16, dev)
    spart = _e((col_tiles(f), M), f32, dev)
    coda_gemm_rowscale_swiglu_bwd(dout, inp["W2"], fwd["y"], fwd["r"], dyhat, spart)
    s = _e((M,), f32, dev)
    coda_row_rms_bwd(spart, s, d)
    dW2 = _e((f, d), f32, dev)
    coda_gemm(fwd["a"], dout, dW2, transA=True)
    dh = _e((M, d), bf16, dev)
    dgp2 = _e((row_tiles32(M), d), f32, dev)
    coda_gemm_resid_norm_stats_bwd(dyhat, inp["W1"], fwd["h"], inp["gamma2"], fwd["r"], s, dh,
                                   dgp2, dresid=dout)
    dgamma2 = _e((d,), f32, dev)
    coda_col_reduce(dgp2, dgamma2)
    dW1 = _e((d, two_f), f32, dev)
    coda_gemm(fwd["hg"], dyhat, dW1, transA=True)
    dWo = _e((d, d), f32, dev)
    coda_gemm(o, dh, dWo, transA=True)
    do = _e((M, d), bf16, dev)
    coda_gemm(dh, inp["Wo"], do, transB=True)
    return {"dqkv_hat": dqh, "s1": s1, "dout": dout, "dgamma1": dgamma1, "dgpart1": dgp1,
            "dgpart2": dgp2, "dWqkv": dWqkv,
            "dyhat": dyhat, "s": s, "dW2": dW2, "dh": dh, "dz": dh, "dgamma2": dgamma2,
            "dW1": dW1, "dWo": dWo, "do": do}


class CapturedStep:
    """A fixed sequence of library calls (same shapes, same buffers every
    time) captured once into a CUDA graph and replayed: one host launch per
    step instead of one per kernel, with the kernels' programmatic
    dependencies kept as graph edges. ``fn`` runs the calls on the current
    stream; it is run ``warmup`` times first (that performs the library's
    one-time per-kernel setup, which must not happen during capture).
    Tensors that ``fn`` allocates come from the graph's private memory pool
    and hold the results of the latest replay."""

    def __init__(self, fn, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.outputs = fn()

    def replay(self):
        self.graph.replay()
        return self.outputs

