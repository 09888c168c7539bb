"""Seeded synthetic inputs for the CODA block workloads.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It only draws random numbers and names shapes: it holds none of the
method's arithmetic (no GEMM, normalisation, activation or loss).

All tensors are drawn from one ``torch.Generator`` per workload, in a fixed
order, in fp32, then rounded to bf16 (round-to-nearest-even, torch's own
conversion). Parity tests draw on the CPU (``device="cpu"``, the default);
the benchmark may draw the same distributions on the GPU's generator to start
faster (different numbers, same recipe). The value distributions follow the workload definitions:
activations and upstream gradients ~N(0,1), weights ~N(0, 0.02^2), RMSNorm
weights ~U[0.5, 1.5], LM-head targets ~U{0, V-1} as int32.
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import torch

__all__ = ["BlockShape", "LMHeadShape", "Block8BShape", "WORKLOADS",
           "mlp_block_inputs", "lmhead_inputs", "block8b_inputs"]


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """GEMM -> residual -> RMSNorm -> GEMM(SwiGLU) -> GEMM block: M tokens,
    hidden width d, MLP width f (the gate/up projection is d x 2f)."""
    name: str
    M: int
    d: int
    f: int
    seed: int
    eps: float = 1e-6


@dataclasses.dataclass(frozen=True)
class LMHeadShape:
    """LM head + cross-entropy: hidden [M, d] times W [d, V]."""
    name: str
    M: int
    d: int
    V: int
    seed: int


@dataclasses.dataclass(frozen=True)
class Block8BShape:
    """Non-attention part of a Llama-3-8B-shaped layer: output projection with
    residual, RMSNorm, SwiGLU MLP with residual, RMSNorm, QKV projection with
    RoPE on the q and k heads."""
    name: str
    M: int
    d: int
    f: int
    seq_len: int
    head_dim: int
    n_q_heads: int
    n_kv_heads: int
    theta: float
    seed: int
    eps: float = 1e-6

    @property
    def n_qkv(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def n_rope_cols(self) -> int:
        return (self.n_q_heads + self.n_kv_heads) * self.head_dim


WORKLOADS = {
    # tiny block, forward (correctness only)
    "tiny_mlp_fwd": BlockShape("tiny_mlp_fwd", M=64, d=256, f=512, seed=0),
    # Llama-3-1B-shaped MLP block, forward
    "llama1b_mlp_fwd": BlockShape("llama1b_mlp_fwd", M=8192, d=2048, f=8192, seed=1),
    # LM head + cross-entropy
    "lmhead_ce": LMHeadShape("lmhead_ce", M=8192, d=2048, V=128256, seed=2),
    # backward of the Llama-3-1B-shaped block
    "llama1b_mlp_bwd": BlockShape("llama1b_mlp_bwd", M=8192, d=2048, f=8192, seed=3),
    # Llama-3-8B-shaped non-attention forward + backward
    "llama8b_block": Block8BShape("llama8b_block", M=16384, d=4096, f=14336, seq_len=4096,
                                  head_dim=128, n_q_heads=32, n_kv_heads=8, theta=500000.0,
                                  seed=4),
}


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def _normal(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=g.device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def _uniform(g: torch.Generator, shape, lo: float, hi: float) -> torch.Tensor:
    t = torch.rand(*shape, generator=g, dtype=torch.float32, device=g.device)
    return (t * (hi - lo) + lo).to(torch.bfloat16)


def mlp_block_inputs(shape: BlockShape, with_grad: bool = True, device="cpu") -> Dict[str, torch.Tensor]:
    """x, z [M,d]; W0 [d,d]; W1 [d,2f] (column 2k = gate k, 2k+1 = up k);
    W2 [f,d]; gamma [d]; dout [M,d] (upstream gradient of the block output).
    All bf16 on the CPU, drawn in exactly this order."""
    g = _gen(shape.seed, device)
    M, d, f = shape.M, shape.d, shape.f
    out = {
        "x": _normal(g, (M, d)),
        "z": _normal(g, (M, d)),
        "W0": _normal(g, (d, d), 0.02),
        "W1": _normal(g, (d, 2 * f), 0.02),
        "W2": _normal(g, (f, d), 0.02),
        "gamma": _uniform(g, (d,), 0.5, 1.5),
    }
    if with_grad:
        out["dout"] = _normal(g, (M, d))
    return out


def ln_block_inputs(shape: BlockShape, with_grad: bool = True, device="cpu") -> Dict[str, torch.Tensor]:
    """mlp_block_inputs plus the LayerNorm shift beta [d] bf16 ~N(0, 0.3^2),
    drawn afterwards from the same generator."""
    g = _gen(shape.seed, device)
    M, d, f = shape.M, shape.d, shape.f
    out = {
        "x": _normal(g, (M, d)),
        "z": _normal(g, (M, d)),
        "W0": _normal(g, (d, d), 0.02),
        "W1": _normal(g, (d, 2 * f), 0.02),
        "W2": _normal(g, (f, d), 0.02),
        "gamma": _uniform(g, (d,), 0.5, 1.5),
    }
    if with_grad:
        out["dout"] = _normal(g, (M, d))
    out["beta"] = _normal(g, (d,), 0.3)
    return out


def lmhead_inputs(shape: LMHeadShape, device="cpu") -> Dict[str, torch.Tensor]:
    """hidden [M,d] bf16 ~N(0,1); W [d,V] bf16 ~N(0,0.02^2); targets int32 [M]."""
    g = _gen(shape.seed, device)
    hidden = _normal(g, (shape.M, shape.d))
    W = _normal(g, (shape.d, shape.V), 0.02)
    targets = torch.randint(0, shape.V, (shape.M,), generator=g, dtype=torch.int64,
                            device=g.device).to(torch.int32)
    return {"hidden": hidden, "W": W, "targets": targets}


def block8b_inputs(shape: Block8BShape, with_grad: bool = True, device="cpu") -> Dict[str, torch.Tensor]:
    """o (attention-output stand-in) and z (residual stream) [M,d]; Wo [d,d];
    W1 [d,2f] gate/up interleaved; W2 [f,d]; gamma2 (pre-MLP norm) and gamma1
    (next pre-attention norm) [d]; Wqkv [d, n_qkv]; upstream gradients dqkv
    [M, n_qkv] (of the rotated q,k and of v) and dres [M,d] (of the residual
    stream leaving the block)."""
    g = _gen(shape.seed, device)
    M, d, f, n = shape.M, shape.d, shape.f, shape.n_qkv
    out = {
        "o": _normal(g, (M, d)),
        "z": _normal(g, (M, d)),
        "Wo": _normal(g, (d, d), 0.02),
        "W1": _normal(g, (d, 2 * f), 0.02),
        "W2": _normal(g, (f, d), 0.02),
        "gamma2": _uniform(g, (d,), 0.5, 1.5),
        "gamma1": _uniform(g, (d,), 0.5, 1.5),
        "Wqkv": _normal(g, (d, n), 0.02),
    }
    if with_grad:
        out["dqkv"] = _normal(g, (M, n))
        out["dres"] = _normal(g, (M, d))
    return out


def positions(M: int, seq_len: int) -> torch.Tensor:
    """Token position of each row: sequences of seq_len tokens laid end to end."""
    return torch.arange(M, dtype=torch.int64) % seq_len
