"""Numerics of the rewritten GEMM-RMSNorm-GEMM against the standard bf16 path
("CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs", Fig. 6
caption: BF16 outputs compared with a high-precision reference on Llama-3-8B
layers, each path's error normalised by the PyTorch path's error).

Layers: Llama-3-8B shapes (d = 4096, 2f = 28672), synthetic weights
(the workloads' distributions; no trained weights exist here), three seeds
standing in for three layers, 2048 tokens each. Reference: the fp64 oracle.
Paths:
  * fused (this library): y = r * ((x W0 + z) * gamma) W1, y as saved for the
    backward (fp16) and also rounded to bf16 for a like-for-like comparison;
  * PyTorch bf16: h = x @ W0 + z (bf16), F.rms_norm (bf16), @ W1 (bf16).
Error: ||y - y_ref||_F / ||y_ref||_F. The test prints the table and asserts
that the fused path's bf16 output is no less accurate than the PyTorch path,
the pages' qualitative claim ("Reading notes on CODA", s5 "Takeaways": the
rewrite keeps accumulations in higher precision longer and lowers the
relative error against PyTorch slightly); they print no values to match.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from coda_inputs import BlockShape, mlp_block_inputs
from oracle import coda_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def _fro(a, ref):
    a = np.asarray(a, dtype=np.float64)
    return float(np.linalg.norm(a - ref) / np.linalg.norm(ref))


def test_gemm_rmsnorm_gemm_error_vs_pytorch_path(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    rows = []
    for layer, seed in enumerate((50, 51, 52)):
        sh = BlockShape(f"llama8b_layer{layer}", M=2048, d=4096, f=14336, seed=seed)
        inp = mlp_block_inputs(sh, with_grad=False)
        g = {k: v.cuda() for k, v in inp.items()}
        fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
        with torch.no_grad():
            h = g["x"] @ g["W0"] + g["z"]
            y_pt = F.rms_norm(h, (sh.d,), g["gamma"], 1e-6) @ g["W1"]
        torch.cuda.synchronize()
        assert coda.get_device_error() == 0
        n = {k: O.to64(v) for k, v in inp.items()}
        y_ref = O.mlp_fwd(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"])["y"]
        e_pt = _fro(O.to64(y_pt), y_ref)
        e_f16 = _fro(O.to64(fw["y"]), y_ref)
        e_bf = _fro(O.to64(fw["y"].to(torch.bfloat16)), y_ref)
        rows.append((sh.name, e_pt, e_f16, e_bf))
    print("\nlayer              err(PyTorch bf16)  err(fused, fp16 y)  err(fused, bf16 y)  "
          "ratio fp16  ratio bf16")
    for name, e_pt, e_f16, e_bf in rows:
        print(f"{name:18s} {e_pt:17.3e} {e_f16:19.3e} {e_bf:19.3e} {e_f16 / e_pt:11.3f} "
              f"{e_bf / e_pt:11.3f}")
    for name, e_pt, e_f16, e_bf in rows:
        assert e_bf <= e_pt * 1.05, name
        assert e_f16 < e_pt, name
