"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (same entry points, same shapes):

  * Llama-3-1B-shaped block forward (M=8192, d=2048, f=8192): every output
    on sampled rows against the oracle (rows are independent in the forward).
  * LM head + CE (8192 x 2048 x 128256): LSE and loss on sampled rows.
  * backward of the 1B block: every output against the full fp64 oracle;
    the same for the LayerNorm variant of the block.
  * Llama-3-8B-shaped block forward + backward (M=16384, d=4096, f=14336):
    per-row outputs on sampled rows; weight gradients through the property
    dW v = A^T (G v) for random v (A, G the GPU's own saved operands, which
    the sampled rows check); dgamma through its per-32-row partials.
  * the same block on one 4096-token sequence at full widths: every weight
    gradient and both dgamma element by element against the full canonical
    oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

from coda_inputs import (WORKLOADS, BlockShape, mlp_block_inputs, ln_block_inputs, lmhead_inputs,
                         block8b_inputs, positions)
from oracle import coda_oracle as O
from tests._util import (TOL_BF16, TOL_F32, assert_close, assert_stat_near_exact,
                         chained_stat_tol, rows_8b_full, sampled_rows, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def test_llama1b_forward_sampled_rows(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = WORKLOADS["llama1b_mlp_fwd"]
    inp = mlp_block_inputs(sh, with_grad=False)
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = sampled_rows(sh.M)
    n = {k: O.to64(v) for k, v in inp.items()}
    ref = O.mlp_fwd(n["x"][rows], n["z"][rows], n["W0"], n["W1"], n["W2"], n["gamma"])
    hg_ref = ref["h"] * n["gamma"][None, :]
    for k, want, tol in (("h", ref["h"], TOL_BF16), ("hg", hg_ref, TOL_BF16),
                         ("r", ref["r"], TOL_F32), ("y", ref["y"], TOL_BF16),
                         ("a", ref["a"], TOL_BF16), ("out", ref["out"], TOL_BF16)):
        assert_close(k, fw[k][torch.from_numpy(rows).cuda()], want, tol)


def test_lmhead_ce_full_size_sampled_rows(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = WORKLOADS["lmhead_ce"]
    inp = lmhead_inputs(sh)
    res = blocks.lmhead_ce(inp["hidden"].cuda(), inp["W"].cuda(), inp["targets"].cuda())
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = sampled_rows(sh.M, 40, 1)
    ref = O.lmhead_ce(O.to64(inp["hidden"][rows]), O.to64(inp["W"]), inp["targets"][rows].numpy())
    assert_close("lse", res["lse"].cpu()[rows], ref["lse"], TOL_F32)
    assert_close("loss", res["loss"].cpu()[rows], ref["loss"], TOL_F32)
    # every row: finite, and LSE >= the target logit's share (loss >= 0)
    loss = res["loss"].cpu()
    assert torch.isfinite(loss).all() and (loss > -1e-3).all()


def test_llama1b_backward_full_oracle(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = WORKLOADS["llama1b_mlp_bwd"]
    inp = mlp_block_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
    bw = blocks.mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["dout"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in inp.items()}
    ref = O.mlp_fwd(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"])
    assert_close("out", fw["out"], ref["out"], TOL_BF16)
    assert_close("r", fw["r"], ref["r"], TOL_F32)
    rb = O.mlp_bwd(ref, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["dout"])
    for k in ("dx", "dz", "dW0", "dW1", "dW2", "dgamma"):
        assert_close(k, bw[k], rb[k], TOL_BF16)
    s_exact = rb["s"]
    del ref, rb
    st = O.mlp_fwd_reparam(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"], store_bf16=True)
    sb = O.mlp_bwd_reparam(st, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["dout"],
                           store_bf16=True, stat_only=True)
    tol = chained_stat_tol("llama1b_mlp_bwd", "s")
    assert_close("s (storage-rounded oracle)", bw["s"], sb["s"], tol)
    assert_stat_near_exact("s (exact oracle)", bw["s"], s_exact, sb["s"], tol)


def test_llama1b_layernorm_block_full_oracle(coda):
    """The LayerNorm variant at the Llama-3-1B MLP shape (M = 8192, d = 2048,
    f = 8192, seed 8), forward and backward, every output against the full
    fp64 canonical oracle; s_a, s_b also against the storage-rounded
    rewritten oracle."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = BlockShape("llama1b_ln_mlp", M=8192, d=2048, f=8192, seed=8)
    inp = ln_block_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.ln_mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"])
    bw = blocks.ln_mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"],
                                 g["dout"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in inp.items()}
    args = (n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"])
    ref = O.ln_mlp_fwd(*args)
    for k in ("h", "y", "a", "out"):
        assert_close(k, fw[k], ref[k], TOL_BF16)
    assert_close("mu", fw["mu"], ref["mu"], TOL_F32)
    assert_close("r", fw["r"], ref["r"], TOL_F32)
    rb = O.ln_mlp_bwd(ref, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"], n["dout"])
    for k in ("dx", "dz", "dW0", "dW1", "dW2", "dgamma", "dbeta"):
        assert_close(k, bw[k], rb[k], TOL_BF16)
    sa_exact, sb_exact = rb["sa"], rb["sb"]
    del ref, rb
    st = O.ln_mlp_fwd_reparam(*args, store_bf16=True)
    sb = O.ln_mlp_bwd_reparam(st, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"],
                              n["dout"], store_bf16=True)
    assert_close("s_a (storage-rounded oracle)", bw["sa"], sb["sa"], TOL_F32)
    assert_close("s_b (storage-rounded oracle)", bw["sb"], sb["sb"], TOL_F32)
    assert_stat_near_exact("s_a (exact oracle)", bw["sa"], sa_exact, sb["sa"])
    assert_stat_near_exact("s_b (exact oracle)", bw["sb"], sb_exact, sb["sb"])


def _proj_check(name, dW, A, G, seed):
    """dW = A^T G (A [M, p], G [M, q]); check dW v = A^T (G v) for random v."""
    rng = np.random.default_rng(seed)
    q = G.shape[1]
    v = rng.standard_normal((q, 2))
    lhs = to64(dW) @ v
    Gv = np.zeros((G.shape[0], 2))
    for i in range(0, G.shape[0], 2048):
        Gv[i:i + 2048] = to64(G[i:i + 2048]) @ v
    rhs = np.zeros((A.shape[1], 2))
    for i in range(0, A.shape[0], 2048):
        rhs += to64(A[i:i + 2048]).T @ Gv[i:i + 2048]
    assert_close(f"{name} (dW v = A^T G v)", lhs, rhs, 1e-3)


def test_llama8b_block_full_size(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = WORKLOADS["llama8b_block"]
    inp = block8b_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    cs = blocks.rope_table(sh.seq_len, sh.head_dim, sh.theta, "cuda")
    fw = blocks.block8b_fwd(g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    bw = blocks.block8b_bwd(fw, g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    # two whole 32-row blocks (for the dgamma partials) plus scattered rows
    rows = rows_8b_full(sh.M)
    n = {k: O.to64(v[rows]) if v.dim() == 2 and v.shape[0] == sh.M else O.to64(v)
         for k, v in inp.items()}
    pos = positions(sh.M, sh.seq_len).numpy()[rows]
    ref = O.block8b_fwd(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                        n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    rb = O.block8b_bwd(ref, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                       n["Wqkv"], n["dqkv"], n["dres"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    ri = torch.from_numpy(rows).cuda()
    for k, want, tol in (("h", ref["h"], TOL_BF16), ("r", ref["r"], TOL_F32),
                         ("out", ref["out"], TOL_BF16), ("r1", ref["r1"], TOL_F32),
                         ("qkv", ref["qkv"], TOL_BF16)):
        assert_close(k, fw[k][ri], want, tol)
    for k in ("dout", "dz", "do"):
        assert_close(k, bw[k][ri], rb[k], TOL_BF16)
    fr = O.block8b_fwd_reparam(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                               n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim, sh.theta, store_bf16=True)
    br = O.block8b_bwd_reparam(fr, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                               n["Wqkv"], n["dqkv"], n["dres"], pos, sh.n_rope_cols, sh.head_dim,
                               sh.theta, store_bf16=True, stat_only=True)
    # s' and s sit at the end of long bf16 storage cascades (h, hg, a, out,
    # outg forward; dqkv_hat, dout backward): where fp32 tensor-core and fp64
    # arithmetic round a stored tensor to different bf16 neighbours they
    # move; the bound is derived from how far the oracle itself moves when it
    # runs in the tensor-core model's fp32 (tests/golden/stat_spread.json).
    # The kernels' own arithmetic is pinned at 1e-3 in test_gpu_stages.py.
    for k in ("s1", "s"):
        tol = chained_stat_tol("llama8b_block", k)
        assert_close(f"{k} (storage-rounded oracle)", bw[k][ri], br[k], tol)
        assert_stat_near_exact(f"{k} (exact oracle)", bw[k][ri], rb[k], br[k], tol)
    # dgamma: the column reduction of its per-32-row partials, and the
    # partials of the two sampled 32-row blocks against the oracle
    for k in ("1", "2"):
        gp = to64(bw["dgpart" + k])
        assert_close(f"dgamma{k} = sum of partials", bw["dgamma" + k], gp.sum(0), 1e-5)
    for blk_rows, j in ((np.arange(0, 32), 0), (np.arange(sh.M - 32, sh.M), sh.M // 32 - 1)):
        nb = {k: O.to64(v[blk_rows]) if v.dim() == 2 and v.shape[0] == sh.M else O.to64(v)
              for k, v in inp.items()}
        pb = positions(sh.M, sh.seq_len).numpy()[blk_rows]
        fb = O.block8b_fwd(nb["o"], nb["z"], nb["Wo"], nb["W1"], nb["W2"], nb["gamma2"],
                           nb["gamma1"], nb["Wqkv"], pb, sh.n_rope_cols, sh.head_dim, sh.theta)
        bb = O.block8b_bwd(fb, nb["o"], nb["Wo"], nb["W1"], nb["W2"], nb["gamma2"], nb["gamma1"],
                           nb["Wqkv"], nb["dqkv"], nb["dres"], pb, sh.n_rope_cols, sh.head_dim,
                           sh.theta)
        assert_close(f"dgamma1 partial of rows {blk_rows[0]}..", bw["dgpart1"][j], bb["dgamma1"], TOL_BF16)
        assert_close(f"dgamma2 partial of rows {blk_rows[0]}..", bw["dgpart2"][j], bb["dgamma2"], TOL_BF16)
    # weight gradients at full size through dW v = A^T (G v)
    _proj_check("dWqkv", bw["dWqkv"], fw["outg"], bw["dqkv_hat"], 1)
    _proj_check("dW2", bw["dW2"], fw["a"], bw["dout"], 2)
    _proj_check("dW1", bw["dW1"], fw["hg"], bw["dyhat"], 3)
    _proj_check("dWo", bw["dWo"], g["o"], bw["dh"], 4)


def test_llama8b_one_sequence_weight_gradients_full_oracle(coda):
    """One 4096-token sequence of the Llama-3-8B-shaped block (d = 4096,
    f = 14336, QKV 6144, RoPE theta 5e5): dWo, dW1, dW2, dWqkv, dgamma1 and
    dgamma2 element by element against the full fp64 canonical oracle."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = dataclasses.replace(WORKLOADS["llama8b_block"], M=4096)
    inp = block8b_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    cs = blocks.rope_table(sh.seq_len, sh.head_dim, sh.theta, "cuda")
    fw = blocks.block8b_fwd(g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    bw = blocks.block8b_bwd(fw, g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    got = {k: to64(bw[k]) for k in ("dWo", "dW1", "dW2", "dWqkv", "dgamma1", "dgamma2")}
    del fw, bw, g
    torch.cuda.empty_cache()
    n = {k: O.to64(v) for k, v in inp.items()}
    pos = positions(sh.M, sh.seq_len).numpy()
    ref = O.block8b_fwd(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                        n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    rb = O.block8b_bwd(ref, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                       n["Wqkv"], n["dqkv"], n["dres"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    for k in ("dWo", "dW1", "dW2", "dWqkv", "dgamma1", "dgamma2"):
        assert_close(f"{k} (one 4096-token sequence)", got[k], rb[k], TOL_BF16)
