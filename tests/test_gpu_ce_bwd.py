"""GPU parity of the LM-head cross-entropy backward (logits recomputed per
vocabulary chunk, never stored) against the fp64 oracle: a ragged shape run
with several chunks (small workspace) and with one chunk, and the full
8192 x 2048 x 128256 shape (dhidden on sampled rows, which are independent;
dW on sampled columns, whose oracle needs every row's log-sum-exp). Also the
fp32 accumulate form of coda_gemm (C += A B) that the backward uses."""
import numpy as np
import pytest
import torch

from coda_inputs import LMHeadShape, WORKLOADS, lmhead_inputs
from oracle import coda_oracle as O
from tests._util import TOL_BF16, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def _dloss(M, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(M, generator=g) + 0.5) / M


@pytest.mark.parametrize("transB", [0, 1])
def test_gemm_fp32_accumulate(coda, transB):
    g = torch.Generator().manual_seed(5)
    M, N, K = 200, 264, 136
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(*((N, K) if transB else (K, N)), generator=g).to(torch.bfloat16)
    C0 = torch.randn(M, N, generator=g)
    C = C0.cuda()
    coda.coda_gemm(A.cuda(), B.cuda(), C, transB=bool(transB), resid=C)
    torch.cuda.synchronize()
    b = to64(B).T if transB else to64(B)
    assert_close("C += A B (fp32)", C, to64(C0) + to64(A) @ b, 1e-5)


@pytest.mark.parametrize("small_ws", [True, False])
def test_ce_bwd_ragged(coda, small_ws):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = LMHeadShape("ce_bwd", M=200, d=136, V=1000, seed=24)
    inp = lmhead_inputs(sh)
    t = inp["targets"]
    t[:4] = torch.tensor([0, 999, 255, 256], dtype=torch.int32)
    dl = _dloss(sh.M, 1)
    h, W = inp["hidden"].cuda(), inp["W"].cuda()
    fw = blocks.lmhead_ce(h, W, t.cuda())
    ws = None
    if small_ws:  # 256-column chunks: 4 chunks, the last one ragged
        ws = torch.empty(sh.M * 256 * 2, dtype=torch.uint8, device="cuda")
    bw = blocks.lmhead_ce_bwd(h, W, t.cuda(), fw["lse"], dl.cuda(), ws=ws)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    ref = O.lmhead_ce_bwd(O.to64(inp["hidden"]), O.to64(inp["W"]), t.numpy(), dl.double().numpy())
    assert_close("dhidden", bw["dhidden"], ref["dhidden"], TOL_BF16)
    assert_close("dW", bw["dW"], ref["dW"], TOL_BF16)


def test_ce_bwd_one_row(coda):
    """One token over the smallest vocabulary (V = 8): one partial tile in
    every GEMM of the backward."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = LMHeadShape("ce_bwd_one", M=1, d=64, V=8, seed=25)
    inp = lmhead_inputs(sh)
    t = inp["targets"]
    dl = _dloss(sh.M, 1)
    h, W = inp["hidden"].cuda(), inp["W"].cuda()
    fw = blocks.lmhead_ce(h, W, t.cuda())
    bw = blocks.lmhead_ce_bwd(h, W, t.cuda(), fw["lse"], dl.cuda())
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    ref = O.lmhead_ce_bwd(O.to64(inp["hidden"]), O.to64(inp["W"]), t.numpy(), dl.double().numpy())
    assert_close("dhidden", bw["dhidden"], ref["dhidden"], TOL_BF16)
    assert_close("dW", bw["dW"], ref["dW"], TOL_BF16)


def test_ce_bwd_full_size(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = WORKLOADS["lmhead_ce"]
    inp = lmhead_inputs(sh)
    dl = _dloss(sh.M, 2)
    h, W, t = inp["hidden"].cuda(), inp["W"].cuda(), inp["targets"].cuda()
    fw = blocks.lmhead_ce(h, W, t)
    bw = blocks.lmhead_ce_bwd(h, W, t, fw["lse"], dl.cuda())
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rng = np.random.default_rng(3)
    rows = np.array(sorted(set(rng.choice(sh.M, 24, replace=False).tolist()) | {0, sh.M - 1}))
    Wd = O.to64(inp["W"])
    ref = O.lmhead_ce_bwd(O.to64(inp["hidden"][rows]), Wd, inp["targets"][rows].numpy(),
                          dl[rows].double().numpy())
    assert_close("dhidden (sampled rows)", bw["dhidden"].cpu()[rows], ref["dhidden"], TOL_BF16)
    cols = np.array(sorted(set(rng.choice(sh.V, 24, replace=False).tolist())
                           | {0, 4095, 4096, 16383, 16384, 114687, 114688, sh.V - 1,
                              int(inp["targets"][0])}))
    dWc = O.lmhead_ce_dW_columns(O.to64(inp["hidden"]), Wd, inp["targets"].numpy(),
                                 dl.double().numpy(), cols)
    assert_close("dW (sampled columns)", bw["dW"].cpu()[:, cols], dWc, TOL_BF16)
    # every row of G sums to zero, so every row of dW sums to zero up to the
    # bf16 rounding of G: at most a few bf16 units of the row's 2-norm
    dW64 = bw["dW"].double()
    ratio = (dW64.sum(1).abs() / dW64.norm(dim=1)).max().item()
    print(f"max |row sum of dW| / ||row||_2 = {ratio:.3e}")
    assert ratio < 1e-2
