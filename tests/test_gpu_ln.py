"""GPU parity of the LayerNorm variant of the block ("CODA: Rewriting
Transformer Blocks as GEMM-Epilogue Programs", abstract: RMSNorm and LayerNorm
compositions) against the fp64 CPU oracle. The library's reading: GEMM 1
emits per-row sums of h and h^2; GEMM 2 applies the delayed normalisation
r (hg W1) - (r mu) w1 + b1 with w1 = gamma W1, b1 = beta W1; the two
LayerNorm-backward statistics are accumulated in the epilogue of the GEMM
that produces dy, and the LayerNorm backward itself is fused into the GEMM
producing dyhat W1^T. Every call goes through the C ABI."""
import pytest
import torch

from coda_inputs import BlockShape, ln_block_inputs
from oracle import coda_oracle as O
from tests._util import TOL_BF16, TOL_F32, TOL_S_EXACT, assert_close

pytestmark = pytest.mark.gpu

SHAPES = [BlockShape("ln_tiny", M=64, d=256, f=512, seed=60),
          BlockShape("ln_ragged", M=200, d=136, f=200, seed=61),
          BlockShape("ln_multi_tile", M=384, d=520, f=392, seed=62)]


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_ln_block_forward_backward(coda, shape):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    inp = ln_block_inputs(shape)
    if shape.name == "ln_ragged":
        # a row whose h is exactly 0: mu = 0, var = 0, r = 1/sqrt(eps), y = beta W1
        inp["x"][0] = 0
        inp["z"][0] = 0
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.ln_mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"])
    bw = blocks.ln_mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"],
                                 g["dout"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in inp.items()}
    args = (n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"])
    ref = O.ln_mlp_fwd(*args)
    rb = O.ln_mlp_bwd(ref, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"], n["dout"])
    rep = O.ln_mlp_fwd_reparam(*args)
    assert_close("h", fw["h"], ref["h"], TOL_BF16)
    assert_close("hg", fw["hg"], rep["hg"], TOL_BF16)
    assert_close("mu", fw["mu"], ref["mu"], TOL_F32)
    assert_close("r", fw["r"], ref["r"], TOL_F32)
    assert_close("w1", fw["w1"], rep["w1"], TOL_F32)
    assert_close("b1", fw["b1"], rep["b1"], TOL_F32)
    assert_close("y", fw["y"], ref["y"], TOL_BF16)
    assert_close("a", fw["a"], ref["a"], TOL_BF16)
    assert_close("out", fw["out"], ref["out"], TOL_BF16)
    # backward against the canonical (chain rule through LayerNorm) oracle
    for k in ("dx", "dz", "dW0", "dW1", "dW2", "dgamma", "dbeta"):
        assert_close(k, bw[k], rb[k], TOL_BF16)
    # the statistics against the rewritten oracle with the fused path's bf16
    # storage points, and against the exact canonical values with the bound
    # that bf16 storage of hg allows (the same reading as s in the RMSNorm path)
    st = O.ln_mlp_fwd_reparam(*args, store_bf16=True)
    sb = O.ln_mlp_bwd_reparam(st, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"],
                              n["dout"], store_bf16=True)
    assert_close("s_a (storage-rounded oracle)", bw["sa"], sb["sa"], TOL_F32)
    assert_close("s_b (storage-rounded oracle)", bw["sb"], sb["sb"], TOL_F32)
    assert_close("s_a (exact oracle)", bw["sa"], rb["sa"], TOL_S_EXACT)
    assert_close("s_b (exact oracle)", bw["sb"], rb["sb"], TOL_S_EXACT)
    assert_close("hhat", bw["hhat"], ref["h2"] / ref["r"][:, None], TOL_BF16)
    assert_close("dyhat", bw["dyhat"], ref["r"][:, None] * rb["dy"], TOL_BF16)


def test_ln_stage_isolated_statistics(coda):
    """s_a, s_b from the GPU's own saved y, r and w1, b1 (no upstream
    storage cascade): the rewritten oracle fed exactly those tensors."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = SHAPES[2]
    inp = ln_block_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.ln_mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"])
    bw = blocks.ln_mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["beta"],
                                 g["dout"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in inp.items()}
    fwd = {k: O.to64(fw[k]) for k in ("h", "hg", "mu", "r", "w1", "b1", "y", "a")}
    sb = O.ln_mlp_bwd_reparam(fwd, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["beta"],
                              n["dout"], store_bf16=True)
    assert_close("s_a (stage-isolated)", bw["sa"], sb["sa"], TOL_F32)
    assert_close("s_b (stage-isolated)", bw["sb"], sb["sb"], TOL_F32)
    assert_close("dh (stage-isolated)", bw["dh"], sb["dh"], TOL_BF16)
    assert_close("hhat (stage-isolated)", bw["hhat"], sb["hhat"], TOL_BF16)
