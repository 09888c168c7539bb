"""CUDA-graph capture of library calls: a whole block forward + backward and
the LM-head CE captured once and replayed give the same bits as the eager
calls (the kernels are deterministic), replay after replay, with the
kernels' programmatic dependencies inside the graph."""
import pytest
import torch

from coda_inputs import BlockShape, LMHeadShape, mlp_block_inputs, lmhead_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def test_graph_replay_matches_eager(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    sh = BlockShape("graph_block", M=1000, d=512, f=776, seed=80)
    g = {k: v.cuda() for k, v in mlp_block_inputs(sh).items()}
    ci = {k: v.cuda() for k, v in lmhead_inputs(LMHeadShape("graph_ce", M=512, d=512, V=5000,
                                                             seed=81)).items()}

    def step():
        fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
        bw = blocks.mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["dout"])
        ce = blocks.lmhead_ce(ci["hidden"], ci["W"], ci["targets"])
        return {"out": fw["out"], "dx": bw["dx"], "dW1": bw["dW1"], "dgamma": bw["dgamma"],
                "s": bw["s"], "loss": ce["loss"]}

    eager = {k: v.clone() for k, v in step().items()}
    torch.cuda.synchronize()
    cap = blocks.CapturedStep(step)
    for _ in range(3):
        out = cap.replay()
        torch.cuda.synchronize()
        assert coda.get_device_error() == 0
        for k, v in eager.items():
            assert torch.equal(out[k], v), k
