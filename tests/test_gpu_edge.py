"""GPU edge cases of the hot path through the C ABI: the closed-form
degenerate cases of the LM-head cross-entropy ("Reading notes on CODA", s2
"Cross-entropy loss": l_i = -h_{i,y_i} + log sum_k exp h_{i,k}) with values
from tests/golden/closed_forms.json, and outputs larger than 4 GiB (64-bit
addressing in the TMA stores and the partial buffers)."""
import json
import os

import numpy as np
import pytest
import torch

from tests._util import TOL_BF16, assert_close, to64

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def test_lmhead_zero_weights_gives_ln_V(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    M, d, V = 300, 64, 128256
    g = torch.Generator().manual_seed(70)
    hidden = torch.randn(M, d, generator=g).to(torch.bfloat16).cuda()
    W = torch.zeros(d, V, dtype=torch.bfloat16, device="cuda")
    t = torch.randint(0, V, (M,), generator=g, dtype=torch.int32).cuda()
    res = blocks.lmhead_ce(hidden, W, t)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    ref = np.full(M, GOLDEN["ln_V_128256"])
    assert_close("lse, W = 0", res["lse"], ref, 1e-6)
    assert_close("loss, W = 0", res["loss"], ref, 1e-6)


def test_lmhead_exact_logits_closed_form(coda):
    """hidden = e_0 and W[0, :] = eight bf16-exact logits, so the logits are
    exactly those values; every target in turn."""
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    gold = GOLDEN["ce_exact8"]
    V, d = 8, 8
    hidden = torch.zeros(V, d, dtype=torch.bfloat16)
    hidden[:, 0] = 1
    W = torch.zeros(d, V, dtype=torch.bfloat16)
    W[0] = torch.tensor(gold["logits"], dtype=torch.bfloat16)
    assert torch.equal(W[0].double(), torch.tensor(gold["logits"], dtype=torch.float64))
    t = torch.arange(V, dtype=torch.int32)
    res = blocks.lmhead_ce(hidden.cuda(), W.cuda(), t.cuda())
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    assert_close("lse, exact logits", res["lse"], np.full(V, gold["lse"]), 1e-6)
    assert_close("loss, exact logits", res["loss"], np.array(gold["loss"]), 1e-6)


def _rows(M, seed):
    rng = np.random.default_rng(seed)
    return np.array(sorted(set(rng.choice(M, 24, replace=False).tolist()) | {0, 1, M - 2, M - 1}))


def test_gemm_output_beyond_4GiB(coda):
    """C = A B with C of 65536 x 32768 bf16 = 4 GiB (more than 2^31 elements)."""
    M, N, K = 65536, 32768, 64
    g = torch.Generator().manual_seed(71)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = _rows(M, 72)
    ref = to64(A)[rows] @ to64(B)
    assert_close("C rows of a 4 GiB output", C[rows].cpu(), ref, TOL_BF16)
    del C
    torch.cuda.empty_cache()


def test_swiglu_saved_copy_beyond_4GiB(coda):
    """The SwiGLU GEMM with a 65536 x 32768 fp16 saved y (4 GiB) and a 2 GiB a."""
    M, two_f, K = 65536, 32768, 64
    g = torch.Generator().manual_seed(73)
    hg = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(K, two_f, generator=g) * 0.1).to(torch.bfloat16)
    r = torch.rand(M, generator=g) + 0.5
    a = torch.empty(M, two_f // 2, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, two_f, dtype=torch.float16, device="cuda")
    coda.coda_gemm_rowscale_swiglu(hg.cuda(), W1.cuda(), r.cuda(), a, y)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = _rows(M, 74)
    yref = (to64(hg)[rows] @ to64(W1)) * r.double().numpy()[rows][:, None]
    aref = yref[:, 0::2] / (1 + np.exp(-yref[:, 0::2])) * yref[:, 1::2]
    assert_close("y rows of a 4 GiB saved copy", y[rows].cpu(), yref, 1e-3)
    assert_close("a rows", a[rows].cpu(), aref, TOL_BF16)
    del a, y
    torch.cuda.empty_cache()
