"""GPU parity of the fused block kernels against the fp64 CPU oracle, at
sizes the oracle finishes in seconds: the tiny workload (M=64, d=256, f=512,
seed 0) and ragged shapes that span several tiles and end in partial tiles in
M, N and K. Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from coda_inputs import BlockShape, LMHeadShape, Block8BShape, WORKLOADS, mlp_block_inputs, \
    lmhead_inputs, block8b_inputs, positions
from oracle import coda_oracle as O
from tests._util import TOL_BF16, TOL_F32, assert_close, assert_stat_near_exact, to64

pytestmark = pytest.mark.gpu

BLOCKS = [WORKLOADS["tiny_mlp_fwd"],
          BlockShape("ragged", M=200, d=136, f=200, seed=11),
          BlockShape("multi_tile", M=384, d=520, f=392, seed=12),
          # one token: every 256-row pair tile holds a single valid row
          BlockShape("one_row", M=1, d=64, f=64, seed=13),
          # rows of 1056 bytes: the epilogues' 32-byte row loads, with a last
          # chunk of 16 columns that falls back to 16-byte loads
          BlockShape("wide_ragged", M=300, d=528, f=264, seed=14),
          # K = 2f = 12320 over 80 tiles: the RMSNorm-backward GEMM takes the
          # two-slab tile with eight epilogue warps, on ragged M and d (the
          # SwiGLU backward, K = d = 1040, its short-K form)
          BlockShape("two_slab_ragged", M=4000, d=1040, f=6160, seed=15)]


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def _run_block(coda, shape, zero_row=False):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    inp = mlp_block_inputs(shape)
    if zero_row:  # a row whose h is exactly 0: r = 1/sqrt(eps)
        inp["x"][0] = 0
        inp["z"][0] = 0
    g = {k: v.cuda() for k, v in inp.items()}
    fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
    bw = blocks.mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["dout"])
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    return inp, fw, bw


@pytest.mark.parametrize("shape", BLOCKS, ids=lambda s: s.name)
def test_block_forward_backward(coda, shape):
    inp, fw, bw = _run_block(coda, shape, zero_row=shape.name == "ragged")
    n = {k: O.to64(v) for k, v in inp.items()}
    ref = O.mlp_fwd(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"])
    rep = O.mlp_fwd_reparam(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"])
    rb = O.mlp_bwd(ref, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["dout"])
    assert_close("h", fw["h"], ref["h"], TOL_BF16)
    assert_close("hg", fw["hg"], rep["hg"], TOL_BF16)
    assert_close("r", fw["r"], ref["r"], TOL_F32)
    assert_close("y", fw["y"], ref["y"], TOL_BF16)
    assert_close("a", fw["a"], ref["a"], TOL_BF16)
    assert_close("out", fw["out"], ref["out"], TOL_BF16)
    # backward against the canonical (autograd-by-hand) oracle
    for k in ("dx", "dz", "dW0", "dW1", "dW2", "dgamma"):
        assert_close(k, bw[k], rb[k], TOL_BF16)
    # s against the oracle's rewritten form with the fused path's bf16 storage
    # points (h, hg, a, dyhat rounded; y saved in fp32), and against the exact
    # canonical form with the bound that bf16 storage of hg allows (s sums
    # products with heavy cancellation, so hg's rounding moves it ~1e-3)
    st = O.mlp_fwd_reparam(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"], store_bf16=True)
    sb = O.mlp_bwd_reparam(st, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["dout"],
                           store_bf16=True)
    assert_close("s (storage-rounded oracle)", bw["s"], sb["s"], TOL_F32)
    assert_stat_near_exact("s (exact oracle)", bw["s"], rb["s"], sb["s"])
    assert_close("dyhat", bw["dyhat"], ref["r"][:, None] * rb["dy"], TOL_BF16)


CE_SHAPES = [LMHeadShape("ce_small", M=200, d=136, V=1000, seed=21),
             LMHeadShape("ce_multi", M=512, d=256, V=8200, seed=22),
             # one token over the smallest vocabulary the entry point takes
             LMHeadShape("ce_one_row", M=1, d=64, V=8, seed=24)]


@pytest.mark.parametrize("shape", CE_SHAPES, ids=lambda s: s.name)
def test_lmhead_ce(coda, shape):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    inp = lmhead_inputs(shape)
    t = inp["targets"]
    # targets on tile edges and at the ends of the vocabulary
    edge = [e for e in (0, shape.V - 1, 255, 256, 511, 512, shape.V - 8) if e < shape.V]
    edge = edge[:shape.M]
    t[:len(edge)] = torch.tensor(edge, dtype=torch.int32)
    res = blocks.lmhead_ce(inp["hidden"].cuda(), inp["W"].cuda(), t.cuda())
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    ref = O.lmhead_ce(O.to64(inp["hidden"]), O.to64(inp["W"]), t.numpy())
    assert_close("lse", res["lse"], ref["lse"], TOL_F32)
    assert_close("loss", res["loss"], ref["loss"], TOL_F32)


def test_lmhead_ce_invalid_target_reports_error(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    inp = lmhead_inputs(LMHeadShape("ce_bad", M=64, d=64, V=512, seed=23))
    t = inp["targets"].clone()
    t[3] = 512  # out of range
    res = blocks.lmhead_ce(inp["hidden"].cuda(), inp["W"].cuda(), t.cuda())
    st = coda.get_device_error()
    assert st == coda.CODA_ERR_INVALID_VALUE
    loss = res["loss"].cpu()
    assert torch.isnan(loss[3]) and torch.isfinite(loss[:3]).all()
    assert coda.get_device_error() == 0


SHAPES_8B = [
    Block8BShape("small_8b", M=256, d=256, f=384, seq_len=128, head_dim=128, n_q_heads=4,
                 n_kv_heads=1, theta=500000.0, seed=31),
    # ragged everywhere: 200 rows = 1.56 sequences of 128 (positions restart
    # inside the second row tile), d and f not multiples of the tile, and
    # 3 q + 1 kv heads, so the QKV GEMM has 640 columns: its last 256-column
    # tile holds the 128 unrotated v columns and 128 columns past the end
    Block8BShape("ragged_8b", M=200, d=136, f=200, seq_len=128, head_dim=128, n_q_heads=3,
                 n_kv_heads=1, theta=500000.0, seed=32),
]


@pytest.mark.parametrize("sh", SHAPES_8B, ids=lambda s: s.name)
def test_block8b_small(coda, sh):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    inp = block8b_inputs(sh)
    g = {k: v.cuda() for k, v in inp.items()}
    cs = blocks.rope_table(sh.seq_len, sh.head_dim, sh.theta, "cuda")
    fw = blocks.block8b_fwd(g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    bw = blocks.block8b_bwd(fw, g, sh.seq_len, sh.head_dim, sh.n_rope_cols, cs)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in inp.items()}
    pos = positions(sh.M, sh.seq_len).numpy()
    ref = O.block8b_fwd(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                        n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    rb = O.block8b_bwd(ref, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                       n["Wqkv"], n["dqkv"], n["dres"], pos, sh.n_rope_cols, sh.head_dim, sh.theta)
    assert_close("h", fw["h"], ref["h"], TOL_BF16)
    assert_close("r", fw["r"], ref["r"], TOL_F32)
    assert_close("out", fw["out"], ref["out"], TOL_BF16)
    assert_close("r1", fw["r1"], ref["r1"], TOL_F32)
    assert_close("qkv", fw["qkv"], ref["qkv"], TOL_BF16)
    for k in ("dout", "dz", "do", "dWo", "dW1", "dW2", "dWqkv", "dgamma1", "dgamma2"):
        assert_close(k, bw[k], rb[k], TOL_BF16)
    fr = O.block8b_fwd_reparam(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                               n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim, sh.theta, store_bf16=True)
    br = O.block8b_bwd_reparam(fr, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"], n["gamma1"],
                               n["Wqkv"], n["dqkv"], n["dres"], pos, sh.n_rope_cols, sh.head_dim,
                               sh.theta, store_bf16=True, stat_only=True)
    assert_close("s1 (storage-rounded oracle)", bw["s1"], br["s1"], TOL_F32)
    assert_close("s (storage-rounded oracle)", bw["s"], br["s"], TOL_F32)
    assert_stat_near_exact("s1 (exact oracle)", bw["s1"], rb["s1"], br["s1"])
    assert_stat_near_exact("s (exact oracle)", bw["s"], rb["s"], br["s"])


def test_saved_fp16_copy_out_of_range_reports_error(coda):
    """A y beyond the fp16 range cannot be saved for the backward: the kernel
    finishes, a is still written, and the host gets CODA_ERR_RANGE once."""
    M, K, two_f = 128, 64, 512
    g = torch.Generator().manual_seed(5)
    hg = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W1 = torch.randn(K, two_f, generator=g).to(torch.bfloat16).cuda()
    r = torch.ones(M, dtype=torch.float32, device="cuda")
    r[7] = 1e6  # row 7: |y| ~ 1e7
    a = torch.empty(M, two_f // 2, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, two_f, dtype=torch.float16, device="cuda")
    coda.coda_gemm_rowscale_swiglu(hg, W1, r, a, y)
    assert coda.get_device_error() == coda.CODA_ERR_RANGE
    assert coda.get_device_error() == 0  # reading the word clears it
    assert torch.isinf(y[7].float()).any() and torch.isfinite(y[:7].float()).all()
    ref = (hg.double() @ W1.double()) * r.double()[:, None]
    a_ref = torch.nn.functional.silu(ref[:, 0::2]) * ref[:, 1::2]
    assert_close("a (rows in range)", a[:7], a_ref[:7].cpu().numpy(), TOL_BF16)
    # the same call without the saved copy has nothing to report
    coda.coda_gemm_rowscale_swiglu(hg, W1, r, a, None)
    assert coda.get_device_error() == 0


def test_rope_table(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    cs = blocks.rope_table(4096, 128, 500000.0, "cuda").cpu().double().numpy()
    c, s = O.rope_cos_sin(np.arange(4096), 128, 500000.0)
    assert np.max(np.abs(cs[..., 0] - c)) < 1e-7
    assert np.max(np.abs(cs[..., 1] - s)) < 1e-7
