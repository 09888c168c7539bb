"""GPU parity of the LayerNorm variant of the block ("CODA: Rewriting
Transformer Blocks as GEMM-Epilogue Programs", abstract: RMSNorm and LayerNorm
compositions) against the fp64 CPU oracle. The library's reading: GEMM 1
emits per-row sums of h and h^2; GEMM 2 applies the delayed normalisation
r (hg W1) - (r mu) w1 + b1 with w1 = gamma W1, b1 = beta W1; the two
LayerNorm-backward statistics are accumulated in the epilogue of the GEMM
that produces dy, and the LayerNorm backward itself is fused into the GEMM
producing dyhat W1^T. Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from coda_inputs import BlockShape, ln_block_inputs
from oracle import coda_oracle as O
from tests._util import TOL_BF16, TOL_F32, assert_close, assert_stat_near_exact

pytestmark = pytest.mark.gpu

SHAPES = [BlockShape("ln_tiny", M=64, d=256, f=512, seed=60),
          BlockShape("ln_ragged", M=200, d=136, f=200, seed=61),
          BlockShape("ln_multi_tile", M=384, d=520, f=392, seed=62),
          BlockShape("ln_one_row", M=1, d=64, f=64, seed=63)]


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
    assert_stat_near_exact("s_a (exact oracle)", bw["sa"], rb["sa"], sb["sa"])
    assert_stat_near_exact("s_b (exact oracle)", bw["sb"], rb["sb"], sb["sb"])
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


def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    edges = [r for b in range(128, M, 128) for r in (b - 1, b)]
    return np.array(sorted(set(rng.choice(M, n, replace=False).tolist()) | set(edges) | {0, M - 1}))


def test_ln_norm_bwd_long_k(coda):
    """The LayerNorm-backward GEMM at K = 2f = 8192 with 8192 rows (many
    tiles per CTA pair, long K): dh and hhat on a row sample covering every
    128-row and pair-tile edge, the dgamma / dbeta partials on 32-row blocks
    around those edges, against the oracle's LayerNorm-backward stage."""
    M, d, two_f = 8192, 2048, 8192
    g = torch.Generator().manual_seed(64)
    dyhat = (torch.randn(M, two_f, generator=g) * 0.05).to(torch.bfloat16)
    W1 = (torch.randn(d, two_f, generator=g) * 0.02).to(torch.bfloat16)
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    gamma = (torch.rand(d, generator=g) + 0.5).to(torch.bfloat16)
    beta = (torch.randn(d, generator=g) * 0.3).to(torch.bfloat16)
    r = torch.rand(M, generator=g) + 0.5
    mu = torch.randn(M, generator=g) * 0.1
    sa = torch.randn(M, generator=g) * 0.01
    sb = torch.randn(M, generator=g) * 0.01
    cu = {k: v.cuda() for k, v in dict(dyhat=dyhat, W1=W1, h=h, gamma=gamma, beta=beta, r=r,
                                        mu=mu, sa=sa, sb=sb).items()}
    dh = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    hhat = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    dgp = torch.empty(coda.row_tiles32(M), d, dtype=torch.float32, device="cuda")
    dbp = torch.empty(coda.row_tiles32(M), d, dtype=torch.float32, device="cuda")
    coda.coda_gemm_resid_ln_stats_bwd(cu["dyhat"], cu["W1"], cu["h"], cu["gamma"], cu["beta"],
                                      cu["r"], cu["mu"], cu["sa"], cu["sb"], dh, dgp, dbp,
                                      hhat=hhat)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = _sample_rows(M, 60, 65)
    n = {k: O.to64(v) for k, v in dict(dyhat=dyhat, W1=W1, h=h, gamma=gamma, beta=beta, r=r,
                                       mu=mu, sa=sa, sb=sb).items()}
    ref = O.ln_norm_bwd_stage(n["dyhat"][rows], n["W1"], n["h"][rows], n["gamma"], n["beta"],
                              n["r"][rows], n["mu"][rows], n["sa"][rows], n["sb"][rows],
                              store_bf16=True)
    assert_close("dh (long K)", dh.cpu()[rows], ref["dh"], TOL_BF16)
    assert_close("hhat (long K)", hhat.cpu()[rows], ref["hhat"], TOL_BF16)
    blocks = [0, 3, 4, 7, 8, 15, 16, 31, 32, 127, 128, M // 32 - 1]
    brows = np.concatenate([np.arange(32 * j, 32 * j + 32) for j in blocks])
    rb = O.ln_norm_bwd_stage(n["dyhat"][brows], n["W1"], n["h"][brows], n["gamma"], n["beta"],
                             n["r"][brows], n["mu"][brows], n["sa"][brows], n["sb"][brows])
    dg_ref = rb["dgamma_rows"].reshape(len(blocks), 32, d).sum(axis=1)
    db_ref = rb["dbeta_rows"].reshape(len(blocks), 32, d).sum(axis=1)
    # the fused path forms P from bf16 operands in fp32 like the oracle; the
    # partials multiply it by the bf16-stored h: compare at the fp32 tolerance
    assert_close("dgamma partials (long K)", dgp.cpu()[blocks], dg_ref, TOL_F32)
    assert_close("dbeta partials (long K)", dbp.cpu()[blocks], db_ref, TOL_F32)


@pytest.mark.parametrize("ln", [0, 1])
def test_resid_stats_long_k(coda, ln):
    """The residual + statistics GEMM at K = 8192 (e.g. a down projection
    feeding the next norm) with 8192 rows: h, hg and the per-tile row
    partials (sum h^2, and sum h for LayerNorm) on a row sample, against
    h = x W + z in fp64."""
    M, K, N = 8192, 8192, 2048
    g = torch.Generator().manual_seed(66 + ln)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(K, N, generator=g) * 0.02).to(torch.bfloat16)
    z = torch.randn(M, N, generator=g).to(torch.bfloat16)
    gamma = (torch.rand(N, generator=g) + 0.5).to(torch.bfloat16)
    h = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    hg = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    psq = torch.empty(coda.col_tiles(N), M, dtype=torch.float32, device="cuda")
    psum = torch.empty(coda.col_tiles(N), M, dtype=torch.float32, device="cuda")
    if ln:
        coda.coda_gemm_resid_ln_stats(x.cuda(), W.cuda(), z.cuda(), gamma.cuda(), h, hg, psq, psum)
    else:
        coda.coda_gemm_resid_norm_stats(x.cuda(), W.cuda(), z.cuda(), gamma.cuda(), h, hg, psq)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rows = _sample_rows(M, 60, 67)
    href = O.to64(x)[rows] @ O.to64(W) + O.to64(z)[rows]
    assert_close("h (long K)", h.cpu()[rows], href, TOL_BF16)
    assert_close("hg (long K)", hg.cpu()[rows], href * O.to64(gamma)[None, :], TOL_BF16)
    tiles = href.reshape(len(rows), -1, 128)  # one partial per 128 columns
    assert_close("sum h^2 partials (long K)", psq.cpu()[:, rows], (tiles ** 2).sum(axis=2).T,
                 TOL_F32)
    if ln:
        assert_close("sum h partials (long K)", psum.cpu()[:, rows], tiles.sum(axis=2).T,
                     TOL_F32)


@pytest.mark.parametrize("d", [2048, 2560])
def test_ln_swiglu_bwd_both_epilogue_forms(coda, d):
    """The LayerNorm SwiGLU backward GEMM runs eight epilogue warps at
    K = d <= 2048 and four above: both forms against the rewritten oracle
    on the same kind of inputs (M = 512, f = 1024, ragged-free): dyhat and
    the three row partials per 128 da columns (sum dy y, sum dy w1,
    sum dy b1)."""
    M, f = 512, 1024
    g = torch.Generator().manual_seed(90 + d)
    dout = torch.randn(M, d, generator=g).to(torch.bfloat16)
    W2 = (torch.randn(f, d, generator=g) * 0.02).to(torch.bfloat16)
    y = torch.randn(M, 2 * f, generator=g).to(torch.float16)
    r = torch.rand(M, generator=g) + 0.5
    w1 = torch.randn(2 * f, generator=g) * 0.1
    b1 = torch.randn(2 * f, generator=g) * 0.1
    cu = {k: v.cuda() for k, v in dict(dout=dout, W2=W2, y=y, r=r, w1=w1, b1=b1).items()}
    dyhat = torch.empty(M, 2 * f, dtype=torch.bfloat16, device="cuda")
    parts = [torch.empty(coda.col_tiles(f), M, dtype=torch.float32, device="cuda") for _ in range(3)]
    coda.coda_gemm_ln_rowscale_swiglu_bwd(cu["dout"], cu["W2"], cu["y"], cu["r"], cu["w1"], cu["b1"],
                                          dyhat, *parts)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    n = {k: O.to64(v) for k, v in dict(dout=dout, W2=W2, y=y, r=r, w1=w1, b1=b1).items()}
    z = np.zeros
    fwd = {"h": z((M, d)), "hg": z((M, d)), "mu": z(M), "r": n["r"], "w1": n["w1"], "b1": n["b1"],
           "y": n["y"], "a": z((M, f))}
    ref = O.ln_mlp_bwd_reparam(fwd, z((M, d)), z((d, d)), z((d, 2 * f)), n["W2"], np.ones(d),
                               z(d), n["dout"], store_bf16=True)
    assert_close(f"dyhat (d={d})", dyhat, ref["dyhat"], TOL_BF16)
    dy = ref["dy"]
    for name, got, vec in (("sum dy y", parts[0], n["y"]), ("sum dy w1", parts[1], n["w1"][None, :]),
                           ("sum dy b1", parts[2], n["b1"][None, :])):
        want = (dy * vec).reshape(M, -1, 256).sum(axis=2).T  # 128 da columns = 256 y columns
        assert_close(f"{name} partials (d={d})", got, want, TOL_F32)
