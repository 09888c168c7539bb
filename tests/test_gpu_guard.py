"""Guard bands around every output (the stand-in for a memory checker): each
output tensor of each entry point sits inside a larger allocation whose other
bytes hold a known pattern, on ragged shapes (M = 200, d = 136, f = 200,
V = 1000, 640 QKV columns: partial tiles in every dimension). After the call
no byte outside the tensor may have changed. For coda_gemm the outputs are
also row-padded (leading dimension > N), so a store into the padding columns
between rows is caught too. Values are checked by the parity tests; here only
where the library writes."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PATTERN = 0xA5
GUARD = 4096
M, D, F, V = 200, 136, 200, 1000
SEQ, HD, NQKV, NROPE = 128, 128, 640, 512


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


class Guarded:
    """A tensor of `shape` (row stride `ld` elements for 2-D) inside a byte
    buffer with GUARD pattern bytes before and after it."""

    def __init__(self, shape, dtype, ld=None):
        self.shape, self.dtype = tuple(shape), dtype
        self.esize = torch.empty((), dtype=dtype).element_size()
        rows = shape[0] if len(shape) == 2 else 1
        cols = shape[-1]
        self.ld = ld if ld is not None else cols
        self.rows, self.cols = rows, cols
        self.nbytes = rows * self.ld * self.esize
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda")
        body = self.raw[GUARD:GUARD + self.nbytes].view(dtype)
        if len(shape) == 2:
            self.t = body.view(rows, self.ld)[:, :cols]
        else:
            self.t = body

    def changed_outside(self):
        raw = self.raw.cpu().numpy()
        inside = np.zeros(raw.size, dtype=bool)
        row_b, used_b = self.ld * self.esize, self.cols * self.esize
        for r in range(self.rows):
            s = GUARD + r * row_b
            inside[s:s + used_b] = True
        bad = np.nonzero((raw != PATTERN) & ~inside)[0]
        return bad


def _check_all(coda, outs):
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    for name, g in outs.items():
        bad = g.changed_outside()
        assert bad.size == 0, (f"{name}: {bad.size} bytes outside the tensor changed, first at "
                               f"offset {int(bad[0]) - GUARD} from its start")


def _bf(*shape, std=1.0, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16)


def _pos(*shape, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.rand(shape, generator=g, device="cuda") + 0.5


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("c_fp32", [0, 1])
def test_gemm_writes_only_its_rows_and_columns(coda, transA, transB, c_fp32):
    N, K = 264, 136
    A = _bf(K, M, seed=1) if transA else _bf(M, K, seed=1)
    B = _bf(N, K, seed=2) if transB else _bf(K, N, seed=2)
    dt = torch.float32 if c_fp32 else torch.bfloat16
    C = Guarded((M, N), dt, ld=N + (4 if c_fp32 else 8))
    outs = {"C": C}
    rowsq = None
    if not transA and not transB and not c_fp32:  # the row sums exist for this form only
        rowsq = Guarded((coda.col_tiles(N), M), torch.float32)
        outs["rowsq_part"] = rowsq
    coda.coda_gemm(A, B, C.t, transA=bool(transA), transB=bool(transB),
                   rowsq_part=rowsq.t if rowsq is not None else None)
    _check_all(coda, outs)


def test_rmsnorm_block_forward_and_backward_outputs(coda):
    x, z, W0 = _bf(M, D, seed=3), _bf(M, D, seed=4), _bf(D, D, std=0.05, seed=5)
    W1, W2 = _bf(D, 2 * F, std=0.05, seed=6), _bf(F, D, std=0.05, seed=7)
    gamma, dout = _bf(D, std=0.2, seed=8) + 1, _bf(M, D, seed=9)
    bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32
    o = {"h": Guarded((M, D), bf), "hg": Guarded((M, D), bf),
         "part": Guarded((coda.col_tiles(D), M), f32), "r": Guarded((M,), f32),
         "a": Guarded((M, F), bf), "y": Guarded((M, 2 * F), f16),
         "dyhat": Guarded((M, 2 * F), bf), "spart": Guarded((coda.col_tiles(F), M), f32),
         "s": Guarded((M,), f32), "dh": Guarded((M, D), bf),
         "dgpart": Guarded((coda.row_tiles32(M), D), f32), "dgamma": Guarded((D,), f32)}
    coda.coda_gemm_resid_norm_stats(x, W0, z, gamma, o["h"].t, o["hg"].t, o["part"].t)
    coda.coda_row_rms(o["part"].t, o["r"].t, D, 1e-6)
    coda.coda_gemm_rowscale_swiglu(o["hg"].t, W1, o["r"].t, o["a"].t, o["y"].t)
    coda.coda_gemm_rowscale_swiglu_bwd(dout, W2, o["y"].t, o["r"].t, o["dyhat"].t, o["spart"].t)
    coda.coda_row_rms_bwd(o["spart"].t, o["s"].t, D)
    coda.coda_gemm_resid_norm_stats_bwd(o["dyhat"].t, W1, o["h"].t, gamma, o["r"].t, o["s"].t,
                                        o["dh"].t, o["dgpart"].t, dresid=dout)
    coda.coda_col_reduce(o["dgpart"].t, o["dgamma"].t)
    _check_all(coda, o)


def test_rope_forward_and_backward_outputs(coda):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    A, W = _bf(M, D, seed=10), _bf(D, NQKV, std=0.05, seed=11)
    r, dq = _pos(M, seed=12), _bf(M, NQKV, seed=13)
    cs = blocks.rope_table(SEQ, HD, 500000.0, "cuda")
    bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32
    o = {"out": Guarded((M, NQKV), bf), "out_f16": Guarded((M, NQKV), f16),
         "dqkv_hat": Guarded((M, NQKV), bf), "s": Guarded((M,), f32)}
    coda.coda_gemm_rope(A, W, r, cs, SEQ, HD, NROPE, o["out"].t, o["out_f16"].t)
    coda.coda_gemm_rope_bwd(dq, o["out_f16"].t, r, cs, SEQ, HD, NROPE, o["dqkv_hat"].t, o["s"].t, D)
    _check_all(coda, o)


def test_lmhead_forward_and_backward_outputs(coda):
    hid, W = _bf(M, D, seed=14), _bf(D, V, std=0.05, seed=15)
    g = torch.Generator(device="cuda").manual_seed(16)
    t = torch.randint(0, V, (M,), generator=g, device="cuda", dtype=torch.int32)
    dl = torch.full((M,), 1.0 / M, device="cuda")
    f32 = torch.float32
    ws = Guarded((coda.coda_lmhead_ce_workspace_size(M, V),), torch.uint8)
    ws_b = Guarded((coda.coda_lmhead_ce_bwd_workspace_size(M, V),), torch.uint8)
    o = {"lse": Guarded((M,), f32), "loss": Guarded((M,), f32), "ws": ws,
         "dhidden": Guarded((M, D), f32), "dW": Guarded((D, V), f32), "ws_bwd": ws_b}
    coda.coda_lmhead_ce(hid, W, t, o["lse"].t, o["loss"].t, ws.t)
    coda.coda_lmhead_ce_bwd(hid, W, t, o["lse"].t, dl, o["dhidden"].t, o["dW"].t, ws_b.t)
    _check_all(coda, o)


def test_layernorm_block_forward_and_backward_outputs(coda):
    x, z, W0 = _bf(M, D, seed=17), _bf(M, D, seed=18), _bf(D, D, std=0.05, seed=19)
    W1, W2 = _bf(D, 2 * F, std=0.05, seed=20), _bf(F, D, std=0.05, seed=21)
    gamma, beta = _bf(D, std=0.2, seed=22) + 1, _bf(D, std=0.2, seed=23)
    dout = _bf(M, D, seed=24)
    w1 = torch.randn(2 * F, device="cuda") * 0.1
    b1 = torch.randn(2 * F, device="cuda") * 0.1
    bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32
    nt, nr = coda.col_tiles(D), coda.row_tiles32(M)
    o = {"h": Guarded((M, D), bf), "hg": Guarded((M, D), bf),
         "psq": Guarded((nt, M), f32), "psum": Guarded((nt, M), f32),
         "r": Guarded((M,), f32), "mu": Guarded((M,), f32),
         "a": Guarded((M, F), bf), "y": Guarded((M, 2 * F), f16),
         "dyhat": Guarded((M, 2 * F), bf), "spart": Guarded((coda.col_tiles(F), M), f32),
         "spart_w": Guarded((coda.col_tiles(F), M), f32),
         "spart_b": Guarded((coda.col_tiles(F), M), f32),
         "s_a": Guarded((M,), f32), "s_b": Guarded((M,), f32),
         "dh": Guarded((M, D), bf), "hhat": Guarded((M, D), bf),
         "dgpart": Guarded((nr, D), f32), "dbpart": Guarded((nr, D), f32)}
    coda.coda_gemm_resid_ln_stats(x, W0, z, gamma, o["h"].t, o["hg"].t, o["psq"].t, o["psum"].t)
    coda.coda_row_ln(o["psq"].t, o["psum"].t, o["r"].t, o["mu"].t, D, 1e-6)
    coda.coda_gemm_ln_rowscale_swiglu(o["hg"].t, W1, o["r"].t, o["mu"].t, w1, b1, o["a"].t,
                                      o["y"].t)
    coda.coda_gemm_ln_rowscale_swiglu_bwd(dout, W2, o["y"].t, o["r"].t, w1, b1, o["dyhat"].t,
                                          o["spart"].t, o["spart_w"].t, o["spart_b"].t)
    coda.coda_row_ln_bwd(o["spart"].t, o["spart_w"].t, o["spart_b"].t, o["s_a"].t, o["s_b"].t, D)
    coda.coda_gemm_resid_ln_stats_bwd(o["dyhat"].t, W1, o["h"].t, gamma, beta, o["r"].t,
                                      o["mu"].t, o["s_a"].t, o["s_b"].t, o["dh"].t,
                                      o["dgpart"].t, o["dbpart"].t, hhat=o["hhat"].t, dresid=dout)
    _check_all(coda, o)


def test_noalloc_lmhead_writes_only_its_outputs(coda):
    hid, W = _bf(M, D, seed=27), _bf(D, V, std=0.05, seed=28)
    g = torch.Generator(device="cuda").manual_seed(29)
    t = torch.randint(0, V, (M,), generator=g, device="cuda", dtype=torch.int32)
    o = {"lse": Guarded((M,), torch.float32), "loss": Guarded((M,), torch.float32)}
    coda.coda_lmhead_ce_noalloc(hid, W, t, o["lse"].t, o["loss"].t)
    _check_all(coda, o)
