"""GPU tests of the plain tcgen05 GEMM through the C ABI (every operand
majorness, bf16 and fp32 outputs, ragged M/N/K tails, more tiles than SMs),
the residual / row-statistic epilogue, and the bounded-wait machinery."""
import numpy as np
import pytest
import torch

from tests._util import TOL_BF16, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("c_fp32", [0, 1])
@pytest.mark.parametrize("MNK", [(200, 264, 136), (128, 256, 64), (8, 8, 8), (16, 8, 24)])
def test_gemm_majorness_ragged(coda, transA, transB, c_fp32, MNK):
    M, N, K = MNK
    A = _rand((K, M) if transA else (M, K), 1)
    B = _rand((N, K) if transB else (K, N), 2)
    Ad = A.cuda()
    Bd = B.cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float32 if c_fp32 else torch.bfloat16,
                   device="cuda")
    coda.coda_gemm(Ad, Bd, C, transA=bool(transA), transB=bool(transB))
    torch.cuda.synchronize()
    a = to64(A).T if transA else to64(A)
    b = to64(B).T if transB else to64(B)
    ref = a @ b
    tol = 1e-5 if c_fp32 else TOL_BF16
    assert_close(f"gemm tA={transA} tB={transB} f32={c_fp32} {MNK}", C, ref, tol)
    assert coda.get_device_error() == 0


def test_gemm_single_row(coda):
    A, B = _rand((1, 40), 11), _rand((40, 24), 12)
    C = torch.empty((1, 24), dtype=torch.float32, device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert_close("gemm M=1", C, to64(A) @ to64(B), 1e-5)


@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 0), (0, 1)])
def test_gemm_many_tiles_per_cta(coda, transA, transB):
    # 32 x 16 = 512 tiles > SM count: each CTA walks several tiles and both
    # TMEM accumulator buffers; K = 320 is 5 k-blocks (ring wraps several times)
    M, N, K = 4096, 4096, 320
    A = _rand((K, M) if transA else (M, K), 3)
    B = _rand((N, K) if transB else (K, N), 4)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C, transA=bool(transA), transB=bool(transB))
    torch.cuda.synchronize()
    a = to64(A).T if transA else to64(A)
    b = to64(B).T if transB else to64(B)
    assert_close("gemm 4096^2 x 320", C, a @ b, 1e-5)


@pytest.mark.parametrize("transA", [1, 0])
@pytest.mark.parametrize("c_fp32", [1, 0])
def test_gemm_two_slab_long_k(coda, transA, c_fp32):
    """Long-K shapes that select the two-slab pair tile (512 rows per CTA
    pair, two MMAs per K step sharing B; with 76 co-resident pairs, 152 such
    tiles against 304 one-slab tiles): ragged M (4000 = 7.8 pair tiles), N
    (4840 = 18.9 column tiles) and K (8232 = 128.6 k-blocks). Checked on a
    row sample that includes every slab and pair-tile boundary."""
    M, N, K = 4000, 4840, 8232
    A = _rand((K, M) if transA else (M, K), 21)
    B = _rand((K, N), 22)
    C = torch.full((M, N), float("nan"), dtype=torch.float32 if c_fp32 else torch.bfloat16,
                   device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C, transA=bool(transA))
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    rng = np.random.default_rng(23)
    edges = [r for b in range(128, M, 128) for r in (b - 1, b)]
    rows = np.array(sorted(set(rng.choice(M, 40, replace=False).tolist()) | set(edges) | {0, M - 1}))
    a = to64(A).T[rows] if transA else to64(A)[rows]
    ref = a @ to64(B)
    got = C.cpu()[rows]
    assert torch.isfinite(got.float()).all()
    assert_close(f"two-slab gemm tA={transA} f32={c_fp32}", got, ref, 1e-5 if c_fp32 else TOL_BF16)


def test_gemm_strided_operands(coda):
    # leading dimensions larger than the logical width (views into wider buffers)
    M, N, K = 136, 72, 96
    Abig = _rand((M, K + 40), 5)
    Bbig = _rand((K, N + 24), 6)
    Cbig = torch.zeros((M, N + 8), dtype=torch.bfloat16, device="cuda")
    Ad, Bd = Abig.cuda(), Bbig.cuda()
    coda.coda_gemm(Ad[:, :K], Bd[:, :N], Cbig[:, :N])
    torch.cuda.synchronize()
    assert_close("gemm strided", Cbig[:, :N], to64(Abig[:, :K]) @ to64(Bbig[:, :N]), TOL_BF16)
    assert torch.all(Cbig[:, N:] == 0), "wrote outside the logical columns"


@pytest.mark.parametrize("MNK", [(200, 520, 72), (64, 256, 256)])
def test_gemm_resid_rowsq(coda, MNK):
    M, N, K = MNK
    A, B, R = _rand((M, K), 7), _rand((K, N), 8, 0.1), _rand((M, N), 9)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    part = torch.empty((coda.col_tiles(N), M), dtype=torch.float32, device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C, resid=R.cuda(), rowsq_part=part)
    torch.cuda.synchronize()
    ref = to64(A) @ to64(B) + to64(R)
    assert_close("gemm+resid", C, ref, TOL_BF16)
    assert_close("row sum of squares", part.sum(0), np.sum(ref * ref, axis=1), 1e-3)


@pytest.mark.parametrize("c_fp32,ld", [(0, 264), (1, 264), (0, 272)])
def test_gemm_resid_row_ends_inside_a_vector(coda, c_fp32, ld):
    """The epilogue reads the residual straight into registers, 32 bytes at a
    time where the row stride is a multiple of 32 bytes and 16 otherwise;
    here each row ends inside such a vector (N = 260 bf16 / 262 fp32), so the
    last elements come from the partial-vector path. Row strides of 264
    elements: 528 bytes (bf16, 16-byte loads) and 1056 bytes (fp32, 32-byte
    loads); 272 bf16 elements: 544 bytes (32-byte loads)."""
    M, K = 200, 72
    N = 262 if c_fp32 else 260
    dt = torch.float32 if c_fp32 else torch.bfloat16
    A, Bbig = _rand((M, K), 17), _rand((K, ld), 18, 0.1)
    B = Bbig[:, :N]  # row stride ld elements (16-byte multiple)
    g = torch.Generator().manual_seed(19)
    Rbig = torch.full((M, ld), float("nan"), dtype=dt)
    Rbig[:, :N] = torch.randn(M, N, generator=g).to(dt)
    Cbig = torch.zeros((M, ld), dtype=dt, device="cuda")
    Rd = Rbig.cuda()
    if c_fp32:  # C += A B: the residual is C itself
        Cbig[:, :N] = Rd[:, :N]
        coda.coda_gemm(A.cuda(), Bbig.cuda()[:, :N], Cbig[:, :N], resid=Cbig[:, :N])
    else:
        Rv = Rd[:, :N]
        Cv = Cbig[:, :N]
        assert Rv.stride() == Cv.stride()
        coda.coda_gemm(A.cuda(), Bbig.cuda()[:, :N], Cv, resid=Rv)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    ref = to64(A) @ to64(B) + to64(Rbig[:, :N])
    assert_close(f"gemm+resid, ragged vector (f32={c_fp32})", Cbig[:, :N], ref,
                 1e-5 if c_fp32 else TOL_BF16)
    assert_close("last columns", Cbig[:, N - 4:N], ref[:, N - 4:], 1e-5 if c_fp32 else TOL_BF16)
    assert torch.all(Cbig[:, N:] == 0), "wrote outside the logical columns"


@pytest.mark.parametrize("MNK,scale_b", [((256, 256, 4096), 0.02), ((256, 512, 2048), 1.0)])
def test_fp32_accumulation_matches_the_tensor_core_model(coda, MNK, scale_b):
    """The oracle's fp32 mode models the tensor-core GEMM as 16-product
    groups added to an fp32 accumulator with truncation (tc_matmul); the
    bounds on the chained statistics s and s' are derived from it. The
    kernel's fp32 output must sit closer to that model than to the exact
    product, err in the same direction (toward zero), and err no more than
    the model does, so that the model is a conservative stand-in."""
    from oracle import coda_oracle as O
    M, N, K = MNK
    A, B = _rand((M, K), 51), _rand((K, N), 52, scale_b)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    coda.coda_gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    gpu = to64(C)
    a, b = to64(A), to64(B)
    exact = a @ b
    model = O.tc_matmul(a, b).astype(np.float64)
    scale = np.max(np.abs(exact))
    e_gpu = np.max(np.abs(gpu - exact)) / scale
    e_model = np.max(np.abs(model - exact)) / scale
    d_gm = np.max(np.abs(gpu - model)) / scale
    bias_gpu = np.mean((gpu - exact) * np.sign(exact)) / np.mean(np.abs(exact))
    bias_model = np.mean((model - exact) * np.sign(exact)) / np.mean(np.abs(exact))
    print(f"fp32 GEMM {MNK}: gpu-exact {e_gpu:.2e} model-exact {e_model:.2e} gpu-model {d_gm:.2e}; "
          f"bias gpu {bias_gpu:.2e} model {bias_model:.2e}")
    assert d_gm < 0.5 * e_gpu
    assert bias_gpu < 0 and bias_model < 0
    assert e_gpu <= e_model and abs(bias_gpu) <= abs(bias_model)


@pytest.mark.parametrize("MNK,skip", [((512, 512, 256), 1), ((600, 1000, 1024), 5)])
def test_production_gemm_wait_runs_out_and_recovers(coda, MNK, skip):
    """The producers of a real GEMM launch leave one k-block of their first
    tile unloaded (coda_debug_skip_kblock): the MMA issuer's wait for it runs
    out under a 50 ms limit, the other roles follow through the CTA's abort
    flag or their own limits, every CTA drains its copies, frees its TMEM and
    returns, and the host reads CODA_ERR_TIMEOUT. The same GEMM then runs
    normally on the same context and matches fp64 (TMEM was released)."""
    M, N, K = MNK
    A, B = _rand((M, K), 61), _rand((K, N), 62, 0.1)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    coda.set_timeout_ms(50)
    coda.lib().coda_debug_skip_kblock(skip)
    try:
        coda.coda_gemm(Ad, Bd, C)
        st = coda.get_device_error()
    finally:
        coda.lib().coda_debug_skip_kblock(-1)
        coda.set_timeout_ms(2000)
    assert st == coda.CODA_ERR_TIMEOUT, f"status {st}"
    assert b"bounded wait" in coda.lib().coda_last_error_string()
    assert coda.get_device_error() == 0  # reading the word cleared it
    C.fill_(float("nan"))
    coda.coda_gemm(Ad, Bd, C)
    assert coda.get_device_error() == 0
    assert_close(f"gemm after a timed-out launch {MNK}", C, to64(A) @ to64(B), TOL_BF16)


def test_bounded_wait_gives_up_without_fault(coda):
    st = coda.coda_selftest_bounded_wait(20)
    assert st == coda.CODA_ERR_TIMEOUT
    # the context is still usable and the error word was cleared
    assert coda.get_device_error() == 0
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
