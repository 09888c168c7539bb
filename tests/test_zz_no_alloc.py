"""GPU test of coda_lmhead_ce_noalloc, the LM-head cross-entropy entry point
for callers that may not allocate device memory (an operator hook handed only
its inputs and outputs, a process whose device memory is reserved up front, a
loop where cudaMalloc / cudaFree are not allowed). It takes its scratch from
an array the library keeps on the device, so it must give the same LSE and
loss as coda_lmhead_ce with a caller-allocated workspace, call after call.

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

from coda_inputs import LMHeadShape, lmhead_inputs
from oracle import coda_oracle as O
from tests._util import TOL_F32, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _with_workspace(coda, inp):
    """Reference: the existing entry point with a caller-allocated workspace."""
    hidden, W, t = inp["hidden"], inp["W"], inp["targets"]
    M, d = hidden.shape
    V = W.shape[1]
    ws = torch.empty(coda.coda_lmhead_ce_workspace_size(M, V), dtype=torch.uint8, device="cuda")
    lse = torch.empty(M, dtype=torch.float32, device="cuda")
    loss = torch.empty(M, dtype=torch.float32, device="cuda")
    st = coda.lib().coda_lmhead_ce(_p(hidden), _p(W), _p(t), _p(lse), _p(loss), _p(ws),
                                   ws.numel(), M, V, d, ctypes.c_void_p(0))
    assert st == 0, coda.lib().coda_last_error_string()
    return lse, loss


def _no_alloc(coda, inp):
    hidden, W, t = inp["hidden"], inp["W"], inp["targets"]
    M, d = hidden.shape
    V = W.shape[1]
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    st = coda.lib().coda_lmhead_ce_noalloc(_p(hidden), _p(W), _p(t), _p(lse), _p(loss), M, V, d,
                                           ctypes.c_void_p(0))
    assert st == 0, coda.lib().coda_last_error_string()
    return lse, loss


def test_no_alloc_matches_workspace_entry_point_twice_in_a_row(coda):
    # first call: the full 128256-class vocabulary on 2048 rows; second call:
    # other inputs and sizes, so that anything the first call left in the
    # shared array would show up in the second call's result
    shapes = [LMHeadShape("noalloc_a", M=2048, d=2048, V=128256, seed=41),
              LMHeadShape("noalloc_b", M=1000, d=512, V=50000, seed=42)]
    for sh in shapes:
        inp = {k: v.cuda() for k, v in lmhead_inputs(sh).items()}
        lse_ref, loss_ref = _with_workspace(coda, inp)
        lse, loss = _no_alloc(coda, inp)
        torch.cuda.synchronize()
        assert coda.get_device_error() == 0
        assert_close(f"lse no-alloc vs workspace ({sh.name})", lse, lse_ref, TOL_F32)
        assert_close(f"loss no-alloc vs workspace ({sh.name})", loss, loss_ref, TOL_F32)
        # and against the fp64 oracle on sampled rows (first, last, scattered)
        rng = np.random.default_rng(sh.seed)
        rows = np.array(sorted({0, sh.M - 1} | set(rng.choice(sh.M, 24, replace=False).tolist())))
        ref = O.lmhead_ce(to64(inp["hidden"][rows]), to64(inp["W"]),
                          inp["targets"][rows].cpu().numpy())
        ri = torch.from_numpy(rows).cuda()
        assert_close(f"lse no-alloc vs oracle ({sh.name})", lse[ri], ref["lse"], TOL_F32)
        assert_close(f"loss no-alloc vs oracle ({sh.name})", loss[ri], ref["loss"], TOL_F32)


def test_no_alloc_rejects_requests_beyond_its_array(coda):
    cap = coda.lib().coda_lmhead_ce_noalloc_capacity()
    V = 128256
    M = 8192  # needs about 33 MB of partials: more than the array holds
    assert coda.lib().coda_lmhead_ce_workspace_size(M, V) > cap
    fake = ctypes.c_void_p(0x10000)
    st = coda.lib().coda_lmhead_ce_noalloc(fake, fake, fake, fake, fake, M, V, 2048,
                                           ctypes.c_void_p(0))
    assert st == coda.CODA_ERR_INVALID_VALUE
    assert b"scratch" in coda.lib().coda_last_error_string()
