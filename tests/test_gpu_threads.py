"""Calls from several host threads at once, each on its own CUDA stream
(the header promises thread-safe, stream-asynchronous calls): every thread's
results must equal, bit for bit, the same calls made from one thread."""
import threading

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


def _work(coda, g, ci):
    from gemm_epilogue_fusion_tcgen05_gb300 import blocks
    fw = blocks.mlp_block_fwd(g["x"], g["z"], g["W0"], g["W1"], g["W2"], g["gamma"])
    bw = blocks.mlp_block_bwd(fw, g["x"], g["W0"], g["W1"], g["W2"], g["gamma"], g["dout"])
    ce = blocks.lmhead_ce(ci["hidden"], ci["W"], ci["targets"])
    return [fw["out"], bw["dx"], bw["dW1"], bw["s"], ce["loss"]]


def test_concurrent_threads_on_own_streams(coda):
    n_threads, iters = 3, 4
    data = []
    for i in range(n_threads):
        g = {k: v.cuda() for k, v in mlp_block_inputs(
            BlockShape(f"thr{i}", M=600 + 128 * i, d=512, f=520, seed=90 + i)).items()}
        ci = {k: v.cuda() for k, v in lmhead_inputs(
            LMHeadShape(f"thr_ce{i}", M=300, d=256, V=3000 + 512 * i, seed=95 + i)).items()}
        data.append((g, ci))
    # single-threaded references on the default stream
    refs = [[t.clone() for t in _work(coda, g, ci)] for g, ci in data]
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0

    results = [None] * n_threads
    errors = []

    def run(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(iters):
                    out = _work(coda, *data[i])
                s.synchronize()
            results[i] = out
        except Exception as e:  # reported below
            errors.append(e)

    th = [threading.Thread(target=run, args=(i,)) for i in range(n_threads)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert coda.get_device_error() == 0
    for i in range(n_threads):
        for got, ref in zip(results[i], refs[i]):
            assert torch.equal(got, ref), f"thread {i}"
