"""The GEMM form choices (one or two 128-row slabs per CTA, four or eight
epilogue warps) for the shapes the library runs, checked on the host: a small
program compiled against core/launch.cuh prints the decisions, no GPU needed.

The expected outcomes are the ones the kernels were measured and tuned for:
two slabs for the long-K weight gradients and norm GEMMs of the 8B block, one
slab where the waves or a short K favour it. The ragged block-parity shape
that tests the two-slab RMSNorm backward is listed too, so a change to the
choice that would stop that test from covering the form fails here."""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gemm_epilogue_fusion_tcgen05_gb300", "csrc")
INC = os.path.join(ROOT, "include")

# (M, N, K, epilogue reads tiles) -> two slabs?
CASES = [
    ((16384, 4096, 14336, 1), 1),   # 8B W2 + residual + statistics
    ((16384, 4096, 28672, 1), 1),   # 8B RMSNorm backward, K = 2f
    ((8192, 2048, 16384, 1), 1),    # 1B RMSNorm backward, K = 2f
    ((4000, 1040, 12320, 1), 1),    # the ragged two-slab block-parity shape
    ((16384, 4096, 4096, 1), 0),    # 8B Wo + residual: short K
    ((16384, 4096, 6144, 1), 0),    # 8B RMSNorm backward for Wqkv, K = 6144
    ((8192, 2048, 8192, 1), 0),     # tile-reading epilogue at K = 8192: no gain measured
    ((4096, 28672, 16384, 0), 1),   # 8B W1 weight gradient, K = tokens
    ((14336, 4096, 16384, 0), 1),   # 8B W2 weight gradient
    ((2048, 16384, 8192, 0), 0),    # 1B W1 weight gradient: 7 one-slab vs 4 two-slab waves
    ((8192, 2048, 8192, 0), 1),     # 1B down projection
    ((8192, 2048, 2048, 0), 0),     # short K
]


@pytest.fixture(scope="module")
def form_choice(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    exe = tmp_path_factory.mktemp("form") / "form_choice"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I", CSRC, "-I", INC, os.path.join(ROOT, "tests", "c", "form_choice.cu"),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    args = [str(v) for (shape, _) in CASES for v in shape]
    run = subprocess.run([str(exe), *args], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    return [json.loads(line) for line in run.stdout.splitlines()]


def test_two_slab_choices(form_choice):
    got = {(d["M"], d["N"], d["K"], d["loads"]): d["two_slabs"] for d in form_choice if "M" in d}
    for shape, want in CASES:
        assert got[shape] == want, f"{shape}: two_slabs = {got[shape]}, expected {want}"


def test_epilogue_warp_choices(form_choice):
    w = form_choice[-1]
    assert w == {"warps_heavy_k2048": 8, "warps_heavy_k4096": 4, "warps_light_k2048": 4}
