"""The boundary from C: include/coda.h compiles as C99 and C++17 (CPU), and
a plain C program links libcoda.so, allocates device memory with the CUDA
runtime and checks a GEMM and the LM-head CE against double-precision loops
(GPU). No Python or PyTorch sits between that program and the library."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "gemm_epilogue_fusion_tcgen05_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_header_compiles(tmp_path, lang):
    cc = shutil.which("gcc" if lang == "c99" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("h.c" if lang == "c99" else "h.cpp")
    src.write_text('#include "coda.h"\nint main(void) { return coda_col_tiles(128) == 1 ? 0 : 1; }\n')
    r = subprocess.run([cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-fsyntax-only", "-I", INC, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_through_the_abi(tmp_path):
    import __graft_entry__ as g
    g.build()
    exe = tmp_path / "use_from_c"
    r = subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Werror",
                        os.path.join(ROOT, "tests", "c", "use_from_c.c"), "-o", str(exe),
                        "-I", INC, "-I", os.path.join(CUDA, "include"),
                        "-L", PKG, "-lcoda", f"-Wl,-rpath,{PKG}",
                        "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                        f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    print(run.stdout)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("OK")
