"""CPU tests of the C-ABI boundary: the library builds for sm_103a, loads
without a GPU, exports every symbol that include/coda.h declares, and rejects
bad arguments with status codes before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__ as g
    g.build()
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    return c.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "coda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(coda_\w+)\s*\(", src)))


def test_header_declares_the_hot_path():
    names = declared_symbols()
    for n in ("coda_gemm_resid_norm_stats", "coda_row_rms", "coda_gemm_rowscale_swiglu",
              "coda_gemm_rope", "coda_lmhead_ce", "coda_gemm_rowscale_swiglu_bwd",
              "coda_row_rms_bwd", "coda_gemm_resid_norm_stats_bwd", "coda_col_reduce",
              "coda_gemm_rope_bwd", "coda_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import gemm_epilogue_fusion_tcgen05_gb300 as c
    for n in declared_symbols():
        assert hasattr(L, n), f"{n} not exported"
        assert n in c.EXPORTS, f"{n} has no binding"


def test_size_queries(L):
    assert L.coda_col_tiles(2048) == 16
    assert L.coda_col_tiles(2049) == 17
    assert L.coda_col_tiles(128) == 1
    assert L.coda_col_tiles(0) == 0
    assert L.coda_row_tiles32(8192) == 256
    assert L.coda_row_tiles32(33) == 2
    # partials (max, sumexp) per 256-column tile plus the target logit, 256-aligned
    M, V = 8192, 128256
    want = ((501 * M * 8 + 255) // 256) * 256 + ((M * 4 + 255) // 256) * 256
    assert L.coda_lmhead_ce_workspace_size(M, V) == want
    assert L.coda_version() >= 100


P = ctypes.c_void_p


def test_invalid_arguments_rejected_on_host(L):
    ok = P(0x10000)       # aligned fake pointer: never dereferenced, checks fail first
    bad = P(0x10001)      # misaligned
    null = None
    # null pointer
    assert L.coda_gemm(null, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 64, 64, 64, None) == 1
    # misaligned pointer
    assert L.coda_gemm(bad, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 64, 64, 64, None) == 1
    # empty and negative sizes
    assert L.coda_gemm(ok, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 0, 64, 64, None) == 1
    assert L.coda_gemm(ok, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 64, -1, 64, None) == 1
    # beyond the largest supported extent (2^30 - 1 per dimension)
    assert L.coda_gemm(ok, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 1 << 30, 64, 64, None) == 1
    # row stride not a multiple of 16 bytes
    assert L.coda_gemm(ok, 65, 0, ok, 64, 0, None, None, ok, 64, 0, 64, 64, 65, None) == 1
    # leading dimension smaller than the row
    assert L.coda_gemm(ok, 32, 0, ok, 64, 0, None, None, ok, 64, 0, 64, 64, 64, None) == 1
    # residual with a transposed operand is not defined
    assert L.coda_gemm(ok, 64, 1, ok, 64, 0, ok, None, ok, 64, 0, 64, 64, 64, None) == 1
    assert b"resid" in L.coda_last_error_string()
    # swiglu: two_f must be a multiple of 16
    assert L.coda_gemm_rowscale_swiglu(ok, ok, ok, ok, None, 64, 24, 64, None) == 1
    # rope: n_rope not a multiple of head_dim
    assert L.coda_gemm_rope(ok, ok, None, ok, 128, 128, 100, ok, None, 64, 256, 64, None) == 1
    # CE: workspace too small
    assert L.coda_lmhead_ce(ok, ok, ok, ok, ok, ok, 16, 64, 512, 64, None) == 1
    assert b"workspace" in L.coda_last_error_string()
    # aux kernels
    assert L.coda_row_rms(null, 8, 64, 256, ctypes.c_float(1e-6), ok, None) == 1
    assert L.coda_row_rms(ok, 0, 64, 256, ctypes.c_float(1e-6), ok, None) == 1
    assert L.coda_col_reduce(ok, 4, 0, ok, None) == 1
    assert L.coda_selftest_bounded_wait(0, None) == 1


def test_error_string_is_never_null(L):
    assert isinstance(L.coda_last_error_string(), bytes)


def test_sources_name_no_closed_copy_call():
    # the batched-memcpy family is closed on this machine; none of the sources may name it
    pat = re.compile(r"(cu|cuda)Memcpy(3D)?Batch" + "Async")
    for d, _, files in os.walk(os.path.join(ROOT, "gemm_epilogue_fusion_tcgen05_gb300")):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".py", ".cpp")):
                assert not pat.search(open(os.path.join(d, f)).read()), f


def _empty_calls(L):
    """Every compute entry point with M = 0 (no rows); the other sizes valid."""
    ok = P(0x10000)
    f = ctypes.c_float(1e-6)
    return {
        "coda_gemm_resid_norm_stats": lambda M: L.coda_gemm_resid_norm_stats(
            ok, ok, ok, ok, ok, ok, ok, M, 64, 64, None),
        "coda_row_rms": lambda M: L.coda_row_rms(ok, 1, M, 64, f, ok, None),
        "coda_gemm_rowscale_swiglu": lambda M: L.coda_gemm_rowscale_swiglu(
            ok, ok, ok, ok, None, M, 64, 64, None),
        "coda_gemm_rope": lambda M: L.coda_gemm_rope(ok, ok, None, ok, 128, 128, 128, ok, None,
                                                     M, 256, 64, None),
        "coda_lmhead_ce": lambda M: L.coda_lmhead_ce(ok, ok, ok, ok, ok, ok, 1 << 20, M, 512, 64,
                                                     None),
        "coda_lmhead_ce_noalloc": lambda M: L.coda_lmhead_ce_noalloc(ok, ok, ok, ok, ok, M, 512,
                                                                     64, None),
        "coda_lmhead_ce_bwd": lambda M: L.coda_lmhead_ce_bwd(ok, ok, ok, ok, ok, ok, ok, ok,
                                                             1 << 20, M, 512, 64, None),
        "coda_gemm_rowscale_swiglu_bwd": lambda M: L.coda_gemm_rowscale_swiglu_bwd(
            ok, ok, ok, ok, ok, ok, M, 64, 64, None),
        "coda_row_rms_bwd": lambda M: L.coda_row_rms_bwd(ok, 1, M, 64, ok, None),
        "coda_gemm_resid_norm_stats_bwd": lambda M: L.coda_gemm_resid_norm_stats_bwd(
            ok, ok, ok, ok, ok, ok, None, ok, ok, M, 64, 128, None),
        "coda_gemm_rope_bwd": lambda M: L.coda_gemm_rope_bwd(ok, ok, ok, ok, 128, 128, 128, ok, ok,
                                                             M, 256, 64, None),
        "coda_gemm_resid_ln_stats": lambda M: L.coda_gemm_resid_ln_stats(
            ok, ok, ok, ok, ok, ok, ok, ok, M, 64, 64, None),
        "coda_row_ln": lambda M: L.coda_row_ln(ok, ok, 1, M, 64, f, ok, ok, None),
        "coda_gemm_ln_rowscale_swiglu": lambda M: L.coda_gemm_ln_rowscale_swiglu(
            ok, ok, ok, ok, ok, ok, ok, None, M, 64, 64, None),
        "coda_gemm_ln_rowscale_swiglu_bwd": lambda M: L.coda_gemm_ln_rowscale_swiglu_bwd(
            ok, ok, ok, ok, ok, ok, ok, ok, ok, ok, M, 64, 64, None),
        "coda_row_ln_bwd": lambda M: L.coda_row_ln_bwd(ok, ok, ok, 1, M, 64, ok, ok, None),
        "coda_gemm_resid_ln_stats_bwd": lambda M: L.coda_gemm_resid_ln_stats_bwd(
            ok, ok, ok, ok, ok, ok, ok, ok, ok, None, ok, None, ok, ok, M, 64, 128, None),
    }


def test_every_entry_point_rejects_empty_and_negative_rows(L):
    """No rows (or a negative count) is an argument error on the host for
    every compute entry point, before any device work."""
    for name, call in _empty_calls(L).items():
        for M in (0, -1):
            assert call(M) == 1, f"{name}(M={M})"
            assert isinstance(L.coda_last_error_string(), bytes)
    covered = set(_empty_calls(L))
    compute = {n for n in declared_symbols()
               if n not in ("coda_gemm", "coda_col_reduce", "coda_rope_table", "coda_col_tiles",
                            "coda_row_tiles32", "coda_lmhead_ce_workspace_size",
                            "coda_lmhead_ce_bwd_workspace_size", "coda_lmhead_ce_noalloc_capacity",
                            "coda_last_error_string",
                            "coda_get_device_error", "coda_set_timeout_ms", "coda_debug_skip_kblock",
                            "coda_selftest_bounded_wait", "coda_version")}
    assert compute <= covered, sorted(compute - covered)


def _run_bad_call(env_value):
    """A child process that makes one call with an argument error."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("CODA_DEBUG", None)
    if env_value is not None:
        env["CODA_DEBUG"] = env_value
    code = ("import ctypes, gemm_epilogue_fusion_tcgen05_gb300 as c; L = c.lib(); "
            "ok = ctypes.c_void_p(0x10000); "
            "print(L.coda_gemm(ok, 64, 0, ok, 64, 0, None, None, ok, 64, 0, 0, 64, 64, None))")
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=120)


def test_coda_debug_echoes_host_errors_to_stderr(L):
    on = _run_bad_call("1")
    assert on.returncode == 0 and on.stdout.strip() == "1"
    assert "libcoda: coda_gemm" in on.stderr
    for quiet in (None, "0"):
        off = _run_bad_call(quiet)
        assert off.returncode == 0 and off.stdout.strip() == "1"
        assert "libcoda:" not in off.stderr
