"""The C ABI library loads and exports every symbol include/gemm.h declares.

Host-side checks only: argument validation that returns before any CUDA call, status
strings, and option parsing.  No kernel is launched and no GPU is needed.
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as p
    return p


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ["gemm_create", "gemm_destroy", "gemm_run", "gemm_run_ex", "gemm_run_host", "conv4d_im2col", "conv4d_forward",
              "gemm_get_device_status", "gemm_set_option", "gemm_launch_count", "gemm_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), "missing export " + name
    assert sorted(pkg.EXPORTS) == sorted(declared_functions())


def test_exports_are_plain_c_symbols(pkg):
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


def test_status_strings(pkg):
    for code in (0, -1, -2, -3, -4, -5):
        assert pkg.status_string(code) not in ("", "unknown status")
    assert pkg.status_string(12345) == "unknown status"


def test_null_handle_is_rejected_without_touching_cuda(pkg):
    lib = pkg.library()
    assert lib.gemm_run(None, 4, 4, 4, 1, 4, 1, 4, 1, 4, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_host(None, 4, 4, 4, 1, 4, 1, 4, 1, 4, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_ex(None, 4, 4, 4, 1.0, 1, 4, 1, 4, 0.0, 1, 4, 0, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_set_option(None, 1, 0) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_get_device_status(None, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_destroy(None) == pkg.GEMM_OK
    assert lib.gemm_create(None, 0) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_launch_count(None) == -1
    ins = (ctypes.c_int64 * 4)(4, 4, 4, 4)
    assert lib.conv4d_im2col(None, 1, 1, ins, ins, 1, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.conv4d_forward(None, 1, 1, ins, 1, 1, ins, 1, 1, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.conv4d_forward_cl(None, 1, 16, ins, 1, 16, ins, 1, pkg.GEMM_BF16, None) == pkg.GEMM_ERR_INVALID_ARG
    probs = (pkg.HostProblem * 1)(pkg.HostProblem(4, 4, 4, 1, 4, 1, 4, 1, 4, 0))
    assert lib.gemm_run_host_batch(None, 1, probs, None) == pkg.GEMM_ERR_INVALID_ARG


def test_create_without_a_gpu_reports_an_error(pkg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = pkg.library().gemm_create(ctypes.byref(h), 0)
    assert rc in (pkg.GEMM_ERR_CUDA, pkg.GEMM_ERR_INVALID_ARG)
    assert not h.value


def test_no_multicast_bulk_copy_in_the_sources():
    """The library may run as one replica per GPU of a node, so no bulk (TMA) copy in its
    sources multicasts to the CTAs of a cluster; the CTA-pair kernel loads its operand
    halves per CTA.  (The pair's MMA commit, which signals barriers in both CTAs of the
    pair, is not a copy.)"""
    csrc = os.path.join(ROOT, "programming_tiled_gemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        for stmt in re.findall(r"cp\.(?:async|reduce\.async)\.bulk[^;\"]*", text):
            assert "multicast" not in stmt, (name, stmt)


def declarations_with_comments():
    """(function name, the comment block right before its declaration) for every function
    the header declares."""
    text = open(HEADER).read()
    # drop type definitions with braces (and the comments inside them), keeping the comment
    # in front: a declaration may follow the option enum its comment also describes
    text = re.sub(r"typedef\s+(?:enum|struct)[^{;]*\{.*?\}\s*\w+\s*;", "", text, flags=re.S)
    out = []
    for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*(typedef[^;]*;\s*)?(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.S):
        if m.group(2):
            continue  # the comment belongs to a type
        out.append((m.group(3), m.group(1)))
    return out


def test_every_declaration_cites_its_passage():
    """Each entry point's comment names the page and the section it implements, or says
    that the pages have no counterpart."""
    found = dict(declarations_with_comments())
    assert sorted(found) == declared_functions()
    for name, comment in found.items():
        flat = " ".join(re.sub(r"^\s*\*", "", line) for line in comment.splitlines())
        flat = " ".join(flat.split())
        cited = re.search(r'"[^"]+", sections? "[^"]+"', flat) or re.search(r'"[^"]+" sections? "[^"]+"', flat)
        assert cited or "no counterpart" in flat, name


def test_noalloc_entry_point_checks_sizes_before_touching_cuda(pkg):
    """The allocation-free entry point applies gemm_run's argument and size checks before
    any CUDA call (the pointers below are never dereferenced)."""
    lib = pkg.library()
    big, huge, p = 1 << 40, 1 << 62, 256
    assert lib.gemm_run_f32_skinny_noalloc(16, big, 64, p, 64, p, big, p, big, 0, None) == pkg.GEMM_ERR_UNSUPPORTED
    assert lib.gemm_run_f32_skinny_noalloc(16, 256, 64, p, 64, p, huge, p, 256, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_f32_skinny_noalloc(33, 256, 64, p, 64, p, 256, p, 256, 0, None) == pkg.GEMM_ERR_UNSUPPORTED
    assert lib.gemm_run_f32_skinny_noalloc(16, 256, 64, p, 63, p, 256, p, 256, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_f32_skinny_noalloc(16, 256, 64, p, 64, p, 256, p, 256, 2000, None) == pkg.GEMM_ERR_INVALID_ARG


def test_debug_library_exports_the_same_symbols(pkg):
    """The debug build (kernels with index checks) exports the same C ABI."""
    path = os.path.join(os.path.dirname(pkg.LIB_PATH), "libgemm_gb300_debug.so")
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), "missing export " + name


LOG_PROBE = r"""
import ctypes, sys
lib = ctypes.CDLL(sys.argv[1])
i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
lib.gemm_run_f32_skinny_noalloc.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, i32, p]
lib.gemm_set_option.argtypes = [p, i32, i64]
assert lib.gemm_run_f32_skinny_noalloc(33, 256, 64, 256, 64, 256, 256, 256, 256, 0, None) == -3
assert lib.gemm_set_option(None, 1, 0) == -1
"""


def run_log_probe(pkg, env_extra):
    env = {k: v for k, v in os.environ.items() if k != "GEMM_LOG"}
    env.update(env_extra)
    return subprocess.run([sys.executable, "-c", LOG_PROBE, pkg.LIB_PATH], capture_output=True, text=True, env=env,
                          timeout=120)


def test_gemm_log_reports_refused_calls_on_stderr(pkg):
    p = run_log_probe(pkg, {"GEMM_LOG": "1"})
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stderr.splitlines() if ln.startswith("[gemm] ")]
    assert any("gemm_run_f32_skinny_noalloc(M 33" in ln and "refused" in ln for ln in lines), p.stderr
    assert any("gemm_set_option(1, 0) refused" in ln for ln in lines), p.stderr


def test_without_gemm_log_nothing_is_printed(pkg):
    for env in ({}, {"GEMM_LOG": "0"}, {"GEMM_LOG": "yes"}):
        p = run_log_probe(pkg, env)
        assert p.returncode == 0, p.stderr
        assert p.stderr == "", p.stderr
