"""The C-ABI library builds, loads and exports every entry point of include/spec_verify.h;
host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_\w+)\s*\(", src, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    B.build()
    return G.load()


def test_header_declares_the_boundary():
    want = {"spec_verify_init", "spec_verify_destroy", "spec_build_tree_mask",
            "spec_verify_greedy", "spec_verify_sample"}
    assert want <= _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in sorted(_declared()):
        assert hasattr(lib, name), name


def test_error_strings(lib):
    assert G.error_string(G.SPEC_OK) == "ok"
    assert "argument" in G.error_string(G.SPEC_ERR_ARG)
    assert G.error_string(12345) == "unknown error code"


def test_host_checks_without_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.spec_verify_init(ctypes.byref(h), 4, 65, 100, 0) == G.SPEC_ERR_UNSUPPORTED
    assert lib.spec_verify_init(ctypes.byref(h), 4, 8, (1 << 21) + 1, 0) == G.SPEC_ERR_UNSUPPORTED
    assert lib.spec_verify_init(ctypes.byref(h), 0, 8, 100, 0) == G.SPEC_ERR_ARG
    assert lib.spec_verify_init(None, 4, 8, 100, 0) == G.SPEC_ERR_ARG
    assert lib.spec_verify_greedy(None, None, 1, 1, 1, 10, None, None, None, None, None, None,
                                  None, None) == G.SPEC_ERR_ARG
    assert lib.spec_verify_sample(None, None, 1, 1, 1, 10, None, None, None, 0, 0, 1.0, None,
                                  None, None, None, None, None, None) == G.SPEC_ERR_ARG
    assert lib.spec_build_tree_mask(None, None, 1, 1, None, None, None, None) == G.SPEC_ERR_ARG
    assert lib.spec_set_node_budget(None, None) == G.SPEC_ERR_ARG
    prm = G.BudgetParams(0.5, 0.5, 0.0, 1, 4, 1)
    assert lib.spec_budget_update(None, ctypes.byref(prm), None, None, None, 1, 4, None, None,
                                  None) == G.SPEC_ERR_ARG
    assert lib.spec_row_stats(None, None, 1, 1, 1, 10, 1.0, None, None, None, None, None, None,
                              None, None) == G.SPEC_ERR_ARG
    assert lib.spec_verify_destroy(None) == G.SPEC_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(G, "LIBRARY", str(tmp_path / "missing.so"))
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        G.load()


def test_nvtx_ranges_compile(tmp_path):
    """The NVTX-instrumented flavour of the entry points (SPEC_NVTX) compiles; a range opens
    and closes around each call without touching its arguments."""
    import subprocess
    obj = tmp_path / "api_nvtx.o"
    r = subprocess.run([B.nvcc(), *B.ARCH, *B.FLAGS, "-DSPEC_NVTX", "-I", B.INCLUDE, "-I",
                        B.CSRC, "-c", os.path.join(B.CSRC, "api.cu"), "-o", str(obj)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert obj.stat().st_size > 0
    src = open(os.path.join(B.CSRC, "api.cu")).read()
    for name in _declared() - {"spec_error_string", "spec_profile_begin", "spec_profile_end",
                               "spec_verify_greedy_noalloc"}:
        assert f'SPEC_RANGE("{name}")' in src, name


def test_release_build_refuses_the_debug_hooks(lib):
    """The debug entry points exist in every build; the release build says it is not the
    debug flavour and refuses the fault-injection and debug-word calls without touching a
    GPU."""
    assert lib.spec_debug_build() == 0
    assert lib.spec_debug_inject_arrival(None, 0, 1) == G.SPEC_ERR_UNSUPPORTED
    assert lib.spec_debug_words(None, None, 0, None) == G.SPEC_ERR_UNSUPPORTED


@pytest.mark.parametrize("src", ["api.cu", "row_stats.cu", "walk_greedy.cu", "kv_commit.cu"])
def test_debug_flavour_compiles(tmp_path, src):
    """The checked flavour (SPEC_DEBUG) of the entry points and kernels compiles for sm_103a."""
    import subprocess
    obj = tmp_path / (src + ".o")
    r = subprocess.run([B.nvcc(), *B.ARCH, *B.FLAGS, "-DSPEC_DEBUG", "-I", B.INCLUDE, "-I",
                        B.CSRC, "-c", os.path.join(B.CSRC, src), "-o", str(obj)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
