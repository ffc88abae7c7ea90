"""CPU-side checks of the C-ABI library: it builds, loads, exports every
symbol include/dseq.h declares, and rejects bad arguments before touching a
GPU.  No compute call runs here."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import embedding_similarity_scan_gb300 as es
from embedding_similarity_scan_gb300 import build as esb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dseq.h")


@pytest.fixture(scope="module")
def lib():
    esb.build()
    return es.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in keywords})


def test_header_declares_the_binding_exports():
    assert sorted(es.EXPORTS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libdseq.so does not export {name}"
    # and they are C symbols (no mangling)
    out = os.popen(f"nm -D --defined-only {es.LIB_PATH}").read()
    for name in _declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} missing from the dynamic symbol table"


def test_library_links_no_cuda_runtime_or_driver_dynamically(lib):
    out = os.popen(f"ldd {es.LIB_PATH}").read()
    assert "libcudart" not in out and "libcuda.so" not in out


def test_argument_errors_before_any_gpu_work(lib):
    h = ctypes.c_void_p()
    assert lib.dseq_create(None, 10, 4, 0, None, ctypes.byref(h)) == es.DSEQ_EINVAL
    assert "NULL" in es.dseq_last_error()
    t = np.zeros((10, 4), np.float32)
    assert lib.dseq_create(t.ctypes.data, 0, 4, 0, None, ctypes.byref(h)) == es.DSEQ_EINVAL
    assert lib.dseq_create(t.ctypes.data, 10, 0, 0, None, ctypes.byref(h)) == es.DSEQ_EINVAL
    assert lib.dseq_create(t.ctypes.data, 10, 20000, 0, None, ctypes.byref(h)) == es.DSEQ_EINVAL
    assert lib.dseq_create(t.ctypes.data, 10, 4, 0, None, None) == es.DSEQ_EINVAL
    assert lib.dseq_run(None, None, 1, 1, None, None, None) == es.DSEQ_EINVAL
    assert lib.dseq_run_trace(None, None, 1, 1, None, None, None, 0, None, None) == es.DSEQ_EINVAL
    i = np.zeros(4, np.int32)
    d = np.zeros(4, np.float32)
    assert lib.bmu_search(None, 4, t.ctypes.data, 10, 4, i.ctypes.data, d.ctypes.data,
                          None) == es.DSEQ_EINVAL
    assert lib.bmu_search(t.ctypes.data, 0, t.ctypes.data, 10, 4, i.ctypes.data,
                          d.ctypes.data, None) == es.DSEQ_EINVAL
    assert lib.bmu_search(t.ctypes.data, 4, t.ctypes.data, 0, 4, i.ctypes.data,
                          d.ctypes.data, None) == es.DSEQ_EINVAL
    lib.dseq_destroy(None)


def test_options(lib):
    assert es.dseq_get_option("engine") == 0
    assert es.dseq_get_option("timeout_ms") == 10000
    assert es.dseq_get_option("pair") == 1
    assert es.dseq_get_option("nonsense") == -1
    with pytest.raises(es.DseqError) as ei:
        es.dseq_set_option("nonsense", 1)
    assert ei.value.code == es.DSEQ_EINVAL
    assert es.dseq_get_option("gram") == 2 and es.dseq_get_option("walk") == 0
    for bad in (("tile_n", 48), ("tile_n", 512), ("engine", 2), ("timeout_ms", 0),
                ("gram", 3), ("walk", 4), ("walk", -1)):
        with pytest.raises(es.DseqError):
            es.dseq_set_option(*bad)
    es.dseq_set_option("tile_n", 96)
    assert es.dseq_get_option("tile_n") == 96
    es.dseq_set_option("tile_n", 0)
    es.dseq_set_option("walk", 2)
    assert es.dseq_get_option("walk") == 2
    es.dseq_set_option("walk", 0)
    assert es.dseq_last_stat("walk") == 0 and es.dseq_last_stat("gram") == 0
    # the process-wide buffer cache: trims to the new limit when lowered;
    # -1 (the default) is half of each device's memory
    assert es.dseq_get_option("cache_mb") == -1
    es.dseq_set_option("cache_mb", 0)
    assert es.dseq_get_option("cache_mb") == 0
    es.dseq_set_option("cache_mb", 4096)
    assert es.dseq_get_option("cache_mb") == 4096
    es.dseq_set_option("cache_mb", -1)
    assert es.dseq_get_option("cache_mb") == -1
    with pytest.raises(es.DseqError):
        es.dseq_set_option("cache_mb", -2)
    assert es.dseq_last_stat("units") == 0 and es.dseq_last_stat("bogus") == -1


def test_test_options_need_opt_in(lib, monkeypatch):
    """Options that change results on purpose (fault injection, the
    epilogue-isolated kernel) are refused unless the process opts in through
    DSEQ_ENABLE_TEST_OPTIONS=1; setting them back to 0 is always allowed."""
    names = ("isolate_epilogue", "fault_skip_arrive", "fault_skip_copy")
    monkeypatch.delenv("DSEQ_ENABLE_TEST_OPTIONS", raising=False)
    for name in names:
        with pytest.raises(es.DseqError) as ei:
            es.dseq_set_option(name, 1)
        assert ei.value.code == es.DSEQ_EINVAL and "DSEQ_ENABLE_TEST_OPTIONS" in str(ei.value)
        es.dseq_set_option(name, 0)
        assert es.dseq_get_option(name) == 0
    monkeypatch.setenv("DSEQ_ENABLE_TEST_OPTIONS", "1")
    for name in names:
        es.dseq_set_option(name, 1)
        assert es.dseq_get_option(name) == 1
        es.dseq_set_option(name, 0)
    with pytest.raises(es.DseqError):
        es.dseq_set_option("isolate_epilogue", 2)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        es.load(str(tmp_path / "libdseq.so"))
