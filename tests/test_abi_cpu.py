"""CPU checks of the boundary: libsc.so loads, exports every function that
include/sc.h declares, and answers host-only calls without a GPU.  No
compute call is made here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def header_functions():
    text = open(os.path.join(ROOT, "include", "sc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sc_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libsc():
    from submanifold_sparse_convolution_hash_gb300 import build
    build.build()
    from submanifold_sparse_convolution_hash_gb300 import binding
    return binding.lib()


def test_header_declares_the_hash_map_and_layer_entry_points():
    fns = header_functions()
    for name in ("sc_hash_build", "sc_kmap_build", "sc_subm_conv_fwd"):
        assert name in fns


def test_library_exports_every_declared_function(libsc):
    missing = [f for f in header_functions() if not hasattr(libsc, f)]
    assert not missing, missing


def test_binding_names_match_header(libsc):
    from submanifold_sparse_convolution_hash_gb300 import binding
    assert set(binding.exported_symbols()) == set(header_functions())


def test_host_only_calls(libsc):
    assert libsc.sc_status_str(0) == b"ok"
    assert libsc.sc_status_str(3) == b"duplicate coordinate"
    assert libsc.sc_launch_count() >= 0
    # argument errors return synchronously, before any CUDA call
    out = ctypes.c_void_p()
    assert libsc.sc_hash_build(None, -1, None, ctypes.byref(out)) == 1
    assert libsc.sc_hash_build(None, 5, None, None) == 1
    assert libsc.sc_kmap_build(None, 3, 3, None, 0, None, ctypes.byref(out)) == 1
    assert libsc.sc_subm_conv_fwd(None, None, None, None, 32, 32, 1, 0, None) == 1
    assert b"NULL" in libsc.sc_last_error()


def test_missing_library_fails_loudly(monkeypatch):
    from submanifold_sparse_convolution_hash_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_LIB_PATH", os.path.join(ROOT, "does-not-exist", "libsc.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "submanifold_sparse_convolution_hash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
