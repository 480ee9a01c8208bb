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
    assert libsc.sc_hash_build(None, -1, None, None, ctypes.byref(out)) == 1
    assert libsc.sc_hash_build(None, 5, None, None, None) == 1
    assert libsc.sc_kmap_build(None, 3, 3, None, 0, None, None, ctypes.byref(out)) == 1
    assert libsc.sc_kmap_view(None, None, None, None, None, None) == 1
    # an allocator with only one of its two callbacks is refused
    from submanifold_sparse_convolution_hash_gb300 import binding
    half_alloc = binding.Allocator(1, None, None)
    assert libsc.sc_hash_build(None, 0, ctypes.byref(half_alloc), None, ctypes.byref(out)) == 1
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


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "sc.h"

int main(void) {
  sc_hash h = NULL;
  if (strcmp(sc_status_str(SC_OK), "ok") != 0) return 2;
  /* argument errors come back synchronously, without touching a device */
  sc_allocator a = {NULL, NULL, NULL};
  if (sc_hash_build(NULL, -1, &a, NULL, &h) != SC_ERR_INVALID_ARG) return 3;
  if (h != NULL) return 4;
  if (sc_last_error() == NULL || strlen(sc_last_error()) == 0) return 5;
  printf("%s\n", sc_last_error());
  return 0;
}
"""


def test_header_serves_a_plain_c_program(libsc, tmp_path):
    """include/sc.h compiles as strict C99, and a C program links against
    libsc.so and gets the synchronous argument errors the header states."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.join(ROOT, "submanifold_sparse_convolution_hash_gb300")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-l:libsc.so", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip()


def test_binding_refuses_host_tensors():
    """No CPU path: a tensor that is not on a CUDA device is refused before
    any library call."""
    import torch
    from submanifold_sparse_convolution_hash_gb300 import binding
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.sc_hash_build(torch.zeros((4, 4), dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.sc_hash_build(torch.zeros((4, 4), dtype=torch.int32).numpy())


def test_readme_names_only_declared_entry_points_and_flags():
    """Every sc_* name (function or type) and SC_* flag the README names is
    declared in include/sc.h, and every declared function appears in the
    README."""
    header = open(os.path.join(ROOT, "include", "sc.h")).read()
    code = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    readme = open(os.path.join(ROOT, "README.md")).read()
    fns = set(header_functions())
    declared = set(re.findall(r"\b(sc_[a-z_]+)\b", code))
    flags = set(re.findall(r"#define (SC_[A-Z0-9_]+)", header))
    named_fns = set(re.findall(r"`(sc_[a-z_]+)`", readme))
    named_flags = set(re.findall(r"`(SC_[A-Z0-9_]+)`", readme))
    assert named_fns <= declared, named_fns - declared
    assert named_flags <= flags, named_flags - flags
    assert fns <= set(re.findall(r"\b(sc_[a-z_]+)\b", readme)), fns - set(re.findall(r"\b(sc_[a-z_]+)\b", readme))
