"""Planted mistakes: each test compiles a copy of the oracle with one plausible
mistake written into its source (a flipped sign, a swapped offset order, a
dropped term, a transposed operand, a missing mirror, a floor for a ceiling,
...) and checks that the pins in test_oracle_pins.py catch it.  A control
build of the unchanged source passes every pin.  Everything runs on the CPU;
the product library is not involved."""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

# (name, text in oracle.cpp, replacement).  Where the text occurs more than
# once (the strided layer restates the submanifold loops), the first
# occurrence, the submanifold one, is mutated.
MUTATIONS = [
    ("offset sign flipped: the input read at Q - d",
     "int64_t x = int64_t(c[1]) + d[0];\n  int64_t y = int64_t(c[2]) + d[1];\n  int64_t z = int64_t(c[3]) + d[2];",
     "int64_t x = int64_t(c[1]) - d[0];\n  int64_t y = int64_t(c[2]) - d[1];\n  int64_t z = int64_t(c[3]) - d[2];"),
    ("offset index order: first axis fastest",
     "for (int k = ndim - 1; k >= 0; --k) {\n    d[k] = idx % K - r;",
     "for (int k = 0; k < ndim; ++k) {\n    d[k] = idx % K - r;"),
    ("dropped term: the last offset never accumulated",
     "for (int v = 0; v < V; ++v) {\n      const int32_t p = neighbour(P, q, &offs[3 * v]);",
     "for (int v = 0; v < V - 1; ++v) {\n      const int32_t p = neighbour(P, q, &offs[3 * v]);"),
    ("ReLU ignored",
     "    if (relu)\n      for (int co = 0; co < c_out; ++co) acc[co] = acc[co] > 0.0 ? acc[co] : 0.0;\n  }\n  return OR_OK;\n}\n\n}  // namespace",
     "    if (relu && false)\n      for (int co = 0; co < c_out; ++co) acc[co] = acc[co] > 0.0 ? acc[co] : 0.0;\n  }\n  return OR_OK;\n}\n\n}  // namespace"),
    ("duplicate coordinates merged instead of rejected",
     "if (!ins.second) return OR_DUPLICATE;",
     "if (!ins.second) continue;"),
    ("input gradient: W_d read transposed",
     "for (int co = 0; co < c_out; ++co) sum += wrow[co] * g[co];",
     "for (int co = 0; co < c_out; ++co) sum += w[int64_t(co) * c_in + ci] * g[co];"),
    ("input gradient: no mirror (the output at c_p + d)",
     "for (int a = 0; a < 3; ++a) neg[3 * v + a] = -neg[3 * v + a];",
     "for (int a = 0; a < 3; ++a) neg[3 * v + a] = +neg[3 * v + a];"),
    ("weight gradient: feature and gradient rows swapped",
     "const double* f = feats + int64_t(p) * c_in;\n      const double* g = gout + q * c_out;",
     "const double* f = feats + q * c_in;\n      const double* g = gout + int64_t(p) * c_out;"),
    ("strided layer: the input read at s o - d",
     "return input_at(P, c_o[0], int64_t(c_o[1]) * stride + d[0], int64_t(c_o[2]) * stride + d[1],\n"
     "                  int64_t(c_o[3]) * sz + d[2]);",
     "return input_at(P, c_o[0], int64_t(c_o[1]) * stride - d[0], int64_t(c_o[2]) * stride - d[1],\n"
     "                  int64_t(c_o[3]) * sz - d[2]);"),
    ("strided output grid: floor(dims / s) instead of the ceiling",
     "int out_extent(int dim, int s) { return (dim + s - 1) / s; }",
     "int out_extent(int dim, int s) { return dim / s; }"),
    ("strided output set: the stride ignored when finding outputs",
     "const int64_t o[3] = {px / stride, py / stride, pz / sz};",
     "const int64_t o[3] = {px, py, pz};"),
]

# The pins run against each build: the pages' worked examples, brute force,
# dense fp64 convolutions and their autograd gradients.
PINS = [
    ("five-point map", lambda: pins.test_five_point_map_matches_worked_example()),
    ("sign quiz", lambda: pins.test_sign_convention_quiz()),
    ("4x5 grid", lambda: pins.test_four_point_grid_counts()),
    ("brute force 3D", lambda: pins.test_kmap_equals_brute_force(3, 3, (6, 7, 5), 60, 2)),
    ("map errors", lambda: pins.test_kmap_errors()),
    ("dense conv 3D", lambda: pins.test_conv_equals_dense_conv(3, 3, (7, 6, 5), 70, 2, 4, 6)),
    ("dense conv 2D", lambda: pins.test_conv_equals_dense_conv(2, 3, (9, 11, 1), 30, 2, 5, 3)),
    ("closed forms", lambda: pins.test_conv_single_site_two_sites_linearity_relu()),
    ("autograd", lambda: pins.test_backward_equals_dense_conv_autograd(3, 3, (7, 6, 5), 70, 2, 4, 6)),
    ("backward closed forms", lambda: pins.test_backward_closed_forms()),
    ("regular 4x5 grid", lambda: pins.test_regular_four_point_grid()),
    ("strided map", lambda: pins.test_strided_map_equals_brute_force(3, 3, 2, (7, 6, 5), 40, 1)),
    ("strided dense conv", lambda: pins.test_strided_conv_equals_dense_conv(3, 3, 2, (8, 7, 6), 50, 1, 4, 4)),
    ("strided input gradient", lambda: pins.test_strided_input_gradient_equals_dense_autograd(3, 3, 2, (7, 6, 8), 40,
                                                                                               3, 2)),
]


def _compile(text, path):
    src = str(path) + ".cpp"
    with open(src, "w") as fh:
        fh.write(text)
    subprocess.run(["g++", "-O1", "-std=c++17", "-fopenmp", "-fPIC", "-shared", src, "-o", str(path)], check=True,
                   capture_output=True)
    return str(path)


def _run_pins(monkeypatch, lib_path):
    """Names of the pins that fail with the oracle loaded from lib_path."""
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "_LIB_PATH", lib_path)
    monkeypatch.setattr(oracle, "build", lambda force=False: lib_path)
    failed = []
    for name, pin in PINS:
        try:
            pin()
        except (Exception, pytest.fail.Exception):  # an assertion, a pytest.raises miss, or a provoked error
            failed.append(name)
    monkeypatch.setattr(oracle, "_lib", None)
    return failed


@pytest.fixture(scope="module")
def source():
    if shutil.which("g++") is None:
        pytest.skip("no C++ compiler")
    return open(SRC).read()


def test_control_build_passes_every_pin(source, tmp_path, monkeypatch):
    lib = _compile(source, tmp_path / "liboracle_control.so")
    assert _run_pins(monkeypatch, lib) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(source, tmp_path, monkeypatch, name, old, new):
    assert source.count(old) >= 1, f"the text to mutate is not in oracle.cpp: {name}"
    lib = _compile(source.replace(old, new, 1), tmp_path / "liboracle_mutant.so")
    failed = _run_pins(monkeypatch, lib)
    assert failed, f"no pin caught: {name}"
