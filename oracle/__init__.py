"""CPU oracle for the submanifold sparse convolution layer.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports, links or calls it, and it imports
nothing from the CUDA library.

The arithmetic lives in ``oracle.cpp`` (plain C++17, fp64, ``std::unordered_map``
keyed on coordinates, a nested loop over outputs x offsets).  This module only
marshals numpy arrays into it and derives the tuple set and per-offset lists
from the neighbour table, which is a relabelling, not a computation.

Pins (tests/test_oracle_pins.py): the pages' worked examples (the 4x5 and 5x5
grids, the 11-tuple map with its 2/1/5/1/2 split, the quiz answer Q = (2, 2)),
the (2L+1)^d dilation counts, mirror symmetry, brute force over all point
pairs, and an fp64 dense convolution from ``torch.nn.functional`` read at the
active sites.  The regular / strided layers are pinned to the same grid
examples (17 then 20 active cells, 30 map entries), the dilation counts,
stride-2 closed forms, brute force, and the strided dense convolution (its
values at the output sites and its support as the output set).  No function
here is parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

STATUS = {0: "ok", 1: "bad argument", 2: "coordinate out of range", 3: "duplicate coordinate"}


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle: {STATUS.get(code, code)}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so next to it (g++, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        lib.oracle_kmap.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
        lib.oracle_kmap.restype = ctypes.c_int
        lib.oracle_subm_conv.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, P,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64,
                                         P, ctypes.c_int]
        lib.oracle_subm_conv.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_subm_conv_bwd_data.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, P,
                                                  ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P, ctypes.c_int]
        lib.oracle_subm_conv_bwd_data.restype = ctypes.c_int
        lib.oracle_subm_conv_bwd_weight.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, P,
                                                    ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
        lib.oracle_subm_conv_bwd_weight.restype = ctypes.c_int
        lib.oracle_hash_only.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P]
        lib.oracle_hash_only.restype = ctypes.c_int
        I64, I = ctypes.c_int64, ctypes.c_int
        lib.oracle_conv_out_coords.argtypes = [P, I64, I, I, I, P, P, I64, P]
        lib.oracle_conv_out_coords.restype = I
        lib.oracle_conv_kmap.argtypes = [P, I64, P, I64, I, I, I, P, P, I]
        lib.oracle_conv_kmap.restype = I
        lib.oracle_conv.argtypes = [P, I64, P, I64, I, I, I, P, P, P, I, I, I, P, I]
        lib.oracle_conv.restype = I
        lib.oracle_conv_bwd_weight.argtypes = [P, I64, P, I64, I, I, I, P, P, P, I, I, P, I]
        lib.oracle_conv_bwd_weight.restype = I
        lib.oracle_conv_bwd_data.argtypes = [P, I64, P, I64, I, I, I, P, P, P, I, I, P, I]
        lib.oracle_conv_bwd_data.restype = I
        lib.oracle_table_build.argtypes = [P, I64, I, I, P, ctypes.POINTER(ctypes.c_int)]
        lib.oracle_table_build.restype = P
        lib.oracle_table_subm_conv.argtypes = [P, P, P, I, I, I, P, I64, P, I]
        lib.oracle_table_subm_conv.restype = I
        lib.oracle_table_free.argtypes = [P]
        lib.oracle_table_free.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _coords(coords):
    return np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))


def _rows(a, n: int) -> np.ndarray:
    """fp64, C-contiguous [n, width] copy of a feature array: a 2-D array as it
    is (it must have n rows), anything else reshaped to n rows.  n may be 0."""
    a = np.asarray(a, dtype=np.float64)
    if a.ndim != 2:
        a = a.reshape(n, -1)
    if a.shape[0] != n:
        raise OracleError(1)
    return np.ascontiguousarray(a)


def _dims(dims):
    d = np.ones(3, dtype=np.int32)
    d[: len(dims)] = dims
    return d


def volume(ndim: int, K: int) -> int:
    return K ** ndim


def offset_index(delta, K: int) -> int:
    """Lexicographic offset index, first spatial axis slowest."""
    r = (K - 1) // 2
    idx = 0
    for d in delta:
        idx = idx * K + (int(d) + r)
    return idx


def offset_of(idx: int, ndim: int, K: int) -> tuple:
    r = (K - 1) // 2
    d = []
    for _ in range(ndim):
        d.append(idx % K - r)
        idx //= K
    return tuple(reversed(d))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def hash_only(coords, ndim: int, K: int, dims) -> None:
    """Builds (and drops) the oracle's coordinate table: step 1 alone."""
    c = _coords(coords)
    st = _load().oracle_hash_only(_ptr(c), c.shape[0], ndim, K, _ptr(_dims(dims)))
    if st:
        raise OracleError(st)


def kmap(coords, ndim: int, K: int, dims, threads: int = 0) -> np.ndarray:
    """Neighbour table int32 [N, K^ndim]: input row at c_q + d, or -1."""
    c = _coords(coords)
    n = c.shape[0]
    V = volume(ndim, K)
    nbr = np.empty((n, V), dtype=np.int32)
    st = _load().oracle_kmap(_ptr(c), n, ndim, K, _ptr(_dims(dims)), _ptr(nbr), threads)
    if st:
        raise OracleError(st)
    return nbr


def tuples(nbr: np.ndarray) -> np.ndarray:
    """The map M as an int64 array of (offset, out, in) rows, sorted."""
    q, v = np.nonzero(nbr >= 0)
    p = nbr[q, v]
    t = np.stack([v.astype(np.int64), q.astype(np.int64), p.astype(np.int64)], axis=1)
    order = np.lexsort((t[:, 2], t[:, 1], t[:, 0]))
    return t[order]


def offset_lists(nbr: np.ndarray) -> list:
    """Per-offset lists [(in_rows, out_rows)] ordered by output row."""
    out = []
    for v in range(nbr.shape[1]):
        q = np.nonzero(nbr[:, v] >= 0)[0]
        out.append((nbr[q, v].astype(np.int64), q.astype(np.int64)))
    return out


def subm_conv(coords, feats, W, ndim: int, K: int, dims, relu: bool = False,
              rows=None, threads: int = 0) -> np.ndarray:
    """fp64 output features [len(rows) or N, C_out] of one submanifold layer."""
    c = _coords(coords)
    n = c.shape[0]
    f = _rows(feats, n)
    w = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
    V, c_in, c_out = w.shape
    if V != volume(ndim, K) or f.shape[1] != c_in:
        raise OracleError(1)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = n if r is None else r.shape[0]
    out = np.empty((nrows, c_out), dtype=np.float64)
    st = _load().oracle_subm_conv(_ptr(c), n, ndim, K, _ptr(_dims(dims)), _ptr(f), _ptr(w),
                                  c_in, c_out, int(bool(relu)), _ptr(r), nrows, _ptr(out), threads)
    if st:
        raise OracleError(st)
    return out


class Table:
    """The coordinate table (step 1) built once and kept, so that layer
    outputs of listed rows can be computed against it repeatedly: used to
    time the table and the rows apart.  subm_conv here equals the module's
    subm_conv for the same arguments."""

    def __init__(self, coords, ndim: int, K: int, dims):
        self._c = _coords(coords)  # the table refers to these coordinates
        self.n = self._c.shape[0]
        self.ndim, self.K = ndim, K
        st = ctypes.c_int(0)
        self._h = _load().oracle_table_build(_ptr(self._c), self.n, ndim, K, _ptr(_dims(dims)), ctypes.byref(st))
        if not self._h:
            raise OracleError(st.value)

    def subm_conv(self, feats, W, relu: bool = False, rows=None, threads: int = 0) -> np.ndarray:
        f = _rows(feats, self.n)
        w = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
        V, c_in, c_out = w.shape
        if V != volume(self.ndim, self.K) or f.shape[1] != c_in:
            raise OracleError(1)
        r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = self.n if r is None else r.shape[0]
        out = np.empty((nrows, c_out), dtype=np.float64)
        st = _load().oracle_table_subm_conv(self._h, _ptr(f), _ptr(w), c_in, c_out, int(bool(relu)), _ptr(r),
                                            nrows, _ptr(out), threads)
        if st:
            raise OracleError(st)
        return out

    def close(self) -> None:
        if self._h:
            _load().oracle_table_free(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def subm_conv_bwd_data(coords, gout, W, ndim: int, K: int, dims, rows=None, threads: int = 0) -> np.ndarray:
    """fp64 gradient with respect to the layer's input features [len(rows) or
    N, C_in], given the gradient with respect to its output [N, C_out]."""
    c = _coords(coords)
    n = c.shape[0]
    w = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
    V, c_in, c_out = w.shape
    g = np.ascontiguousarray(np.asarray(gout, dtype=np.float64).reshape(n, c_out))
    if V != volume(ndim, K):
        raise OracleError(1)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = n if r is None else r.shape[0]
    out = np.empty((nrows, c_in), dtype=np.float64)
    st = _load().oracle_subm_conv_bwd_data(_ptr(c), n, ndim, K, _ptr(_dims(dims)), _ptr(g), _ptr(w), c_in, c_out,
                                           _ptr(r), nrows, _ptr(out), threads)
    if st:
        raise OracleError(st)
    return out


def subm_conv_bwd_weight(coords, feats, gout, ndim: int, K: int, dims, threads: int = 0) -> np.ndarray:
    """fp64 gradient with respect to the weights [K^ndim, C_in, C_out]."""
    c = _coords(coords)
    n = c.shape[0]
    f = _rows(feats, n)
    g = _rows(gout, n)
    V = volume(ndim, K)
    out = np.empty((V, f.shape[1], g.shape[1]), dtype=np.float64)
    st = _load().oracle_subm_conv_bwd_weight(_ptr(c), n, ndim, K, _ptr(_dims(dims)), _ptr(f), _ptr(g), f.shape[1],
                                             g.shape[1], _ptr(out), threads)
    if st:
        raise OracleError(st)
    return out


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values once to a storage dtype (RN-even), returned as fp64."""
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # bfloat16 keeps 8 significant bits and fp32's exponent range: round
        # the fp64 value straight to a multiple of its bf16 quantum, ties to
        # even (np.rint), with the quantum floored at 2^-133 (subnormals).
        x = np.asarray(x, dtype=np.float64)
        _, e = np.frexp(x)
        e = np.maximum(e, -125)
        return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    raise ValueError(dtype)


def subm_conv_stack(coords, feats, Ws, ndim: int, K: int, dims, dtype: str,
                    threads: int = 0) -> list:
    """Layer outputs of a stack sharing one map: ReLU between layers, none
    after the last; each layer's output rounded once to ``dtype`` (as stored)
    before it feeds the next layer."""
    outs = []
    x = np.asarray(feats, dtype=np.float64)
    for li, W in enumerate(Ws):
        y = subm_conv(coords, x, W, ndim, K, dims, relu=(li + 1 < len(Ws)), threads=threads)
        y = round_to(y, dtype)
        outs.append(y)
        x = y
    return outs


# --------------------------------------------------------------------------
# Regular (stride 1: dilating) and strided layers: the output set differs
# from the input set ("SparseConvNet: from hash table to rulebook", sections
# 2 and 3).  Output o reads the input at stride * o + d through W_d.
# --------------------------------------------------------------------------

def conv_out_coords(coords, ndim: int, K: int, stride: int, dims) -> np.ndarray:
    """Output sites int32 [N_out, 4] of a regular / strided layer, sorted by
    (batch, x, y, z): every o with an active input at stride * o + d."""
    c = _coords(coords)
    n = c.shape[0]
    cap = n * volume(ndim, K)
    out = np.empty((max(cap, 1), 4), dtype=np.int32)
    n_out = ctypes.c_int64(0)
    st = _load().oracle_conv_out_coords(_ptr(c), n, ndim, K, stride, _ptr(_dims(dims)), _ptr(out), cap,
                                        ctypes.byref(n_out))
    if st:
        raise OracleError(st)
    return out[: n_out.value].copy()


def conv_out_extent(dims, ndim: int, stride: int) -> tuple:
    """Extents of the output grid: ceil(dims / stride) on the strided axes."""
    d = list(_dims(dims))
    axes = 3 if ndim == 3 else 2
    return tuple((d[a] + stride - 1) // stride if a < axes else d[a] for a in range(3))


def conv_kmap(coords, out_coords, ndim: int, K: int, stride: int, dims, threads: int = 0) -> np.ndarray:
    """Neighbour table int32 [N_out, K^ndim]: input row at stride * c_q + d, or -1."""
    c, o = _coords(coords), _coords(out_coords)
    V = volume(ndim, K)
    nbr = np.empty((o.shape[0], V), dtype=np.int32)
    st = _load().oracle_conv_kmap(_ptr(c), c.shape[0], _ptr(o), o.shape[0], ndim, K, stride, _ptr(_dims(dims)),
                                  _ptr(nbr), threads)
    if st:
        raise OracleError(st)
    return nbr


def sparse_conv(coords, out_coords, feats, W, ndim: int, K: int, stride: int, dims, relu: bool = False,
                threads: int = 0) -> np.ndarray:
    """fp64 output features [N_out, C_out] of one regular / strided layer."""
    c, o = _coords(coords), _coords(out_coords)
    n = c.shape[0]
    f = _rows(feats, n)
    w = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
    V, c_in, c_out = w.shape
    if V != volume(ndim, K) or f.shape[1] != c_in:
        raise OracleError(1)
    out = np.empty((o.shape[0], c_out), dtype=np.float64)
    st = _load().oracle_conv(_ptr(c), n, _ptr(o), o.shape[0], ndim, K, stride, _ptr(_dims(dims)), _ptr(f), _ptr(w),
                             c_in, c_out, int(bool(relu)), _ptr(out), threads)
    if st:
        raise OracleError(st)
    return out


def sparse_conv_bwd_weight(coords, out_coords, feats, gout, ndim: int, K: int, stride: int, dims,
                           threads: int = 0) -> np.ndarray:
    """fp64 weight gradient [K^ndim, C_in, C_out] of a regular / strided layer."""
    c, o = _coords(coords), _coords(out_coords)
    f = _rows(feats, c.shape[0])
    g = _rows(gout, o.shape[0])
    V = volume(ndim, K)
    out = np.empty((V, f.shape[1], g.shape[1]), dtype=np.float64)
    st = _load().oracle_conv_bwd_weight(_ptr(c), c.shape[0], _ptr(o), o.shape[0], ndim, K, stride,
                                        _ptr(_dims(dims)), _ptr(f), _ptr(g), f.shape[1], g.shape[1], _ptr(out),
                                        threads)
    if st:
        raise OracleError(st)
    return out


def sparse_conv_bwd_data(coords, out_coords, gout, W, ndim: int, K: int, stride: int, dims,
                         threads: int = 0) -> np.ndarray:
    """fp64 input gradient [N, C_in] of a regular / strided layer, given the
    gradient with respect to its output [N_out, C_out]."""
    c, o = _coords(coords), _coords(out_coords)
    w = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
    V, c_in, c_out = w.shape
    g = np.ascontiguousarray(np.asarray(gout, dtype=np.float64).reshape(o.shape[0], c_out))
    if V != volume(ndim, K):
        raise OracleError(1)
    out = np.empty((c.shape[0], c_in), dtype=np.float64)
    st = _load().oracle_conv_bwd_data(_ptr(c), c.shape[0], _ptr(o), o.shape[0], ndim, K, stride, _ptr(_dims(dims)),
                                      _ptr(g), _ptr(w), c_in, c_out, _ptr(out), threads)
    if st:
        raise OracleError(st)
    return out
