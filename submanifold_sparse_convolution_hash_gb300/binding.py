"""Thin ctypes binding over libsc (include/sc.h), with the same names.

Argument marshalling only: torch tensors become device pointers, sizes and a
stream; every step of the layer runs in libsc's CUDA kernels.  There is no
CPU path: if libsc.so is missing, or a tensor is not on a CUDA device, the
calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsc.so")
_lib = None

SC_RELU = 0x1
SC_VARIANT_FUSED = 0x10
SC_VARIANT_WS = 0x20
SC_VARIANT_SIMT = 0x40
SC_VARIANT_SPLIT = 0x80
SC_KMAP_NO_SYNC = 0x100
SC_KMAP_ORDER = 0x200
SC_KMAP_NO_ORDER = 0x400
SC_KMAP_SORT = 0x800
SC_KMAP_NO_SORT = 0x1000
SC_KMAP_TRANSPOSE = 0x2000
SC_KMAP_HALF = 0x4000
SC_KMAP_SPLIT = 0x8000
SC_KMAP_TILE_TABLE = 0x10000
VARIANTS = {"fused": SC_VARIANT_FUSED, "ws": SC_VARIANT_WS, "simt": SC_VARIANT_SIMT, "split": SC_VARIANT_SPLIT}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
STATUS = {0: "SC_OK", 1: "SC_ERR_INVALID_ARG", 2: "SC_ERR_OUT_OF_RANGE", 3: "SC_ERR_DUPLICATE_COORD",
          4: "SC_ERR_TABLE_FULL", 5: "SC_ERR_UNSUPPORTED", 6: "SC_ERR_CUDA", 7: "SC_ERR_OOM",
          8: "SC_ERR_TIMEOUT"}


class ScError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libsc.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libsc.so is not built: run `python -m submanifold_sparse_convolution_hash_gb300.build`"
                               " or __graft_entry__.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, I32, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
        sig = {
            "sc_hash_build": ([P, I64, P, P, P], I32),
            "sc_hash_query": ([P, P, I64, P, P], I32),
            "sc_hash_info": ([P, P, P], I32),
            "sc_hash_check": ([P, P], I32),
            "sc_hash_destroy": ([P, P], I32),
            "sc_hash_build_conv_out": ([P, I32, I32, I32, P, P, P, P], I32),
            "sc_hash_coords": ([P, P, P], I32),
            "sc_kmap_build_conv": ([P, P, I32, I32, I32, P, U, P, P, P], I32),
            "sc_kmap_build": ([P, I32, I32, P, U, P, P, P], I32),
            "sc_kmap_view": ([P, P, P, P, P, P], I32),
            "sc_kmap_info": ([P, P, P, P, P], I32),
            "sc_kmap_check": ([P, P], I32),
            "sc_kmap_export": ([P, P, P, P, P, P], I32),
            "sc_kmap_destroy": ([P, P], I32),
            "sc_subm_conv_fwd": ([P, P, P, P, I32, I32, I32, U, P], I32),
            "sc_subm_conv_bwd_data": ([P, P, P, P, I32, I32, I32, U, P], I32),
            "sc_subm_conv_bwd_weight": ([P, P, P, P, I32, I32, I32, U, P], I32),
            "sc_subm_conv_tune": ([P, P, P, P, I32, I32, I32, U, I32, P, P], I32),
            "sc_subm_conv_fwd_noalloc": ([P, P, P, P, I32, I32, I32, U, P], I32),
            "sc_set_allocator": ([P, P, P], I32),
            "sc_status_str": ([I32], ctypes.c_char_p),
            "sc_last_error": ([], ctypes.c_char_p),
            "sc_launch_count": ([], I64),
            "sc_profile_enable": ([I32], None),
            "sc_profile_only": ([ctypes.c_char_p], None),
            "sc_profile_collect": ([], I32),
            "sc_profile_reset": ([], None),
            "sc_profile_get": ([I32, P, P, P], I32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def exported_symbols() -> list:
    return [n for n in ("sc_hash_build", "sc_hash_query", "sc_hash_info", "sc_hash_check", "sc_hash_destroy",
                        "sc_hash_build_conv_out", "sc_hash_coords", "sc_kmap_build_conv",
                        "sc_kmap_build", "sc_kmap_info", "sc_kmap_check", "sc_kmap_export", "sc_kmap_view",
                        "sc_kmap_destroy",
                        "sc_subm_conv_fwd", "sc_subm_conv_tune", "sc_subm_conv_fwd_noalloc",
                        "sc_subm_conv_bwd_data", "sc_subm_conv_bwd_weight", "sc_set_allocator",
                        "sc_status_str", "sc_last_error",
                        "sc_launch_count", "sc_profile_enable", "sc_profile_only", "sc_profile_collect",
                        "sc_profile_reset",
                        "sc_profile_get")]


def _check(st: int, what: str):
    if st != 0:
        raise ScError(st, f"{what}: {lib().sc_last_error().decode()}")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


class Hash:
    """Handle of a coordinate hash table built by sc_hash_build."""

    def __init__(self, handle, n: int, capacity: int, device):
        self._h = handle
        self.n = n
        self.capacity = capacity
        self.device = device

    def query(self, coords: torch.Tensor, stream=None) -> torch.Tensor:
        """Row id of each (batch, x, y, z) query, -1 when absent (sc_hash_query)."""
        q = _dev(coords, "coords")
        rows = torch.empty(q.shape[0], dtype=torch.int32, device=q.device)
        _check(lib().sc_hash_query(self._h, _ptr(q), q.shape[0], _ptr(rows), _stream(stream)), "sc_hash_query")
        return rows

    def check(self, stream=None):
        _check(lib().sc_hash_check(self._h, _stream(stream)), "sc_hash_check")

    def coords(self, stream=None) -> torch.Tensor:
        """int32 [n, 4] (batch, x, y, z) of every row (sc_hash_coords)."""
        out = torch.empty((self.n, 4), dtype=torch.int32, device=self.device)
        _check(lib().sc_hash_coords(self._h, _ptr(out), _stream(stream)), "sc_hash_coords")
        return out

    def destroy(self, stream=None):
        if self._h:
            lib().sc_hash_destroy(self._h, _stream(stream))
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class KernelMap:
    """Handle of a kernel map built by sc_kmap_build."""

    def __init__(self, handle, n: int, ndim: int, K: int, dims, device, n_in: int | None = None,
                 stride: int = 1):
        self._h = handle
        self.n = n
        self.n_in = n if n_in is None else n_in
        self.stride = stride
        self.identity = n_in is None  # submanifold: the centre list is the identity
        self.ndim = ndim
        self.K = K
        self.volume = K ** ndim
        self.dims = tuple(dims)
        self.device = device

    def map_size(self, stream=None) -> int:
        """|M|, centre tuples included (sc_kmap_info)."""
        m = ctypes.c_int64(0)
        _check(lib().sc_kmap_info(self._h, None, None, ctypes.byref(m), _stream(stream)), "sc_kmap_info")
        return m.value

    def check(self, stream=None):
        _check(lib().sc_kmap_check(self._h, _stream(stream)), "sc_kmap_check")

    def nbr(self, stream=None) -> torch.Tensor:
        out = torch.empty((self.n, self.volume), dtype=torch.int32, device=self.device)
        _check(lib().sc_kmap_export(self._h, _ptr(out), None, None, None, _stream(stream)), "sc_kmap_export")
        return out

    def offsets(self, stream=None) -> torch.Tensor:
        out = torch.empty(self.volume + 1, dtype=torch.int64, device=self.device)
        _check(lib().sc_kmap_export(self._h, None, _ptr(out), None, None, _stream(stream)), "sc_kmap_export")
        return out

    def lists(self, stream=None):
        """(offs [V+1], in_rows [L], out_rows [L]): the per-offset lists (a
        submanifold map's centre segment is empty, its tuples implicit)."""
        offs = self.offsets(stream)
        L = self.map_size(stream) - (self.n if self.identity else 0)
        i = torch.empty(max(L, 0), dtype=torch.int32, device=self.device)
        o = torch.empty(max(L, 0), dtype=torch.int32, device=self.device)
        _check(lib().sc_kmap_export(self._h, None, None, _ptr(i) if L else None, _ptr(o) if L else None,
                                    _stream(stream)), "sc_kmap_export")
        return offs, i, o

    def view(self):
        """Borrowed, zero-copy device tensors of the products (sc_kmap_view):
        {"nbr": int32 [n, V], "offs": int64 [V+1], "in": int32 [L], "out":
        int32 [L], "map_size": |M|}.  They alias memory the handle owns: valid
        while this map is alive (each tensor keeps a reference to it), and not
        to be written."""
        nbr, offs, i, o = (ctypes.c_void_p() for _ in range(4))
        ms = ctypes.c_int64()
        _check(lib().sc_kmap_view(self._h, ctypes.byref(nbr), ctypes.byref(offs), ctypes.byref(i), ctypes.byref(o),
                                  ctypes.byref(ms)), "sc_kmap_view")
        L = ms.value - (self.n if self.identity else 0)

        def wrap(ptr, shape, typestr):
            n_el = 1
            for d in shape:
                n_el *= d
            if n_el == 0 or not ptr.value:
                return torch.empty(shape, dtype=torch.int64 if typestr == "<i8" else torch.int32, device=self.device)
            owner = self

            class _Borrowed:
                # torch takes only writable interfaces; the memory is read-only by contract
                __cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr.value, False),
                                            "version": 3, "strides": None}
                keep = owner  # the map outlives the tensor's view of it
            return torch.as_tensor(_Borrowed(), device=self.device)

        return {"nbr": wrap(nbr, (self.n, self.volume), "<i4"), "offs": wrap(offs, (self.volume + 1,), "<i8"),
                "in": wrap(i, (max(L, 0),), "<i4"), "out": wrap(o, (max(L, 0),), "<i4"), "map_size": ms.value}

    def destroy(self, stream=None):
        if self._h:
            lib().sc_kmap_destroy(self._h, _stream(stream))
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def sc_hash_build(coords: torch.Tensor, stream=None, allocator=None) -> Hash:
    """Hash table over int32 coords [N, 4] = (batch, x, y, z) on a CUDA device."""
    c = _dev(coords, "coords")
    if c.dtype != torch.int32 or c.dim() != 2 or c.shape[1] != 4:
        raise ValueError("coords must be int32 [N, 4]")
    h = ctypes.c_void_p()
    _check(lib().sc_hash_build(_ptr(c), c.shape[0], _alloc_arg(allocator), _stream(stream), ctypes.byref(h)),
           "sc_hash_build")
    n = ctypes.c_int64()
    cap = ctypes.c_int64()
    lib().sc_hash_info(h, ctypes.byref(n), ctypes.byref(cap))
    return Hash(h, n.value, cap.value, c.device)


def sc_kmap_build(h: Hash, ndim: int, K: int, dims, sync: bool = True, order: bool | None = None,
                  sort: bool | None = None, half: bool = False, split: bool = False, stream=None,
                  allocator=None, tile_table: bool = False) -> KernelMap:
    """Kernel map of a K^ndim submanifold convolution over the hashed points.

    order: True / False forces the locality order on / off; None leaves the
    library's default (on for n >= 262144).  sort: the same for the
    signature sort of the convolution's rows (default on for n >= 262144 when
    K^ndim <= 128).  half: build it by the half probe (mirror symmetry); the
    map is the same.  split: also compute the row orders of column splitting
    (K^ndim <= 32), which the "split" layer variant uses.  tile_table: also
    build the fused layer's tile-transposed index table (K^ndim <= 128),
    which pays when the map serves several layers."""
    d = (ctypes.c_int32 * 3)(*(list(dims) + [1] * (3 - len(dims))))
    m = ctypes.c_void_p()
    flags = 0 if sync else SC_KMAP_NO_SYNC
    if half:
        flags |= SC_KMAP_HALF
    if split:
        flags |= SC_KMAP_SPLIT
    if tile_table:
        flags |= SC_KMAP_TILE_TABLE
    if order is True:
        flags |= SC_KMAP_ORDER
    elif order is False:
        flags |= SC_KMAP_NO_ORDER
    if sort is True:
        flags |= SC_KMAP_SORT
    elif sort is False:
        flags |= SC_KMAP_NO_SORT
    _check(lib().sc_kmap_build(h._h, ndim, K, d, flags, _alloc_arg(allocator), _stream(stream), ctypes.byref(m)),
           "sc_kmap_build")
    return KernelMap(m, h.n, ndim, K, list(d), h.device)


def sc_hash_build_conv_out(h: Hash, ndim: int, K: int, stride: int, dims, stream=None, allocator=None) -> Hash:
    """Output set of a regular (stride 1: dilating) or strided layer over the
    points of `h`: every o with an input at stride * o + d (synchronises)."""
    d = (ctypes.c_int32 * 3)(*(list(dims) + [1] * (3 - len(dims))))
    o = ctypes.c_void_p()
    _check(lib().sc_hash_build_conv_out(h._h, ndim, K, stride, d, _alloc_arg(allocator), _stream(stream),
                                        ctypes.byref(o)),
           "sc_hash_build_conv_out")
    n = ctypes.c_int64()
    cap = ctypes.c_int64()
    lib().sc_hash_info(o, ctypes.byref(n), ctypes.byref(cap))
    return Hash(o, n.value, cap.value, h.device)


def sc_kmap_build_conv(h_in: Hash, h_out: Hash, ndim: int, K: int, stride: int, dims, sync: bool = True,
                       order: bool | None = None, sort: bool | None = None, transpose: bool = False, stream=None,
                       allocator=None, tile_table: bool = False) -> KernelMap:
    """Kernel map of a regular / strided layer: rows = the points of `h_out`,
    neighbours = rows of `h_in` at stride * o + d.  transpose: the transposed
    map (rows = the points of `h_in`, neighbours = the outputs whose windows
    hold them, at the mirrored offset), which sc_subm_conv_bwd_data takes.
    tile_table: as for sc_kmap_build."""
    d = (ctypes.c_int32 * 3)(*(list(dims) + [1] * (3 - len(dims))))
    m = ctypes.c_void_p()
    flags = 0 if sync else SC_KMAP_NO_SYNC
    if transpose:
        flags |= SC_KMAP_TRANSPOSE
    if tile_table:
        flags |= SC_KMAP_TILE_TABLE
    if order is True:
        flags |= SC_KMAP_ORDER
    elif order is False:
        flags |= SC_KMAP_NO_ORDER
    if sort is True:
        flags |= SC_KMAP_SORT
    elif sort is False:
        flags |= SC_KMAP_NO_SORT
    _check(lib().sc_kmap_build_conv(h_in._h, h_out._h, ndim, K, stride, d, flags, _alloc_arg(allocator),
                                    _stream(stream), ctypes.byref(m)),
           "sc_kmap_build_conv")
    if transpose:
        return KernelMap(m, h_in.n, ndim, K, list(d), h_in.device, n_in=h_out.n, stride=stride)
    return KernelMap(m, h_out.n, ndim, K, list(d), h_in.device, n_in=h_in.n, stride=stride)


def _conv_args(kmap, feats, W, out):
    f = _dev(feats, "feats")
    w = _dev(W, "W")
    if f.dtype not in _DTYPES or w.dtype != f.dtype:
        raise ValueError("feats and W must share one dtype: float32, float16 or bfloat16")
    if (w.dim() != 3 or w.shape[0] != kmap.volume or f.dim() != 2 or f.shape[1] != w.shape[1]
            or f.shape[0] != kmap.n_in):
        raise ValueError("shapes must be feats [N_in, C_in], W [K^ndim, C_in, C_out]")
    c_out = w.shape[2]
    if out is None:
        out = torch.empty((kmap.n, c_out), dtype=f.dtype, device=f.device)
    else:
        _dev(out, "out")
        if out.dtype != f.dtype or tuple(out.shape) != (kmap.n, c_out):
            raise ValueError("out must be [N, C_out] of the feats dtype")
    return f, w, out, f.shape[1], c_out, _DTYPES[f.dtype]


def sc_subm_conv_fwd(kmap: KernelMap, feats: torch.Tensor, W: torch.Tensor, out: torch.Tensor | None = None,
                     relu: bool = False, variant: str | None = None, stream=None) -> torch.Tensor:
    """out[q] = act(sum over map tuples (p, q, d) of feats[p] @ W[d]).  feats has
    the map's input rows (kmap.n_in), out its rows (kmap.n): the same for a
    submanifold map, the output set's for a regular / strided one."""
    f, w, out, c_in, c_out, dt = _conv_args(kmap, feats, W, out)
    flags = (SC_RELU if relu else 0) | (VARIANTS[variant] if variant else 0)
    _check(lib().sc_subm_conv_fwd(kmap._h, _ptr(f), _ptr(w), _ptr(out), c_in, c_out, dt, flags,
                                  _stream(stream)), "sc_subm_conv_fwd")
    return out


def sc_subm_conv_bwd_data(kmap: KernelMap, gout: torch.Tensor, W: torch.Tensor, gin: torch.Tensor | None = None,
                          variant: str | None = None, stream=None) -> torch.Tensor:
    """Gradient of a (ReLU-free) layer's loss with respect to its input
    features: gin[p] = sum over map tuples (p, q, d) of gout[q] @ W[d]^T.
    kmap: the layer's submanifold map, or the transposed map of a regular /
    strided layer (sc_kmap_build_conv(..., transpose=True)): gout has
    kmap.n_in rows (the layer's outputs), gin kmap.n (its inputs)."""
    g = _dev(gout, "gout")
    w = _dev(W, "W")
    if g.dtype not in _DTYPES or w.dtype != g.dtype:
        raise ValueError("gout and W must share one dtype: float32, float16 or bfloat16")
    if (w.dim() != 3 or w.shape[0] != kmap.volume or g.dim() != 2 or g.shape[1] != w.shape[2]
            or g.shape[0] != kmap.n_in):
        raise ValueError("shapes must be gout [N_out, C_out], W [K^ndim, C_in, C_out] (a submanifold map: "
                         "N_out = N; a transposed map: N_out = the layer's output count)")
    c_in, c_out = w.shape[1], w.shape[2]
    if gin is None:
        gin = torch.empty((kmap.n, c_in), dtype=g.dtype, device=g.device)
    elif gin.dtype != g.dtype or tuple(gin.shape) != (kmap.n, c_in):
        raise ValueError("gin must be [N, C_in] of the gout dtype")
    _check(lib().sc_subm_conv_bwd_data(kmap._h, _ptr(g), _ptr(w), _ptr(_dev(gin, "gin")), c_in, c_out,
                                       _DTYPES[g.dtype], VARIANTS[variant] if variant else 0, _stream(stream)),
           "sc_subm_conv_bwd_data")
    return gin


def sc_subm_conv_bwd_weight(kmap: KernelMap, feats: torch.Tensor, gout: torch.Tensor, dW: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Gradient with respect to the weights: dW[d] = sum over map tuples
    (p, q, d) of feats[p]^T gout[q]."""
    f = _dev(feats, "feats")
    g = _dev(gout, "gout")
    if f.dtype not in _DTYPES or g.dtype != f.dtype:
        raise ValueError("feats and gout must share one dtype: float32, float16 or bfloat16")
    if f.dim() != 2 or g.dim() != 2 or f.shape[0] != kmap.n_in or g.shape[0] != kmap.n:
        raise ValueError("shapes must be feats [N_in, C_in], gout [N, C_out]")
    c_in, c_out = f.shape[1], g.shape[1]
    if dW is None:
        dW = torch.empty((kmap.volume, c_in, c_out), dtype=f.dtype, device=f.device)
    elif dW.dtype != f.dtype or tuple(dW.shape) != (kmap.volume, c_in, c_out):
        raise ValueError("dW must be [K^ndim, C_in, C_out] of the feats dtype")
    _check(lib().sc_subm_conv_bwd_weight(kmap._h, _ptr(f), _ptr(g), _ptr(_dev(dW, "dW")), c_in, c_out,
                                         _DTYPES[f.dtype], 0, _stream(stream)), "sc_subm_conv_bwd_weight")
    return dW


def sc_subm_conv_tune(kmap: KernelMap, feats: torch.Tensor, W: torch.Tensor, out: torch.Tensor | None = None,
                      relu: bool = False, reps: int = 3, stream=None) -> str:
    """Times the variants on this map, caches the fastest, returns its name."""
    f, w, out, c_in, c_out, dt = _conv_args(kmap, feats, W, out)
    chosen = ctypes.c_uint(0)
    _check(lib().sc_subm_conv_tune(kmap._h, _ptr(f), _ptr(w), _ptr(out), c_in, c_out, dt,
                                   SC_RELU if relu else 0, reps, _stream(stream), ctypes.byref(chosen)),
           "sc_subm_conv_tune")
    return VARIANT_NAMES[chosen.value]


_ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
_FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)
_torch_allocator = None  # the callbacks stay alive: buffers they made are freed through them


class Allocator(ctypes.Structure):
    """sc_allocator: a caller's device allocator for one build call."""
    _fields_ = [("alloc", ctypes.c_void_p), ("free", ctypes.c_void_p), ("ctx", ctypes.c_void_p)]


def _alloc_arg(allocator):
    return ctypes.byref(allocator) if allocator is not None else None


def torch_allocator() -> Allocator:
    """An sc_allocator over PyTorch's caching allocator, for the allocator
    argument of the build calls (the callbacks live as long as the module)."""
    _torch_callbacks()
    return Allocator(ctypes.cast(_torch_allocator[0], ctypes.c_void_p).value,
                     ctypes.cast(_torch_allocator[1], ctypes.c_void_p).value, None)


def _torch_callbacks():
    global _torch_allocator
    if _torch_allocator is None:
        def _alloc(nbytes, stream, ctx):
            try:
                return torch.cuda.caching_allocator_alloc(int(nbytes), stream=int(stream or 0))
            except Exception:
                return None

        def _free(ptr, stream, ctx):
            torch.cuda.caching_allocator_delete(int(ptr))

        _torch_allocator = (_ALLOC_FN(_alloc), _FREE_FN(_free))
    return _torch_allocator


def use_torch_allocator(on: bool = True):
    """Route the library's device memory through PyTorch's caching allocator
    (on) or back to CUDA's stream-ordered pool (off) (sc_set_allocator)."""
    if not on:
        _check(lib().sc_set_allocator(None, None, None), "sc_set_allocator")
        return
    _torch_callbacks()
    a = ctypes.cast(_torch_allocator[0], ctypes.c_void_p)
    f = ctypes.cast(_torch_allocator[1], ctypes.c_void_p)
    _check(lib().sc_set_allocator(a, f, None), "sc_set_allocator")


def launch_count() -> int:
    return int(lib().sc_launch_count())


def profile_enable(on: bool = True):
    lib().sc_profile_enable(1 if on else 0)


def profile_only(name_prefix: str | None = None):
    """Time only kernels whose profile name starts with `name_prefix`."""
    lib().sc_profile_only(name_prefix.encode() if name_prefix else None)


def profile_reset():
    lib().sc_profile_reset()


def profile_collect() -> dict:
    """{kernel name: (launches, total ms)} accumulated since the last reset."""
    L = lib()
    _check(L.sc_profile_collect(), "sc_profile_collect")
    out = {}
    i = 0
    name = ctypes.c_char_p()
    n = ctypes.c_int64()
    ms = ctypes.c_double()
    while L.sc_profile_get(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms)) == 0:
        out[name.value.decode()] = (n.value, ms.value)
        i += 1
    return out
