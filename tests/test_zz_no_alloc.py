"""The no-allocation convolution entry point, sc_subm_conv_fwd_noalloc.

Some callers cannot allocate device memory when they run a layer: programs
that plan all device memory up front, runtimes that own every allocation,
or latency-critical code that cannot accept an allocation that may block or
fail.  This entry point serves them: its packed weights live in a fixed
4 MiB device array inside the library.

These checks call it through the C ABI and compare its output element by
element with the CPU oracle's fp64 layer, within the parity tolerance used
everywhere else, max|gpu - ref| <= 5e-3 * max(1, max|ref|), on two calls in
a row (the array keeps the previous call's contents).  With PyTorch's
caching allocator plugged in as the library's allocator, a call must not
allocate through it.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close
from submanifold_sparse_convolution_hash_gb300 import binding as sc
from submanifold_sparse_convolution_hash_gb300 import scenes

pytestmark = pytest.mark.gpu

_DT = {torch.float16: 1, torch.bfloat16: 2}
_NAME = {torch.float16: "f16", torch.bfloat16: "bf16"}


def _noalloc(kmap, f, W, out, relu=False):
    """Direct C-ABI call; returns the status code."""
    L = sc.lib()
    return L.sc_subm_conv_fwd_noalloc(kmap._h, ctypes.c_void_p(f.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), f.shape[1], W.shape[2], _DT[f.dtype],
                                      sc.SC_RELU if relu else 0,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs(n, V, c_in, c_out, dt, seed):
    f = torch.from_numpy(scenes.features(seed, n, c_in)).to(dt)
    W = torch.from_numpy(scenes.weights(seed + 1, V, c_in, c_out)).to(dt)
    return f.cuda(), W.cuda(), f.double().numpy(), W.double().numpy()


def _allocs():
    torch.cuda.synchronize()
    return torch.cuda.memory_stats().get("allocation.all.allocated", 0)


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row():
    s = scenes.lidar_scan(91, 3000, (160, 160, 41))
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, 3, 3, s.dims)
    cases = [(32, 64, torch.float16, False), (64, 32, torch.bfloat16, True)]
    for i, (c_in, c_out, dt, relu) in enumerate(cases):
        f, W, f64, W64 = _inputs(s.n, 27, c_in, c_out, dt, 200 + 2 * i)
        ref = oracle.subm_conv(s.coords, f64, W64, 3, 3, s.dims, relu=relu)
        out = torch.full((s.n, c_out), float("nan"), dtype=dt, device="cuda")
        assert _noalloc(m, f, W, out, relu) == 0, sc.lib().sc_last_error()
        torch.cuda.synchronize()
        assert_close(out, ref, _NAME[dt], f"call {i}")


def test_noalloc_at_the_largest_kernel_that_fits_the_buffer():
    """5x5x5 with C_in = C_out = 128: 125 * 128 * 128 * 2 = 4,096,000 bytes,
    just under the 4 MiB bound; two calls with different weights."""
    s = scenes.indoor_scene(93, 2500, (48, 48, 24), extent=(8, 30), radius=(3, 8))
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, 3, 5, s.dims)
    for call in range(2):
        f, W, f64, W64 = _inputs(s.n, 125, 128, 128, torch.bfloat16, 400 + 2 * call)
        ref = oracle.subm_conv(s.coords, f64, W64, 3, 5, s.dims)
        out = torch.full((s.n, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(m, f, W, out) == 0, sc.lib().sc_last_error()
        torch.cuda.synchronize()
        assert_close(out, ref, "bf16", f"5x5x5 call {call}")


def test_noalloc_on_a_strided_map():
    s = scenes.lidar_scan(94, 3000, (160, 160, 41))
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    ho = sc.sc_hash_build_conv_out(h, 3, 3, 2, s.dims)
    m = sc.sc_kmap_build_conv(h, ho, 3, 3, 2, s.dims)
    oc = ho.coords().cpu().numpy()
    f, W, f64, W64 = _inputs(s.n, 27, 32, 32, torch.float16, 500)
    ref = oracle.sparse_conv(s.coords, oc, f64, W64, 3, 3, 2, s.dims)
    out = torch.full((ho.n, 32), float("nan"), dtype=torch.float16, device="cuda")
    assert _noalloc(m, f, W, out) == 0, sc.lib().sc_last_error()
    torch.cuda.synchronize()
    assert_close(out, ref, "f16", "stride 2")


def test_noalloc_allocates_nothing():
    """With the library's allocator set to PyTorch's caching allocator, any
    library allocation would show in torch's allocation counter; the
    no-allocation call leaves it unchanged (the weight-stationary call, which
    allocates its packed weights and fp32 sums, moves it)."""
    s = scenes.lidar_scan(95, 3000, (160, 160, 41))
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, 3, 3, s.dims)
    f, W, f64, W64 = _inputs(s.n, 27, 32, 32, torch.float16, 600)
    out = torch.empty((s.n, 32), dtype=torch.float16, device="cuda")
    out2 = torch.empty_like(out)
    assert _noalloc(m, f, W, out) == 0, sc.lib().sc_last_error()  # first call on the device: set-up
    sc.use_torch_allocator(True)
    try:
        before = _allocs()
        for _ in range(3):
            assert _noalloc(m, f, W, out) == 0, sc.lib().sc_last_error()
        assert _allocs() == before
        sc.sc_subm_conv_fwd(m, f, W, out=out2, variant="ws")
        assert _allocs() > before
    finally:
        sc.use_torch_allocator(False)
    assert_close(out, oracle.subm_conv(s.coords, f64, W64, 3, 3, s.dims), "f16", "after the allocation check")


def test_noalloc_empty_input():
    h = sc.sc_hash_build(torch.empty((0, 4), dtype=torch.int32, device="cuda"))
    m = sc.sc_kmap_build(h, 3, 3, (16, 16, 16))
    f = torch.empty((0, 32), dtype=torch.float16, device="cuda")
    W = torch.zeros((27, 32, 32), dtype=torch.float16, device="cuda")
    out = torch.empty((0, 32), dtype=torch.float16, device="cuda")
    assert _noalloc(m, f, W, out) == 0, sc.lib().sc_last_error()
    torch.cuda.synchronize()


def test_noalloc_rejects_weights_beyond_the_fixed_buffer():
    s = scenes.indoor_scene(92, 2000, (40, 40, 24), extent=(8, 30), radius=(3, 8))
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, 3, 5, s.dims)  # V = 125
    # 125 * 256 * 256 * 2 bytes = 16 MB > 4 MiB
    f = torch.zeros((s.n, 256), dtype=torch.float16, device="cuda")
    W = torch.zeros((125, 256, 256), dtype=torch.float16, device="cuda")
    out = torch.empty((s.n, 256), dtype=torch.float16, device="cuda")
    assert _noalloc(m, f, W, out) == 5  # SC_ERR_UNSUPPORTED
    assert b"4 MiB" in sc.lib().sc_last_error()
    # 125 * 128 * 144 * 2 = 4,608,000 bytes: one step past the bound
    f = torch.zeros((s.n, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((125, 128, 144), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((s.n, 144), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(m, f, W, out) == 5
