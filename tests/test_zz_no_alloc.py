"""The no-allocation convolution entry point, sc_subm_conv_fwd_noalloc.

Some callers cannot allocate device memory when they run a layer: programs
that plan all device memory up front, runtimes that own every allocation,
or latency-critical code that cannot accept an allocation that may block or
fail.  This entry point serves them: its packed weights live in a fixed
4 MiB device array inside the library.  These checks call it through the C
ABI and compare it with sc_subm_conv_fwd (fused variant) on two calls in a
row, within the parity tolerance used everywhere else:
max|a - b| <= 5e-3 * max(1, max|b|).

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from submanifold_sparse_convolution_hash_gb300 import binding as sc
from submanifold_sparse_convolution_hash_gb300 import scenes

pytestmark = pytest.mark.gpu

_DT = {torch.float16: 1, torch.bfloat16: 2}


def _noalloc(kmap, f, W, out, relu=False):
    """Direct C-ABI call; returns the status code."""
    L = sc.lib()
    return L.sc_subm_conv_fwd_noalloc(kmap._h, ctypes.c_void_p(f.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), f.shape[1], W.shape[2], _DT[f.dtype],
                                      sc.SC_RELU if relu else 0,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max()), 5e-3 * max(1.0, float(np.abs(b).max()))


def test_noalloc_matches_fused_on_two_calls_in_a_row():
    s = scenes.lidar_scan(91, 3000, (160, 160, 41))
    c = torch.from_numpy(s.coords).cuda()
    h = sc.sc_hash_build(c)
    m = sc.sc_kmap_build(h, 3, 3, s.dims)
    cases = [(32, 64, torch.float16, False), (64, 32, torch.bfloat16, True)]
    for i, (c_in, c_out, dt, relu) in enumerate(cases):
        f = torch.from_numpy(scenes.features(200 + i, s.n, c_in)).to(dt).cuda()
        W = torch.from_numpy(scenes.weights(300 + i, 27, c_in, c_out)).to(dt).cuda()
        ref = sc.sc_subm_conv_fwd(m, f, W, relu=relu, variant="fused")
        out = torch.full((s.n, c_out), float("nan"), dtype=dt, device="cuda")
        st = _noalloc(m, f, W, out, relu)
        assert st == 0, sc.lib().sc_last_error()
        torch.cuda.synchronize()
        err, bound = _close(out, ref)
        assert err <= bound, f"call {i}: {err} > {bound}"


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
