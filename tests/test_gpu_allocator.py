"""The caller's allocator (sc_set_allocator): with PyTorch's caching
allocator plugged in, the library's handles and temporaries come from
torch's pool, results still match the oracle, and buffers made by one
allocator go back to it after the setting changes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close
from submanifold_sparse_convolution_hash_gb300 import binding as sc
from submanifold_sparse_convolution_hash_gb300 import scenes

pytestmark = pytest.mark.gpu


def _allocs():
    torch.cuda.synchronize()
    return torch.cuda.memory_stats().get("allocation.all.allocated", 0)


def test_torch_allocator_serves_the_library():
    s = scenes.lidar_scan(61, 3000, (160, 160, 41))
    coords = torch.from_numpy(s.coords).cuda()
    f = torch.from_numpy(scenes.features(62, s.n, 32)).half().cuda()
    W = torch.from_numpy(scenes.weights(63, 27, 32, 32)).half().cuda()
    out = torch.empty((s.n, 32), dtype=torch.float16, device="cuda")
    sc.use_torch_allocator(True)
    try:
        before = _allocs()
        h = sc.sc_hash_build(coords)
        m = sc.sc_kmap_build(h, 3, 3, s.dims)
        sc.sc_subm_conv_fwd(m, f, W, out=out, variant="fused")  # reads W's slices by TMA: no temporary
        ws = sc.sc_subm_conv_fwd(m, f, W, variant="ws")          # packed weights + fp32 accumulator
        dW = sc.sc_subm_conv_bwd_weight(m, f, out)
        after = _allocs()
        # hash arena, map arena, the temporaries of the weight-stationary call
        # and the weight gradient (torch allocations made by the test itself:
        # ws and dW outputs)
        assert after - before >= 2 + 3 + 2
    finally:
        sc.use_torch_allocator(False)
    assert np.array_equal(m.nbr().cpu().numpy(), oracle.kmap(s.coords, 3, 3, s.dims))
    ref = oracle.subm_conv(s.coords, f.double().cpu().numpy(), W.double().cpu().numpy(), 3, 3, s.dims)
    assert_close(out, ref, "f16", "fused, torch allocator")
    assert_close(ws, ref, "f16", "weight-stationary, torch allocator")
    ref_dw = oracle.subm_conv_bwd_weight(s.coords, f.double().cpu().numpy(), out.double().cpu().numpy(), 3, 3,
                                         s.dims)
    assert float(np.abs(dW.double().cpu().numpy() - ref_dw).max()) <= 5e-3 * max(1.0, float(np.abs(ref_dw).max()))
    # the handles were made by torch's allocator and go back to it although
    # the default pool is set again
    m.destroy()
    h.destroy()
    torch.cuda.synchronize()
    # the default pool serves the next build
    h2 = sc.sc_hash_build(coords)
    m2 = sc.sc_kmap_build(h2, 3, 3, s.dims)
    assert np.array_equal(m2.nbr().cpu().numpy(), oracle.kmap(s.coords, 3, 3, s.dims))


def test_allocator_arguments():
    with pytest.raises(sc.ScError) as e:
        sc._check(sc.lib().sc_set_allocator(sc.ctypes.c_void_p(1), None, None), "sc_set_allocator")
    assert e.value.code == 1
    sc.use_torch_allocator(False)


def test_allocator_argument_of_a_build_call():
    """A build call given an sc_allocator takes the handle's memory from it
    (here PyTorch's caching allocator), whatever the process-wide setting;
    the map's later buffers (sc_kmap_view) come from it too."""
    s = scenes.lidar_scan(64, 3000, (160, 160, 41))
    coords = torch.from_numpy(s.coords).cuda()
    sc.use_torch_allocator(False)  # process-wide: the stream-ordered pool
    alloc = sc.torch_allocator()
    before = _allocs()
    h = sc.sc_hash_build(coords, allocator=alloc)
    m = sc.sc_kmap_build(h, 3, 3, s.dims, order=True, allocator=alloc)
    after_build = _allocs()
    assert after_build - before >= 2  # the hash arena and the map arena
    v = m.view()  # materialises the exported forms from the same allocator
    assert _allocs() - after_build >= 1
    assert np.array_equal(v["nbr"].cpu().numpy(), oracle.kmap(s.coords, 3, 3, s.dims))
    # a build without the argument leaves torch's pool alone
    mid = _allocs()
    h2 = sc.sc_hash_build(coords)
    m2 = sc.sc_kmap_build(h2, 3, 3, s.dims)
    assert _allocs() == mid
    del v
    m.destroy()
    h.destroy()
    m2.destroy()
    h2.destroy()
    torch.cuda.synchronize()
