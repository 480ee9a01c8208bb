"""Maps built with SC_KMAP_TILE_TABLE: the fused layer reads its neighbour
indices from the tile-transposed table instead of nbr.  The results must not
change: the layer, its input gradient, regular / strided and transposed maps
against the CPU oracle at the parity tolerance, with every row order, and the
map's own products (nbr, lists) bit-exact as before."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TORCH_DT, assert_close, layer_inputs
from submanifold_sparse_convolution_hash_gb300 import ScError, scenes
from submanifold_sparse_convolution_hash_gb300 import binding as sc

pytestmark = pytest.mark.gpu

SCENES = {
    "uniform2d_dense": scenes.uniform_2d(21, (40, 40), 900),
    "lidar": scenes.lidar_scan(61, 3000, (160, 160, 41)),
    "indoor": scenes.indoor_scene(62, 4000, (48, 48, 32), extent=(8, 40), radius=(3, 10)),
    "batch": scenes.batch_of_scans(63, 3, 1200, (120, 120, 41)),
}

CASES = [
    # scene, K, c_in, c_out, dtype, relu
    ("lidar", 3, 32, 32, "f16", True),
    ("lidar", 3, 32, 64, "f16", False),
    ("indoor", 3, 64, 64, "bf16", True),
    ("batch", 3, 64, 128, "f16", False),
    ("batch", 3, 128, 256, "f16", True),   # two tiles per unit
    ("batch", 3, 256, 256, "bf16", False),
    ("indoor", 5, 128, 128, "bf16", False),
    ("uniform2d_dense", 5, 16, 48, "bf16", True),
    ("uniform2d_dense", 9, 16, 32, "f16", False),  # V = 81: 64-point map units
    ("lidar", 1, 32, 32, "f16", False),
]


def build(s, K, order=None, sort=None, half=False):
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, s.ndim, K, s.dims, order=order, sort=sort, half=half, tile_table=True)
    return h, m


@pytest.mark.parametrize("order,sort,half", [(False, False, False), (True, False, False), (False, True, False),
                                             (True, True, False), (True, True, True)])
@pytest.mark.parametrize("name,K,c_in,c_out,dtype,relu", CASES)
def test_layer_and_input_gradient_on_a_tile_table_map(name, K, c_in, c_out, dtype, relu, order, sort, half):
    s = SCENES[name]
    h, m = build(s, K, order=order, sort=sort, half=half)
    assert np.array_equal(m.nbr().cpu().numpy(), oracle.kmap(s.coords, s.ndim, K, s.dims))
    f, w, f64, w64 = layer_inputs(s, K, c_in, c_out, dtype, seed=17 + c_in + K)
    out = torch.full((s.n, c_out), float("nan"), dtype=f.dtype, device="cuda")
    sc.sc_subm_conv_fwd(m, f, w, out=out, relu=relu, variant="fused")
    torch.cuda.synchronize()
    ref = oracle.subm_conv(s.coords, f64, w64, s.ndim, K, s.dims, relu=relu)
    assert_close(out, ref, dtype, f"tile table {name} K={K} {c_in}->{c_out}")
    g = torch.from_numpy(scenes.features(5 + c_out, s.n, c_out)).to(f.dtype).cuda()
    gin = sc.sc_subm_conv_bwd_data(m, g, w, variant="fused")
    torch.cuda.synchronize()
    gref = oracle.subm_conv_bwd_data(s.coords, g.double().cpu().numpy(), w64, s.ndim, K, s.dims)
    assert_close(gin, gref, dtype, f"tile table input gradient {name} K={K}")
    m.check()


def test_the_no_allocation_layer_on_a_tile_table_map():
    s = SCENES["lidar"]
    h, m = build(s, 3, order=True, sort=True)
    f, w, f64, w64 = layer_inputs(s, 3, 32, 32, "f16", seed=3)
    out = torch.full((s.n, 32), float("nan"), dtype=f.dtype, device="cuda")
    sc.sc_subm_conv_fwd(m, f, w, out=out, variant="fused")
    out2 = torch.full_like(out, float("nan"))
    import ctypes
    st = sc.lib().sc_subm_conv_fwd_noalloc(m._h, ctypes.c_void_p(f.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                           ctypes.c_void_p(out2.data_ptr()), 32, 32, 1, 0,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out, out2)  # the same kernel on the same map and inputs
    assert_close(out, oracle.subm_conv(s.coords, f64, w64, 3, 3, s.dims), "f16", "noalloc, tile table")


@pytest.mark.parametrize("name,K,stride,c_in,c_out,dtype,sort", [
    ("lidar", 3, 2, 32, 64, "f16", None), ("indoor", 5, 2, 48, 32, "bf16", True),
    ("batch", 3, 2, 128, 256, "bf16", True), ("lidar", 3, 1, 32, 32, "f16", True),
])
def test_strided_and_transposed_maps_with_a_tile_table(name, K, stride, c_in, c_out, dtype, sort):
    s = SCENES[name]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    ho = sc.sc_hash_build_conv_out(h, s.ndim, K, stride, s.dims)
    m = sc.sc_kmap_build_conv(h, ho, s.ndim, K, stride, s.dims, order=True if sort else None, sort=sort,
                              tile_table=True)
    oc = ho.coords().cpu().numpy()
    V = K ** s.ndim
    dt = TORCH_DT[dtype]
    f = torch.from_numpy(scenes.features(7, s.n, c_in)).to(dt).cuda()
    W = torch.from_numpy(scenes.weights(8, V, c_in, c_out)).to(dt).cuda()
    out = torch.full((ho.n, c_out), float("nan"), dtype=dt, device="cuda")
    sc.sc_subm_conv_fwd(m, f, W, out=out, variant="fused")
    torch.cuda.synchronize()
    ref = oracle.sparse_conv(s.coords, oc, f.double().cpu().numpy(), W.double().cpu().numpy(), s.ndim, K, stride,
                             s.dims)
    assert_close(out, ref, dtype, f"strided tile table {name} K={K} s={stride}")
    mt = sc.sc_kmap_build_conv(h, ho, s.ndim, K, stride, s.dims, order=True if sort else None, sort=sort,
                               transpose=True, tile_table=True)
    g = torch.from_numpy(scenes.features(31, ho.n, c_out)).to(dt).cuda()
    gin = sc.sc_subm_conv_bwd_data(mt, g, W)
    torch.cuda.synchronize()
    gref = oracle.sparse_conv_bwd_data(s.coords, oc, g.double().cpu().numpy(), W.double().cpu().numpy(), s.ndim, K,
                                       stride, s.dims)
    assert_close(gin, gref, dtype, f"transposed tile table {name} K={K} s={stride}")
    m.check()
    mt.check()


def test_tile_table_arguments_and_empty_input():
    s = SCENES["indoor"]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    with pytest.raises(ScError) as e:  # V = 343 > 128
        sc.sc_kmap_build(h, 3, 7, s.dims, tile_table=True)
    assert e.value.code == 5
    with pytest.raises(ScError) as e:  # not with column splitting
        sc.sc_kmap_build(h, 3, 3, s.dims, split=True, tile_table=True)
    assert e.value.code == 5
    he = sc.sc_hash_build(torch.empty((0, 4), dtype=torch.int32, device="cuda"))
    me = sc.sc_kmap_build(he, 3, 3, (16, 16, 16), tile_table=True)
    out = sc.sc_subm_conv_fwd(me, torch.empty((0, 32), dtype=torch.float16, device="cuda"),
                              torch.zeros((27, 32, 32), dtype=torch.float16, device="cuda"), variant="fused")
    assert out.shape == (0, 32)
