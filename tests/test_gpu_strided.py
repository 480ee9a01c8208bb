"""GPU parity of regular (stride 1: dilating) and strided layers against the
CPU oracle.

The output set must equal the oracle's as a set of coordinates (bit-exact).
The GPU numbers its output rows in table order, so the map and the features
are checked against the oracle evaluated on the GPU's own output coordinates:
the neighbour table element by element, the per-offset lists as pair sets,
and the features within max|gpu - ref| <= 5e-3 * max(1, max|ref|) (f16 /
bf16 with fp32 accumulation) or 1e-5 * max(1, max|ref|) (fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TORCH_DT, assert_close, gpu_lists_by_offset
from submanifold_sparse_convolution_hash_gb300 import binding as sc
from submanifold_sparse_convolution_hash_gb300 import scenes

pytestmark = pytest.mark.gpu

SC = {
    "lidar": scenes.lidar_scan(51, 3000, (160, 160, 41)),
    "indoor": scenes.indoor_scene(52, 4000, (48, 48, 32), extent=(8, 40), radius=(3, 10)),
    "batch": scenes.batch_of_scans(53, 3, 1200, (120, 120, 41)),
    "uniform2d": scenes.uniform_2d(1001, (64, 64), 200),
}


def build(s, K, stride, order=None, sort=None):
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    ho = sc.sc_hash_build_conv_out(h, s.ndim, K, stride, s.dims)
    m = sc.sc_kmap_build_conv(h, ho, s.ndim, K, stride, s.dims, order=order, sort=sort)
    return h, ho, m


def sort_rows(c):
    c = np.asarray(c)
    return c[np.lexsort((c[:, 3], c[:, 2], c[:, 1], c[:, 0]))] if len(c) else c.reshape(0, 4)


GEOM = [("lidar", 3, 1), ("lidar", 3, 2), ("indoor", 3, 2), ("indoor", 5, 2), ("indoor", 3, 3),
        ("batch", 3, 2), ("batch", 1, 2), ("uniform2d", 3, 1), ("uniform2d", 3, 2), ("uniform2d", 5, 3)]


@pytest.mark.parametrize("order", [False, True])
@pytest.mark.parametrize("name,K,stride", GEOM)
def test_output_set_and_map_match_oracle(name, K, stride, order):
    s = SC[name]
    h, ho, m = build(s, K, stride, order=order)
    oc = ho.coords().cpu().numpy()
    ref_set = oracle.conv_out_coords(s.coords, s.ndim, K, stride, s.dims)
    assert ho.n == len(ref_set)
    assert np.array_equal(sort_rows(oc), ref_set), "output set differs from the oracle"
    # the GPU's table agrees with its own coordinate list
    assert np.array_equal(ho.query(torch.from_numpy(oc).cuda()).cpu().numpy(), np.arange(ho.n))
    nbr_ref = oracle.conv_kmap(s.coords, oc, s.ndim, K, stride, s.dims)
    assert np.array_equal(m.nbr().cpu().numpy(), nbr_ref), "neighbour table differs from the oracle"
    lists, offs = gpu_lists_by_offset(m)
    assert m.map_size() == int((nbr_ref >= 0).sum()) == int(offs[-1])
    for v, (pi, qi) in enumerate(lists):
        q = np.nonzero(nbr_ref[:, v] >= 0)[0]
        want = set(zip(nbr_ref[q, v].tolist(), q.tolist()))
        assert set(zip(pi.tolist(), qi.tolist())) == want, f"offset {v} list differs"
    m.check()


CONV = [
    # scene, K, stride, c_in, c_out, dtype, variant
    ("lidar", 3, 1, 32, 32, "f16", "fused"),
    ("lidar", 3, 2, 32, 64, "f16", "fused"),
    ("indoor", 3, 2, 64, 64, "bf16", "fused"),
    ("indoor", 5, 2, 48, 32, "bf16", "fused"),
    ("batch", 3, 2, 64, 128, "f16", "fused"),
    ("batch", 3, 3, 128, 256, "bf16", "fused"),
    ("batch", 1, 2, 32, 32, "f16", "fused"),
    ("uniform2d", 3, 2, 16, 16, "f32", "simt"),
    ("uniform2d", 3, 1, 16, 32, "f16", "simt"),
    ("lidar", 3, 2, 16, 16, "f32", None),
]


@pytest.mark.parametrize("relu,sort", [(False, None), (True, None), (False, True), (True, True)])
@pytest.mark.parametrize("name,K,stride,c_in,c_out,dtype,variant", CONV)
def test_conv_matches_oracle(name, K, stride, c_in, c_out, dtype, variant, relu, sort):
    """sort: the layer on a map whose output rows are signature-sorted."""
    s = SC[name]
    h, ho, m = build(s, K, stride, order=True if sort else None, sort=sort)
    oc = ho.coords().cpu().numpy()
    V = K ** s.ndim
    f = scenes.features(7 + stride, s.n, c_in)
    W = scenes.weights(8 + K, V, c_in, c_out, std=1.0 if dtype == "f32" else None)
    dt = TORCH_DT[dtype]
    ft, wt = torch.from_numpy(f).to(dt).cuda(), torch.from_numpy(W).to(dt).cuda()
    out = torch.full((ho.n, c_out), float("nan"), dtype=dt, device="cuda")
    sc.sc_subm_conv_fwd(m, ft, wt, out=out, relu=relu, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.sparse_conv(s.coords, oc, ft.double().cpu().numpy(), wt.double().cpu().numpy(), s.ndim, K, stride,
                             s.dims, relu=relu)
    assert_close(out, ref, dtype, f"{name} K={K} s={stride} {c_in}->{c_out} {dtype} {variant}")


@pytest.mark.parametrize("name,K,stride,c_in,c_out,dtype", [
    ("lidar", 3, 2, 32, 32, "f16"), ("indoor", 3, 1, 64, 64, "bf16"), ("batch", 3, 2, 128, 64, "f16"),
    ("uniform2d", 3, 2, 16, 16, "f32"),
])
def test_weight_gradient_matches_oracle(name, K, stride, c_in, c_out, dtype):
    s = SC[name]
    h, ho, m = build(s, K, stride)
    oc = ho.coords().cpu().numpy()
    dt = TORCH_DT[dtype]
    f = torch.from_numpy(scenes.features(21, s.n, c_in)).to(dt).cuda()
    g = torch.from_numpy(scenes.features(22, ho.n, c_out)).to(dt).cuda()
    dW = sc.sc_subm_conv_bwd_weight(m, f, g)
    torch.cuda.synchronize()
    ref = oracle.sparse_conv_bwd_weight(s.coords, oc, f.double().cpu().numpy(), g.double().cpu().numpy(), s.ndim, K,
                                        stride, s.dims)
    scale = max(1.0, float(np.abs(ref).max()))
    err = float(np.abs(dW.double().cpu().numpy() - ref).max())
    assert err <= (1e-5 if dtype == "f32" else 5e-3) * scale, f"{name}: {err}"


def test_regular_then_submanifold_chain():
    """A dilating layer's output set feeds a submanifold layer as its input."""
    s = SC["indoor"]
    h, ho, m = build(s, 3, 1)
    oc = ho.coords().cpu().numpy()
    f = torch.from_numpy(scenes.features(3, s.n, 32)).half().cuda()
    W1 = torch.from_numpy(scenes.weights(4, 27, 32, 64)).half().cuda()
    W2 = torch.from_numpy(scenes.weights(5, 27, 64, 32)).half().cuda()
    y = sc.sc_subm_conv_fwd(m, f, W1, relu=True)
    m2 = sc.sc_kmap_build(ho, 3, 3, s.dims)
    z = sc.sc_subm_conv_fwd(m2, y, W2)
    torch.cuda.synchronize()
    ref1 = oracle.sparse_conv(s.coords, oc, f.double().cpu().numpy(), W1.double().cpu().numpy(), 3, 3, 1, s.dims,
                              relu=True)
    assert_close(y, ref1, "f16", "dilating layer")
    ref2 = oracle.subm_conv(oc, y.double().cpu().numpy(), W2.double().cpu().numpy(), 3, 3, s.dims)
    assert_close(z, ref2, "f16", "submanifold layer on the dilated set")


def test_unsupported_paths_and_empty_input():
    s = SC["lidar"]
    h, ho, m = build(s, 3, 2)
    W = torch.zeros((27, 32, 32), dtype=torch.float16, device="cuda")
    # the input gradient needs the transposed map; the forward map is refused
    g = torch.zeros((m.n_in, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(sc.ScError) as e:
        sc.sc_subm_conv_bwd_data(m, g, W)
    assert e.value.code == 5
    f = torch.zeros((s.n, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(sc.ScError) as e:
        sc.sc_subm_conv_fwd(m, f, W, variant="ws")
    assert e.value.code == 5
    with pytest.raises(ValueError):
        sc.sc_subm_conv_fwd(m, f[:10], W)  # feats must have the input's rows
    # empty input: empty output set, empty map, empty layer
    h0 = sc.sc_hash_build(torch.zeros((0, 4), dtype=torch.int32, device="cuda"))
    o0 = sc.sc_hash_build_conv_out(h0, 3, 3, 2, (8, 8, 8))
    assert o0.n == 0 and o0.coords().shape == (0, 4)
    m0 = sc.sc_kmap_build_conv(h0, o0, 3, 3, 2, (8, 8, 8))
    assert m0.map_size() == 0
    out = sc.sc_subm_conv_fwd(m0, torch.zeros((0, 16), dtype=torch.float16, device="cuda"),
                              torch.zeros((27, 16, 16), dtype=torch.float16, device="cuda"))
    assert out.shape == (0, 16)


@pytest.mark.parametrize("sort", [None, True])
def test_full_size_strided_layer_on_lidar_scan(sort):
    """The LiDAR workload (1440 x 1440 x 41, ~100k voxels) through a stride-2
    3x3x3 layer, C 32 -> 64 f16: the output set in full, the map in full, the
    features on sampled output rows (sort: with the signature-sorted rows)."""
    w, s = scenes.workload(1)
    h, ho, m = build(s, 3, 2, order=True if sort else None, sort=sort)
    oc = ho.coords().cpu().numpy()
    assert np.array_equal(sort_rows(oc), oracle.conv_out_coords(s.coords, 3, 3, 2, s.dims))
    nbr_ref = oracle.conv_kmap(s.coords, oc, 3, 3, 2, s.dims)
    assert np.array_equal(m.nbr().cpu().numpy(), nbr_ref)
    f = torch.from_numpy(scenes.features(w.seed, s.n, 32)).half().cuda()
    W = torch.from_numpy(scenes.weights(w.seed, 27, 32, 64)).half().cuda()
    out = sc.sc_subm_conv_fwd(m, f, W)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.linspace(0, ho.n - 1, 2048).astype(np.int64),
                                     np.arange(max(0, ho.n - 200), ho.n)]))
    ref = oracle.sparse_conv(s.coords, oc[rows], f.double().cpu().numpy(), W.double().cpu().numpy(), 3, 3, 2, s.dims)
    assert_close(out[torch.from_numpy(rows).cuda()], ref, "f16", "full-size strided layer")


@pytest.mark.parametrize("name,K,stride,c_in,c_out,dtype,order", [
    ("lidar", 3, 2, 32, 32, "f16", False), ("lidar", 3, 1, 32, 64, "f16", True),
    ("indoor", 3, 2, 64, 64, "bf16", True), ("indoor", 5, 2, 32, 48, "bf16", False),
    ("indoor", 3, 3, 64, 32, "f16", False), ("batch", 3, 2, 128, 256, "bf16", False),
    ("batch", 1, 2, 32, 32, "f16", False), ("uniform2d", 3, 2, 16, 16, "f32", False),
    ("uniform2d", 5, 3, 16, 32, "f16", False),
])
def test_transposed_map_and_input_gradient(name, K, stride, c_in, c_out, dtype, order):
    """The transposed map holds, for each input p, the outputs whose windows
    contain it at the mirrored offset; the input gradient runs on it (with the
    row order, also on signature-sorted rows)."""
    s = SC[name]
    h, ho, m = build(s, K, stride)
    mt = sc.sc_kmap_build_conv(h, ho, s.ndim, K, stride, s.dims, order=order, sort=True if order else None,
                               transpose=True)
    assert mt.n == s.n and mt.n_in == ho.n
    oc = ho.coords().cpu().numpy()
    V = K ** s.ndim
    fwd = oracle.conv_kmap(s.coords, oc, s.ndim, K, stride, s.dims)
    want = np.full((s.n, V), -1, dtype=np.int32)
    q, v = np.nonzero(fwd >= 0)
    want[fwd[q, v], V - 1 - v] = q  # a relabelling of the forward tuples
    assert np.array_equal(mt.nbr().cpu().numpy(), want), "transposed neighbour table differs"
    assert mt.map_size() == m.map_size()
    dt = TORCH_DT[dtype]
    g = torch.from_numpy(scenes.features(31, ho.n, c_out)).to(dt).cuda()
    W = torch.from_numpy(scenes.weights(32, V, c_in, c_out, std=1.0 if dtype == "f32" else None)).to(dt).cuda()
    gin = sc.sc_subm_conv_bwd_data(mt, g, W)
    torch.cuda.synchronize()
    ref = oracle.sparse_conv_bwd_data(s.coords, oc, g.double().cpu().numpy(), W.double().cpu().numpy(), s.ndim, K,
                                      stride, s.dims)
    assert_close(gin, ref, dtype, f"{name} K={K} s={stride} input gradient")
    mt.check()
