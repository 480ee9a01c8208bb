"""GPU parity: hash table, kernel map and convolution against the CPU oracle.

Sizes here finish in the oracle within seconds and still span several
128-row tiles plus a ragged tail.  Maps must match bit for bit; features
within max|gpu - ref| <= 5e-3 * max(1, max|ref|) (f16/bf16 inputs, fp32
accumulation) or 1e-5 * max(1, max|ref|) (fp32).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, gpu_lists_by_offset, layer_inputs
from submanifold_sparse_convolution_hash_gb300 import ScError, scenes
from submanifold_sparse_convolution_hash_gb300 import binding as sc

pytestmark = pytest.mark.gpu


def small_scenes():
    return {
        "uniform2d": scenes.uniform_2d(1000, (64, 64), 200),
        "uniform2d_dense": scenes.uniform_2d(21, (40, 40), 900),
        "lidar": scenes.lidar_scan(31, 3000, (160, 160, 41)),
        "indoor": scenes.indoor_scene(32, 4000, (48, 48, 32), extent=(8, 40), radius=(3, 10)),
        "batch": scenes.batch_of_scans(33, 3, 1200, (120, 120, 41)),
    }


SCENES = small_scenes()


def build(scene, K, sync=True, order=None, sort=None, half=False):
    c = torch.from_numpy(scene.coords).cuda()
    h = sc.sc_hash_build(c)
    m = sc.sc_kmap_build(h, scene.ndim, K, scene.dims, sync=sync, order=order, sort=sort, half=half)
    return c, h, m


# ------------------------------------------------------------------ hash --

def test_hash_query_finds_every_row_and_misses_absent_keys():
    s = SCENES["lidar"]
    c, h, m = build(s, 3)
    rows = h.query(c).cpu().numpy()
    np.testing.assert_array_equal(rows, np.arange(s.n))
    # shifted coordinates: present iff the shifted point is in the set
    q = s.coords.copy()
    q[:, 3] += 1
    present = {tuple(r) for r in s.coords.tolist()}
    index = {tuple(r): i for i, r in enumerate(s.coords.tolist())}
    want = np.array([index.get(tuple(r), -1) for r in q.tolist()])
    np.testing.assert_array_equal(h.query(torch.from_numpy(q).cuda()).cpu().numpy(), want)
    assert (want >= 0).any() and (want < 0).any()
    # other batch, out-of-field values
    q2 = np.array([[1, 10, 10, 10], [-1, 0, 0, 0], [0, 65535, 0, 0], [0, -3, 1, 1]], dtype=np.int32)
    np.testing.assert_array_equal(h.query(torch.from_numpy(q2).cuda()).cpu().numpy(), [-1, -1, -1, -1])
    assert len(present) == s.n
    assert h.capacity >= s.n and (h.capacity & (h.capacity - 1)) == 0


# ------------------------------------------------------------------- map --

@pytest.mark.parametrize("name,K", [("uniform2d", 3), ("uniform2d_dense", 5), ("uniform2d_dense", 9), ("lidar", 3),
                                    ("indoor", 3), ("indoor", 5), ("batch", 3), ("lidar", 1), ("indoor", 7)])
@pytest.mark.parametrize("sync,order,sort", [(True, False, False), (False, False, False), (True, True, False),
                                             (False, True, False), (True, False, True), (False, True, True)])
@pytest.mark.parametrize("half", [False, True])
def test_kmap_bit_exact(name, K, sync, order, sort, half):
    """half: the half-probe build (mirror symmetry, "Sparse inputs and sparse
    convolution", section "A symmetry you can check") must give the same map."""
    s = SCENES[name]
    c, h, m = build(s, K, sync, order, sort, half)
    if not sync:
        m.check()
    ref = oracle.kmap(s.coords, s.ndim, K, s.dims)
    nbr = m.nbr().cpu().numpy()
    np.testing.assert_array_equal(nbr, ref)
    lists, offs = gpu_lists_by_offset(m)
    ref_lists = oracle.offset_lists(ref)
    centre = (K ** s.ndim - 1) // 2
    for v, ((gi, go), (ri, ro)) in enumerate(zip(lists, ref_lists)):
        if v == centre:
            assert len(gi) == 0  # the identity is implied, not listed
            np.testing.assert_array_equal(ri, np.arange(s.n))
            continue
        # the order inside a segment is unspecified: compare as sets
        k = np.lexsort((gi, go))
        np.testing.assert_array_equal(go[k], ro)
        np.testing.assert_array_equal(gi[k], ri)
    assert m.map_size() == len(oracle.tuples(ref))
    assert offs[-1] == m.map_size() - s.n


@pytest.mark.parametrize("n", [1, 100, 50_000])
def test_isolated_points_one_per_block(n):
    """Every point in its own 2x2x2 block (even coordinates, no two in one
    block): the table holds n occupied blocks, its design maximum, and the
    map of isolated points has only centre tuples."""
    rng = scenes.SplitMix64(77, 1)
    cells = np.unique(rng.integers(0, 2048 * 2048 * 32, 2 * n))[:n]
    rng.permutation(len(cells))
    x, rest = np.divmod(cells, 2048 * 32)
    y, z = np.divmod(rest, 32)
    coords = np.stack([np.zeros_like(x), 2 * x, 2 * y, 2 * z], axis=1).astype(np.int32)[:n]
    c = torch.from_numpy(coords).cuda()
    h = sc.sc_hash_build(c)
    np.testing.assert_array_equal(h.query(c).cpu().numpy(), np.arange(len(coords)))
    m = sc.sc_kmap_build(h, 3, 3, (4096, 4096, 64))
    assert m.map_size() == len(coords)
    ref = oracle.kmap(coords, 3, 3, (4096, 4096, 64))
    np.testing.assert_array_equal(m.nbr().cpu().numpy(), ref)


@pytest.mark.parametrize("order", [False, True])
def test_kmap_is_deterministic(order):
    """The neighbour table and segment sizes repeat exactly; each segment
    holds the same pairs (the order inside a segment is unspecified)."""
    s = SCENES["lidar"]
    _, _, m1 = build(s, 3, order=order)
    _, _, m2 = build(s, 3, order=order)
    assert torch.equal(m1.nbr(), m2.nbr())
    (o1, i1, q1), (o2, i2, q2) = m1.lists(), m2.lists()
    assert torch.equal(o1, o2)
    for v in range(len(o1) - 1):
        a, b = int(o1[v]), int(o1[v + 1])
        assert sorted(zip(q1[a:b].tolist(), i1[a:b].tolist())) == sorted(zip(q2[a:b].tolist(), i2[a:b].tolist()))


def test_five_point_worked_example_on_gpu():
    coords = np.array([[0, 1, 1, 0], [0, 2, 2, 0], [0, 2, 4, 0], [0, 3, 2, 0], [0, 4, 3, 0]], dtype=np.int32)
    h = sc.sc_hash_build(torch.from_numpy(coords).cuda())
    m = sc.sc_kmap_build(h, 2, 3, (5, 5, 1))
    assert m.map_size() == 11
    offs = m.offsets().cpu().numpy()
    counts = np.diff(offs)
    counts[4] = 5  # centre: the identity over the five points
    oi = lambda d: oracle.offset_index(d, 3)
    assert counts[oi((-1, -1))] == 2 and counts[oi((-1, 0))] == 1 and counts[oi((0, 0))] == 5
    assert counts[oi((1, 0))] == 1 and counts[oi((1, 1))] == 2 and int((counts > 0).sum()) == 5


# -------------------------------------------------------------- features --

CONV_CASES = [
    # scene, K, c_in, c_out, dtype, relu, variant
    ("lidar", 3, 32, 32, "f16", False, "fused"),
    ("lidar", 3, 32, 32, "f16", True, "ws"),
    ("indoor", 3, 64, 64, "bf16", False, "fused"),
    ("indoor", 3, 64, 64, "bf16", True, "ws"),
    ("batch", 3, 32, 64, "f16", True, "fused"),
    ("batch", 3, 64, 128, "f16", False, "fused"),
    ("batch", 3, 128, 256, "f16", True, "fused"),
    ("batch", 3, 256, 256, "f16", False, "fused"),
    ("batch", 3, 256, 256, "f16", False, "ws"),
    ("indoor", 5, 128, 128, "bf16", False, "fused"),
    ("indoor", 5, 128, 128, "bf16", False, "ws"),
    ("uniform2d", 3, 16, 16, "f16", False, "fused"),
    ("uniform2d_dense", 5, 16, 48, "bf16", True, "fused"),
    ("uniform2d_dense", 5, 48, 16, "bf16", True, "ws"),
    ("uniform2d_dense", 7, 32, 32, "bf16", False, "fused"),  # 2D with V = 49 > 32: direction signature
    ("uniform2d_dense", 9, 16, 32, "f16", False, "fused"),   # V = 81: 64-point map-build units
    ("indoor", 5, 64, 32, "f16", True, "fused"),
    ("lidar", 1, 32, 32, "f16", False, "fused"),
    ("lidar", 1, 32, 32, "f16", False, "ws"),
    ("indoor", 7, 32, 32, "bf16", False, None),  # V = 343: auto picks weight-stationary
    ("lidar", 3, 32, 32, "f16", False, "simt"),
    ("uniform2d", 3, 16, 16, "f32", False, None),
    ("uniform2d", 3, 16, 16, "f32", True, "simt"),
    ("lidar", 3, 32, 16, "f32", False, None),
]


@pytest.mark.parametrize("order,sort", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("name,K,c_in,c_out,dtype,relu,variant", CONV_CASES)
def test_conv_matches_oracle(name, K, c_in, c_out, dtype, relu, variant, order, sort):
    s = SCENES[name]
    c, h, m = build(s, K, order=order, sort=sort)
    f, w, f64, w64 = layer_inputs(s, K, c_in, c_out, dtype, seed=7 + c_in + K,
                                  w_std=1.0 if dtype == "f32" else None)
    out = sc.sc_subm_conv_fwd(m, f, w, relu=relu, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.subm_conv(s.coords, f64, w64, s.ndim, K, s.dims, relu=relu)
    assert_close(out, ref, dtype, f"{name} K={K} {c_in}->{c_out} {dtype} {variant}")
    m.check()


HALF_CASES = [
    ("lidar", 3, 32, 32, "f16", False),
    ("indoor", 3, 64, 64, "bf16", True),
    ("batch", 3, 64, 128, "f16", False),
    ("indoor", 5, 128, 128, "bf16", False),
    ("uniform2d_dense", 5, 16, 48, "bf16", True),
    ("uniform2d_dense", 9, 16, 32, "f16", False),
]


@pytest.mark.parametrize("order,sort", [(False, False), (True, True)])
@pytest.mark.parametrize("name,K,c_in,c_out,dtype,relu", HALF_CASES)
def test_conv_on_half_probe_map(name, K, c_in, c_out, dtype, relu, order, sort):
    """The layer on a map built by the half probe (its tile and row masks are
    derived from the finished table)."""
    s = SCENES[name]
    c, h, m = build(s, K, order=order, sort=sort, half=True)
    f, w, f64, w64 = layer_inputs(s, K, c_in, c_out, dtype, seed=9 + c_in + K)
    for variant in ("fused", "ws"):
        out = sc.sc_subm_conv_fwd(m, f, w, relu=relu, variant=variant)
        torch.cuda.synchronize()
        ref = oracle.subm_conv(s.coords, f64, w64, s.ndim, K, s.dims, relu=relu)
        assert_close(out, ref, dtype, f"half probe {name} K={K} {variant}")
    m.check()


def test_half_probe_is_submanifold_only():
    s = SCENES["lidar"]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    ho = sc.sc_hash_build_conv_out(h, 3, 3, 2, s.dims)
    d = (ctypes.c_int32 * 3)(*s.dims)
    m = ctypes.c_void_p()
    st = sc.lib().sc_kmap_build_conv(h._h, ho._h, 3, 3, 2, d, sc.SC_KMAP_HALF, None, None, ctypes.byref(m))
    assert st == 5  # SC_ERR_UNSUPPORTED


def test_every_row_written_once_no_stale_values():
    """Output buffer pre-filled with NaN: every row must be overwritten."""
    s = SCENES["lidar"]
    c, h, m = build(s, 3)
    f, w, f64, w64 = layer_inputs(s, 3, 32, 32, "f16", seed=3)
    ref = oracle.subm_conv(s.coords, f64, w64, 3, 3, s.dims)
    for variant in ("fused", "ws", "simt"):
        out = torch.full((s.n, 32), float("nan"), dtype=torch.float16, device="cuda")
        sc.sc_subm_conv_fwd(m, f, w, out=out, variant=variant)
        assert_close(out, ref, "f16", variant)


def test_tune_picks_a_variant_and_result_matches():
    s = SCENES["indoor"]
    c, h, m = build(s, 3)
    f, w, f64, w64 = layer_inputs(s, 3, 64, 64, "bf16", seed=4)
    out = torch.empty((s.n, 64), dtype=torch.bfloat16, device="cuda")
    name = sc.sc_subm_conv_tune(m, f, w, out=out, reps=2)
    assert name in ("fused", "ws")
    ref = oracle.subm_conv(s.coords, f64, w64, 3, 3, s.dims)
    assert_close(out, ref, "bf16", "tuned")
    out2 = sc.sc_subm_conv_fwd(m, f, w)
    assert_close(out2, ref, "bf16", "after tune")


def test_map_reused_across_a_layer_stack():
    """One map, several layers, ReLU between them; each layer checked with
    the oracle fed the GPU's own input, and the stack end to end."""
    s = SCENES["batch"]
    c, h, m = build(s, 3)
    widths = [32, 32, 64, 64, 128]
    x = torch.from_numpy(scenes.features(11, s.n, widths[0])).half().cuda()
    x0 = x.double().cpu().numpy()
    Ws = [torch.from_numpy(scenes.weights(12 + i, 27, widths[i], widths[i + 1])).half().cuda()
          for i in range(len(widths) - 1)]
    for i, W in enumerate(Ws):
        relu = i + 1 < len(Ws)
        y = sc.sc_subm_conv_fwd(m, x, W, relu=relu)
        ref = oracle.subm_conv(s.coords, x.double().cpu().numpy(), W.double().cpu().numpy(), 3, 3, s.dims,
                               relu=relu)
        assert_close(y, ref, "f16", f"layer {i}")
        x = y
    ref_stack = oracle.subm_conv_stack(s.coords, x0, [W.double().cpu().numpy() for W in Ws], 3, 3, s.dims, "f16")
    assert_close(x, ref_stack[-1], "f16", "stack end to end")


# ------------------------------------------------------------ edge cases --

def test_empty_and_single_point():
    h = sc.sc_hash_build(torch.zeros((0, 4), dtype=torch.int32, device="cuda"))
    m = sc.sc_kmap_build(h, 3, 3, (8, 8, 8))
    assert m.map_size() == 0
    f = torch.zeros((0, 32), dtype=torch.float16, device="cuda")
    W = torch.randn((27, 32, 32), dtype=torch.float16, device="cuda")
    assert sc.sc_subm_conv_fwd(m, f, W).shape == (0, 32)
    one = torch.tensor([[0, 3, 3, 3]], dtype=torch.int32, device="cuda")
    m1 = sc.sc_kmap_build(sc.sc_hash_build(one), 3, 3, (8, 8, 8))
    assert m1.map_size() == 1
    f1 = torch.randn((1, 32), device="cuda").half()
    for v in ("fused", "ws", "simt"):
        out = sc.sc_subm_conv_fwd(m1, f1, W, variant=v)
        ref = f1.double().cpu().numpy() @ W[13].double().cpu().numpy()
        assert_close(out, ref, "f16", v)


@pytest.mark.parametrize("n", [127, 128, 129, 255, 257, 1000])
def test_ragged_tile_counts(n):
    s = scenes.uniform_2d(500 + n, (64, 64), n)
    c, h, m = build(s, 3)
    f, w, f64, w64 = layer_inputs(s, 3, 16, 32, "bf16", seed=n)
    ref = oracle.subm_conv(s.coords, f64, w64, 2, 3, s.dims)
    for v in ("fused", "ws"):
        assert_close(sc.sc_subm_conv_fwd(m, f, w, variant=v), ref, "bf16", f"n={n} {v}")


def test_error_reporting():
    dup = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32, device="cuda")
    h = sc.sc_hash_build(dup)
    with pytest.raises(ScError) as e:
        h.check()
    assert e.value.code == 3
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(h, 3, 3, (4, 4, 4))
    assert e.value.code == 3
    ok = torch.tensor([[0, 1, 1, 1], [0, 5, 2, 2]], dtype=torch.int32, device="cuda")
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(sc.sc_hash_build(ok), 3, 3, (4, 4, 4))  # x = 5 outside dims
    assert e.value.code == 2
    neg = torch.tensor([[0, -1, 1, 1]], dtype=torch.int32, device="cuda")
    with pytest.raises(ScError) as e:
        sc.sc_hash_build(neg).check()
    assert e.value.code == 2
    h2 = sc.sc_hash_build(torch.tensor([[0, 1, 1, 1]], dtype=torch.int32, device="cuda"))
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(h2, 3, 4, (4, 4, 4))
    assert e.value.code == 1
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(h2, 4, 3, (4, 4, 4))
    assert e.value.code == 1
    m = sc.sc_kmap_build(h2, 3, 3, (4, 4, 4))
    f = torch.zeros((1, 24), dtype=torch.float16, device="cuda")
    with pytest.raises(ScError) as e:
        sc.sc_subm_conv_fwd(m, f, torch.zeros((27, 24, 24), dtype=torch.float16, device="cuda"))
    assert e.value.code == 5
    with pytest.raises(ScError) as e:  # fp32 on the tensor-core kernel
        sc.sc_subm_conv_fwd(m, torch.zeros((1, 16), device="cuda"), torch.zeros((27, 16, 16), device="cuda"),
                            variant="fused")
    assert e.value.code == 5
    with pytest.raises(ValueError):
        sc.sc_hash_build(torch.zeros((4, 4), dtype=torch.int32))  # host tensor: no CPU path
    # the library is still usable after every error above
    assert sc.sc_kmap_build(sc.sc_hash_build(ok), 3, 3, (8, 8, 8)).map_size() == 2


def test_launch_count_and_profile():
    s = SCENES["lidar"]
    before = sc.launch_count()
    sc.profile_reset()
    sc.profile_enable(True)
    try:
        c, h, m = build(s, 3)
        f, w, _, _ = layer_inputs(s, 3, 32, 32, "f16", seed=1)
        sc.sc_subm_conv_fwd(m, f, w, variant="fused")
        prof = sc.profile_collect()
    finally:
        sc.profile_enable(False)
    launched = sc.launch_count() - before
    # insert, the single-pass map build, the fused conv (which reads the
    # weight slices from W by TMA: no pack)
    assert launched == 3
    for k in ("hash_insert", "kmap_build", "subm_conv_fused"):
        assert k in prof and prof[k][0] == 1 and prof[k][1] > 0
    assert "pack_weights" not in prof


def test_profile_only_brackets_the_named_kernels():
    s = SCENES["lidar"]
    sc.profile_reset()
    sc.profile_only("subm_conv")
    sc.profile_enable(True)
    try:
        c, h, m = build(s, 3)
        f, w, _, _ = layer_inputs(s, 3, 32, 32, "f16", seed=1)
        sc.sc_subm_conv_fwd(m, f, w, variant="fused")
        prof = sc.profile_collect()
    finally:
        sc.profile_enable(False)
        sc.profile_only(None)
    timed = {k for k, (launches, _) in prof.items() if launches}
    assert timed == {"subm_conv_fused"} and prof["subm_conv_fused"][0] == 1


@pytest.mark.parametrize("order", [False, True])
@pytest.mark.parametrize("K", [3, 5])
def test_coordinates_at_the_top_of_the_key_fields(K, order):
    """Points in the far corner of the largest grid (every axis 65535 wide,
    coordinates up to 65534) and at the largest batch id, next to points at
    the origin: the map bit-exact, the layer within the bar, and a stride-2
    layer's output set (extents 32768) exact."""
    rng = np.random.default_rng(K)
    dims = (65535, 65535, 65535)
    corner = np.stack(np.meshgrid(np.arange(65528, 65535), np.arange(65528, 65535), np.arange(65530, 65535),
                                  indexing="ij"), -1).reshape(-1, 3)
    corner = corner[rng.random(len(corner)) < 0.45]
    origin = np.stack(np.meshgrid(np.arange(0, 6), np.arange(0, 6), np.arange(0, 4), indexing="ij"), -1).reshape(-1, 3)
    origin = origin[rng.random(len(origin)) < 0.5]
    coords = np.concatenate([np.c_[np.full(len(corner), 65534), corner], np.c_[np.zeros(len(corner), int), corner],
                             np.c_[np.full(len(origin), 65534), origin], np.c_[np.zeros(len(origin), int), origin]])
    coords = coords[rng.permutation(len(coords))].astype(np.int32)
    c = torch.from_numpy(coords).cuda()
    h = sc.sc_hash_build(c)
    m = sc.sc_kmap_build(h, 3, K, dims, order=order)
    nbr_ref = oracle.kmap(coords, 3, K, dims)
    assert np.array_equal(m.nbr().cpu().numpy(), nbr_ref)
    V = K ** 3
    f = torch.from_numpy(scenes.features(K, len(coords), 32)).half().cuda()
    W = torch.from_numpy(scenes.weights(K + 1, V, 32, 32)).half().cuda()
    out = sc.sc_subm_conv_fwd(m, f, W)
    ref = oracle.subm_conv(coords, f.double().cpu().numpy(), W.double().cpu().numpy(), 3, K, dims)
    assert_close(out, ref, "f16", f"K={K} at the top of the key fields")
    ho = sc.sc_hash_build_conv_out(h, 3, K, 2, dims)
    oc = ho.coords().cpu().numpy()
    want = oracle.conv_out_coords(coords, 3, K, 2, dims)
    got = oc[np.lexsort((oc[:, 3], oc[:, 2], oc[:, 1], oc[:, 0]))]
    assert np.array_equal(got, want)
    assert int(oc[:, 1:].max()) <= 32767
    ms = sc.sc_kmap_build_conv(h, ho, 3, K, 2, dims, order=order)
    assert np.array_equal(ms.nbr().cpu().numpy(), oracle.conv_kmap(coords, oc, 3, K, 2, dims))
    m.check()
    ms.check()


def test_full_table_is_reported(monkeypatch):
    """A table forced too small (developer capacity override) makes the
    insert latch SC_ERR_TABLE_FULL after probing every entry; the map build
    reports it and the library stays usable.  Every probe loop is bounded by
    the table's size, so nothing waits."""
    rng = np.random.default_rng(4)
    pts = np.unique(rng.integers(0, 200, size=(400, 3)) * 2, axis=0)  # one point per 2x2x2 block
    coords = torch.from_numpy(np.c_[np.zeros(len(pts), int), pts].astype(np.int32)).cuda()
    monkeypatch.setenv("SC_DEV_HASH_CAPACITY", "16")
    h = sc.sc_hash_build(coords)
    monkeypatch.delenv("SC_DEV_HASH_CAPACITY")
    assert h.capacity == 16
    with pytest.raises(ScError) as e:
        h.check()
    assert e.value.code == 4
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(h, 3, 3, (400, 400, 400))
    assert e.value.code == 4
    h2 = sc.sc_hash_build(coords)
    assert h2.capacity >= 2 * len(pts)
    m2 = sc.sc_kmap_build(h2, 3, 3, (400, 400, 400))
    assert np.array_equal(m2.nbr().cpu().numpy(), oracle.kmap(coords.cpu().numpy(), 3, 3, (400, 400, 400)))


@pytest.mark.parametrize("name,K,order,half", [("lidar", 3, False, False), ("lidar", 3, True, False),
                                               ("indoor", 5, True, False), ("indoor", 3, True, True),
                                               ("uniform2d_dense", 5, False, True)])
def test_kmap_view_matches_oracle(name, K, order, half):
    """sc_kmap_view (borrowed device pointers, the rulebook grouped by
    offset): the neighbour table in input row order, equal to the oracle's,
    and the CSR lists, equal to the oracle's per-offset lists as pair sets;
    a second call returns the same pointers."""
    s = SCENES[name]
    c, h, m = build(s, K, sync=False, order=order, half=half)
    L = sc.lib()
    ptrs = [ctypes.c_void_p() for _ in range(4)]
    ms = ctypes.c_int64()
    assert L.sc_kmap_view(m._h, *(ctypes.byref(p) for p in ptrs), ctypes.byref(ms)) == 0, L.sc_last_error()
    again = [ctypes.c_void_p() for _ in range(4)]
    assert L.sc_kmap_view(m._h, *(ctypes.byref(p) for p in again), None) == 0
    assert [p.value for p in ptrs] == [p.value for p in again]
    v = m.view()
    ref = oracle.kmap(s.coords, s.ndim, K, s.dims)
    assert v["nbr"].data_ptr() == ptrs[0].value
    np.testing.assert_array_equal(v["nbr"].cpu().numpy(), ref)
    assert ms.value == v["map_size"] == len(oracle.tuples(ref))
    offs = v["offs"].cpu().numpy()
    gi, go = v["in"].cpu().numpy(), v["out"].cpu().numpy()
    centre = (K ** s.ndim - 1) // 2
    for off, ((ri, ro)) in enumerate(oracle.offset_lists(ref)):
        a, b = offs[off], offs[off + 1]
        if off == centre:
            assert a == b  # the identity is implied
            continue
        k = np.lexsort((gi[a:b], go[a:b]))
        np.testing.assert_array_equal(go[a:b][k], ro)
        np.testing.assert_array_equal(gi[a:b][k], ri)


SPLIT_CASES = [
    ("lidar", 3, 32, 32, "f16", False),
    ("indoor", 3, 64, 64, "bf16", True),
    ("batch", 3, 128, 256, "f16", True),
    ("batch", 3, 256, 256, "f16", False),
    ("uniform2d_dense", 5, 16, 48, "bf16", True),
]


@pytest.mark.parametrize("order", [False, True])
@pytest.mark.parametrize("name,K,c_in,c_out,dtype,relu", SPLIT_CASES)
def test_conv_with_column_splitting(name, K, c_in, c_out, dtype, relu, order):
    """Column splitting ("TorchSparse optimizations", section "TorchSparse++"):
    two launches over the two halves of the offset range, each in its own
    signature-sorted row order, fp32 partial sums between them.  The layer,
    its input gradient and the unsplit kernel on the same map all match the
    oracle."""
    s = SCENES[name]
    c, h, m = build(s, K, order=order, sort=True)
    hs = sc.sc_hash_build(c)
    ms = sc.sc_kmap_build(hs, s.ndim, K, s.dims, order=order, split=True)
    np.testing.assert_array_equal(ms.nbr().cpu().numpy(), m.nbr().cpu().numpy())
    f, w, f64, w64 = layer_inputs(s, K, c_in, c_out, dtype, seed=11 + c_in + K)
    ref = oracle.subm_conv(s.coords, f64, w64, s.ndim, K, s.dims, relu=relu)
    for variant in ("split", "fused"):
        out = torch.full((s.n, c_out), float("nan"), dtype=f.dtype, device="cuda")
        sc.sc_subm_conv_fwd(ms, f, w, out=out, relu=relu, variant=variant)
        torch.cuda.synchronize()
        assert_close(out, ref, dtype, f"column split {name} K={K} {c_in}->{c_out} {variant}")
    g = torch.from_numpy(scenes.features(77, s.n, c_out)).to(f.dtype).cuda()
    gin = sc.sc_subm_conv_bwd_data(ms, g, w, variant="split")
    torch.cuda.synchronize()
    ref_g = oracle.subm_conv_bwd_data(s.coords, g.double().cpu().numpy(), w64, s.ndim, K, s.dims)
    assert_close(gin, ref_g, dtype, f"column split input gradient {name}")
    ms.check()


def test_column_splitting_arguments():
    s = SCENES["indoor"]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    with pytest.raises(ScError) as e:  # V = 125 > 32
        sc.sc_kmap_build(h, 3, 5, s.dims, split=True)
    assert e.value.code == 5
    with pytest.raises(ScError) as e:
        sc.sc_kmap_build(h, 3, 3, s.dims, split=True, sort=False)
    assert e.value.code == 1
    m = sc.sc_kmap_build(h, 3, 3, s.dims)  # no split orders: the split variant is refused
    f = torch.zeros((s.n, 32), dtype=torch.float16, device="cuda")
    w = torch.zeros((27, 32, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(ScError) as e:
        sc.sc_subm_conv_fwd(m, f, w, variant="split")
    assert e.value.code == 5
