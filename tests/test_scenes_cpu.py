"""Seeded scene generators: determinism, uniqueness, ranges, sizes."""
import numpy as np

from submanifold_sparse_convolution_hash_gb300 import scenes


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    r = scenes.SplitMix64.__new__(scenes.SplitMix64)
    r.state = 0
    got = [int(v) for v in r.u64(3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_is_uniform_enough():
    u = scenes.SplitMix64(5).uniform(200000)
    assert 0 <= u.min() and u.max() < 1
    assert abs(u.mean() - 0.5) < 0.005
    z = scenes.SplitMix64(6).normal(200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def _check_scene(s, n_lo, n_hi):
    c = s.coords
    assert c.dtype == np.int32 and c.shape[1] == 4
    assert n_lo <= s.n <= n_hi
    assert len(np.unique(c, axis=0)) == s.n
    for a in range(3):
        assert c[:, 1 + a].min() >= 0 and c[:, 1 + a].max() < s.dims[a]


def test_scenes_deterministic_and_valid():
    a = scenes.lidar_scan(3, 5000, (200, 200, 41))
    b = scenes.lidar_scan(3, 5000, (200, 200, 41))
    np.testing.assert_array_equal(a.coords, b.coords)
    _check_scene(a, 4000, 6000)
    c = scenes.indoor_scene(4, 20000, (96, 96, 48))
    _check_scene(c, 20000, 40000)
    d = scenes.batch_of_scans(5, 3, 2000, (120, 120, 41))
    assert set(np.unique(d.coords[:, 0])) == {0, 1, 2}
    _check_scene(d, 4500, 7500)
    e = scenes.uniform_2d(1000, (64, 64), 200)
    _check_scene(e, 200, 200)
    assert (e.coords[:, 3] == 0).all()
    # rows come out in a random order, not sorted
    assert not (np.diff(a.coords[:, 1]) >= 0).all()


def test_workload_sizes_match_the_five_configs():
    w0, s0 = scenes.workload(0)
    assert s0.n == 200 and w0.K == 3 and w0.channels == (16, 16) and w0.dtype == "f32"
    w1, s1 = scenes.workload(1)
    assert 90_000 <= s1.n <= 110_000 and s1.dims == (1440, 1440, 41) and w1.channels == (32, 32)
    w3, _ = scenes.workload(3, scale=0.05)
    assert w3.channels == (32, 32, 64, 64, 128, 128, 256, 256, 256)


def test_features_and_weights():
    f = scenes.features(1, 100, 32)
    assert f.shape == (100, 32) and f.dtype == np.float32
    w = scenes.weights(1, 27, 32, 64)
    assert w.shape == (27, 32, 64)
    assert abs(w.std() * np.sqrt(27 * 32) - 1) < 0.05
    np.testing.assert_array_equal(f, scenes.features(1, 100, 32))


def test_threaded_feature_draw_equals_one_serial_pass():
    """Features are drawn in 2^22-value chunks on threads; each chunk starts
    at the counter a serial pass reaches there."""
    n, c = 70_000, 64  # two chunks, the second one short
    f = scenes.features(5, n, c)
    rng = scenes.SplitMix64(5, 10)
    parts = []
    for s in range(0, n * c, 1 << 22):
        parts.append(rng.normal(min(1 << 22, n * c - s)).astype(np.float32))
    np.testing.assert_array_equal(f.reshape(-1), np.concatenate(parts))
