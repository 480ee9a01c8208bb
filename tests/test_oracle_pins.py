"""Pins for the CPU oracle, against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the pages'
worked examples (tests/golden/), brute force over all point pairs, and an fp64
dense convolution computed by torch.nn.functional on a dense grid.
"""
import itertools

import numpy as np
import pytest
import torch

from conftest import read_golden

import oracle
from submanifold_sparse_convolution_hash_gb300 import scenes


# ---------------------------------------------------------------------------
# helpers (independent of the oracle)
# ---------------------------------------------------------------------------

def grid_points(golden):
    pts = {}
    grid = None
    for row in golden:
        if row[0] == "grid":
            grid = (int(row[1]), int(row[2]))
        elif row[0] == "point":
            pts[row[1]] = (int(row[2]), int(row[3]))
    names = sorted(pts, key=lambda s: int(s[1:]))
    coords = np.array([[0, pts[n][0], pts[n][1], 0] for n in names], dtype=np.int32)
    return grid, names, coords


def dense_dilate(active, K):
    """Regular output definition on a grid: an output is active when any
    active input lies inside its KxK(xK) window, the window clipped to the
    grid (same padding)."""
    r = K // 2
    out = np.zeros_like(active)
    for idx in np.argwhere(active):
        sl = tuple(slice(max(i - r, 0), min(i + r + 1, s)) for i, s in zip(idx, active.shape))
        out[sl] = True
    return out


def brute_force_tuples(coords, ndim, K, dims):
    """All (offset, out, in) with c_in - c_out = d, |d|_inf <= r, same batch."""
    r = K // 2
    n = coords.shape[0]
    res = []
    for q in range(n):
        for p in range(n):
            if coords[p, 0] != coords[q, 0]:
                continue
            d = coords[p, 1:1 + ndim] - coords[q, 1:1 + ndim]
            if ndim == 2 and coords[p, 3] != coords[q, 3]:
                continue
            if np.all(np.abs(d) <= r):
                res.append((oracle.offset_index(d, K), q, p))
    res.sort()
    return np.array(res, dtype=np.int64).reshape(-1, 3)


def random_scene(seed, n, dims, ndim, batches=1):
    rng = scenes.SplitMix64(seed, 99)
    X, Y, Z = dims
    tot = X * Y * (Z if ndim == 3 else 1)
    pts = []
    for b in range(batches):
        cells = rng.permutation(tot)[:n]
        if ndim == 3:
            x, rem = cells // (Y * Z), cells % (Y * Z)
            y, z = rem // Z, rem % Z
        else:
            x, y, z = cells // Y, cells % Y, np.zeros_like(cells)
        pts.append(np.stack([np.full_like(x, b), x, y, z], axis=1))
    c = np.concatenate(pts).astype(np.int32)
    return c[rng.permutation(c.shape[0])]


def dense_conv_reference(coords, feats, W, ndim, K, dims):
    """fp64 dense convolution (torch, cross-correlation, zero padding) over the
    whole grid, read back at the active sites."""
    r = K // 2
    n, c_in = feats.shape
    c_out = W.shape[2]
    out = np.zeros((n, c_out))
    for b in np.unique(coords[:, 0]):
        sel = np.nonzero(coords[:, 0] == b)[0]
        if ndim == 3:
            grid = torch.zeros((1, c_in) + tuple(dims), dtype=torch.float64)
            c = torch.from_numpy(coords[sel].astype(np.int64))
            grid[0, :, c[:, 1], c[:, 2], c[:, 3]] = torch.from_numpy(feats[sel]).T
            w = torch.from_numpy(W).reshape(K, K, K, c_in, c_out).permute(4, 3, 0, 1, 2).contiguous()
            y = torch.nn.functional.conv3d(grid, w, padding=r)
            out[sel] = y[0, :, c[:, 1], c[:, 2], c[:, 3]].T.numpy()
        else:
            grid = torch.zeros((1, c_in, dims[0], dims[1]), dtype=torch.float64)
            c = torch.from_numpy(coords[sel].astype(np.int64))
            grid[0, :, c[:, 1], c[:, 2]] = torch.from_numpy(feats[sel]).T
            w = torch.from_numpy(W).reshape(K, K, c_in, c_out).permute(3, 2, 0, 1).contiguous()
            y = torch.nn.functional.conv2d(grid, w, padding=r)
            out[sel] = y[0, :, c[:, 1], c[:, 2]].T.numpy()
    return out


# ---------------------------------------------------------------------------
# the pages' worked examples
# ---------------------------------------------------------------------------

def test_five_point_map_matches_worked_example():
    g = read_golden("five_point_map.txt")
    grid, names, coords = grid_points(g)
    nbr = oracle.kmap(coords, 2, 3, (grid[0], grid[1], 1))
    got = {tuple(t) for t in oracle.tuples(nbr).tolist()}
    want = set()
    for row in g:
        if row[0] == "tuple":
            p, q = int(row[1][1:]), int(row[2][1:])
            want.add((oracle.offset_index((int(row[3]), int(row[4])), 3), q, p))
    assert got == want
    total = [int(r[1]) for r in g if r[0] == "total"][0]
    assert len(got) == total == 11
    counts = np.bincount(oracle.tuples(nbr)[:, 0], minlength=9)
    nonempty = [int(r[1]) for r in g if r[0] == "nonempty_offsets"][0]
    assert int((counts > 0).sum()) == nonempty == 5
    split = [r[1:] for r in g if r[0] == "rows_per_nonempty_offset"][0]
    for item in split:
        d, k = item.split(":")
        dx, dy = (int(v) for v in d.split(","))
        assert counts[oracle.offset_index((dx, dy), 3)] == int(k)
    # the isolated point P2 appears only in the centre group
    t = oracle.tuples(nbr)
    assert set(map(tuple, t[(t[:, 1] == 2) | (t[:, 2] == 2)].tolist())) == {(4, 2, 2)}


def test_five_point_update_rule_closed_form():
    """The weight-stationary equations printed under the gather/scatter figure
    (f1 += f0 W(-1,-1), f4 += f3 W(-1,-1)) are the W(-1,-1) part of the
    oracle's output; with W zero elsewhere they are the whole output."""
    g = read_golden("five_point_map.txt")
    grid, names, coords = grid_points(g)
    rng = np.random.default_rng(5)
    f = rng.standard_normal((5, 4))
    W = np.zeros((9, 4, 3))
    W[oracle.offset_index((-1, -1), 3)] = rng.standard_normal((4, 3))
    out = oracle.subm_conv(coords, f, W, 2, 3, (5, 5, 1))
    Wm = W[oracle.offset_index((-1, -1), 3)]
    want = np.zeros((5, 3))
    want[1] = f[0] @ Wm
    want[4] = f[3] @ Wm
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-14)
    # full weights: Q1 receives (P0, W(-1,-1)), (P1, W(0,0)), (P3, W(1,0))
    W = rng.standard_normal((9, 4, 3))
    out = oracle.subm_conv(coords, f, W, 2, 3, (5, 5, 1))
    oi = lambda d: oracle.offset_index(d, 3)
    want_q1 = f[0] @ W[oi((-1, -1))] + f[1] @ W[oi((0, 0))] + f[3] @ W[oi((1, 0))]
    np.testing.assert_allclose(out[1], want_q1, rtol=1e-13, atol=1e-13)


def test_sign_convention_quiz():
    g = read_golden("sign_quiz.txt")
    kv = {r[0]: r[1:] for r in g if r[0] in ("input", "offset", "output")}
    g5 = read_golden("five_point_map.txt")
    grid, names, coords = grid_points(g5)
    nbr = oracle.kmap(coords, 2, 3, (5, 5, 1))
    pin = [i for i in range(5) if tuple(coords[i, 1:3]) == tuple(int(v) for v in kv["input"])][0]
    qout = [i for i in range(5) if tuple(coords[i, 1:3]) == tuple(int(v) for v in kv["output"])][0]
    v = oracle.offset_index(tuple(int(x) for x in kv["offset"]), 3)
    assert nbr[qout, v] == pin  # (P3, Q1, W(1,0))
    assert (pin, qout) == (3, 1)
    # P0's dense window: the output at (0,0) uses W(1,1), the one at (2,2) W(-1,-1)
    for row in g:
        if row[0] in ("window_corner", "window_centre"):
            qx, qy, dx, dy = (int(x) for x in row[1:])
            assert (1 - qx, 1 - qy) == (dx, dy)


def test_four_point_grid_counts():
    g = read_golden("four_point_grid.txt")
    kv = {r[0]: r[1:] for r in g}
    grid, names, coords = grid_points(g)
    active = np.zeros(grid, dtype=bool)
    active[coords[:, 1], coords[:, 2]] = True
    one = dense_dilate(active, 3)
    two = dense_dilate(one, 3)
    assert one.sum() == int(kv["dense_active_after_1"][0])
    assert {f"{i},{j}" for i, j in np.argwhere(~one)} == set(kv["dense_empty_after_1"])
    assert two.sum() == int(kv["dense_active_after_2"][0])
    # submanifold: the output set is the input set, layer after layer
    nbr = oracle.kmap(coords, 2, 3, (4, 5, 1))
    assert nbr.shape[0] == int(kv["submanifold_outputs"][0])
    m = len(oracle.tuples(nbr))
    assert m == int(kv["entries_submanifold"][0])
    # zero-skipping entries: every in-grid output of each active input's window
    zs = sum(int(dense_dilate(np.eye(1, 20, 5 * i + j, dtype=bool).reshape(4, 5), 3).sum())
             for i, j in coords[:, 1:3])
    assert zs == int(kv["entries_zero_skipping"][0])
    assert 20 * 9 == int(kv["entries_dense"][0])
    per = int(kv["macs_per_entry_c64"][0])
    assert per == 64 * 64
    assert m * per == int(kv["macs_submanifold_c64"][0])
    assert zs * per == int(kv["macs_zero_skipping_c64"][0])
    assert 180 * per == int(kv["macs_dense_c64"][0])
    # P0's window keeps exactly the two listed tuples
    t = oracle.tuples(nbr)
    p0 = {(int(v), int(q)) for v, q, p in t.tolist() if p == 0}
    want = {(oracle.offset_index((int(r[3]), int(r[4])), 3), int(r[2][1:])) for r in g if r[0] == "p0_tuple"}
    assert p0 == want


def test_dilation_counts():
    for row in read_golden("dilation.txt"):
        ndim, L, want = int(row[1]), int(row[2]), int(row[3])
        shape = (11,) * ndim
        a = np.zeros(shape, dtype=bool)
        a[(5,) * ndim] = True
        for _ in range(L):
            a = dense_dilate(a, 3)
        assert a.sum() == want == (2 * L + 1) ** ndim
    # submanifold never dilates: one site stays one site with one tuple
    for ndim, K in ((3, 3), (3, 5), (2, 3)):
        nbr = oracle.kmap(np.array([[0, 5, 5, 5 if ndim == 3 else 0]]), ndim, K, (11, 11, 11 if ndim == 3 else 1))
        assert nbr.shape == (1, K ** ndim) and (nbr >= 0).sum() == 1 and nbr[0, (K ** ndim - 1) // 2] == 0


# ---------------------------------------------------------------------------
# brute force and invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ndim,K,dims,n,batches", [
    (2, 3, (12, 9, 1), 40, 1), (2, 5, (10, 10, 1), 35, 2),
    (3, 3, (6, 7, 5), 60, 2), (3, 5, (6, 6, 6), 50, 1), (3, 1, (4, 4, 4), 10, 1),
    (3, 7, (9, 9, 8), 80, 2), (2, 7, (12, 11, 1), 50, 1),
])
def test_kmap_equals_brute_force(ndim, K, dims, n, batches):
    coords = random_scene(ndim * 100 + K * 10 + n, n, dims, ndim, batches)
    nbr = oracle.kmap(coords, ndim, K, dims)
    np.testing.assert_array_equal(oracle.tuples(nbr), brute_force_tuples(coords, ndim, K, dims))


def test_kmap_invariants_on_lidar_like_scene():
    s = scenes.lidar_scan(7, 3000, (120, 120, 41))
    nbr = oracle.kmap(s.coords, 3, 3, s.dims)
    V = 27
    counts = (nbr >= 0).sum(axis=0)
    # centre column is the identity, and only it
    np.testing.assert_array_equal(nbr[:, V // 2], np.arange(s.n))
    # count(d) == count(-d); (p, q, d) in M <=> (q, p, -d) in M
    np.testing.assert_array_equal(counts, counts[::-1])
    t = oracle.tuples(nbr)
    mirrored = np.stack([V - 1 - t[:, 0], t[:, 2], t[:, 1]], axis=1)
    mirrored = mirrored[np.lexsort((mirrored[:, 2], mirrored[:, 1], mirrored[:, 0]))]
    np.testing.assert_array_equal(t, mirrored)
    # translation invariance (shift kept inside the grid)
    c2 = s.coords.copy()
    c2[:, 1] += 3
    c2[:, 2] -= 2
    np.testing.assert_array_equal(oracle.kmap(c2, 3, 3, s.dims), nbr)
    # permutation equivariance of row ids
    perm = np.random.default_rng(1).permutation(s.n)
    inv = np.argsort(perm)
    nbr_p = oracle.kmap(s.coords[perm], 3, 3, s.dims)
    expect = np.where(nbr[perm] >= 0, inv[np.maximum(nbr[perm], 0)], -1)
    np.testing.assert_array_equal(nbr_p, expect)


def test_kmap_errors():
    c = np.array([[0, 1, 1, 1], [0, 1, 1, 1]])
    with pytest.raises(oracle.OracleError) as e:
        oracle.kmap(c, 3, 3, (4, 4, 4))
    assert e.value.code == 3
    with pytest.raises(oracle.OracleError) as e:
        oracle.kmap(np.array([[0, 4, 1, 1]]), 3, 3, (4, 4, 4))
    assert e.value.code == 2
    with pytest.raises(oracle.OracleError) as e:
        oracle.kmap(np.array([[0, 1, 1, 1]]), 3, 4, (4, 4, 4))
    assert e.value.code == 1
    assert oracle.kmap(np.zeros((0, 4)), 3, 3, (4, 4, 4)).shape == (0, 27)


# ---------------------------------------------------------------------------
# features
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ndim,K,dims,n,batches,cin,cout", [
    (2, 3, (9, 11, 1), 30, 2, 5, 3), (3, 3, (7, 6, 5), 70, 2, 4, 6), (3, 5, (7, 7, 6), 60, 1, 3, 2),
    (2, 5, (10, 9, 1), 40, 1, 3, 3), (3, 7, (9, 8, 9), 90, 1, 2, 3), (3, 1, (5, 5, 5), 30, 2, 4, 3),
    (3, 5, (8, 7, 6), 60, 3, 2, 2),
])
def test_conv_equals_dense_conv(ndim, K, dims, n, batches, cin, cout):
    coords = random_scene(7 + n, n, dims, ndim, batches)
    rng = np.random.default_rng(n)
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((K ** ndim, cin, cout))
    got = oracle.subm_conv(coords, f, W, ndim, K, dims)
    want = dense_conv_reference(coords, f, W, ndim, K, dims)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # the kept-table entry point (used to time the oracle) gives the same rows
    with oracle.Table(coords, ndim, K, dims) as t:
        np.testing.assert_allclose(t.subm_conv(f, W), want, rtol=1e-12, atol=1e-12)
        rows = np.arange(coords.shape[0])[::-3]
        np.testing.assert_allclose(t.subm_conv(f, W, rows=rows), want[rows], rtol=1e-12, atol=1e-12)


def test_conv_single_site_two_sites_linearity_relu():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((27, 4, 5))
    f = rng.standard_normal((2, 4))
    one = oracle.subm_conv(np.array([[0, 2, 2, 2]]), f[:1], W, 3, 3, (5, 5, 5))
    np.testing.assert_allclose(one[0], f[0] @ W[13], rtol=1e-14)
    # q at (2,2,2), p at q + d with d = (1,0,-1): out_q = f_q Wc + f_p W_d,
    # out_p = f_p Wc + f_q W_{-d}
    c = np.array([[0, 2, 2, 2], [0, 3, 2, 1]])
    d = oracle.offset_index((1, 0, -1), 3)
    md = oracle.offset_index((-1, 0, 1), 3)
    two = oracle.subm_conv(c, f, W, 3, 3, (5, 5, 5))
    np.testing.assert_allclose(two[0], f[0] @ W[13] + f[1] @ W[d], rtol=1e-13)
    np.testing.assert_allclose(two[1], f[1] @ W[13] + f[0] @ W[md], rtol=1e-13)
    # linearity in features and in weights
    s = scenes.lidar_scan(11, 800, (60, 60, 41))
    f1, f2 = rng.standard_normal((2, s.n, 4))
    W2 = rng.standard_normal(W.shape)
    conv = lambda ff, ww: oracle.subm_conv(s.coords, ff, ww, 3, 3, s.dims)
    np.testing.assert_allclose(conv(2 * f1 - f2, W), 2 * conv(f1, W) - conv(f2, W), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(conv(f1, W + W2), conv(f1, W) + conv(f1, W2), rtol=1e-11, atol=1e-11)
    # ReLU and row subsets
    full = conv(f1, W)
    rl = oracle.subm_conv(s.coords, f1, W, 3, 3, s.dims, relu=True)
    np.testing.assert_array_equal(rl, np.maximum(full, 0))
    rows = np.array([5, 0, s.n - 1, 5])
    np.testing.assert_array_equal(oracle.subm_conv(s.coords, f1, W, 3, 3, s.dims, rows=rows), full[rows])


def test_mac_count_independent_of_grouping():
    s = scenes.lidar_scan(12, 1500, (80, 80, 41))
    nbr = oracle.kmap(s.coords, 3, 3, s.dims)
    per_offset = (nbr >= 0).sum(axis=0)
    m = int(per_offset.sum())
    assert m == len(oracle.tuples(nbr))
    assert per_offset[13] == s.n  # the centre map has one entry per point
    # grouping offsets into any partition leaves the MAC total unchanged
    groups = [list(range(0, 13)), [13], list(range(14, 27))]
    assert sum(int(per_offset[g].sum()) for g in groups) * 32 * 32 == m * 32 * 32


def test_round_to_matches_library_rounding():
    x = np.random.default_rng(0).standard_normal(20000) * 10
    x32 = x.astype(np.float32).astype(np.float64)  # exactly representable in fp32
    want = torch.from_numpy(x32).float().to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_to(x32, "bf16"), want)
    np.testing.assert_array_equal(oracle.round_to(x, "f16"), x.astype(np.float16).astype(np.float64))
    # ties go to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 in bf16
    assert oracle.round_to(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8]), "bf16").tolist() == [1.0, 1 + 2 ** -6]


def test_stack_rounds_between_layers():
    s = scenes.lidar_scan(13, 600, (50, 50, 41))
    rng = np.random.default_rng(4)
    f = rng.standard_normal((s.n, 8)).astype(np.float16).astype(np.float64)
    Ws = [rng.standard_normal((27, 8, 8)) / 8 for _ in range(3)]
    outs = oracle.subm_conv_stack(s.coords, f, Ws, 3, 3, s.dims, "f16")
    x = f
    for li, W in enumerate(Ws):
        y = oracle.subm_conv(s.coords, x, W, 3, 3, s.dims, relu=li < 2).astype(np.float16).astype(np.float64)
        np.testing.assert_array_equal(outs[li], y)
        x = y
    assert (outs[0] >= 0).all() and (outs[1] >= 0).all() and (outs[2] < 0).any()


# ---------------------------------------------------------------------------
# backward (the layer is linear in f and in W)
# ---------------------------------------------------------------------------

def dense_conv_grads(coords, feats, W, gout, ndim, K, dims):
    """Gradients of sum(out * gout) for the fp64 dense convolution (torch
    autograd) with zeros at inactive sites, outputs read at active sites:
    (d/d feats at active sites, d/d W in the [V, C_in, C_out] layout)."""
    r = K // 2
    n, c_in = feats.shape
    c_out = W.shape[2]
    Wt = torch.from_numpy(W.copy()).requires_grad_(True)
    gin = np.zeros((n, c_in))
    total = 0
    for b in np.unique(coords[:, 0]):
        sel = np.nonzero(coords[:, 0] == b)[0]
        c = torch.from_numpy(coords[sel].astype(np.int64))
        if ndim == 3:
            grid = torch.zeros((1, c_in) + tuple(dims), dtype=torch.float64)
            grid[0, :, c[:, 1], c[:, 2], c[:, 3]] = torch.from_numpy(feats[sel]).T
            grid.requires_grad_(True)
            w = Wt.reshape(K, K, K, c_in, c_out).permute(4, 3, 0, 1, 2)
            y = torch.nn.functional.conv3d(grid, w, padding=r)[0, :, c[:, 1], c[:, 2], c[:, 3]].T
        else:
            grid = torch.zeros((1, c_in, dims[0], dims[1]), dtype=torch.float64)
            grid[0, :, c[:, 1], c[:, 2]] = torch.from_numpy(feats[sel]).T
            grid.requires_grad_(True)
            w = Wt.reshape(K, K, c_in, c_out).permute(3, 2, 0, 1)
            y = torch.nn.functional.conv2d(grid, w, padding=r)[0, :, c[:, 1], c[:, 2]].T
        loss = (y * torch.from_numpy(gout[sel])).sum()
        g_grid, = torch.autograd.grad(loss, grid, retain_graph=True)
        if ndim == 3:
            gin[sel] = g_grid[0, :, c[:, 1], c[:, 2], c[:, 3]].T.numpy()
        else:
            gin[sel] = g_grid[0, :, c[:, 1], c[:, 2]].T.numpy()
        total = total + loss
    gW, = torch.autograd.grad(total, Wt)
    return gin, gW.numpy()


@pytest.mark.parametrize("ndim,K,dims,n,batches,cin,cout", [
    (2, 3, (9, 11, 1), 30, 2, 5, 3), (3, 3, (7, 6, 5), 70, 2, 4, 6), (3, 5, (7, 7, 6), 60, 1, 3, 2),
    (2, 5, (10, 9, 1), 40, 1, 3, 3), (3, 7, (9, 8, 9), 90, 1, 2, 3), (3, 1, (5, 5, 5), 30, 2, 4, 3),
])
def test_backward_equals_dense_conv_autograd(ndim, K, dims, n, batches, cin, cout):
    coords = random_scene(17 + n, n, dims, ndim, batches)
    rng = np.random.default_rng(3 * n)
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((K ** ndim, cin, cout))
    g = rng.standard_normal((coords.shape[0], cout))
    want_gin, want_gW = dense_conv_grads(coords, f, W, g, ndim, K, dims)
    np.testing.assert_allclose(oracle.subm_conv_bwd_data(coords, g, W, ndim, K, dims), want_gin, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(oracle.subm_conv_bwd_weight(coords, f, g, ndim, K, dims), want_gW, rtol=1e-12,
                               atol=1e-11)


def test_backward_adjoint_identities():
    """<conv_W(f), g> = <f, dgrad_W(g)> = <W, wgrad(f, g)> (bilinear form)."""
    coords = random_scene(5, 120, (10, 9, 8), 3, 2)
    rng = np.random.default_rng(11)
    n = coords.shape[0]
    f = rng.standard_normal((n, 6))
    W = rng.standard_normal((27, 6, 5))
    g = rng.standard_normal((n, 5))
    lhs = float(np.sum(oracle.subm_conv(coords, f, W, 3, 3, (10, 9, 8)) * g))
    mid = float(np.sum(f * oracle.subm_conv_bwd_data(coords, g, W, 3, 3, (10, 9, 8))))
    rhs = float(np.sum(W * oracle.subm_conv_bwd_weight(coords, f, g, 3, 3, (10, 9, 8))))
    assert abs(lhs - mid) <= 1e-9 * max(1.0, abs(lhs))
    assert abs(lhs - rhs) <= 1e-9 * max(1.0, abs(lhs))


def test_backward_closed_forms():
    """Two sites at offset d: out[q] = f[q] W_c + f[p] W_d (c_p = c_q + d),
    out[p] = f[p] W_c + f[q] W_-d, so d/d f[p] = g[p] W_c^T + g[q] W_d^T and
    d/d W_d = f[p]^T g[q]; an offset with no pair gets a zero gradient."""
    coords = np.array([[0, 2, 2, 2], [0, 3, 2, 1]], dtype=np.int32)  # p - q = (1, 0, -1)
    q, p = 0, 1
    d = oracle.offset_index((1, 0, -1), 3)
    md = oracle.offset_index((-1, 0, 1), 3)
    c = 13
    rng = np.random.default_rng(2)
    f = rng.standard_normal((2, 3))
    W = rng.standard_normal((27, 3, 4))
    g = rng.standard_normal((2, 4))
    gin = oracle.subm_conv_bwd_data(coords, g, W, 3, 3, (6, 6, 6))
    np.testing.assert_allclose(gin[p], W[c] @ g[p] + W[d] @ g[q], rtol=1e-13)
    np.testing.assert_allclose(gin[q], W[c] @ g[q] + W[md] @ g[p], rtol=1e-13)
    gW = oracle.subm_conv_bwd_weight(coords, f, g, 3, 3, (6, 6, 6))
    np.testing.assert_allclose(gW[d], np.outer(f[p], g[q]), rtol=1e-13)
    np.testing.assert_allclose(gW[md], np.outer(f[q], g[p]), rtol=1e-13)
    np.testing.assert_allclose(gW[c], np.outer(f[p], g[p]) + np.outer(f[q], g[q]), rtol=1e-13)
    others = [v for v in range(27) if v not in (d, md, c)]
    assert np.all(gW[others] == 0)


def test_backward_data_rows_subset_equals_full():
    coords = random_scene(9, 80, (8, 8, 8), 3, 1)
    rng = np.random.default_rng(4)
    g = rng.standard_normal((coords.shape[0], 3))
    W = rng.standard_normal((27, 5, 3))
    full = oracle.subm_conv_bwd_data(coords, g, W, 3, 3, (8, 8, 8))
    rows = np.array([0, 7, 3, 79, 41])
    np.testing.assert_array_equal(oracle.subm_conv_bwd_data(coords, g, W, 3, 3, (8, 8, 8), rows=rows), full[rows])


# ---------------------------------------------------------------------------
# regular (dilating) and strided layers: the output set differs from the input
# ("SparseConvNet: from hash table to rulebook", sections 2 and 3)
# ---------------------------------------------------------------------------

def dense_strided(coords, feats, W, ndim, K, stride, dims):
    """fp64 dense convolution (torch, cross-correlation, zero padding r,
    stride s) of each batch's scattered features: {batch: [c_out, *out_ext]}.
    Output o reads the inputs at s * o + d, d in [-r, r]."""
    r = K // 2
    c_in, c_out = W.shape[1], W.shape[2]
    res = {}
    for b in np.unique(coords[:, 0]):
        sel = np.nonzero(coords[:, 0] == b)[0]
        c = torch.from_numpy(coords[sel].astype(np.int64))
        f = torch.from_numpy(np.asarray(feats)[sel]).T
        if ndim == 3:
            grid = torch.zeros((1, c_in) + tuple(dims), dtype=torch.float64)
            grid[0, :, c[:, 1], c[:, 2], c[:, 3]] = f
            w = torch.from_numpy(W).reshape(K, K, K, c_in, c_out).permute(4, 3, 0, 1, 2).contiguous()
            res[int(b)] = torch.nn.functional.conv3d(grid, w, padding=r, stride=stride)[0]
        else:
            # 2D: the planes z are independent; stride and offsets act on (x, y)
            outs = []
            for z in range(dims[2]):
                grid = torch.zeros((1, c_in, dims[0], dims[1]), dtype=torch.float64)
                m = c[:, 3] == z
                grid[0, :, c[m, 1], c[m, 2]] = f[:, m]
                w = torch.from_numpy(W).reshape(K, K, c_in, c_out).permute(3, 2, 0, 1).contiguous()
                outs.append(torch.nn.functional.conv2d(grid, w, padding=r, stride=stride)[0])
            res[int(b)] = torch.stack(outs, dim=-1)
    return res


def read_dense(res, out_coords):
    c_out = next(iter(res.values())).shape[0]
    rows = [res[int(b)][:, x, y, z].numpy() for b, x, y, z in out_coords]
    return np.stack(rows) if rows else np.zeros((0, c_out))


def test_regular_four_point_grid():
    """17 of 20 cells after one dilating layer (empties (0,3), (0,4), (3,0)),
    all 20 after a second; the first layer's map holds the 30 entries of the
    zero-skipping count."""
    g = read_golden("four_point_grid.txt")
    kv = {r[0]: r[1:] for r in g}
    grid, names, coords = grid_points(g)
    dims = (grid[0], grid[1], 1)
    one = oracle.conv_out_coords(coords, 2, 3, 1, dims)
    assert len(one) == int(kv["dense_active_after_1"][0])
    empty = {f"{i},{j}" for i in range(grid[0]) for j in range(grid[1])} - {f"{x},{y}" for _, x, y, _ in one}
    assert empty == set(kv["dense_empty_after_1"])
    two = oracle.conv_out_coords(one, 2, 3, 1, dims)
    assert len(two) == int(kv["dense_active_after_2"][0])
    nbr = oracle.conv_kmap(coords, one, 2, 3, 1, dims)
    assert int((nbr >= 0).sum()) == int(kv["entries_zero_skipping"][0])
    # the oracle's output set is the independent dense dilation of the grid
    active = np.zeros(grid, dtype=bool)
    active[coords[:, 1], coords[:, 2]] = True
    assert {(x, y) for _, x, y, _ in one} == {tuple(ij) for ij in np.argwhere(dense_dilate(active, 3))}


def test_regular_dilation_counts():
    """One site grows to (2L+1)^d sites after L dilating layers of width 3."""
    for row in read_golden("dilation.txt"):
        ndim, L, want = int(row[1]), int(row[2]), int(row[3])
        dims = (11, 11, 11 if ndim == 3 else 1)
        c = np.array([[0, 5, 5, 5 if ndim == 3 else 0]], dtype=np.int32)
        for _ in range(L):
            c = oracle.conv_out_coords(c, ndim, 3, 1, dims)
        assert len(c) == want == (2 * L + 1) ** ndim


def test_strided_single_site_closed_forms():
    """Stride 2, width 3: output o reads inputs 2o - 1 .. 2o + 1, so an odd
    site 5 feeds o = 2 (offset +1) and o = 3 (offset -1) on each axis, an even
    site 4 only o = 2 (offset 0)."""
    dims = (11, 11, 11)
    odd = oracle.conv_out_coords(np.array([[0, 5, 5, 5]]), 3, 3, 2, dims)
    assert sorted(map(tuple, odd[:, 1:].tolist())) == sorted(itertools.product((2, 3), repeat=3))
    nbr = oracle.conv_kmap(np.array([[0, 5, 5, 5]]), odd, 3, 3, 2, dims)
    for (b, x, y, z), row in zip(odd, nbr):
        d = tuple(5 - 2 * v for v in (x, y, z))
        assert (row >= 0).sum() == 1 and row[oracle.offset_index(d, 3)] == 0
    even = oracle.conv_out_coords(np.array([[0, 4, 4, 4]]), 3, 3, 2, dims)
    assert even.tolist() == [[0, 2, 2, 2]]
    # width 1, stride 2: only even sites have an output, at half the coordinate
    pts = np.array([[0, 4, 6, 2], [0, 5, 6, 2], [1, 8, 0, 10]], dtype=np.int32)
    o = oracle.conv_out_coords(pts, 3, 1, 2, dims)
    assert o.tolist() == [[0, 2, 3, 1], [1, 4, 0, 5]]
    assert oracle.conv_out_extent((11, 11, 11), 3, 2) == (6, 6, 6)
    assert oracle.conv_out_extent((11, 10, 3), 2, 2) == (6, 5, 3)


def brute_force_strided(coords, out_coords, ndim, K, stride, dims):
    """(offset, out, in) for every pair with c_in - stride * c_out in
    [-r, r]^ndim, same batch (and same plane in 2D)."""
    r = K // 2
    res = []
    for q, co in enumerate(out_coords):
        for p, ci in enumerate(coords):
            if ci[0] != co[0] or (ndim == 2 and ci[3] != co[3]):
                continue
            d = ci[1:1 + ndim] - stride * co[1:1 + ndim]
            if np.all(np.abs(d) <= r):
                res.append((oracle.offset_index(d, K), q, p))
    res.sort()
    return np.array(res, dtype=np.int64).reshape(-1, 3)


@pytest.mark.parametrize("ndim,K,stride,dims,n,batches", [
    (2, 3, 1, (9, 8, 1), 25, 1), (2, 3, 2, (9, 8, 2), 30, 2), (2, 5, 3, (12, 10, 1), 30, 1),
    (3, 3, 1, (6, 5, 6), 30, 2), (3, 3, 2, (7, 6, 5), 40, 1), (3, 5, 2, (6, 6, 6), 30, 1),
    (3, 1, 2, (6, 6, 6), 30, 1), (3, 3, 3, (8, 7, 9), 40, 2),
])
def test_strided_map_equals_brute_force(ndim, K, stride, dims, n, batches):
    c = random_scene(ndim * 100 + K * 10 + stride, n, dims, ndim, batches)
    o = oracle.conv_out_coords(c, ndim, K, stride, dims)
    t = oracle.tuples(oracle.conv_kmap(c, o, ndim, K, stride, dims))
    assert np.array_equal(t, brute_force_strided(c, o, ndim, K, stride, dims))
    # every output has at least one tuple; every input reaches an output when
    # the windows s * o + [-r, r] tile the axis without gaps (s <= r + 1)
    assert set(t[:, 1].tolist()) == set(range(len(o)))
    if stride <= K // 2 + 1:
        assert set(t[:, 2].tolist()) == set(range(len(c)))


@pytest.mark.parametrize("ndim,K,stride,dims,n,batches,cin,cout", [
    (2, 3, 1, (10, 9, 1), 30, 1, 3, 4), (2, 3, 2, (10, 9, 2), 40, 2, 2, 5), (2, 5, 2, (11, 12, 1), 30, 1, 4, 3),
    (3, 3, 1, (7, 6, 5), 40, 2, 3, 2), (3, 3, 2, (8, 7, 6), 50, 1, 4, 4), (3, 5, 3, (9, 8, 7), 40, 1, 2, 3),
    (3, 1, 2, (6, 6, 6), 80, 1, 3, 3),
])
def test_strided_conv_equals_dense_conv(ndim, K, stride, dims, n, batches, cin, cout):
    c = random_scene(ndim * 1000 + K * 100 + stride, n, dims, ndim, batches)
    rng = np.random.default_rng(7)
    f = rng.standard_normal((c.shape[0], cin))
    W = rng.standard_normal((K ** ndim, cin, cout))
    o = oracle.conv_out_coords(c, ndim, K, stride, dims)
    got = oracle.sparse_conv(c, o, f, W, ndim, K, stride, dims)
    dense = dense_strided(c, f, W, ndim, K, stride, dims)
    assert np.allclose(got, read_dense(dense, o), rtol=1e-12, atol=1e-12)
    # the output set is the support of the dense layer on the active-site
    # indicator with a kernel of ones
    ind = dense_strided(c, np.ones((c.shape[0], 1)), np.ones((K ** ndim, 1, 1)), ndim, K, stride, dims)
    support = sorted((b, *map(int, idx[1:])) for b, g in ind.items() for idx in np.argwhere(g.numpy() > 0.5))
    assert [tuple(r) for r in o.tolist()] == support
    relu = oracle.sparse_conv(c, o, f, W, ndim, K, stride, dims, relu=True)
    assert np.array_equal(relu, np.maximum(got, 0.0))


def test_strided_conv_at_stride_one_agrees_with_submanifold_on_input_sites():
    c = random_scene(5, 60, (8, 7, 6), 3, 2)
    rng = np.random.default_rng(3)
    f = rng.standard_normal((c.shape[0], 3))
    W = rng.standard_normal((27, 3, 2))
    o = oracle.conv_out_coords(c, 3, 3, 1, (8, 7, 6))
    full = oracle.sparse_conv(c, o, f, W, 3, 3, 1, (8, 7, 6))
    at = {tuple(r): k for k, r in enumerate(o.tolist())}
    idx = np.array([at[tuple(r)] for r in c.tolist()])
    assert np.allclose(full[idx], oracle.subm_conv(c, f, W, 3, 3, (8, 7, 6)), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ndim,K,stride,dims,n,cin,cout", [
    (3, 3, 2, (7, 6, 8), 40, 3, 2), (2, 3, 1, (9, 9, 1), 30, 2, 3), (3, 5, 2, (6, 7, 6), 30, 2, 2),
])
def test_strided_weight_gradient_equals_dense_autograd(ndim, K, stride, dims, n, cin, cout):
    c = random_scene(ndim * 7 + K + stride, n, dims, ndim, 1)
    rng = np.random.default_rng(11)
    f = rng.standard_normal((c.shape[0], cin))
    W = rng.standard_normal((K ** ndim, cin, cout))
    o = oracle.conv_out_coords(c, ndim, K, stride, dims)
    g = rng.standard_normal((o.shape[0], cout))
    dW = oracle.sparse_conv_bwd_weight(c, o, f, g, ndim, K, stride, dims)
    Wt = torch.from_numpy(W).requires_grad_(True)
    r = K // 2
    ext = oracle.conv_out_extent(dims, ndim, stride)
    cc = torch.from_numpy(c.astype(np.int64))
    oo = torch.from_numpy(o.astype(np.int64))
    if ndim == 3:
        grid = torch.zeros((1, cin) + tuple(dims), dtype=torch.float64)
        grid[0, :, cc[:, 1], cc[:, 2], cc[:, 3]] = torch.from_numpy(f).T
        w = Wt.reshape(K, K, K, cin, cout).permute(4, 3, 0, 1, 2)
        y = torch.nn.functional.conv3d(grid, w, padding=r, stride=stride)[0]
        gy = torch.zeros((cout,) + ext, dtype=torch.float64)
        gy[:, oo[:, 1], oo[:, 2], oo[:, 3]] = torch.from_numpy(g).T
    else:
        grid = torch.zeros((1, cin, dims[0], dims[1]), dtype=torch.float64)
        grid[0, :, cc[:, 1], cc[:, 2]] = torch.from_numpy(f).T
        w = Wt.reshape(K, K, cin, cout).permute(3, 2, 0, 1)
        y = torch.nn.functional.conv2d(grid, w, padding=r, stride=stride)[0]
        gy = torch.zeros((cout,) + ext[:2], dtype=torch.float64)
        gy[:, oo[:, 1], oo[:, 2]] = torch.from_numpy(g).T
    (y * gy).sum().backward()
    assert np.allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("ndim,K,stride,dims,n,cin,cout", [
    (3, 3, 2, (7, 6, 8), 40, 3, 2), (2, 3, 1, (9, 9, 1), 30, 2, 3), (3, 5, 2, (6, 7, 6), 30, 2, 2),
    (3, 3, 3, (8, 7, 9), 40, 2, 3), (2, 5, 2, (11, 9, 2), 40, 3, 2),
])
def test_strided_input_gradient_equals_dense_autograd(ndim, K, stride, dims, n, cin, cout):
    c = random_scene(ndim * 11 + K + 3 * stride, n, dims, ndim, 1)
    rng = np.random.default_rng(13)
    f = rng.standard_normal((c.shape[0], cin))
    W = rng.standard_normal((K ** ndim, cin, cout))
    o = oracle.conv_out_coords(c, ndim, K, stride, dims)
    g = rng.standard_normal((o.shape[0], cout))
    gin = oracle.sparse_conv_bwd_data(c, o, g, W, ndim, K, stride, dims)
    r = K // 2
    ext = oracle.conv_out_extent(dims, ndim, stride)
    cc = torch.from_numpy(c.astype(np.int64))
    oo = torch.from_numpy(o.astype(np.int64))
    Wt = torch.from_numpy(W)
    if ndim == 3:
        grid = torch.zeros((1, cin) + tuple(dims), dtype=torch.float64, requires_grad=True)
        y = torch.nn.functional.conv3d(grid, Wt.reshape(K, K, K, cin, cout).permute(4, 3, 0, 1, 2), padding=r,
                                       stride=stride)[0]
        gy = torch.zeros((cout,) + ext, dtype=torch.float64)
        gy[:, oo[:, 1], oo[:, 2], oo[:, 3]] = torch.from_numpy(g).T
        (y * gy).sum().backward()
        want = grid.grad[0][:, cc[:, 1], cc[:, 2], cc[:, 3]].T.numpy()
    else:
        assert dims[2] <= 2
        want = np.zeros_like(gin)
        for z in range(dims[2]):
            grid = torch.zeros((1, cin, dims[0], dims[1]), dtype=torch.float64, requires_grad=True)
            y = torch.nn.functional.conv2d(grid, Wt.reshape(K, K, cin, cout).permute(3, 2, 0, 1), padding=r,
                                           stride=stride)[0]
            gy = torch.zeros((cout,) + ext[:2], dtype=torch.float64)
            mo = oo[:, 3] == z
            gy[:, oo[mo, 1], oo[mo, 2]] = torch.from_numpy(g[mo.numpy()]).T
            (y * gy).sum().backward()
            mc = (cc[:, 3] == z).numpy()
            want[mc] = grid.grad[0][:, cc[mc, 1], cc[mc, 2]].T.numpy()
    assert np.allclose(gin, want, rtol=1e-10, atol=1e-10)
    # adjoint identity: <conv(f), g> = <f, gin>
    lhs = float((oracle.sparse_conv(c, o, f, W, ndim, K, stride, dims) * g).sum())
    assert abs(lhs - float((f * gin).sum())) <= 1e-9 * max(1.0, abs(lhs))


def test_empty_scene_gives_empty_outputs_and_zero_weight_gradients():
    """No active site: every layer output has no rows, and a weight gradient,
    a sum over the map's tuples, is the empty sum 0.  The kept table agrees."""
    c = np.zeros((0, 4), dtype=np.int32)
    o = np.zeros((0, 4), dtype=np.int32)
    dims = (8, 8, 8)
    W = np.ones((27, 16, 8))
    assert oracle.kmap(c, 3, 3, dims).shape == (0, 27)
    assert oracle.subm_conv(c, np.zeros((0, 16)), W, 3, 3, dims, relu=True).shape == (0, 8)
    assert oracle.subm_conv_bwd_data(c, np.zeros((0, 8)), W, 3, 3, dims).shape == (0, 16)
    gw = oracle.subm_conv_bwd_weight(c, np.zeros((0, 16)), np.zeros((0, 8)), 3, 3, dims)
    assert gw.shape == (27, 16, 8) and not gw.any()
    outs = oracle.subm_conv_stack(c, np.zeros((0, 16)), [np.ones((27, 16, 16))] * 2, 3, 3, dims, "f16")
    assert [x.shape for x in outs] == [(0, 16), (0, 16)]
    with oracle.Table(c, 3, 3, dims) as t:
        assert t.subm_conv(np.zeros((0, 16)), W).shape == (0, 8)
    assert oracle.conv_out_coords(c, 3, 3, 2, dims).shape == (0, 4)
    assert oracle.sparse_conv(c, o, np.zeros((0, 16)), W, 3, 3, 2, dims).shape == (0, 8)
    assert oracle.sparse_conv_bwd_data(c, o, np.zeros((0, 8)), W, 3, 3, 2, dims).shape == (0, 16)
    gw = oracle.sparse_conv_bwd_weight(c, o, np.zeros((0, 16)), np.zeros((0, 8)), 3, 3, 2, dims)
    assert gw.shape == (27, 16, 8) and not gw.any()


def test_feature_rows_must_match_the_points():
    """A feature array whose row count differs from the number of points is
    an argument error, not silently reshaped."""
    c = np.array([[0, 1, 1, 1], [0, 2, 1, 1]], dtype=np.int32)
    W = np.ones((27, 4, 4))
    with pytest.raises(oracle.OracleError):
        oracle.subm_conv(c, np.zeros((4, 4)), W, 3, 3, (8, 8, 8))
    with pytest.raises(oracle.OracleError):
        oracle.subm_conv_bwd_weight(c, np.zeros((2, 4)), np.zeros((1, 8)), 3, 3, (8, 8, 8))
