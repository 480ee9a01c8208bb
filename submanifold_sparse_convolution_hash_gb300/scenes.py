"""Seeded synthetic voxel scenes and layer tensors.

This module only draws inputs: coordinates, features and weights.  It holds
none of the layer's arithmetic (no hashing, no neighbour search, no
convolution), so the CPU reference checks and the CUDA path can both take their
inputs from here without sharing any computation.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used in its counter form: the
k-th draw of a stream with state s is mix(s + k * 0x9E3779B97F4A7C15).

Scene families, following the densities and map-size regimes that the source
pages describe for outdoor LiDAR frames and indoor scans ("Sparse inputs and
sparse convolution", opening section; "TorchSparse optimizations", section
"Measured"):

* ``uniform_2d``   -- cells drawn uniformly without replacement on a 2D grid.
* ``lidar_scan``   -- a jittered ground disk plus axis-aligned box shells and
                      vertical cylinder shells standing on it.
* ``indoor_scene`` -- 1-voxel-thick axis-aligned walls/floors and sphere
                      shells, added until the voxel budget is reached.

Every scene is emitted as int32 coords ``[N, 4] = (batch, x, y, z)`` in a
seeded random permutation (no spatial locality in row order), duplicates
removed.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def _mix64_int(v: int) -> int:
    return int(_mix64(np.array([v & _M64], dtype=np.uint64))[0])


class SplitMix64:
    """Counter-form SplitMix64 stream; every call advances the counter."""

    def __init__(self, seed: int, stream: int = 0):
        # distinct streams of one seed start from well separated states
        self.state = _mix64_int((seed & _M64) ^ _mix64_int(0x5EED0000 + stream))

    def u64(self, n: int) -> np.ndarray:
        k = np.arange(1, n + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            z = np.uint64(self.state) + k * np.uint64(_GAMMA)
        self.state = (self.state + n * _GAMMA) & _M64
        return _mix64(z)

    def uniform(self, n: int) -> np.ndarray:
        """Doubles in [0, 1) from the top 53 bits."""
        return (self.u64(n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)

    def integers(self, lo: int, hi: int, n: int) -> np.ndarray:
        """Integers in [lo, hi)."""
        return (lo + np.floor(self.uniform(n) * (hi - lo))).astype(np.int64)

    def normal(self, n: int) -> np.ndarray:
        """Standard normals by the Box-Muller transform."""
        m = (n + 1) // 2
        u1 = self.uniform(m)
        u2 = self.uniform(m)
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * np.pi * u2
        return np.concatenate([r * np.cos(t), r * np.sin(t)])[:n]

    def permutation(self, n: int) -> np.ndarray:
        return np.argsort(self.u64(n), kind="stable")


@dataclass
class Scene:
    """A voxel scene: int32 coords [N, 4] (batch, x, y, z) plus its grid."""

    name: str
    coords: np.ndarray
    dims: tuple  # (X, Y, Z) spatial extents; Z = 1 for 2D scenes
    ndim: int
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.coords.shape[0])


def _emit(points_xyz: np.ndarray, batch: int, rng: SplitMix64) -> np.ndarray:
    """Deduplicate (x, y, z) rows, then emit them in a seeded random order."""
    pts = np.unique(points_xyz.astype(np.int64), axis=0)
    perm = rng.permutation(pts.shape[0])
    pts = pts[perm]
    out = np.empty((pts.shape[0], 4), dtype=np.int32)
    out[:, 0] = batch
    out[:, 1:] = pts
    return out


# ----------------------------------------------------------------------------
# 2D uniform cells
# ----------------------------------------------------------------------------

def uniform_2d(seed: int = 1000, grid=(64, 64), n: int = 200) -> Scene:
    """``n`` distinct cells of a 2D grid, drawn uniformly without replacement."""
    X, Y = grid
    if n > X * Y:
        raise ValueError("more cells than the grid holds")
    rng = SplitMix64(seed, 0)
    cells = rng.permutation(X * Y)[:n]
    coords = np.zeros((n, 4), dtype=np.int32)
    coords[:, 1] = cells // Y
    coords[:, 2] = cells % Y
    return Scene("uniform_2d", coords, (X, Y, 1), 2, seed, {"grid": grid})


# ----------------------------------------------------------------------------
# LiDAR-like scan
# ----------------------------------------------------------------------------

def _box_shell(x0, y0, z0, a, b, h):
    g = np.ones((a, b, h), dtype=bool)
    if a > 2 and b > 2 and h > 2:
        g[1:-1, 1:-1, 1:-1] = False
    p = np.argwhere(g)
    p[:, 0] += x0
    p[:, 1] += y0
    p[:, 2] += z0
    return p


def _cylinder_shell(xc, yc, z0, r, h):
    R = int(math.ceil(r)) + 1
    xs = np.arange(-R, R + 1)
    dx, dy = np.meshgrid(xs, xs, indexing="ij")
    d = np.sqrt(dx * dx + dy * dy)
    ring = np.abs(d - r) < 0.5
    cap = d <= r
    parts = []
    ring_xy = np.stack([dx[ring], dy[ring]], axis=1)
    for z in range(h):
        p = np.empty((ring_xy.shape[0], 3), dtype=np.int64)
        p[:, :2] = ring_xy
        p[:, 2] = z
        parts.append(p)
    cap_xy = np.stack([dx[cap], dy[cap]], axis=1)
    p = np.empty((cap_xy.shape[0], 3), dtype=np.int64)
    p[:, :2] = cap_xy
    p[:, 2] = h - 1
    parts.append(p)
    p = np.concatenate(parts)
    p[:, 0] += xc
    p[:, 1] += yc
    p[:, 2] += z0
    return p


def _clip(p, dims):
    m = np.all((p >= 0) & (p < np.asarray(dims)), axis=1)
    return p[m]


def lidar_scan(seed: int = 1001, n_target: int = 100_000, dims=(1440, 1440, 41),
               batch: int = 0, n_boxes: int = 40, n_cyl: int = 20,
               ground_z: int = 8, ground_share: float = 0.6) -> Scene:
    """Outdoor-scan stand-in: ground disk with +-1 voxel jitter and objects.

    The ground disk is centred on the grid and sized so that it supplies about
    ``ground_share`` of ``n_target`` voxels.  Box shells (sides 4-40 in x/y,
    4-20 in z) and vertical cylinder shells (radius 2-8, height 10-35) stand on
    the ground inside that disk.  The object sizes are drawn once from those
    ranges, then all scaled by one common factor so that the objects supply
    the rest of the budget; N lands within a few percent of ``n_target``.
    """
    X, Y, Z = dims
    rng = SplitMix64(seed, 1)
    cx, cy = X // 2, Y // 2
    r_disk0 = math.sqrt(ground_share * n_target / math.pi)
    # object draws (unit-interval variates, scaled below)
    bu = rng.uniform(n_boxes * 5).reshape(n_boxes, 5)
    cu = rng.uniform(n_cyl * 4).reshape(n_cyl, 4)

    def place(u_r, u_t, margin):
        rr = max(r_disk0 - margin, 1.0) * math.sqrt(u_r)
        t = 2 * math.pi * u_t
        return int(cx + rr * math.cos(t)), int(cy + rr * math.sin(t))

    def objects(scale):
        parts = []
        for i in range(n_boxes):
            a = max(2, int(round((4 + bu[i, 0] * 36) * scale)))
            b = max(2, int(round((4 + bu[i, 1] * 36) * scale)))
            h = max(2, int(round((4 + bu[i, 2] * 16) * scale)))
            x0, y0 = place(bu[i, 3], bu[i, 4], 20)
            parts.append(_box_shell(x0 - a // 2, y0 - b // 2, ground_z + 1, a, b, h))
        for i in range(n_cyl):
            r = max(1.5, (2 + cu[i, 0] * 6) * scale)
            h = max(2, int(round((10 + cu[i, 1] * 25) * scale)))
            x0, y0 = place(cu[i, 2], cu[i, 3], 12)
            parts.append(_cylinder_shell(x0, y0, ground_z + 1, r, h))
        p = _clip(np.concatenate(parts), dims)
        return np.unique(p, axis=0)

    budget = (1.0 - ground_share) * n_target
    scale = 1.0
    obj = objects(scale)
    for _ in range(4):
        scale *= math.sqrt(budget / max(obj.shape[0], 1))
        obj = objects(scale)
    # ground disk sized to fill the remaining budget
    n_ground = max(n_target - obj.shape[0], 0)
    r_disk = math.sqrt(n_ground / math.pi)
    R = int(math.ceil(r_disk))
    gx, gy = np.meshgrid(np.arange(cx - R, cx + R + 1), np.arange(cy - R, cy + R + 1), indexing="ij")
    inside = (gx - cx) ** 2 + (gy - cy) ** 2 <= r_disk * r_disk
    gx = gx[inside].ravel()
    gy = gy[inside].ravel()
    jitter = rng.integers(-1, 2, gx.shape[0])
    ground = np.stack([gx, gy, ground_z + jitter], axis=1)
    pts = _clip(np.concatenate([ground, obj]), dims)
    coords = _emit(pts, batch, rng)
    return Scene("lidar_scan", coords, tuple(dims), 3, seed,
                 {"n_target": n_target, "object_scale": scale, "ground_radius": r_disk})


# ----------------------------------------------------------------------------
# Indoor-like scene
# ----------------------------------------------------------------------------

def indoor_scene(seed: int = 1002, n_target: int = 1_000_000, dims=(512, 512, 128),
                 extent=(32, 256), radius=(8, 40)) -> Scene:
    """Indoor-scan stand-in: walls, floors and sphere shells until N >= n_target.

    Each object is, with probabilities 0.3/0.3/0.2/0.2, a 1-voxel-thick plane
    normal to x, to y or to z (in-plane extents uniform in ``extent``,
    clipped to the grid) or a sphere shell (radius uniform in ``radius``).
    """
    X, Y, Z = dims
    occ = np.zeros(dims, dtype=bool)
    rng = SplitMix64(seed, 2)
    count = 0
    n_obj = 0
    while count < n_target:
        u = rng.uniform(8)
        kind = u[0]
        lo, hi = extent
        if kind < 0.8:
            if kind < 0.3:
                axis = 0
            elif kind < 0.6:
                axis = 1
            else:
                axis = 2
            ext = [X, Y, Z]
            pos = int(u[1] * ext[axis])
            sl = [None, None, None]
            sl[axis] = slice(pos, pos + 1)
            others = [a for a in range(3) if a != axis]
            for j, a in enumerate(others):
                length = int(lo + u[2 + 2 * j] * (hi - lo))
                start = int(u[3 + 2 * j] * max(ext[a] - 1, 1))
                sl[a] = slice(start, min(start + length, ext[a]))
            region = occ[tuple(sl)]
            before = int(region.sum())
            region[...] = True
            count += region.size - before
        else:
            r = radius[0] + u[1] * (radius[1] - radius[0])
            c = (u[2] * X, u[3] * Y, u[4] * Z)
            R = int(math.ceil(r)) + 1
            box = [slice(max(int(c[a]) - R, 0), min(int(c[a]) + R + 1, dims[a])) for a in range(3)]
            xs = [np.arange(b.start, b.stop) + 0.5 - c[a] for a, b in enumerate(box)]
            d = np.sqrt(xs[0][:, None, None] ** 2 + xs[1][None, :, None] ** 2 + xs[2][None, None, :] ** 2)
            shell = np.abs(d - r) < 0.5
            region = occ[tuple(box)]
            before = int(region.sum())
            region |= shell
            count += int(region.sum()) - before
        n_obj += 1
    pts = np.argwhere(occ)
    del occ
    coords = _emit(pts, 0, rng)
    return Scene("indoor_scene", coords, tuple(dims), 3, seed, {"n_target": n_target, "objects": n_obj})


def batch_of_scans(seed: int = 1003, n_scans: int = 4, n_target: int = 120_000,
                   dims=(1440, 1440, 41)) -> Scene:
    """``n_scans`` LiDAR-like scans (seeds seed+b) stacked with batch index b."""
    parts = [lidar_scan(seed + b, n_target, dims, batch=b).coords for b in range(n_scans)]
    coords = np.concatenate(parts)
    rng = SplitMix64(seed, 3)
    coords = coords[rng.permutation(coords.shape[0])]
    return Scene("batch_of_scans", np.ascontiguousarray(coords), tuple(dims), 3, seed,
                 {"n_scans": n_scans, "n_target": n_target})


# ----------------------------------------------------------------------------
# Features and weights
# ----------------------------------------------------------------------------

def features(seed: int, n: int, c: int, std: float = 1.0) -> np.ndarray:
    """float32 [n, c] ~ N(0, std^2)."""
    rng = SplitMix64(seed, 10)
    out = np.empty(n * c, dtype=np.float32)
    step = 1 << 22
    # chunk k starts at the counter the serial draw would reach there (each
    # normal(m) call consumes 2 * ceil(m / 2) counters), so the chunks can be
    # drawn on threads and the values equal one serial pass
    jobs = []
    state = rng.state
    for s in range(0, n * c, step):
        m = min(step, n * c - s)
        jobs.append((s, m, state))
        state = (state + 2 * ((m + 1) // 2) * _GAMMA) & _M64

    def draw(job):
        s, m, st = job
        r = SplitMix64.__new__(SplitMix64)
        r.state = st
        out[s:s + m] = (r.normal(m) * std).astype(np.float32)

    if len(jobs) > 1:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
            list(ex.map(draw, jobs))
    else:
        for j in jobs:
            draw(j)
    return out.reshape(n, c)


def weights(seed: int, volume: int, c_in: int, c_out: int, std: float | None = None) -> np.ndarray:
    """float32 [volume, c_in, c_out] ~ N(0, std^2); std defaults to 1/sqrt(volume*c_in)."""
    if std is None:
        std = 1.0 / math.sqrt(volume * c_in)
    rng = SplitMix64(seed, 11)
    return (rng.normal(volume * c_in * c_out) * std).astype(np.float32).reshape(volume, c_in, c_out)


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    scene_fn: object
    K: int
    channels: tuple  # layer widths: (c0, c1, ...) -> len-1 layers
    dtype: str  # "f32" | "f16" | "bf16"
    seed: int
    w_std_unit: bool = False  # True: W ~ N(0,1) instead of 1/sqrt(V*C_in)


def workload(idx: int, scale: float = 1.0, replica: int = 0) -> tuple:
    """(Workload, Scene) for workload ``idx`` (0..4); ``scale`` < 1 shrinks N and grid.
    ``replica`` > 0 draws another scene of the same recipe (scene seed shifted
    by 7919 * replica; weights unchanged), one per independent replica.

    0: 2D 64x64, 200 cells, 3x3, C 16, fp32, W ~ N(0,1)
    1: LiDAR-like 1440x1440x41, ~100k, 3x3x3, C 32, fp16
    2: indoor-like 512x512x128, ~1M, 3x3x3, C 64, bf16
    3: 4 LiDAR-like scans ~120k each, 3x3x3, 8 layers 32->...->256, fp16
    4: 2048x2048x64, ~2M, 5x5x5, C 128, bf16
    """
    r = 7919 * replica

    def sdims(d, keep_z=True):
        f = math.sqrt(scale)
        return tuple(max(16, int(d[a] * f)) if (a < 2 or not keep_z) else d[a] for a in range(3))

    if idx == 0:
        w = Workload("2d_uniform_64x64_n200_k3_c16_f32", None, 3, (16, 16), "f32", 1000, True)
        return w, uniform_2d(1000 + r, (64, 64), max(8, int(200 * scale)) if scale < 1 else 200)
    if idx == 1:
        w = Workload("lidar_1440x1440x41_n100k_k3_c32_f16", None, 3, (32, 32), "f16", 1001)
        return w, lidar_scan(1001 + r, int(100_000 * scale), sdims((1440, 1440, 41)))
    if idx == 2:
        w = Workload("indoor_512x512x128_n1m_k3_c64_bf16", None, 3, (64, 64), "bf16", 1002)
        return w, indoor_scene(1002 + r, int(1_000_000 * scale), sdims((512, 512, 128)))
    if idx == 3:
        w = Workload("lidar_batch4x120k_k3_8layers_32to256_f16", None, 3,
                     (32, 32, 64, 64, 128, 128, 256, 256, 256), "f16", 1003)
        return w, batch_of_scans(1003 + r, 4, int(120_000 * scale), sdims((1440, 1440, 41)))
    if idx == 4:
        w = Workload("surfaces_2048x2048x64_n2m_k5_c128_bf16", None, 5, (128, 128), "bf16", 1004)
        return w, indoor_scene(1004 + r, int(2_000_000 * scale), sdims((2048, 2048, 64)))
    raise ValueError(idx)
