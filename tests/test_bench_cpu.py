"""Host logic of bench.py (no GPU): the algorithmic-byte models behind the
roofline, the staleness check of recorded DRAM traffic, and the parsing of
sampled clocks and throttle reasons."""
import hashlib
import json
import os

import bench


def test_algorithmic_bytes_of_the_fused_layer():
    N, V, M, s = 1000, 27, 9000, 2
    # gathered rows M C_in s, one write per output row N C_out s, the
    # neighbour table 4 N V, the weights V C_in C_out s
    want = M * 32 * s + N * 64 * s + 4 * N * V + V * 32 * 64 * s
    assert bench.algo_bytes_step("subm_conv_fused", N, V, M, [(32, 64)], s, 0) == want
    # two layers add up; the backward pass adds each layer's input gradient (64 -> 32)
    two = bench.algo_bytes_step("subm_conv_fused", N, V, M, [(32, 64), (64, 64)], s, 0)
    assert two == want + (M * 64 * s + N * 64 * s + 4 * N * V + V * 64 * 64 * s)
    bwd = bench.algo_bytes_step("subm_conv_fused", N, V, M, [(32, 64)], s, 0, backward=True)
    assert bwd == want + (M * 64 * s + N * 32 * s + 4 * N * V + V * 64 * 32 * s)


def test_algorithmic_bytes_of_map_and_gradient_kernels():
    N, V, M, s = 1000, 27, 9000, 2
    lists = 8 * (M - N)  # the centre's tuples are implicit in a submanifold map
    assert bench.algo_bytes_step("kmap_build", N, V, M, [(32, 32)], s, 0) == 8 * N + 4 * N * V + lists
    assert bench.algo_bytes_step("hash_insert", N, V, M, [(32, 32)], s, 0) == 28 * N
    wg = bench.algo_bytes_step("subm_conv_wgrad", N, V, M, [(32, 64)], s, 0)
    assert wg == M * (32 + 64) * s + 4 * V * 32 * 64 + lists
    # a strided layer's map lists every tuple and has n_out rows
    n_out = 400
    assert bench.algo_bytes_step("kmap_build", N, V, M, [(32, 32)], s, 0, n_out=n_out) == \
        8 * n_out + 4 * n_out * V + 8 * M
    assert bench.algo_bytes_step("no_such_kernel", N, V, M, [(32, 32)], s, 0) is None
    # the tile-transposed table: table and row order read, table written
    assert bench.algo_bytes_step("tile_table", N, V, M, [(32, 32)], s, 0) == 8 * N * V + 4 * N
    assert "tile_table" in bench.MAP_KERNELS


def test_recorded_traffic_is_dropped_once_the_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// version 1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"k@w": {"source": "kernel.cu", "sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
                   "dram_bytes_per_launch": 1234}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k", "w") == 1234
    assert bench.recorded_traffic("k", "other") is None
    src.write_text("// version 2\n")
    assert bench.recorded_traffic("k", "w") is None


def test_committed_traffic_records_name_existing_sources():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, r in d.items():
        assert os.path.exists(os.path.join(bench.ROOT, r["source"])), key
        assert r["dram_bytes_per_launch"] > 0 and len(r["sha256"]) == 64
        assert r["command"].startswith("ncu ") and "--clock-control none" in r["command"], key


def test_clock_summary_reads_reasons():
    c = bench.ClockSampler("00000000:01:00.0")
    for ln, ph in [("2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active", "timed"),
                   ("1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active", "timed"),
                   ("garbage", "timed")]:
        s = c.parse_smi_line(ln, ph)
        if s:
            c.samples.append(s)
    s = c.summary(("timed",), min_samples=1)
    assert s["samples"] == 2 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz"] == (2070.0 + 1980.0) / 2


def test_clock_summary_widens_to_the_load_phases_when_the_timed_steps_are_short():
    c = bench.ClockSampler("00000000:01:00.0")
    c.samples += [("warmup", 2000.0, 2070.0, frozenset())] * 30
    c.samples += [("timed", 2070.0, 2070.0, frozenset({"sw_power_cap"}))] * 3
    c.samples += [("idle", 500.0, 2070.0, frozenset({"hw_slowdown"}))] * 50
    s = c.summary(("timed",), 10, ("warmup", "timed"))
    # too few timed samples: the summary covers warm-up + timed, never idle
    assert s["samples"] == 33 and s["samples_timed"] == 3 and s["window"] == ["warmup", "timed"]
    assert s["sm_mhz"] == 2000.0 and s["reasons"] == ["sw_power_cap"]
    s = c.summary(("timed",), 3, ("warmup", "timed"))
    assert s["samples"] == 3 and s["window"] == ["timed"] and s["sm_mhz"] == 2070.0


def test_default_workload_is_the_largest_single_gpu_configuration(monkeypatch):
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert a.workload == 4 and a.gpus == 1 and a.scale == 1.0
    from submanifold_sparse_convolution_hash_gb300 import scenes
    w, _ = scenes.workload(4, scale=0.001)
    assert w.K == 5 and w.channels == (128, 128) and w.dtype == "bf16"


def test_map_build_time_counts_every_map_kernel():
    """Every named launch of the hash / map source that runs inside a map
    build (not the export, query or coordinate read-back helpers) is in the
    bench's map-build kernel set."""
    import re
    src = open(os.path.join(bench.ROOT, "submanifold_sparse_convolution_hash_gb300", "csrc", "hash_kmap.cu")).read()
    names = set(re.findall(r'SC_LAUNCH\("([a-z_0-9]+)"', src))
    helpers = {"hash_query", "hash_coords", "kmap_compact", "kmap_unpermute"}
    assert names - helpers <= set(bench.MAP_KERNELS), sorted(names - helpers - set(bench.MAP_KERNELS))
    assert not set(bench.MAP_KERNELS) & helpers


def test_unique_bytes_model_is_the_stricter_one():
    N, V, M, s = 1000, 27, 9000, 2
    # rows once: N C_in s in, N C_out s out, the neighbour table, the weights
    assert bench.unique_bytes_op("conv", N, V, M, 32, 64, s) == N * 32 * s + N * 64 * s + 4 * N * V + V * 32 * 64 * s
    assert bench.unique_bytes_op("wgrad", N, V, M, 32, 64, s) == N * (32 + 64) * s + 8 * (M - N) + 4 * V * 32 * 64
    fwd = bench.unique_bytes_step(N, V, M, [(32, 64)], s)
    assert fwd < bench.algo_bytes_step("subm_conv_fused", N, V, M, [(32, 64)], s, 0)
    bwd = bench.unique_bytes_step(N, V, M, [(32, 64)], s, backward=True)
    assert bwd == fwd + bench.unique_bytes_op("conv", N, V, M, 64, 32, s) + bench.unique_bytes_op("wgrad", N, V, M, 32,
                                                                                                   64, s)
    # a strided layer: n_out output rows, every tuple listed
    assert bench.unique_bytes_op("conv", N, V, M, 32, 32, s, n_out=400) == \
        N * 32 * s + 400 * 32 * s + 4 * 400 * V + V * 32 * 32 * s
    assert bench.unique_bytes_op("wgrad", N, V, M, 32, 32, s, n_out=400) == \
        N * 32 * s + 400 * 32 * s + 8 * M + 4 * V * 32 * 32


def test_map_build_hbm_fraction():
    # two modelled kernels of 1 ms each per step over 4 steps, one unmodelled
    prof = {"hash_insert": (4, 4.0), "kmap_build": (4, 4.0), "sig_count": (4, 40.0), "subm_conv_fused": (4, 1.0)}
    nbytes = {"hash_insert": 1e9, "kmap_build": 3e9}
    frac = bench.map_build_hbm_frac(prof, 4, nbytes.get, 1000.0)
    assert frac == round(4e9 / 2e-3 / 1e12, 4)  # 2 TB/s of 1 TB/s
    assert bench.map_build_hbm_frac({"subm_conv_fused": (1, 1.0)}, 1, nbytes.get, 1000.0) is None


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference times the CPU oracle on this host and prints
    the contract's JSON line (no GPU involved)."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "Mvoxels/s"
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True and d["steps"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "Mvoxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cfg = d["config"]
    assert cfg["workload"].startswith("lidar_") and cfg["layers"] == [[32, 32]] and cfg["K"] == 3
    # |M| counted from the oracle's map; the same keys the GPU arm's config carries
    from submanifold_sparse_convolution_hash_gb300 import scenes
    import oracle
    w, s = scenes.workload(1)
    assert cfg["N"] == s.n and cfg["map_size"] == int((oracle.kmap(s.coords, 3, 3, s.dims) >= 0).sum())
    assert cfg == bench.workload_config(w, s, cfg["map_size"], 1)
    assert "hash + map + layers" in cb["sample"]


def test_the_two_oracle_timings_estimate_the_same_quantity():
    """cpu_baseline (one large sample) and the reference arm's steps (small
    samples) time the oracle the same way: the coordinate table's build once,
    the sampled rows against a kept table, scaled to N.  Their estimates of
    the whole-scene rate agree within timing noise."""
    import statistics
    w, s = bench.make_workload(1, 0, 0.3)
    cb = bench.cpu_oracle_sampled(w, s, 1.0)
    table, ins, rows, t_table = bench.oracle_sampled_plan(w, s, 0.02)
    ref = statistics.median(s.n / bench.oracle_sampled_pass(w, s, table, ins, rows, t_table) / 1e6
                            for _ in range(9))
    table.close()
    assert len(rows) < s.n
    assert 0.6 < ref / cb["value"] < 1.6, (ref, cb["value"])


def test_tile_table_policy():
    """auto: only when one map serves several layers; never with column
    splitting or above 128 offsets (the library refuses those)."""
    assert bench.use_tile_table("auto", 8, 27, False)
    assert not bench.use_tile_table("auto", 1, 27, False)
    assert not bench.use_tile_table("auto", 1, 125, False)
    assert bench.use_tile_table("on", 1, 125, False)
    assert not bench.use_tile_table("on", 8, 343, False)
    assert not bench.use_tile_table("on", 8, 27, True)
    assert not bench.use_tile_table("off", 8, 27, False)
