#!/usr/bin/env python3
"""Benchmark of the submanifold sparse convolution hot path on one GPU.

One step = one pass of the whole path over one synthetic scene:
    sc_hash_build -> sc_kmap_build -> sc_subm_conv_fwd (every layer)
By default on the largest single-GPU workload: 2048x2048x64 grid, ~2M
voxels on synthetic surfaces, 5x5x5 kernel (125 offsets), C_in = C_out =
128, bf16 features and weights, fp32 accumulation.  --workload 0..3 selects
the others (2D 200 cells; LiDAR ~100k C 32; indoor ~1M C 64; four LiDAR
scans with an 8-layer stack 32 -> 256).

Prints one JSON line.  `value` is Mvoxels/s over the timed steps with inputs
resident in device memory and L2 flushed (a 256 MB write) before every step,
outside the per-step CUDA events.  `e2e` is the same metric with pinned host
inputs copied in and the output copied back inside every step, through the
public API calls: asynchronous map builds with each step's error status
checked, double-buffered so one step's copies overlap the previous step's
layers.  `roofline` reports the dominant kernel's
algorithmic bytes over its average event-timed launch duration against the
measured HBM copy bandwidth.  `cpu_baseline` times the CPU oracle on a
bounded sample of the same scene on this host's cores (the coordinate table
over every point, then the map rows and fp64 outputs of evenly spaced rows,
scaled to the scene).  `clocks` summarises read-only NVML samples of the SM
clock and its throttle reasons, taken from the first warm-up step to the end
of the timed steps.

--layer-type regular | strided replaces the workload's layer stack by its
first layer as a dilating (stride 1) or strided layer: a step is then
sc_hash_build -> sc_hash_build_conv_out -> sc_kmap_build_conv -> the layer.

--impl reference times the CPU oracle alone (the reference arm).
Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica on
its own scene (replicas only; no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
# the kernels of the map build (hash insert, output set, row order, map,
# signature sort, the fused layer's tile table): their event-timed sum is the
# step's map-build kernel time
MAP_KERNELS = ("hash_insert", "out_mark", "out_count", "out_scan", "out_number", "order_count", "order_partials",
               "order_apply", "order_scatter", "kmap_clear", "kmap_build", "kmap_masks", "sig_count", "sig_partials",
               "sig_scan", "sig_scatter", "sig_present", "tile_table")
sys.path.insert(0, ROOT)

METRIC = "subm-conv layer effective TFLOP/s, Mvoxels/s & % roofline; kernel-map build ms"
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4,
                    help="0..4; the default, 4, is the largest single-GPU configuration (2M voxels, 5x5x5, C 128 bf16)")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="shrink the scene (N and grid) for small profiling captures; the workload name records it")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extras of the default line: the training step and the stride-2 layer of the same "
                         "workload, each measured by a child run of this script")
    ap.add_argument("--backward", action="store_true",
                    help="a training step: after the forward layers, the input and weight gradients of every "
                         "layer (a seeded output gradient, ReLU masks applied)")
    ap.add_argument("--variant", choices=["fused", "ws", "simt", "split"], default=None,
                    help="run every layer with this variant instead of the measured choice")
    ap.add_argument("--layer-type", choices=["submanifold", "regular", "strided"], default="submanifold",
                    help="regular: a dilating layer (stride 1, output set grown by the kernel window); strided: "
                         "a layer on the grid coarsened by --stride; both run the workload's first layer only")
    ap.add_argument("--stride", type=int, default=2, help="stride of --layer-type strided")
    ap.add_argument("--kmap-half", action="store_true",
                    help="build submanifold maps with the half probe (mirror symmetry) instead of the full probe")
    ap.add_argument("--kmap-sort", choices=["auto", "on", "off"], default="auto",
                    help="signature sort of the map's rows: the library's default (auto: at 262,144 rows and more), "
                         "always, or never")
    ap.add_argument("--kmap-split", action="store_true",
                    help="also build the row orders of column splitting (K^ndim <= 32), so each layer's measured "
                         "variant choice includes the split kernel")
    ap.add_argument("--kmap-tile-table", choices=["auto", "on", "off"], default="auto",
                    help="build the fused layer's tile-transposed index table with the map (SC_KMAP_TILE_TABLE): "
                         "auto = when one map serves several layers (the eight-layer stack), else not")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def make_workload(idx: int, rank: int, scale: float = 1.0):
    from submanifold_sparse_convolution_hash_gb300 import scenes
    return scenes.workload(idx, scale=scale, replica=rank)  # each replica draws its own scene of the recipe


def layer_tensors(w, s):
    from submanifold_sparse_convolution_hash_gb300 import scenes
    V = w.K ** s.ndim
    c_in, c_out = w.channels[0], w.channels[1]
    f = scenes.features(w.seed, s.n, c_in)
    W = scenes.weights(w.seed, V, c_in, c_out, std=1.0 if w.w_std_unit else None)
    return f, W


# ------------------------------------------------------------- algorithmic bytes --
def algo_bytes_step(kernel: str, N: int, V: int, M: int, layers, s: int, ntiles: int, backward: bool = False,
                    n_out: int | None = None):
    """Bytes a kernel must move at minimum in one step (summed over its
    launches in that step); None for kernels without a stated model.  With
    `backward`, the convolution kernels also run each layer's input gradient
    (a layer from c_out to c_in channels).  n_out: output rows of a regular /
    strided layer (its map lists every tuple, the centre's included)."""
    No = N if n_out is None else n_out
    lists = 8 * (M - N) if n_out is None else 8 * M
    conv_layers = list(layers) + ([(co, ci) for ci, co in layers] if backward else [])
    conv = sum(M * ci * s + No * co * s + 4 * No * V + V * ci * co * s for ci, co in conv_layers)
    table = {
        # coords in; row keys out; one row slot per point
        "hash_insert": 16 * N + 8 * N + 4 * N,
        # row keys in; neighbour table and (in, out) lists out
        "kmap_build": 8 * No + 4 * No * V + lists,
        # the half probe's clear of the columns before the centre, and its mask
        # pass (reads the table once, writes the tile masks)
        "kmap_clear": 4 * No * ((V - 1) // 2),
        "kmap_masks": 4 * No * V + 16 * ((No + 127) // 128),
        # the fused layer's tile-transposed table: the table and the row
        # order read, the same entries written in tile order
        "tile_table": 8 * No * V + 4 * No,
        "order_count": 8 * N,
        "order_scatter": 8 * N + 4 * N,
        "pack_weights": sum(2 * V * ci * co * s for ci, co in conv_layers),
        # gathered neighbour rows + one write per output row + neighbour table + weights
        "subm_conv_fused": conv,
        "subm_conv_split": conv,
        "subm_conv_simt": conv,
        # weight gradient: both gathered rows of every tuple, the list indices
        # (the centre list is implicit), the fp32 gradient written once
        "subm_conv_wgrad": sum(M * (ci + co) * s + 4 * V * ci * co for ci, co in layers) + lists * len(layers),
    }
    return table.get(kernel)


def unique_bytes_op(op: str, N: int, V: int, M: int, ci: int, co: int, s: int, n_out: int | None = None):
    """The stricter byte model of one layer op: every input row, output row,
    neighbour-table entry and weight moved once (the algorithmic model counts
    a gathered row once per tuple).  op "conv": a layer from ci to co channels
    (an input gradient is the layer from co to ci); op "wgrad": a weight
    gradient (both row sets once, the lists, the fp32 gradient written)."""
    No = N if n_out is None else n_out
    if op == "conv":
        return N * ci * s + No * co * s + 4 * No * V + V * ci * co * s
    lists = 8 * (M - N) if n_out is None else 8 * M
    return N * ci * s + No * co * s + lists + 4 * V * ci * co


def unique_bytes_step(N: int, V: int, M: int, layers, s: int, backward: bool = False, n_out: int | None = None):
    """unique_bytes_op summed over the layer ops of one step: each layer, and
    with `backward` its input gradient and weight gradient."""
    total = sum(unique_bytes_op("conv", N, V, M, ci, co, s, n_out) for ci, co in layers)
    if backward:
        total += sum(unique_bytes_op("conv", N, V, M, co, ci, s, n_out) + unique_bytes_op("wgrad", N, V, M, ci, co, s,
                                                                                        n_out) for ci, co in layers)
    return total


def map_build_hbm_frac(prof_all: dict, steps: int, bytes_of, hbm_gbs: float):
    """Algorithmic bytes over time of the map-build kernels that have a byte
    model (prof_all: name -> (launches, total ms) over `steps` steps;
    bytes_of(name): bytes per step or None), as a fraction of `hbm_gbs`."""
    b = t_ms = 0.0
    for k in MAP_KERNELS:
        if k not in prof_all:
            continue
        kb = bytes_of(k)
        if kb:
            b += kb
            t_ms += prof_all[k][1] / steps
    return round(b / (t_ms / 1e3) / (hbm_gbs * 1e9), 4) if t_ms > 0 else None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu
    summary, or None if absent or taken on a different version of the
    kernel's source file."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{kernel}@{workload}")
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != d["sha256"]:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    """Read-only sampling of the GPU's SM clock, power draw and clock-event
    (throttle) reasons while the bench runs.

    In-process NVML (libnvidia-ml) every `period` seconds from a thread; the
    device is found by its PCI bus id (else its UUID), never by index, so
    CUDA_VISIBLE_DEVICES cannot point the sampler at another GPU.  Without
    NVML it runs `nvidia-smi -i <bus id> -lms 100`.  Every sample carries the
    phase set by mark() (warm-up, breakdown, timed ...).  Queries only:
    nothing here changes a clock, a power limit or any other setting."""

    # clock-event reason bits of NVML's current-reasons mask
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
    SMI_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, bus_id: str | None = None, uuid: str | None = None, period: float = 0.005):
        self.bus_id, self.uuid, self.period = bus_id, uuid, period
        self.samples = []  # (phase, sm_mhz, sm_max_mhz, reasons frozenset)
        self.phase = "idle"
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None

    @staticmethod
    def for_torch_device(dev_index: int, period: float = 0.005):
        import torch
        p = torch.cuda.get_device_properties(dev_index)
        bus = None
        if hasattr(p, "pci_bus_id"):
            bus = f"{getattr(p, 'pci_domain_id', 0):08X}:{p.pci_bus_id:02X}:{getattr(p, 'pci_device_id', 0):02X}.0"
        uuid = str(getattr(p, "uuid", "")) or None
        return ClockSampler(bus, uuid, period)

    def mark(self, phase: str):
        self.phase = phase

    # ---- NVML
    def _nvml_open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.bus_id:
            ok = nv.nvmlDeviceGetHandleByPciBusId_v2(self.bus_id.encode(), ctypes.byref(h)) == 0
        if not ok and self.uuid:
            for u in (self.uuid, "GPU-" + self.uuid):
                if nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        if not ok:
            raise OSError("NVML: device not found by bus id or UUID")
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return nv, h, reasons_fn

    def _nvml_loop(self, nv, h, reasons_fn):
        import ctypes
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and  # 1 = SM clock
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons_fn(h, ctypes.byref(rs)) == 0):
                r = frozenset(nm for bit, nm in self.REASONS.items() if rs.value & bit)
                self.samples.append((self.phase, float(clk.value), float(mx.value), r))
            time.sleep(self.period)

    # ---- nvidia-smi fallback
    def parse_smi_line(self, line: str, phase: str = "idle"):
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            return None
        try:
            sm, mx = float(parts[0]), float(parts[1])
        except ValueError:
            return None
        r = frozenset(nm for nm, v in zip(self.SMI_NAMES, parts[4:8]) if v.lower() == "active")
        return (phase, sm, mx, r)

    def _smi_loop(self):
        for line in self._proc.stdout:
            s = self.parse_smi_line(line, self.phase)
            if s:
                self.samples.append(s)

    def __enter__(self):
        try:
            nv, h, fn = self._nvml_open()
            self.source = "nvml"
            self._t = threading.Thread(target=self._nvml_loop, args=(nv, h, fn), daemon=True)
            self._t.start()
            return self
        except (OSError, AttributeError):
            pass
        if self.bus_id or self.uuid:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", self.bus_id or ("GPU-" + self.uuid), f"--query-gpu={self.SMI_FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self._t = threading.Thread(target=self._smi_loop, daemon=True)
                self._t.start()
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._t:
            self._t.join(timeout=5)

    def summary(self, phases=("timed",), min_samples: int = 10, load_phases=None):
        """Median SM MHz, max SM MHz and the union of the reasons over the
        samples of `phases`; if those are fewer than `min_samples`, over the
        samples of every phase in `load_phases` (all GPU-busy phases), which
        the `window` key then names."""
        def pick(ph):
            return [s for s in self.samples if s[0] in ph]
        sel, window = pick(phases), list(phases)
        if len(sel) < min_samples and load_phases:
            sel, window = pick(load_phases), list(load_phases)
        out = {"samples": len(sel), "samples_timed": len(pick(phases)), "window": window, "source": self.source}
        if not sel:
            out.update({"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
            return out
        out.update({"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": max(s[2] for s in sel),
                    "reasons": sorted(set().union(*(s[3] for s in sel)))})
        return out


# ---------------------------------------------------------------------- CPU --
def oracle_layer_inputs(w, s):
    """fp64 (feats, W) of every layer of the workload for timing the oracle:
    the first layer's seeded inputs, and seeded features of the right width
    for the later layers (their values do not change the oracle's time)."""
    from submanifold_sparse_convolution_hash_gb300 import scenes
    V = w.K ** s.ndim
    layers = list(zip(w.channels[:-1], w.channels[1:]))

    def rnd(a):
        return a.astype(np.float64)

    feats_by_width = {}
    out = []
    for li, (ci, co) in enumerate(layers):
        if li == 0:
            f = rnd(scenes.features(w.seed, s.n, ci))
            W = rnd(scenes.weights(w.seed, V, ci, co, std=1.0 if w.w_std_unit else None))
        else:
            if ci not in feats_by_width:
                feats_by_width[ci] = rnd(scenes.features(w.seed + 50 + ci, s.n, ci))
            f = feats_by_width[ci]
            W = rnd(scenes.weights(w.seed + li, V, ci, co))
        out.append((f, W))
    return out


def oracle_sampled_plan(w, s, seconds: float):
    """Sizes a bounded sample of the oracle's work on the workload: the
    coordinate table over all N, timed on its own (median of three builds),
    and evenly spaced output rows whose layer outputs take about `seconds`
    against a table built once.  Returns (table, inputs, rows, t_table)."""
    import oracle
    oracle.build()
    ins = oracle_layer_inputs(w, s)
    t_tab = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.hash_only(s.coords, s.ndim, w.K, s.dims)
        t_tab.append(time.perf_counter() - t0)
    t_table = statistics.median(t_tab)
    table = oracle.Table(s.coords, s.ndim, w.K, s.dims)
    # at least 64 rows per thread, so every thread of the oracle's loop works
    kmin = min(s.n, 64 * max(1, oracle.max_threads()))
    probe = np.linspace(0, s.n - 1, kmin).astype(np.int64)
    per_row = 0.0
    for f, W in ins:
        t0 = time.perf_counter()
        table.subm_conv(f, W, rows=probe)
        per_row += (time.perf_counter() - t0) / len(probe)
    k = int(max(kmin, min(s.n, seconds / max(per_row, 1e-12))))
    rows = np.linspace(0, s.n - 1, k).astype(np.int64)
    return table, ins, rows, t_table


def oracle_sampled_pass(w, s, table, ins, rows, t_table) -> float:
    """One oracle pass on the sample, scaled to the whole scene (seconds):
    t_table (the coordinate table over all N) plus, layer by layer, the time
    of the sampled rows' V neighbour lookups (their map rows) and fp64
    outputs against the kept table, scaled by N / k."""
    total = t_table
    for f, W in ins:
        t0 = time.perf_counter()
        table.subm_conv(f, W, rows=rows)
        total += (time.perf_counter() - t0) * s.n / len(rows)
    return total


def oracle_sample_text(w, s, k: int) -> str:
    V = w.K ** s.ndim
    nl = len(w.channels) - 1
    return (f"coordinate table (hash) over all N={s.n}, its build timed on its own (median of 3, t_table); "
            f"then for {k} evenly spaced output rows the row's {V} neighbour lookups (its map row) and its "
            f"fp64 output in each of the {nl} layer(s), against that table; time scaled to N as "
            f"t_table + t_rows * N / {k}; phases: hash + map + layers, as in the GPU step")


def cpu_oracle_sampled(w, s, seconds: float):
    """cpu_baseline of the GPU line: the oracle on a bounded sample."""
    import oracle
    t0 = time.perf_counter()
    table, ins, rows, t_table = oracle_sampled_plan(w, s, seconds)
    t = oracle_sampled_pass(w, s, table, ins, rows, t_table)
    table.close()
    el = time.perf_counter() - t0
    return {"value": round(s.n / t / 1e6, 4), "unit": "Mvoxels/s", "cores": oracle.max_threads(),
            "host_cpus": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": oracle_sample_text(w, s, len(rows)) + f"; one pass, {el:.1f} s of CPU work"}


def cpu_oracle_run(s, K, f, W, seconds: float, stride: int = 0):
    """Times the oracle on the full scene (regular / strided layer: output
    set + map + layer; stride > 0), repeated to ~`seconds`."""
    import oracle
    f64 = f.astype(np.float64)
    W64 = W.astype(np.float64)
    t0 = time.perf_counter()
    passes = 0
    while True:
        oc = oracle.conv_out_coords(s.coords, s.ndim, K, stride, s.dims)
        oracle.conv_kmap(s.coords, oc, s.ndim, K, stride, s.dims)
        oracle.sparse_conv(s.coords, oc, f64, W64, s.ndim, K, stride, s.dims)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds or el * (passes + 1) / passes > 3 * seconds:
            break
    return {"value": s.n * passes / el / 1e6, "unit": "Mvoxels/s", "cores": oracle.max_threads(),
            "host_cpus": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"full scene (N={s.n}) x {passes} pass(es): output set + map + fp64 layer, {el:.1f} s"}


def use_tile_table(mode: str, n_layers: int, V: int, split: bool) -> bool:
    """Whether the map is built with the fused layer's tile table
    (SC_KMAP_TILE_TABLE): "on", "off", or "auto" = when one map serves more
    than one layer (the pass costs more than a single layer gains).  Never
    with column splitting or above 128 offsets, which the library refuses."""
    if split or V > 128:
        return False
    return mode == "on" or (mode == "auto" and n_layers > 1)


def workload_config(w, s, M: int, world: int, layer_type: str = "submanifold", stride: int = 1,
                    n_out: int | None = None, backward: bool = False, scale: float = 1.0):
    """The line's `config`: what the workload is, identical in both arms."""
    cfg = {"workload": w.name if scale == 1.0 else f"{w.name}_scale{scale:g}", "N": s.n, "map_size": int(M),
           "K": w.K, "ndim": s.ndim, "dims": list(s.dims), "layers": [list(l) for l in zip(w.channels[:-1], w.channels[1:])],
           "layer_type": layer_type, "stride": stride, "N_out": int(s.n if n_out is None else n_out),
           "pass": "forward+backward" if backward else "forward",
           "l2": "GPU arm: flushed before every step (256 MB write, outside the events); CPU arm: no flush",
           "parallelism": "replicas" if world > 1 else "single"}
    if layer_type != "submanifold":
        cfg["layers"] = cfg["layers"][:1]
    return cfg


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this host's cores.

    Each step is one oracle pass on a bounded sample of the workload, the
    same estimate as the GPU line's cpu_baseline: the coordinate table's
    build time over the whole scene (timed once, before the steps), plus,
    for a fixed set of evenly spaced output rows, their map rows and fp64
    outputs in every layer against that table, scaled to the whole scene
    (oracle_sampled_pass).  The sample is sized so that warm-up plus timed
    steps take a few minutes.  |M| for the config is counted from the
    oracle's own map (outside the timed steps).
    """
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w, s = make_workload(args.workload, 0, args.scale)
    M = int((oracle.kmap(s.coords, s.ndim, w.K, s.dims) >= 0).sum())
    budget = 150.0 / max(1, args.steps + args.warmup)
    table, ins, rows, t_table = oracle_sampled_plan(w, s, budget)
    for _ in range(args.warmup):
        oracle_sampled_pass(w, s, table, ins, rows, t_table)
    times = [oracle_sampled_pass(w, s, table, ins, rows, t_table) for _ in range(args.steps)]
    table.close()
    ms = 1e3 * statistics.mean(times)
    value = s.n / (ms / 1e3) / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "Mvoxels/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, s, M, world, scale=args.scale),
        "cpu_baseline": {"value": round(value, 4), "unit": "Mvoxels/s", "cores": oracle.max_threads(),
                         "host_cpus": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": oracle_sample_text(w, s, len(rows))},
        "e2e": {"value": round(value, 4), "unit": "Mvoxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- GPU --
def reduce_over_ranks(total_s: float, n_units: int, device, world: int):
    """(slowest rank's timed seconds, voxels processed by all ranks).  Each
    rank is an independent replica; this is the only collective and it runs
    after the timed region."""
    if world <= 1:
        return float(total_s), float(n_units)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(total_s), float(n_units)], dtype=torch.float64, device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(tmax[0].item()), float(t[1].item())


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from submanifold_sparse_convolution_hash_gb300 import binding as sc

    w, s = make_workload(args.workload, rank, args.scale)
    from submanifold_sparse_convolution_hash_gb300 import scenes as sc_scenes
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
    esize = 4 if w.dtype == "f32" else 2
    V = w.K ** s.ndim
    layers = list(zip(w.channels[:-1], w.channels[1:]))  # (c_in, c_out) of each layer on the one map
    general = args.layer_type != "submanifold"
    if general:
        layers = layers[:1]
        if args.backward:
            raise SystemExit("--backward runs submanifold layers only (the input gradient of a regular or strided "
                             "layer needs the transposed map)")
    conv_stride = args.stride if args.layer_type == "strided" else 1
    f_np, W0 = layer_tensors(w, s)
    Ws = [torch.from_numpy(W0).to(tdt).to(dev)]
    for li, (ci, co) in enumerate(layers[1:], start=1):
        Ws.append(torch.from_numpy(sc_scenes.weights(w.seed + li, V, ci, co)).to(tdt).to(dev))
    c_in, c_out = layers[0]
    coords = torch.from_numpy(s.coords).to(dev)
    feats = torch.from_numpy(f_np).to(tdt).to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    sort_arg = {"auto": None, "on": True, "off": False}[args.kmap_sort]
    tile_table = use_tile_table(args.kmap_tile_table, len(layers), V, args.kmap_split)

    def build_map(c, sync):
        """hash -> kernel map (submanifold), or hash -> output set -> map
        (regular / strided; the output set's count is read on the host)."""
        h = sc.sc_hash_build(c)
        if not general:
            return (h,), sc.sc_kmap_build(h, s.ndim, w.K, s.dims, sync=sync, half=args.kmap_half,
                                          split=args.kmap_split, sort=sort_arg, tile_table=tile_table)
        ho = sc.sc_hash_build_conv_out(h, s.ndim, w.K, conv_stride, s.dims)
        return (h, ho), sc.sc_kmap_build_conv(h, ho, s.ndim, w.K, conv_stride, s.dims, sync=sync, sort=sort_arg,
                                              tile_table=tile_table)

    # variant of each layer chosen from measured time on this map
    hs0, m0 = build_map(coords, True)
    M = m0.map_size()
    n_out = m0.n
    outs = [torch.empty((n_out, co), dtype=tdt, device=dev) for _, co in layers]
    variants = []
    x = feats
    for li, W in enumerate(Ws):
        relu = li + 1 < len(Ws)
        if args.variant:
            variants.append(args.variant)
        else:
            variants.append(sc.sc_subm_conv_tune(m0, x, W, out=outs[li], relu=relu, reps=5))
        x = outs[li]
    ntiles = (s.n + 31) // 32

    if args.backward:
        gout_last = torch.from_numpy(sc_scenes.features(w.seed + 99, s.n, layers[-1][1])).to(tdt).to(dev)
        gins = [torch.empty((s.n, ci), dtype=tdt, device=dev) for ci, _ in layers]
        dWs = [torch.empty_like(W) for W in Ws]

    def step():
        h, m = build_map(coords, False)
        xin = feats
        for li, W in enumerate(Ws):
            sc.sc_subm_conv_fwd(m, xin, W, out=outs[li], relu=li + 1 < len(Ws), variant=variants[li])
            xin = outs[li]
        if args.backward:
            g = gout_last
            for li in range(len(Ws) - 1, -1, -1):
                if li + 1 < len(Ws):  # ReLU after this layer: pass the gradient where the output was positive
                    g = g * (outs[li] > 0)
                sc.sc_subm_conv_bwd_weight(m, feats if li == 0 else outs[li - 1], g, dW=dWs[li])
                sc.sc_subm_conv_bwd_data(m, g, Ws[li], gin=gins[li], variant=variants[li])
                g = gins[li]
        return h, m

    # clocks are sampled from the first warm-up step to the end of the timed
    # steps, each sample tagged with its phase
    clk = ClockSampler.for_torch_device(dev.index if dev.index is not None else torch.cuda.current_device())
    clk.__enter__()
    clk.mark("warmup")
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    # per-kernel breakdown from an untimed pass with every launch bracketed;
    # it also names the dominant kernel, the only one bracketed while timing
    keep = []
    sc.profile_reset()
    sc.profile_only(None)
    sc.profile_enable(True)
    bd_steps = min(args.steps, 100)
    clk.mark("breakdown")
    for _ in range(bd_steps):
        flush.zero_()
        keep.append(step())
        if len(keep) > 4:
            keep.pop(0)
    torch.cuda.synchronize()
    sc.profile_enable(False)
    prof_all = sc.profile_collect()
    keep.clear()
    dom = max(prof_all, key=lambda k: prof_all[k][1])

    # each forward layer alone (events around its call on one map, flushed
    # L2 before every layer), untimed pass: per-layer roofline fractions
    layer_detail = []
    if len(layers) > 1 and not args.backward:
        hs_l, m_l = build_map(coords, False)
        reps = min(bd_steps, 20)
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
              for _ in layers]
        for rep in range(reps):
            xin = feats
            for li, W in enumerate(Ws):
                flush.zero_()
                ev[li][rep][0].record(stream)
                sc.sc_subm_conv_fwd(m_l, xin, W, out=outs[li], relu=li + 1 < len(Ws), variant=variants[li])
                ev[li][rep][1].record(stream)
                xin = outs[li]
        torch.cuda.synchronize()
        for li, (ci, co) in enumerate(layers):
            t_l = statistics.median(a.elapsed_time(b) for a, b in ev[li]) / 1e3
            b_l = algo_bytes_step("subm_conv_fused", s.n, V, M, [(ci, co)], esize, ntiles, False, None)
            roof_l = max(2.0 * M * ci * co / (load_peaks()["bf16_tflops"] * 1e12), b_l / (load_peaks()["hbm_gbs"] * 1e9))
            layer_detail.append({"c_in": ci, "c_out": co, "us": round(t_l * 1e6, 2),
                                 "roofline_frac": round(roof_l / t_l, 4), "variant": variants[li]})
        del hs_l, m_l

    # map build end to end (sc_hash_build .. sc_kmap_build, events on the
    # stream, no per-kernel brackets), untimed pass
    map_e2e = []
    clk.mark("map_build")
    for _ in range(bd_steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h, m = build_map(coords, False)
        e1.record(stream)
        keep.append((h, m, e0, e1))
        if len(keep) > 4:
            keep.pop(0)
        map_e2e.append((e0, e1))
    torch.cuda.synchronize()
    keep.clear()
    map_e2e_ms = statistics.median(a.elapsed_time(b) for a, b in map_e2e)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    keep = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sc.profile_reset()
    sc.profile_only(dom)
    sc.profile_enable(True)
    launches0 = sc.launch_count()
    clk.mark("timed")
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        keep.append(step())
        ends[i].record(stream)
        if len(keep) > 4:
            keep.pop(0)
    torch.cuda.synchronize()
    clk.mark("after")
    clk.__exit__(None, None, None)
    launches = sc.launch_count() - launches0
    sc.profile_enable(False)
    sc.profile_only(None)
    prof = sc.profile_collect()  # the dominant kernel's launches inside the timed region
    keep.clear()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_s = sum(step_ms) / 1e3
    total_s, n_total = reduce_over_ranks(total_s, s.n, dev, world)
    # error status of the last map (outside the timed region)
    h_chk, m_chk = step()
    m_chk.check()
    torch.cuda.synchronize()

    value = n_total * args.steps / total_s / 1e6
    ms_per_step = 1e3 * total_s / args.steps
    flops = sum(2.0 * M * ci * co for ci, co in layers) * (3 if args.backward else 1)
    per_kernel = {}
    tot_all = sum(v[1] for v in prof_all.values()) or 1.0
    for k, (n_l, tot) in prof_all.items():
        per_kernel[k] = {"launches_per_step": round(n_l / bd_steps, 3), "avg_us": round(1e3 * tot / max(n_l, 1), 3),
                         "share": round(tot / tot_all, 4)}
    # the layers' kernels: the convolution kernels, and the weight pack of a
    # layer that packs its weights (the weight-stationary and CUDA-core
    # variants; the fused kernel reads W's slices by TMA and launches none)
    conv_k = [k for k in prof_all if k.startswith("subm_conv") or k in ("pack_weights", "cast_out", "wgrad_cast")]
    conv_ms = sum(prof_all[k][1] for k in conv_k) / bd_steps
    map_ms = sum(prof_all[k][1] for k in MAP_KERNELS if k in prof_all) / bd_steps
    peaks = load_peaks()
    ab_step = algo_bytes_step(dom, s.n, V, M, layers, esize, ntiles, args.backward, n_out if general else None)
    launches_per_step = prof[dom][0] / args.steps
    ab = ab_step / launches_per_step if ab_step else None
    avg_s = prof[dom][1] / prof[dom][0] / 1e3
    achieved = ab / avg_s / 1e9 if ab else None
    roofline = {"kernel": dom, "launches_timed": prof[dom][0], "bound": "hbm", "achieved": round(achieved, 1) if achieved else None,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4) if achieved else None,
                "traffic": recorded_traffic(dom, w.name), "peak_source": f"{peaks['source']} hbm_gbs",
                "algorithmic_bytes_per_launch": ab}
    # each layer op's roofline time: the slower of its FLOPs at tensor peak
    # and its algorithmic bytes at HBM bandwidth; summed over the ops of a
    # step (forward layers; with --backward also their input and weight
    # gradients)
    def roof_s(kernel, ci, co):
        return max(2.0 * M * ci * co / (peaks["bf16_tflops"] * 1e12),
                   algo_bytes_step(kernel, s.n, V, M, [(ci, co)], esize, ntiles, False, n_out if general else None)
                   / (peaks["hbm_gbs"] * 1e9))
    conv_roof_s = sum(roof_s("subm_conv_fused", ci, co) for ci, co in layers)
    if args.backward:
        conv_roof_s += sum(roof_s("subm_conv_fused", co, ci) + roof_s("subm_conv_wgrad", ci, co) for ci, co in layers)
    # the same with the stricter unique-bytes model of each layer op
    def roof_unique_s(op, ci, co):
        return max(2.0 * M * ci * co / (peaks["bf16_tflops"] * 1e12),
                   unique_bytes_op(op, s.n, V, M, ci, co, esize, n_out if general else None) / (peaks["hbm_gbs"] * 1e9))
    conv_unique_s = sum(roof_unique_s("conv", ci, co) for ci, co in layers)
    if args.backward:
        conv_unique_s += sum(roof_unique_s("conv", co, ci) + roof_unique_s("wgrad", ci, co) for ci, co in layers)

    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "Mvoxels/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, s, M, world, args.layer_type, conv_stride, n_out, args.backward, args.scale),
        "run": {"variant": variants, "variant_choice": "given" if args.variant else "measured", "kmap_sync": False,
                "kmap_probe": "half (mirror symmetry)" if args.kmap_half else "full",
                "column_split_orders": bool(args.kmap_split), "kmap_sort": args.kmap_sort,
                "kmap_tile_table": bool(tile_table)},
        "layer_tflops": round(flops / (conv_ms / 1e3) / 1e12, 3) if conv_ms else None,
        "layer_ms": round(conv_ms, 5),
        "layer_roofline_frac": round(conv_roof_s / (conv_ms / 1e3), 4) if conv_ms else None,
        "layer_unique_roofline_frac": round(conv_unique_s / (conv_ms / 1e3), 4) if conv_ms else None,
        "kmap_build_hbm_frac": map_build_hbm_frac(
            prof_all, bd_steps,
            lambda k: algo_bytes_step(k, s.n, V, M, layers, esize, ntiles, args.backward, n_out if general else None),
            peaks["hbm_gbs"]),
        "kmap_build_ms": round(map_e2e_ms, 5),
        "kmap_build_kernels_ms": round(map_ms, 5),
        "roofline": roofline,
        "per_kernel": per_kernel,
        "per_kernel_source": f"untimed pass of {bd_steps} steps, every launch bracketed by CUDA events",
        "layers_detail": layer_detail or None,
        "gpu_launches": launches,
        "clocks": clk.summary(("timed",), 10, ("warmup", "breakdown", "map_build", "timed")),
    }

    # the child runs first: measured after the end-to-end run's 300 steps
    # (whose buffers and pooled maps this process still holds), the 2M-voxel
    # training step read 22.6 ms against 11.2 ms measured alone
    if not args.no_extras and rank == 0 and world == 1 and not args.backward and not general:
        torch.cuda.synchronize()
        line["extras"] = run_extras(args)
    if not args.no_e2e and rank == 0:
        line["e2e"] = run_e2e(args, w, s, f_np, Ws, tdt, dev, variants, world, build_map, n_out)
    if args.backward:
        # the weight gradient against its own algorithmic bytes (both gathered
        # rows of every tuple, the lists, the fp32 gradient)
        if "subm_conv_wgrad" in prof_all:
            t_w = prof_all["subm_conv_wgrad"][1] / 1e3 / bd_steps
            b_w = algo_bytes_step("subm_conv_wgrad", s.n, V, M, layers, esize, ntiles, False, None)
            line["wgrad_roofline_frac"] = round(b_w / t_w / (peaks["hbm_gbs"] * 1e9), 4)
    if not args.no_cpu_baseline and rank == 0:
        if general:
            line["cpu_baseline"] = cpu_oracle_run(s, w.K, feats.float().cpu().numpy(), W0, args.cpu_seconds,
                                                  conv_stride)
        else:
            line["cpu_baseline"] = cpu_oracle_sampled(w, s, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_extras(args):
    """The training step (--backward) and the stride-2 layer (--layer-type
    strided) of the same workload, each measured by a child run of this
    script with the same timing rules (L2 flushed per step, CUDA events),
    after this run's own timed steps.  Returns their key figures."""
    # up to 200 timed steps: a stride-2 step at 1M voxels is 0.5 ms (with its
    # host read-back of the output count), and 20 of them read up to 4x slow
    # from one host stall
    base = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", str(args.workload), "--scale",
            str(args.scale), "--steps", str(min(args.steps, 200)), "--warmup", str(args.warmup), "--no-e2e",
            "--no-cpu-baseline", "--no-extras"]
    keys = ("value", "ms_per_step", "layer_ms", "layer_roofline_frac", "layer_unique_roofline_frac",
            "wgrad_roofline_frac", "kmap_build_ms", "clocks")
    out = {}
    for name, extra in (("training_step", ["--backward"]), ("stride2_layer", ["--layer-type", "strided"])):
        try:
            r = subprocess.run(base + extra, capture_output=True, text=True, timeout=900, cwd=ROOT)
            lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
            if r.returncode != 0 or not lines:
                out[name] = {"error": (r.stderr or "no output")[-300:]}
                continue
            d = json.loads(lines[-1])
            e = {k: d[k] for k in keys if k in d}
            e["pass"] = d["config"]["pass"]
            if name == "stride2_layer":
                e["N_out"] = d["config"]["N_out"]
                e["map_size"] = d["config"]["map_size"]
            out[name] = e
        except (subprocess.SubprocessError, OSError, ValueError) as ex:
            out[name] = {"error": str(ex)[-300:]}
    return out


def run_e2e(args, w, s, f_np, Ws_dev, tdt, dev, variants, world, build_map, n_out):
    """Same metric through the public calls with host buffers: every step
    copies its coordinates, features and all layer weights from pinned host
    memory, builds the map asynchronously, runs every layer, copies the last
    layer's output back into pinned host memory, and has its map's error
    status checked (sc_kmap_check).  Steps are double-buffered: the input
    copies (one stream) and the output copies (another) overlap the layers of
    the neighbouring steps, and step i-1's status is read (on a fourth
    stream, after its layers) while step i runs."""
    import torch
    from submanifold_sparse_convolution_hash_gb300 import binding as sc
    cs = torch.cuda.current_stream(dev)  # layers
    xs = torch.cuda.Stream(dev)           # host -> device copies
    ds = torch.cuda.Stream(dev)           # device -> host copies
    ks = torch.cuda.Stream(dev)           # status reads
    c_h = torch.from_numpy(s.coords).pin_memory()
    f_h = torch.from_numpy(f_np).to(tdt).pin_memory()
    W_h = [W.cpu().pin_memory() for W in Ws_dev]
    co_last = Ws_dev[-1].shape[2]
    o_h = [torch.empty((n_out, co_last), dtype=tdt).pin_memory() for _ in range(2)]
    c_d = [torch.empty_like(c_h, device=dev) for _ in range(2)]
    f_d = [torch.empty_like(f_h, device=dev) for _ in range(2)]
    W_d = [[torch.empty_like(W, device=dev) for W in W_h] for _ in range(2)]
    outs = [[torch.empty((n_out, W.shape[2]), dtype=tdt, device=dev) for W in W_h] for _ in range(2)]
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("h2d", "comp", "d2h")}
    used = [False, False]
    pending = []  # (buffer, handles) of the step whose status is still to be read

    def check_oldest():
        k, hs, m = pending.pop(0)
        ks.wait_event(ev["comp"][k])
        m.check(stream=ks)  # reads the status words on ks: waits for that step's layers only

    def step(i):
        k = i % 2
        with torch.cuda.stream(xs):
            if used[k]:
                xs.wait_event(ev["comp"][k])  # step i-2's layers are done with buffer k
            c_d[k].copy_(c_h, non_blocking=True)
            f_d[k].copy_(f_h, non_blocking=True)
            for Wd, Wh in zip(W_d[k], W_h):
                Wd.copy_(Wh, non_blocking=True)
            ev["h2d"][k].record(xs)
        cs.wait_event(ev["h2d"][k])
        if used[k]:
            cs.wait_event(ev["d2h"][k])  # step i-2's output copy is done with outs[k]
        hs, m = build_map(c_d[k], False)
        x = f_d[k]
        for li, W in enumerate(W_d[k]):
            x = sc.sc_subm_conv_fwd(m, x, W, out=outs[k][li], relu=li + 1 < len(W_d[k]), variant=variants[li])
        ev["comp"][k].record(cs)
        used[k] = True
        with torch.cuda.stream(ds):
            ds.wait_event(ev["comp"][k])
            o_h[k].copy_(x, non_blocking=True)
            ev["d2h"][k].record(ds)
        pending.append((k, hs, m))
        if len(pending) > 1:
            check_oldest()

    for i in range(3):
        step(i)
    while pending:
        check_oldest()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(cs)
    for i in range(args.e2e_steps):
        step(i)
    while pending:
        check_oldest()
    b.record(ds)  # after the last output copy
    b.synchronize()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.e2e_steps
    bi = c_h.numel() * 4 + f_h.numel() * f_h.element_size() + sum(W.numel() * W.element_size() for W in W_h)
    bo = o_h[0].numel() * o_h[0].element_size()
    return {"value": round(s.n / (ms / 1e3) / 1e6, 4), "unit": "Mvoxels/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo), "steps": args.e2e_steps,
            "schedule": "double-buffered: input and output copies on their own streams overlap the "
                        "neighbouring steps' layers; asynchronous map build, status checked per step"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
