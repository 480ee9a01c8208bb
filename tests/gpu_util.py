"""Shared helpers for the GPU parity tests: seeded inputs as tensors, the
oracle-side reference, and the tolerance the parity bar fixes."""
import numpy as np
import torch

import oracle
from submanifold_sparse_convolution_hash_gb300 import scenes

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def tol(dtype: str, ref: np.ndarray) -> float:
    """max|gpu - ref| bound: 5e-3 * max(1, max|ref|) for f16/bf16 inputs with
    fp32 accumulation, 1e-5 * max(1, max|ref|) for fp32."""
    scale = max(1.0, float(np.abs(ref).max()) if ref.size else 1.0)
    return (1e-5 if dtype == "f32" else 5e-3) * scale


def layer_inputs(scene, K, c_in, c_out, dtype, seed, w_std=None):
    """(feats, W) as device tensors in `dtype` and their exact fp64 values."""
    V = K ** scene.ndim
    f = scenes.features(seed, scene.n, c_in)
    w = scenes.weights(seed, V, c_in, c_out, std=w_std)
    ft = torch.from_numpy(f).to(TORCH_DT[dtype])
    wt = torch.from_numpy(w).to(TORCH_DT[dtype])
    return ft.cuda(), wt.cuda(), ft.double().numpy(), wt.double().numpy()


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    g = gpu.double().cpu().numpy()
    err = float(np.abs(g - ref).max()) if ref.size else 0.0
    bound = tol(dtype, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert err <= bound, f"{what}: max|gpu-ref| = {err:.3e} > {bound:.3e}"
    return err


def oracle_lists(nbr: np.ndarray):
    return oracle.offset_lists(nbr)


def gpu_lists_by_offset(kmap):
    offs, i, o = kmap.lists()
    offs = offs.cpu().numpy()
    i = i.cpu().numpy()
    o = o.cpu().numpy()
    return [(i[offs[v]:offs[v + 1]].astype(np.int64), o[offs[v]:offs[v + 1]].astype(np.int64))
            for v in range(len(offs) - 1)], offs
