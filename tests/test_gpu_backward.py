"""GPU parity of the backward pass (input and weight gradients) against the
CPU oracle, on the seeded scenes of the forward tests: every variant, both
row orders and the signature sort, max|gpu - ref| <= 5e-3 * max(1, max|ref|)
(f16/bf16 inputs, fp32 accumulation) or 1e-5 * max(1, max|ref|) (fp32)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TORCH_DT, assert_close
from submanifold_sparse_convolution_hash_gb300 import binding as sc
from submanifold_sparse_convolution_hash_gb300 import scenes

pytestmark = pytest.mark.gpu

SC = {
    "lidar": scenes.lidar_scan(41, 3000, (160, 160, 41)),
    "indoor": scenes.indoor_scene(42, 4000, (48, 48, 32), extent=(8, 40), radius=(3, 10)),
    "batch": scenes.batch_of_scans(43, 3, 1200, (120, 120, 41)),
    "uniform2d": scenes.uniform_2d(1000, (64, 64), 200),
}


def tensors(s, K, c_in, c_out, dtype, seed):
    V = K ** s.ndim
    f = scenes.features(seed, s.n, c_in)
    g = scenes.features(seed + 1, s.n, c_out)
    w = scenes.weights(seed + 2, V, c_in, c_out, std=1.0 if dtype == "f32" else None)
    dt = TORCH_DT[dtype]
    ft, gt, wt = (torch.from_numpy(a).to(dt) for a in (f, g, w))
    return ft.cuda(), gt.cuda(), wt.cuda(), ft.double().numpy(), gt.double().numpy(), wt.double().numpy()


BWD_CASES = [
    # scene, K, c_in, c_out, dtype, variant (input gradient)
    ("lidar", 3, 32, 32, "f16", "fused"),
    ("lidar", 3, 32, 64, "f16", "ws"),
    ("indoor", 3, 64, 64, "bf16", "fused"),
    ("batch", 3, 64, 128, "f16", "fused"),
    ("batch", 3, 128, 256, "f16", "fused"),
    ("batch", 3, 256, 256, "bf16", "fused"),
    ("indoor", 5, 128, 128, "bf16", "fused"),
    ("indoor", 5, 32, 48, "bf16", "ws"),
    ("lidar", 3, 32, 16, "f32", "simt"),
    ("uniform2d", 3, 16, 16, "f32", None),
    ("uniform2d", 5, 16, 32, "f16", "fused"),
]


@pytest.mark.parametrize("order,sort", [(False, False), (True, True)])
@pytest.mark.parametrize("name,K,c_in,c_out,dtype,variant", BWD_CASES)
def test_bwd_data_matches_oracle(name, K, c_in, c_out, dtype, variant, order, sort):
    s = SC[name]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, s.ndim, K, s.dims, order=order, sort=sort)
    f, g, w, f64, g64, w64 = tensors(s, K, c_in, c_out, dtype, seed=c_in + K)
    gin = sc.sc_subm_conv_bwd_data(m, g, w, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.subm_conv_bwd_data(s.coords, g64, w64, s.ndim, K, s.dims)
    assert_close(gin, ref, dtype, f"{name} K={K} {c_in}->{c_out} {dtype} {variant}")
    m.check()


@pytest.mark.parametrize("name,K,c_in,c_out,dtype", [
    ("lidar", 3, 32, 32, "f16"), ("indoor", 3, 64, 64, "bf16"), ("batch", 3, 128, 256, "f16"),
    ("indoor", 5, 48, 16, "bf16"), ("uniform2d", 3, 16, 16, "f32"), ("lidar", 1, 16, 32, "f16"),
    # tensor-core shapes: two M halves (c_in 256), padded M panels (c_in 192, 48),
    # three N panels (c_out 48), wide N (c_out 128, 256), one accumulator buffer
    ("batch", 3, 256, 256, "bf16"), ("indoor", 3, 64, 128, "f16"), ("lidar", 3, 192, 64, "bf16"),
    ("lidar", 3, 32, 48, "f16"), ("indoor", 3, 128, 32, "bf16"), ("uniform2d", 5, 16, 32, "f16"),
])
def test_bwd_weight_matches_oracle(name, K, c_in, c_out, dtype):
    s = SC[name]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, s.ndim, K, s.dims, sync=False)
    f, g, w, f64, g64, w64 = tensors(s, K, c_in, c_out, dtype, seed=3 * c_in + K)
    dW = sc.sc_subm_conv_bwd_weight(m, f, g)
    torch.cuda.synchronize()
    ref = oracle.subm_conv_bwd_weight(s.coords, f64, g64, s.ndim, K, s.dims)
    # the fp32 sums run over up to N products (the centre offset): the bound
    # scales with their magnitude
    scale = max(1.0, float(np.abs(ref).max()))
    err = float(np.abs(dW.double().cpu().numpy() - ref).max())
    tol = (1e-5 if dtype == "f32" else 5e-3) * scale
    assert err <= tol, f"{name} {dtype}: {err} > {tol}"


def test_backward_adjoint_on_gpu():
    """<conv(f), g> = <f, dgrad(g)> = <W, wgrad(f, g)> with the GPU's three
    kernels (fp32)."""
    s = SC["indoor"]
    h = sc.sc_hash_build(torch.from_numpy(s.coords).cuda())
    m = sc.sc_kmap_build(h, 3, 3, s.dims)
    f, g, w, *_ = tensors(s, 3, 16, 32, "f32", seed=5)
    lhs = float((sc.sc_subm_conv_fwd(m, f, w).double() * g.double()).sum())
    mid = float((f.double() * sc.sc_subm_conv_bwd_data(m, g, w).double()).sum())
    rhs = float((w.double() * sc.sc_subm_conv_bwd_weight(m, f, g).double()).sum())
    assert abs(lhs - mid) <= 1e-4 * max(1.0, abs(lhs))
    assert abs(lhs - rhs) <= 1e-4 * max(1.0, abs(lhs))


def test_backward_empty_map():
    h = sc.sc_hash_build(torch.zeros((0, 4), dtype=torch.int32, device="cuda"))
    m = sc.sc_kmap_build(h, 3, 3, (8, 8, 8))
    f = torch.zeros((0, 16), dtype=torch.float16, device="cuda")
    g = torch.zeros((0, 32), dtype=torch.float16, device="cuda")
    W = torch.randn((27, 16, 32), device="cuda").half()
    assert sc.sc_subm_conv_bwd_data(m, g, W).shape == (0, 16)
    dW = sc.sc_subm_conv_bwd_weight(m, f, g)
    assert dW.shape == (27, 16, 32) and int(torch.count_nonzero(dW)) == 0
