// CUDA-core submanifold convolution: one thread per (table row, output
// channel), walking the row's neighbour-table entries in offset order and
// accumulating feats[p, ci] * W[d, ci, co] with fp32 FMAs (exam sheet
// "Sparse convolution for point clouds", "The map and the update rule").
// It is the path for fp32 layers, which the f16-kind tensor-core MMA does not
// take, and a forced variant for f16/bf16.  Threads of a warp share the
// output row and read consecutive W columns, so W loads coalesce and the
// feature row is a broadcast.

#include "sc_internal.cuh"

namespace sc {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) k_conv_simt(const T* __restrict__ feats, const T* __restrict__ W,
                                                   T* __restrict__ out, const int* __restrict__ nbr,
                                                   const int* __restrict__ order, int64_t n, int V, int c_in,
                                                   int c_out, int relu, int wt) {
  const int64_t total = n * c_out;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t q = idx / c_out;
    const int co = static_cast<int>(idx - q * c_out);
    float acc = 0.0f;
    for (int v = 0; v < V; ++v) {
      const int j = __ldg(nbr + q * V + v);
      if (j < 0) continue;
      const T* f = feats + static_cast<int64_t>(j) * c_in;
      if (wt) {  // W'[v][ci][co] = W[V-1-v][co][ci]
        const T* w = W + (static_cast<int64_t>(V - 1 - v) * c_out + co) * c_in;
        for (int ci = 0; ci < c_in; ++ci) acc = fmaf(to_f(f[ci]), to_f(w[ci]), acc);
      } else {
        const T* w = W + static_cast<int64_t>(v) * c_in * c_out + co;
        for (int ci = 0; ci < c_in; ++ci) acc = fmaf(to_f(f[ci]), to_f(w[static_cast<int64_t>(ci) * c_out]), acc);
      }
    }
    if (relu) acc = fmaxf(acc, 0.0f);
    const int64_t dst = order ? static_cast<int64_t>(__ldg(order + q)) : q;
    out[dst * c_out + co] = from_f<T>(acc);
  }
}

template <typename T>
sc_status launch(const ConvArgs& a) {
  const int64_t total = a.m->n * a.c_out;
  int64_t g = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (g > cap) g = cap;
  SC_LAUNCH("subm_conv_simt", a.stream,
            k_conv_simt<T><<<static_cast<int>(g), 256, 0, a.stream>>>(
                static_cast<const T*>(a.feats), static_cast<const T*>(a.W), static_cast<T*>(a.out), a.m->nbr,
                a.m->order, a.m->n, a.m->V, a.c_in, a.c_out, a.relu ? 1 : 0, a.wt ? 1 : 0));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "subm_conv_simt launch");
}

}  // namespace

sc_status conv_simt(const ConvArgs& a) {
  if (a.m->n == 0) return SC_OK;
  switch (a.dtype) {
    case SC_F32: return launch<float>(a);
    case SC_F16: return launch<__half>(a);
    case SC_BF16: return launch<__nv_bfloat16>(a);
  }
  return set_error(SC_ERR_UNSUPPORTED, "dtype");
}

}  // namespace sc
