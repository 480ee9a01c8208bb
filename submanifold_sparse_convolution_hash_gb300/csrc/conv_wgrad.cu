// Weight gradient of a submanifold convolution layer:
//   dW[d] = sum over the tuples (p, q, d) of feats[p]^T gout[q]
// (the layer is linear in W; the tuples are those of the forward update rule,
// exam sheet "Sparse convolution for point clouds", "The map and the update
// rule").  The tuples of offset d are the map's list of d (the identity for
// the centre), so every product is a real pair: no zero rows.
//
// One block per (offset, chunk of kChunk tuples, 64 x 64 tile of dW[d]):
// 32 tuples at a time, the block stages their feature and gradient rows in
// shared memory as fp32 and every thread accumulates a 4 x 4 patch of the
// tile with FMAs; the tile is added to an fp32 buffer with atomics, which one
// cast kernel turns into the output dtype.

#include <type_traits>

#include "sc_internal.cuh"

namespace sc {
namespace {

constexpr int kChunk = 4096;  // tuples per block
constexpr int kStep = 32;     // tuples staged at a time
constexpr int kTile = 64;     // dW tile edge

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__half>(const __half* p) { return __half2float(__ldg(p)); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

// grid: x = chunk of the offset's tuples, y = offset, z = dW tile
template <typename T>
__global__ void __launch_bounds__(256) k_wgrad(const T* __restrict__ feats, const T* __restrict__ gout,
                                               const int* __restrict__ in_rows, const int* __restrict__ out_rows,
                                               const int64_t* __restrict__ offs, int64_t n, int V, int c_in,
                                               int c_out, float* __restrict__ dw) {
  __shared__ float s_f[kStep][kTile + 1];
  __shared__ float s_g[kStep][kTile + 1];
  __shared__ int s_p[kStep], s_q[kStep];
  const int v = blockIdx.y;
  const int centre = (V - 1) / 2;
  const int64_t count = v == centre ? n : __ldg(offs + v + 1) - __ldg(offs + v);
  const int64_t e0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  if (e0 >= count) return;
  const int64_t e1 = min(count, e0 + kChunk);
  const int tiles_co = (c_out + kTile - 1) / kTile;
  const int ci0 = (blockIdx.z / tiles_co) * kTile, co0 = (blockIdx.z % tiles_co) * kTile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 4 x 4 patch at (ty * 4, tx * 4)
  float acc[4][4] = {};
  const int64_t lb = static_cast<int64_t>(v) * n;  // offset v's list in the strided lists
  for (int64_t e = e0; e < e1; e += kStep) {
    const int ne = static_cast<int>(min(static_cast<int64_t>(kStep), e1 - e));
    if (threadIdx.x < kStep) {
      int p = -1, q = -1;
      if (threadIdx.x < ne) {
        if (v == centre) {  // the identity: every row with itself
          p = q = static_cast<int>(e + threadIdx.x);
        } else {
          p = __ldg(in_rows + lb + e + threadIdx.x);
          q = __ldg(out_rows + lb + e + threadIdx.x);
        }
      }
      s_p[threadIdx.x] = p;
      s_q[threadIdx.x] = q;
    }
    __syncthreads();
    // rows: kStep x 64 features and gradients, 8 elements per thread each
    for (int k = threadIdx.x; k < kStep * kTile; k += 256) {
      const int t = k / kTile, c = k % kTile;
      const int p = s_p[t], q = s_q[t];
      s_f[t][c] = (p >= 0 && ci0 + c < c_in) ? ld_f<T>(feats + static_cast<int64_t>(p) * c_in + ci0 + c) : 0.f;
      s_g[t][c] = (q >= 0 && co0 + c < c_out) ? ld_f<T>(gout + static_cast<int64_t>(q) * c_out + co0 + c) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int t = 0; t < kStep; ++t) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = s_f[t][ty * 4 + i];
        b[i] = s_g[t][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = ci0 + ty * 4 + i;
    if (ci >= c_in) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int co = co0 + tx * 4 + j;
      if (co < c_out) atomicAdd(dw + (static_cast<int64_t>(v) * c_in + ci) * c_out + co, acc[i][j]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_from_f32(const float* __restrict__ src, T* __restrict__ dst, int64_t count) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float x = __ldg(src + i);
    if constexpr (std::is_same_v<T, float>) dst[i] = x;
    else if constexpr (std::is_same_v<T, __half>) dst[i] = __float2half_rn(x);
    else dst[i] = __float2bfloat16_rn(x);
  }
}

template <typename T>
sc_status run(const KernelMap* m, const void* feats, const void* gout, void* dW, int c_in, int c_out,
              cudaStream_t s) {
  const int64_t count = static_cast<int64_t>(m->V) * c_in * c_out;
  float* acc = nullptr;
  sc_status st = dev_alloc(reinterpret_cast<void**>(&acc), sizeof(float) * count, s);
  if (st) return st;
  cudaError_t e = cudaMemsetAsync(acc, 0, sizeof(float) * count, s);
  if (e != cudaSuccess) {
    dev_free(acc, s);
    return set_cuda_error(e, "wgrad accumulator clear");
  }
  if (m->n > 0) {
    const int tiles = ((c_in + kTile - 1) / kTile) * ((c_out + kTile - 1) / kTile);
    const dim3 grid(static_cast<unsigned>((m->n + kChunk - 1) / kChunk), static_cast<unsigned>(m->V),
                    static_cast<unsigned>(tiles));
    SC_LAUNCH("subm_conv_wgrad", s,
              k_wgrad<T><<<grid, 256, 0, s>>>(static_cast<const T*>(feats), static_cast<const T*>(gout), m->in_rows,
                                              m->out_rows, m->offs, m->n, m->V, c_in, c_out, acc));
  }
  int g = static_cast<int>((count + 255) / 256);
  if (g > device_sm_count() * 16) g = device_sm_count() * 16;
  SC_LAUNCH("wgrad_cast", s, k_from_f32<T><<<g, 256, 0, s>>>(acc, static_cast<T*>(dW), count));
  e = cudaGetLastError();
  dev_free(acc, s);
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "wgrad launch");
}

}  // namespace

sc_status conv_bwd_weight(const KernelMap* m, const void* feats, const void* gout, void* dW, int c_in, int c_out,
                          sc_dtype dtype, cudaStream_t s) {
  switch (dtype) {
    case SC_F32: return run<float>(m, feats, gout, dW, c_in, c_out, s);
    case SC_F16: return run<__half>(m, feats, gout, dW, c_in, c_out, s);
    case SC_BF16: return run<__nv_bfloat16>(m, feats, gout, dW, c_in, c_out, s);
  }
  return set_error(SC_ERR_UNSUPPORTED, "dtype");
}

}  // namespace sc
