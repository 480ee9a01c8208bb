// Weight gradient of a submanifold convolution layer:
//   dW[d] = sum over the tuples (p, q, d) of feats[p]^T gout[q]
// (the layer is linear in W; the tuples are those of the forward update rule,
// exam sheet "Sparse convolution for point clouds", "The map and the update
// rule").  The tuples of offset d are the map's list of d (the identity for
// the centre), so every product is a real pair: no zero rows.
//
// f16 / bf16: a tcgen05 GEMM per offset, dW[d] (c_in x c_out) = A B with
// A = feats rows gathered by the list (K = tuples, M = c_in) and B = gout
// rows (N = c_out).  Both operands land in shared memory exactly as gathered,
// one row per tuple, which is the MN-major layout of A and B: each 16-byte
// chunk of a row goes to its swizzled place in a panel of 16, 32 or 64
// channels, and the MMA reads the panels with MN-major descriptors.  A work
// unit is a run of one offset's list (a few K tiles); its fp32 tile of dW[d]
// is accumulated in TMEM and added into an fp32 buffer with vector atomics
// by the epilogue warps, which one cast kernel rounds to the dtype.  CTA:
// NPW producer warps (cp.async gathers; each thread's arrival on a stage
// barrier fires when its copies land), one MMA warp, four epilogue warps.
// c_in above 128 takes two M = 128 halves (two accumulators).  c_in that is
// one panel wide (16, 32, 64) uses M = 128 with every M atom reading the same
// panel (atom stride 0); the extra rows of D are copies and are not stored.
// Other widths that are not a multiple of 128 pad A's panels up to the next
// 128 channels; the rows of D past c_in are never stored.
//
// fp32 (CUDA cores): one block per (offset, chunk of kChunk tuples, 64 x 64
// tile of dW[d]): 32 tuples at a time, the block stages their feature and
// gradient rows in shared memory and every thread accumulates a 4 x 4 patch
// of the tile with FMAs; the tile is added to the fp32 buffer with atomics.

#include <type_traits>

#include "sc_internal.cuh"
#include "tc_ptx.cuh"

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
                                               int c_out, int identity, float* __restrict__ dw) {
  __shared__ float s_f[kStep][kTile + 1];
  __shared__ float s_g[kStep][kTile + 1];
  __shared__ int s_p[kStep], s_q[kStep];
  const int v = blockIdx.y;
  const int centre = (V - 1) / 2;
  const bool implicit = v == centre && identity;  // the identity list of a submanifold map
  const int64_t count = implicit ? n : __ldg(offs + v + 1) - __ldg(offs + v);
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
        if (implicit) {  // every row with itself
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

// ------------------------------------------------------- tensor-core path --
constexpr int kWgMaxStages = 4;
constexpr int kWgBarriers = 2 * kWgMaxStages + 5;  // full[S], empty[S], acc_full[2], acc_empty[2], done

struct WgParams {
  const uint8_t* feats;  // [n, c_in] 2-byte elements
  const uint8_t* gout;   // [n, c_out]
  const int* in_rows;    // offset v's list at v * n
  const int* out_rows;
  const int64_t* offs;   // [V+1]
  float* dw;             // [V, c_in, c_out] fp32, zeroed
  int64_t n;
  int V, c_in, c_out;
  int nc;                // chunks per offset list
  int num_units;         // V * nc
  int rba, rbb;          // bytes per panel row of A (feature channels) and B (gradient channels)
  int a_bytes, b_bytes;  // one stage's A and B
  int a_half;            // bytes between A's two M = 128 halves
  uint32_t lbo_a, lbo_b; // bytes between panels (M / N atoms)
  int n_m;               // M halves (1 or 2)
  int identity;          // the centre list is the identity (submanifold map)
  int stages, acc_cols, nbuf, tmem_cols;
  int* status;
};

__device__ __forceinline__ int64_t list_count(const WgParams& p, int v) {
  return v == (p.V - 1) / 2 && p.identity ? p.n : __ldg(p.offs + v + 1) - __ldg(p.offs + v);
}

// Work unit u: chunk c = u / V of offset v = u % V, the list entries
// [c count / nc, (c + 1) count / nc) (possibly none).  Every list runs in row
// order, so chunk c of every offset covers about the same rows: units that run
// at the same time share a spatial window of the rows and reuse them in L2.
__device__ __forceinline__ void unit_decode(const WgParams& p, int u, int& v, int64_t& e0, int& len) {
  const int c = u / p.V;
  v = u - c * p.V;
  const int64_t cnt = list_count(p, v);
  e0 = cnt * c / p.nc;
  len = static_cast<int>(cnt * (c + 1) / p.nc - e0);
}

// log2 of (128 / row bytes): the shift of the swizzle's row bits
__device__ __forceinline__ int swz_shift(int rb) { return rb == 128 ? 0 : (rb == 64 ? 1 : 2); }
__host__ __device__ constexpr uint32_t swz_layout(int rb) { return rb == 128 ? 2u : (rb == 64 ? 4u : 6u); }

template <bool BF16, int NPW, int KT>
__global__ void __launch_bounds__((NPW + 5) * 32, NPW == 4 ? 3 : 2) k_wgrad_tc(const WgParams p) {
  constexpr int TW = KT / NPW;  // tuples per producer warp and stage
  static_assert(TW >= 1 && TW <= 32 && KT % 16 == 0, "a producer warp holds one index pair per lane");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages, NB = p.nbuf;
  const int stage_bytes = p.a_bytes + p.b_bytes;  // a multiple of 1024
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * stage_bytes);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kWgBarriers);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kWgMaxStages);
  const uint32_t accf0 = smem_u32(bars + 2 * kWgMaxStages), acce0 = smem_u32(bars + 2 * kWgMaxStages + 2);
  const uint32_t done_bar = smem_u32(bars + 2 * kWgMaxStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, NPW * 32);  // one copy-completion arrival per producer thread
      mbar_init(empty0 + 8 * s, 1);        // one tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);
    }
    mbar_init(done_bar, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == NPW) {
    tmem_alloc(smem_u32(s_tmem), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp < NPW) {
    // ======================================================= producers
    // A warp instruction copies whole rows: lane = row step * (chunks per
    // row) + chunk, so each lane keeps one 16-byte chunk position of the
    // feature rows (A) and one of the gradient rows (B) and walks the rows.
    const int cia = p.c_in / 8, cib = p.c_out / 8;  // 16-byte chunks per row
    const int rpa = 32 / cia, rpb = 32 / cib;        // rows per warp instruction
    const int ra = lane / cia, ca = lane - ra * cia;
    const int rb = lane / cib, cb = lane - rb * cib;
    const bool acta = ra < rpa, actb = rb < rpb;     // lanes past the last whole row idle
    const int cpra = p.rba / 16, cprb = p.rbb / 16;  // chunks per panel row
    const uint32_t cola = static_cast<uint32_t>((ca / cpra) * KT * p.rba);  // this chunk's panel
    const uint32_t colb = static_cast<uint32_t>((cb / cprb) * KT * p.rbb);
    const int cca = ca % cpra, ccb = cb % cprb;
    const int sha = swz_shift(p.rba), shb = swz_shift(p.rbb);
    const size_t rowa = static_cast<size_t>(p.c_in) * 2, rowb = static_cast<size_t>(p.c_out) * 2;
    const int t0w = warp * TW;  // this warp's first tuple (K row) of a stage
    const int centre = (p.V - 1) / 2;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < p.num_units && !*s_abort; u += gridDim.x) {
      int v, len;
      int64_t e0;
      unit_decode(p, u, v, e0, len);
      if (len == 0) continue;
      const int64_t lb = static_cast<int64_t>(v) * p.n + e0;
      const int nkt = (len + KT - 1) / KT;
      // lane j < TW holds the (feature row, gradient row) of tuple t0w + j
      auto fetch = [&](int kt, int& pp, int& qq) {
        const int t = kt * KT + t0w + lane;
        pp = qq = -1;
        if (lane < TW && t < len) {
          if (v == centre && p.identity) {
            pp = qq = static_cast<int>(e0 + t);
          } else {
            pp = __ldg(p.in_rows + lb + t);
            qq = __ldg(p.out_rows + lb + t);
          }
        }
      };
      // indices of this K tile and the next two, loads in flight
      int pc, qc, p1, q1;
      fetch(0, pc, qc);
      fetch(1, p1, q1);
      for (int kt = 0; kt < nkt; ++kt, ++it) {
        int p2, q2;
        fetch(kt + 2, p2, q2);
        const int s = static_cast<int>(it % S);
        const uint32_t ph = (it / S) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * s, ph ^ 1u, s_abort))) {
          *s_abort = 1;
          break;
        }
        const uint32_t a_st = smem_u32(smem + s * stage_bytes);
        const uint32_t b_st = a_st + static_cast<uint32_t>(p.a_bytes);
        for (int r0 = 0; r0 < TW; r0 += rpa) {
          const int tl = r0 + ra;
          const int pr = __shfl_sync(0xffffffffu, pc, tl < TW ? tl : 0);
          if (acta && tl < TW) {
            const int t = t0w + tl;  // K row of the stage
            const uint32_t dst = a_st + cola + static_cast<uint32_t>(t * p.rba) +
                                 (static_cast<uint32_t>(cca ^ ((t >> sha) & (cpra - 1))) << 4);
            cp_async_16(dst, p.feats + static_cast<size_t>(pr < 0 ? 0 : pr) * rowa + ca * 16, pr >= 0 ? 16u : 0u);
          }
        }
        for (int r0 = 0; r0 < TW; r0 += rpb) {
          const int tl = r0 + rb;
          const int qr = __shfl_sync(0xffffffffu, qc, tl < TW ? tl : 0);
          if (actb && tl < TW) {
            const int t = t0w + tl;
            const uint32_t dst = b_st + colb + static_cast<uint32_t>(t * p.rbb) +
                                 (static_cast<uint32_t>(ccb ^ ((t >> shb) & (cprb - 1))) << 4);
            cp_async_16(dst, p.gout + static_cast<size_t>(qr < 0 ? 0 : qr) * rowb + cb * 16, qr >= 0 ? 16u : 0u);
          }
        }
        cp_async_arrive_noinc(full0 + 8 * s);
        pc = p1;
        qc = q1;
        p1 = p2;
        q1 = q2;
      }
    }
    cp_async_wait_all();
  } else if (warp == NPW) {
    // ======================================================= MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_mn(BF16, 128, p.c_out);
      const uint32_t base = smem_u32(smem);
      const uint64_t da0 = smem_desc_mn(base, p.lbo_a, 8u * p.rba, swz_layout(p.rba));
      const uint64_t db0 = smem_desc_mn(base + p.a_bytes, p.lbo_b, 8u * p.rbb, swz_layout(p.rbb));
      uint32_t it = 0;
      int j = 0;
      for (int u = blockIdx.x; u < p.num_units && !*s_abort; u += gridDim.x) {
        int v, len;
        int64_t e0;
        unit_decode(p, u, v, e0, len);
        if (len == 0) continue;
        const int nkt = (len + KT - 1) / KT;
        const int b = j % NB;
        if (!mbar_wait(acce0 + 8 * b, ((j / NB) & 1) ^ 1, s_abort)) {
          *s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * p.n_m * p.acc_cols);
        uint32_t accumulate = 0;
        for (int kt = 0; kt < nkt; ++kt, ++it) {
          const int s = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(full0 + 8 * s, ph, s_abort)) {
            *s_abort = 1;
            break;
          }
          // the producers' cp.async writes are generic-proxy writes: order
          // them before the tensor core's reads
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < KT / 16; ++k) {
            // K step k: tuples 16k .. 16k + 15 = two 8-row atoms of each panel
            for (int h = 0; h < p.n_m; ++h) {
              const uint64_t ad = da0 + static_cast<uint64_t>((s * stage_bytes + h * p.a_half + k * 16 * p.rba) >> 4);
              const uint64_t bd = db0 + static_cast<uint64_t>((s * stage_bytes + k * 16 * p.rbb) >> 4);
              tc_mma(d + static_cast<uint32_t>(h * p.acc_cols), ad, bd, idesc, accumulate);
            }
            accumulate = 1;
          }
          tc_commit(empty0 + 8 * s);
        }
        tc_commit(accf0 + 8 * b);
        ++j;
      }
      tc_commit(done_bar);
      if (!mbar_drain(done_bar, 0)) *s_abort = 1;
    }
    __syncwarp();
  } else {
    // ======================================================= epilogue (warps NPW+1 .. NPW+4)
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    int j = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
      int v, len;
      int64_t e0;
      unit_decode(p, u, v, e0, len);
      if (len == 0) continue;
      const int b = j % NB;
      if (*s_abort || !mbar_wait(accf0 + 8 * b, (j / NB) & 1, s_abort)) {
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      for (int h = 0; h < p.n_m; ++h) {
        if (h * 128 + q * 32 >= p.c_in) continue;  // this quadrant holds no row of dW[v]
        const int ci = h * 128 + q * 32 + lane;
        const uint32_t trow = tmem + static_cast<uint32_t>((b * p.n_m + h) * p.acc_cols) +
                              (static_cast<uint32_t>(q * 32) << 16);
        const int64_t row = ci < p.c_in ? (static_cast<int64_t>(v) * p.c_in + ci) * p.c_out : -1;
        for (int c0 = 0; c0 < p.c_out; c0 += 16) {
          float a[16];
          tmem_ld16(trow + static_cast<uint32_t>(c0), a);  // the whole warp loads; rows past c_in are dropped
          if (row >= 0) {
            float4* dst = reinterpret_cast<float4*>(p.dw + row + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              atomicAdd(dst + k, make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
      ++j;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == NPW) {
    tc_fence_after();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
  if (threadIdx.x == 0 && *s_abort) atomicOr(p.status, kDevErrTimeout);
}

struct WgPlan {
  int kt, npw, stages, cps;
  size_t smem;
  WgParams prm;  // the shape fields
};

int panel_row_bytes(int c) { return c % 64 == 0 ? 128 : (c % 32 == 0 ? 64 : 32); }

// Shape of the tensor-core launch: K tile of 128 tuples while a stage stays
// within 48 KB, else 64; as many stages (2..4) as fit 96 KB; two TMEM
// accumulators where 512 columns allow, so the epilogue overlaps the next
// unit.  False if c_in needs more than two M halves.
bool wg_plan(int c_in, int c_out, WgPlan* pl) {
  WgParams& p = pl->prm;
  p.rba = panel_row_bytes(c_in);
  p.rbb = panel_row_bytes(c_out);
  const int panels_a = c_in * 2 / p.rba, atoms_half = 256 / p.rba;
  for (int kt = 128; kt >= 64; kt -= 64) {
    if (panels_a == 1) {  // every M atom reads the one panel
      p.n_m = 1;
      p.a_bytes = kt * p.rba;
      p.lbo_a = 0;
      p.a_half = 0;
    } else {
      p.n_m = (panels_a + atoms_half - 1) / atoms_half;
      p.a_bytes = p.n_m * atoms_half * kt * p.rba;
      p.lbo_a = static_cast<uint32_t>(kt * p.rba);
      p.a_half = atoms_half * kt * p.rba;
    }
    p.b_bytes = kt * c_out * 2;
    p.lbo_b = static_cast<uint32_t>(kt * p.rbb);
    pl->kt = kt;
    if (p.a_bytes + p.b_bytes <= 48 * 1024) break;
  }
  if (p.n_m > 2) return false;
  const int stage = p.a_bytes + p.b_bytes;
  int st = (96 * 1024) / stage;
  p.stages = st < 2 ? 2 : (st > kWgMaxStages ? kWgMaxStages : st);
  int cols = 32;
  while (cols < c_out) cols <<= 1;
  p.acc_cols = cols;
  if (p.n_m * cols > 512) return false;
  p.nbuf = 2 * p.n_m * cols <= 512 ? 2 : 1;
  p.tmem_cols = p.nbuf * p.n_m * cols;
  pl->smem = 1024 + static_cast<size_t>(p.stages) * stage + 8 * kWgBarriers + 16;
  if (pl->smem > 220 * 1024) return false;
  int cps = static_cast<int>((220 * 1024) / pl->smem);
  if (cps * p.tmem_cols > 512) cps = 512 / p.tmem_cols;
  if (cps > 3) cps = 3;
  pl->npw = cps >= 3 ? 4 : 8;  // 12 to 16 gathering warps per SM
  pl->cps = cps < 1 ? 1 : cps;
  return true;
}

template <bool BF16, int NPW, int KT>
sc_status launch_wgrad_tc(const WgParams& prm, const WgPlan& pl, cudaStream_t s) {
  auto kern = k_wgrad_tc<BF16, NPW, KT>;
  sc_status st = kernel_setup(reinterpret_cast<const void*>(kern), pl.smem, nullptr);
  if (st) return st;
  const int slots = device_sm_count() * pl.cps;
  const int grid = prm.num_units < slots ? prm.num_units : slots;
  SC_LAUNCH("subm_conv_wgrad", s, kern<<<grid, (NPW + 5) * 32, pl.smem, s>>>(prm));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "wgrad launch");
}

template <bool BF16>
sc_status dispatch_wgrad_tc(const WgParams& prm, const WgPlan& pl, cudaStream_t s) {
  if (pl.kt == 128)
    return pl.npw == 4 ? launch_wgrad_tc<BF16, 4, 128>(prm, pl, s) : launch_wgrad_tc<BF16, 8, 128>(prm, pl, s);
  return pl.npw == 4 ? launch_wgrad_tc<BF16, 4, 64>(prm, pl, s) : launch_wgrad_tc<BF16, 8, 64>(prm, pl, s);
}

// The tensor-core weight gradient into the zeroed fp32 buffer `acc`.  Needs
// the map's host counts (the per-offset list lengths set the work units).
sc_status wgrad_tc(const KernelMap* m, const WgPlan& pl, const void* feats, const void* gout, float* acc, int c_in,
                   int c_out, bool bf16, cudaStream_t s) {
  WgParams prm = pl.prm;
  prm.feats = static_cast<const uint8_t*>(feats);
  prm.gout = static_cast<const uint8_t*>(gout);
  prm.in_rows = m->in_rows;
  prm.out_rows = m->out_rows;
  prm.offs = m->offs;
  prm.dw = acc;
  prm.n = m->n;
  prm.V = m->V;
  prm.c_in = c_in;
  prm.c_out = c_out;
  prm.status = m->status;
  prm.identity = m->identity ? 1 : 0;
  // about four units per resident CTA, at least two K tiles each on average
  const int64_t total = m->map_size_host;
  const int64_t slots = static_cast<int64_t>(device_sm_count()) * pl.cps;
  int64_t nc = (4 * slots + m->V - 1) / m->V;
  const int64_t nc_max = total / (static_cast<int64_t>(m->V) * 2 * pl.kt);
  if (nc > nc_max) nc = nc_max;
  if (nc < 1) nc = 1;
  prm.nc = static_cast<int>(nc);
  prm.num_units = static_cast<int>(nc * m->V);
  return bf16 ? dispatch_wgrad_tc<true>(prm, pl, s) : dispatch_wgrad_tc<false>(prm, pl, s);
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
  WgPlan pl;
  if (m->n > 0 && !std::is_same_v<T, float> && m->host_valid && wg_plan(c_in, c_out, &pl)) {
    st = wgrad_tc(m, pl, feats, gout, acc, c_in, c_out, std::is_same_v<T, __nv_bfloat16>, s);
    if (st) {
      dev_free(acc, s);
      return st;
    }
  } else if (m->n > 0) {
    const int tiles = ((c_in + kTile - 1) / kTile) * ((c_out + kTile - 1) / kTile);
    const dim3 grid(static_cast<unsigned>((m->n + kChunk - 1) / kChunk), static_cast<unsigned>(m->V),
                    static_cast<unsigned>(tiles));
    SC_LAUNCH("subm_conv_wgrad", s,
              k_wgrad<T><<<grid, 256, 0, s>>>(static_cast<const T*>(feats), static_cast<const T*>(gout), m->in_rows,
                                              m->out_rows, m->offs, m->n, m->V, c_in, c_out,
                                              m->identity ? 1 : 0, acc));
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
