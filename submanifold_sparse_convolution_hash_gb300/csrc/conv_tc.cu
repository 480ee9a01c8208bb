// Tensor-core (tcgen05) submanifold convolution kernels for sm_103a.
//
// Update rule: out[q] += feats[p] @ W[d] for every tuple (p, q, d) of the map
// (exam sheet "Sparse convolution for point clouds", "The map and the update
// rule"; "Sparse inputs and sparse convolution", "The map is the computation").
//
// Two dataflows share one persistent, warp-specialised kernel:
//
//  * Output-stationary implicit GEMM ("TorchSparse optimizations", section
//    "TorchSparse++": each block owns a tile of output rows, walks the
//    weights, fetches the matching input rows on demand and writes each output
//    once).  A tile is 128 output rows; its K dimension is the concatenation
//    over offsets d of the C_in input channels.  An offset with no neighbour
//    in any of the tile's rows is skipped (the map build records, per tile,
//    which offsets occur); absent neighbours inside a present offset are zero
//    rows.  That remaining waste is the lockstep redundancy the section
//    describes.
//
//  * Weight-stationary gather -> GEMM -> scatter ("Sparse inputs and sparse
//    convolution", section "Gather, matmul, scatter").  A tile is 128 tuples
//    of one offset: gather their input rows, multiply by W[d], scatter-add the
//    fp32 products with vector atomics.  The centre offset (identity map)
//    writes its product with plain stores first.
//
// CTA ((NPW + 6) warps; as many per SM as shared memory and TMEM allow, each
// taking tiles round-robin):
//   NPW producer warps (4, 8 or 16): per pipeline stage, each thread
//              cp.asyncs 16-byte chunks of its warp's tile rows' neighbour
//              feature rows into a swizzled K-major tile (a warp instruction
//              covers whole rows; a missing neighbour is a zero-filled copy of
//              size 0, skipped when that row of the buffer is already zero).
//              A stage holds G (offset, channel-panel) sub-blocks.  Each
//              thread's arrival on the stage barrier fires when its copies
//              land (cp.async.mbarrier.arrive.noinc), so a warp never waits
//              for its own copies.
//   1 warp     weight loader: one thread loads the matching W slices into
//              each stage, by TMA straight from W (cp.async.bulk.tensor: the
//              slice lands swizzled; a layer's B is MN-major, an input
//              gradient's K-major) or by bulk copies from a pre-swizzled image
//              (widths that fit no TMA box, the weight-stationary modes, the
//              no-allocation entry point), and prefetches the next tile's
//              neighbour-table block into L2.
//   1 warp     MMA issuer: allocates TMEM (two accumulators of C_out fp32 columns); lane 0
//              issues tcgen05.mma (M = 128, N = C_out, K = 16) and commits.
//   4 warps    epilogue: TMEM lane quadrant (warp % 4) -> registers -> global,
//              overlapping the next tile's mainloop through the second
//              accumulator; output rows are transposed across groups of four
//              lanes, so each store instruction writes 64 contiguous bytes of
//              8 rows.
// The row gathers use the load/store path: a TMA tile::gather4 moves four
// rows per instruction but its row rate, not its byte rate, bounds it, and
// for 32-256 byte rows that rate is several times below what cp.async from
// four warps sustains.
//
// Every mbarrier wait is bounded (about two seconds of %globaltimer); on
// expiry the CTA latches kDevErrTimeout, stops issuing work, waits (bounded)
// for what it issued, and still frees its TMEM.

#include <cuda.h>  // CUtensorMap and its encoding enums (the encoder is resolved at run time)

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "sc_internal.cuh"
#include "tc_ptx.cuh"

// Packed-weight buffer of sc_subm_conv_fwd_noalloc: a fixed, file-scope
// device array, so that entry point needs no allocation.  Every GPU that
// loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_weights[sc::kNoAllocWeightBytes];

namespace sc {
namespace {

constexpr int kRows = 128;        // rows per tile (MMA M)
constexpr int kMaxStages = 8;
constexpr int kAhead = 2;  // offsets whose neighbour indices a producer loads ahead (measured: 2 > 1, 3)
constexpr int kBarriers = 2 * kMaxStages + 5;  // full[S], empty[S], acc_full[2], acc_empty[2], done

enum Mode { kOutputStationary = 0, kWsScatter = 1, kWsCentre = 2 };

struct TcParams {
  // how the weight loader fetches each (offset, panel) slice of W (wmode 1
  // and 2 read W by TMA through the tensor map passed as the kernel's
  // second, __grid_constant__ argument):
  //   0: bulk copy from a packed image (wimg)
  //   1: TMA from W [V][c_in][c_out] (a layer): B MN-major, boxes of wnb
  //      output channels x BK input channels, wnb-column swizzle
  //   2: TMA from W [V][c_out][c_in] of the forward layer whose input
  //      gradient this is (W'[v] = W[V-1-v]^T): B K-major, one box of c_out
  //      rows x BK channels, the same layout as the packed image
  int wmode;
  int wnb;
  const uint8_t* feats;      // [n, c_in] 2-byte elements
  const uint8_t* wimg;       // wmode 0: packed weight images [V][P][c_out rows][BK*2 bytes]
  uint8_t* out;              // output-stationary: [n, c_out] 2-byte elements
  float* acc;                // weight-stationary: fp32 [n, c_out]
  const int* nbr;            // [n, V]
  const int* order;          // [n] input row of each tile row (null: identity); tiles are runs of 128 rows
  const int* perm;           // [n] table row of each tile row (null: identity; set by the signature sort)
  const int* tnbr;           // or null: the map's tile-transposed index table, [tiles][V][128] in tile row order
  const uint4* present;      // [tiles]: 128-bit mask of the offsets present in each 128-row tile
  const int* in_rows;        // weight-stationary lists: offset v's at v * n
  const int* out_rows;
  const int64_t* offs;       // [V+1]
  const int* ws_tiles;       // [V+1]
  int64_t n;
  int num_tiles;             // 128-row tiles (output-stationary) or tuple tiles (weight-stationary scatter)
  int num_units;             // work units: ceil(num_tiles / T)
  int V, c_in, c_out, relu, stages, group, acc_cols, tmem_cols;
  int nbuf;                  // accumulator buffers (2: the epilogue overlaps the next unit)
  int* status;
  // column splitting (output-stationary): this launch walks only the
  // offsets of one part of the offset range, in that part's row order;
  // epi 0 casts and stores the output (one part), 1 stores the fp32 partial
  // sums in acc, 2 adds acc to them and casts and stores the output
  int epi;
  int centre_in;             // the centre offset (every row's own) belongs to this launch's offsets
};

// Next offset after v whose bit is set in the 4-word mask m (V if none).
__device__ __forceinline__ int next_present(const uint4& m, int v, int V) {
  const int u = v + 1;
  const uint32_t w[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lo = 32 * k;
    if (u < lo + 32) {
      const uint32_t x = u <= lo ? w[k] : (w[k] & (0xFFFFFFFFu << (u - lo)));
      if (x) {
        const int r = lo + __ffs(x) - 1;
        return r < V ? r : V;
      }
    }
  }
  return V;
}

// The tile's present-offset mask with the centre offset added (every tile has
// at least one row, and every row has itself as a neighbour).
__device__ __forceinline__ uint4 tile_mask(const TcParams& p, int tile) {
  uint4 m = __ldg(p.present + tile);
  if (!p.centre_in) return m;
  const int c = (p.V - 1) / 2;
  const uint32_t bit = 1u << (c & 31);
  if (c < 32) m.x |= bit; else if (c < 64) m.y |= bit; else if (c < 96) m.z |= bit; else m.w |= bit;
  return m;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// A work unit: T consecutive 128-row tiles (output-stationary; the T tiles
// share every weight slice the CTA loads) or one 128-row tile of tuples
// (weight-stationary, T = 1).
struct TileInfo {
  int64_t row0;  // first output row (output-stationary, centre)
  int64_t lb;    // first list entry (weight-stationary scatter)
  int nrows;     // rows of the unit, up to 128 T
  int v;         // the offset of a weight-stationary tile
};

template <int MODE, int T>
__device__ __forceinline__ TileInfo tile_info(const TcParams& p, int u) {
  TileInfo t;
  t.row0 = 0;
  t.lb = 0;
  t.v = (p.V - 1) / 2;
  if (MODE == kWsScatter) {
    int lo = 0, hi = p.V;  // largest v with ws_tiles[v] <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.ws_tiles + mid) <= u) lo = mid; else hi = mid;
    }
    t.v = lo;
    // offset lo's list starts at lo * n and holds offs[lo + 1] - offs[lo] entries
    const int64_t seg = static_cast<int64_t>(lo) * p.n;
    const int64_t seg_end = seg + (__ldg(p.offs + lo + 1) - __ldg(p.offs + lo));
    t.lb = seg + static_cast<int64_t>(u - __ldg(p.ws_tiles + lo)) * kRows;
    t.nrows = static_cast<int>(min(static_cast<int64_t>(kRows), seg_end - t.lb));
  } else {
    t.row0 = static_cast<int64_t>(u) * kRows * T;
    t.nrows = static_cast<int>(min(static_cast<int64_t>(kRows) * T, p.n - t.row0));
  }
  return t;
}

// Offsets present in any tile of an output-stationary unit, centre included.
template <int T>
__device__ __forceinline__ uint4 unit_mask(const TcParams& p, int u) {
  uint4 m = tile_mask(p, u * T);
#pragma unroll
  for (int k = 1; k < T; ++k) {
    if (u * T + k < p.num_tiles) {
      const uint4 x = tile_mask(p, u * T + k);
      m.x |= x.x;
      m.y |= x.y;
      m.z |= x.z;
      m.w |= x.w;
    }
  }
  return m;
}

template <int MODE, int T>
__device__ __forceinline__ int unit_kblocks(const TcParams& p, int u, int P) {
  if (MODE != kOutputStationary) return P;
  const uint4 m = unit_mask<T>(p, u);
  return (__popc(m.x) + __popc(m.y) + __popc(m.z) + __popc(m.w)) * P;
}

// Register budget: 4 producer warps run three CTAs per SM, 8 run two, 16 one.
// TT (output-stationary): the neighbour indices come from the map's
// tile-transposed table (p.tnbr) instead of nbr through perm.
template <int BK, int MODE, bool BF16, int NPW, int T, bool TT>
__global__ void __launch_bounds__((NPW + 6) * 32, NPW == 4 ? 3 : (NPW == 8 ? 2 : 1))
    k_conv_tc(const TcParams p, const __grid_constant__ CUtensorMap wmap) {
  constexpr int ROWB = BK * 2;          // bytes per tile row (= swizzle width)
  constexpr int A_PART = kRows * ROWB;  // one 128-row MMA operand of a sub-block
  constexpr int A_SUB = T * A_PART;     // one (offset, panel) sub-block of A
  constexpr int CPR = ROWB / 16;        // 16-byte chunks per row
  constexpr int RW = kRows * T / NPW;   // unit rows per producer warp
  constexpr int RSTEP = 32 / CPR;       // rows covered by one warp instruction
  constexpr int RPT = RW / RSTEP;       // copy instructions per producer thread and sub-block
  static_assert(RPT >= 1 && RW <= 32 && kRows % RW == 0, "producer warps must cover whole rows of one part");
  static_assert(MODE == kOutputStationary || T == 1, "weight-stationary units are single tiles");
  constexpr uint32_t LAYOUT = layout_code<BK>();
  constexpr uint32_t SBO = 8 * ROWB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages, G = p.group, NB = p.nbuf;
  const int B_SUB = p.c_out * ROWB;
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * G * A_SUB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * G * B_SUB);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kBarriers);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_dirty = s_tmem + 4;  // [NPW][S * G] zero-row masks of the producer warps

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.c_in / BK;
  const int V = p.V;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const uint32_t accf0 = smem_u32(bars + 2 * kMaxStages), acce0 = smem_u32(bars + 2 * kMaxStages + 2);
  const uint32_t done_bar = smem_u32(bars + 2 * kMaxStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // one copy-completion arrival per producer thread + the weight loader's expect_tx
      mbar_init(full0 + 8 * s, NPW * 32 + 1);
      mbar_init(empty0 + 8 * s, 1);  // one tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);   // one tcgen05.commit per unit
      mbar_init(acce0 + 8 * b, 4);   // one arrival per epilogue warp
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
    const int chunk = lane % CPR;      // 16-byte chunk of a row
    const int rw0 = RW * warp;         // this warp's unit rows: rw0 .. rw0 + RW - 1, all in one part
    const int part_off = (rw0 / kRows) * A_PART;
    const int rp0 = rw0 % kRows;       // first of them within the part
    // per (stage, sub-block): bit j set while row rw0 + j of that buffer may
    // hold data; clear bits are rows known to be zero, which an absent
    // neighbour then needs no zero-filling copy for
    uint32_t* dirty = s_dirty + warp * S * G;
    for (int e = lane; e < S * G; e += 32) dirty[e] = 0xFFFFFFFFu;
    __syncwarp();
    uint32_t it = 0;
    for (int u = blockIdx.x; u < p.num_units && !*s_abort; u += gridDim.x) {
      const TileInfo t = tile_info<MODE, T>(p, u);
      uint4 m = make_uint4(0, 0, 0, 0);
      int v = t.v;
      if (MODE == kOutputStationary) {
        m = unit_mask<T>(p, u);
        v = next_present(m, -1, V);
      }
      const int nkb = unit_kblocks<MODE, T>(p, u, P);
      // Lane j < RW of warp w fetches the source row of unit row RW w + j for
      // an offset; the warp's lanes then take the rows they copy by shuffle,
      // so each offset costs one index load per row, issued an offset ahead.
      // this lane's row of the neighbour table (the tile row itself, or the
      // row the signature sort put there)
      // (TT: this lane's entries in the tile-transposed table, 128 apart per
      // offset; a warp's rows of one offset are consecutive ints)
      int64_t trow_lane = 0;
      if (MODE == kOutputStationary && lane < RW && rw0 + lane < t.nrows) {
        const int64_t k = t.row0 + rw0 + lane;
        if constexpr (TT) trow_lane = (k >> 7) * static_cast<int64_t>(V) * 128 + (k & 127);
        else trow_lane = p.perm ? static_cast<int64_t>(__ldg(p.perm + k)) : k;
      }
      auto fetch = [&](int vv) -> int {
        const int r = rw0 + lane;
        if (vv >= V || lane >= RW || r >= t.nrows) return -1;
        if constexpr (MODE == kOutputStationary && TT) return __ldg(p.tnbr + trow_lane + static_cast<int64_t>(vv) * 128);
        if (MODE == kOutputStationary) return __ldg(p.nbr + trow_lane * V + vv);
        if (MODE == kWsScatter) return __ldg(p.in_rows + t.lb + r);
        return static_cast<int>(t.row0 + r);
      };
      int src[RPT];
      uint32_t valid = 0;  // bit j: row rw0 + j has a neighbour for the current offset
      auto spread = [&](int cur) {
        valid = __ballot_sync(0xffffffffu, cur >= 0);
#pragma unroll
        for (int k = 0; k < RPT; ++k) src[k] = __shfl_sync(0xffffffffu, cur, lane / CPR + RSTEP * k);
      };
      spread(fetch(v));
      // neighbour indices of the next kAhead present offsets, loads in flight
      int va[kAhead], na[kAhead];
      {
        int vv = v;
#pragma unroll
        for (int d = 0; d < kAhead; ++d) {
          vv = MODE == kOutputStationary ? next_present(m, vv, V) : V;
          va[d] = vv;
          na[d] = MODE == kOutputStationary ? fetch(vv) : -1;
        }
      }
      int pnl = 0;
      for (int kb = 0; kb < nkb; kb += G, ++it) {
        const int s = static_cast<int>(it % S);
        const uint32_t ph = (it / S) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * s, ph ^ 1u, s_abort))) {
          *s_abort = 1;
          break;
        }
        const int gc = min(G, nkb - kb);
        for (int g = 0; g < gc; ++g) {
          const uint32_t a_base = smem_u32(sA + (s * G + g) * A_SUB + part_off);
          const uint32_t was = dirty[s * G + g];
#pragma unroll
          for (int k = 0; k < RPT; ++k) {
            const int rl = lane / CPR + RSTEP * k;
            const int r = rp0 + rl;  // row within the part
            const int j = src[k];
            if (((valid | was) >> rl) & 1u) {
              const uint8_t* g_src = p.feats + (static_cast<size_t>(j < 0 ? 0 : j) * p.c_in +
                                                static_cast<size_t>(pnl) * BK) * 2 + chunk * 16;
              cp_async_16(a_base + r * ROWB + ((chunk ^ swz<BK>(r)) << 4), g_src, j >= 0 ? 16u : 0u);
            }
          }
          __syncwarp();
          if (lane == 0) dirty[s * G + g] = valid;
          if (++pnl == P) {
            pnl = 0;
            if (MODE == kOutputStationary) {
              v = va[0];
              if (v < V) {
                spread(na[0]);
#pragma unroll
                for (int d = 0; d + 1 < kAhead; ++d) {
                  va[d] = va[d + 1];
                  na[d] = na[d + 1];
                }
                va[kAhead - 1] = next_present(m, va[kAhead - 1], V);
                na[kAhead - 1] = fetch(va[kAhead - 1]);
              }
            }
          }
        }
        // every thread's arrival fires once its copies of this stage landed
        cp_async_arrive_noinc(full0 + 8 * s);
      }
    }
    cp_async_wait_all();
  } else if (warp == NPW + 5) {
    // ======================================================= weight loader
    // One thread walks the producers' (unit, offset, panel) sequence and
    // bulk-copies the matching W slices into each stage, arming the stage's
    // barrier with their byte count; it also prefetches each next unit's block
    // of the neighbour table into L2.
    if (lane == 0) {
      uint32_t it = 0;
      // each unit's block of neighbour indices into L2: its tiles of the
      // tile-transposed table, or its rows of nbr when those are contiguous
      auto prefetch_unit = [&](int uu) {
        const TileInfo tu = tile_info<MODE, T>(p, uu);
        if constexpr (TT) {
          const int nt = (tu.nrows + kRows - 1) / kRows;
          bulk_prefetch_l2(p.tnbr + (tu.row0 >> 7) * static_cast<int64_t>(V) * 128,
                           static_cast<uint32_t>(nt) * static_cast<uint32_t>(V) * 512u);
        } else {
          const uint32_t bytes = (static_cast<uint32_t>(tu.nrows) * V * 4) & ~15u;
          if (bytes) bulk_prefetch_l2(p.nbr + tu.row0 * V, bytes);
        }
      };
      if (MODE == kOutputStationary && (TT || !p.perm) && static_cast<int>(blockIdx.x) < p.num_units)
        prefetch_unit(blockIdx.x);
      for (int u = blockIdx.x; u < p.num_units && !*s_abort; u += gridDim.x) {
        uint4 m = make_uint4(0, 0, 0, 0);
        int bv = tile_info<MODE, T>(p, u).v;
        if (MODE == kOutputStationary) {
          m = unit_mask<T>(p, u);
          bv = next_present(m, -1, V);
          const int nu = u + gridDim.x;
          if (nu < p.num_units && (TT || !p.perm)) prefetch_unit(nu);
        }
        const int nkb = unit_kblocks<MODE, T>(p, u, P);
        int bp = 0;
        for (int kb = 0; kb < nkb; kb += G, ++it) {
          const int s = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, s_abort)) {
            *s_abort = 1;
            break;
          }
          const int gc = min(G, nkb - kb);
          mbar_arrive_expect_tx(full0 + 8 * s, static_cast<uint32_t>(gc * B_SUB));
          for (int g = 0; g < gc; ++g) {
            const uint32_t dstb = smem_u32(sB + (s * G + g) * B_SUB);
            if (p.wmode == 1) {
              // W[v] rows bp * BK .. + BK (input channels), wnb output channels per box
              const int y = bv * p.c_in + bp * BK;
              for (int i = 0; i * p.wnb < p.c_out; ++i)
                tma_load_2d(dstb + static_cast<uint32_t>(i * BK * p.wnb * 2), &wmap, i * p.wnb, y, full0 + 8 * s);
            } else if (p.wmode == 2) {
              // rows (V-1-v) * c_out .. + c_out of the forward W, channels bp * BK .. + BK
              tma_load_2d(dstb, &wmap, bp * BK, (V - 1 - bv) * p.c_out, full0 + 8 * s);
            } else {
              bulk_g2s(dstb, p.wimg + (static_cast<size_t>(bv) * P + bp) * B_SUB, static_cast<uint32_t>(B_SUB),
                       full0 + 8 * s);
            }
            if (++bp == P) {
              bp = 0;
              if (MODE == kOutputStationary) bv = next_present(m, bv, V);
            }
          }
        }
      }
      // the weight copies of the last stages have landed before the CTA may exit
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t k = first; k < it; ++k)
        if (!mbar_drain(full0 + 8 * (k % S), (k / S) & 1u)) *s_abort = 1;
    }
    __syncwarp();
  } else if (warp == NPW) {
    // ======================================================= MMA issuer
    if (lane == 0) {
      // B MN-major (wmode 1: the slice as W holds it, output channels
      // contiguous) or K-major (the packed image's layout)
      const bool b_mn = p.wmode == 1;
      const uint32_t idesc = make_idesc(BF16, kRows, p.c_out) | (b_mn ? (1u << 16) : 0u);
      // descriptor halves: low = start address >> 4 (14 bits; shared memory
      // is below 256 KB, so offsets add without carry) | LBO; high = SBO,
      // version 1, swizzle layout
      const uint64_t d0 = smem_desc(smem_u32(sA), SBO, LAYOUT);
      const uint32_t desc_hi = static_cast<uint32_t>(d0 >> 32);
      const uint32_t a_lo0 = static_cast<uint32_t>(d0);
      uint32_t b_lo0, b_hi, b_step;
      if (b_mn) {
        // rows of wnb * 2 bytes (one input channel each), 8-row atoms along
        // K, boxes of wnb output channels BK rows apart along N; a K = 16
        // step advances 16 rows
        const uint32_t rb = static_cast<uint32_t>(p.wnb * 2);
        const uint64_t bd = smem_desc_mn(smem_u32(sB), BK * rb, 8 * rb, rb == 128 ? 2u : (rb == 64 ? 4u : 6u));
        b_lo0 = static_cast<uint32_t>(bd);
        b_hi = static_cast<uint32_t>(bd >> 32);
        b_step = 16 * rb / 16;
      } else {
        b_lo0 = static_cast<uint32_t>(smem_desc(smem_u32(sB), SBO, LAYOUT));
        b_hi = desc_hi;
        b_step = 2;  // 16 channels of a K-major row: 32 bytes
      }
      uint32_t it = 0;
      int j = 0;
      // output-stationary: each unit's offset mask is loaded one unit ahead,
      // so the issuer does not wait on it when the unit's first stage is
      // already full (measured: 100k voxels 37.9 -> 37.0 us; no change at
      // 1M and 2M voxels)
      uint4 m_nx = make_uint4(0, 0, 0, 0);
      if (MODE == kOutputStationary && static_cast<int>(blockIdx.x) < p.num_units) m_nx = unit_mask<T>(p, blockIdx.x);
      for (int u = blockIdx.x; u < p.num_units && !*s_abort; u += gridDim.x, ++j) {
        int nkb = P;
        if (MODE == kOutputStationary) {
          nkb = (__popc(m_nx.x) + __popc(m_nx.y) + __popc(m_nx.z) + __popc(m_nx.w)) * P;
          if (u + static_cast<int>(gridDim.x) < p.num_units) m_nx = unit_mask<T>(p, u + gridDim.x);
        }
        const int b = j % NB;
        if (!mbar_wait(acce0 + 8 * b, ((j / NB) & 1) ^ 1, s_abort)) {
          *s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * T * p.acc_cols);
        uint32_t accumulate = 0;
        for (int kb = 0; kb < nkb; kb += G, ++it) {
          const int s = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(full0 + 8 * s, ph, s_abort)) {
            *s_abort = 1;
            break;
          }
          // the producers' cp.async writes are generic-proxy writes: order
          // them before the tensor core's (async-proxy) reads
          fence_proxy_async_smem();
          tc_fence_after();
          const int gc = min(G, nkb - kb);
          for (int g = 0; g < gc; ++g) {
            const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(((s * G + g) * A_SUB) >> 4);
            const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(((s * G + g) * B_SUB) >> 4);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
              for (int tp = 0; tp < T; ++tp)
                tc_mma_lohi2(d + static_cast<uint32_t>(tp * p.acc_cols), a_lo + tp * (A_PART >> 4) + 2 * k, desc_hi,
                             b_lo + b_step * k, b_hi, idesc, accumulate);
              accumulate = 1;
            }
          }
          tc_commit(empty0 + 8 * s);
        }
        tc_commit(accf0 + 8 * b);  // arrives once every MMA of the unit has completed
      }
      // all tcgen05 work of this thread has completed before TMEM is released
      tc_commit(done_bar);
      if (!mbar_drain(done_bar, 0)) *s_abort = 1;
    }
    __syncwarp();
  } else {
    // ======================================================= epilogue (warps NPW+1 .. NPW+4)
    const int q = warp & 3;             // TMEM lane quadrant of this warp
    int j = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++j) {
      const TileInfo t = tile_info<MODE, T>(p, u);
      const int b = j % NB;
      if (*s_abort || !mbar_wait(accf0 + 8 * b, (j / NB) & 1, s_abort)) {
        *s_abort = 1;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int tp = 0; tp < T; ++tp) {
        const int r = tp * kRows + q * 32 + lane;  // unit row held by this thread
        const uint32_t trow = tmem + static_cast<uint32_t>((b * T + tp) * p.acc_cols) +
                              (static_cast<uint32_t>(q * 32) << 16);
        int dst_row = -1;
        if (r < t.nrows) {
          if (MODE == kWsScatter) dst_row = __ldg(p.out_rows + t.lb + r);
          else if (MODE == kOutputStationary && p.order) dst_row = __ldg(p.order + t.row0 + r);
          else dst_row = static_cast<int>(t.row0 + r);
        }
        if (MODE == kOutputStationary && p.epi == 0 && (p.c_out & 31) == 0) {
          // 32 columns at a time, transposed across groups of four lanes so
          // that a store instruction writes 64 contiguous bytes of each of 8
          // rows (instead of 16 bytes of each of 32): lane 4 g + c stores
          // 16-byte chunk c of rows 4 g + i, i = 0..3
          int drow[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) drow[i] = __shfl_sync(0xffffffffu, dst_row, (lane & ~3) + i);
          const int c = lane & 3;
          for (int c0 = 0; c0 < p.c_out; c0 += 32) {
            float a[32];
            tmem_ld32(trow + static_cast<uint32_t>(c0), a);
            if (p.relu) {
#pragma unroll
              for (int k = 0; k < 32; ++k) a[k] = fmaxf(a[k], 0.0f);
            }
            uint4 x[4];  // x[k]: columns c0 + 8 k .. c0 + 8 k + 7 of this lane's row
#pragma unroll
            for (int k = 0; k < 4; ++k)
              x[k] = make_uint4(pack2<BF16>(a[8 * k], a[8 * k + 1]), pack2<BF16>(a[8 * k + 2], a[8 * k + 3]),
                                pack2<BF16>(a[8 * k + 4], a[8 * k + 5]), pack2<BF16>(a[8 * k + 6], a[8 * k + 7]));
            // butterfly over lane distances 2 and 1: afterwards lane 4 g + c
            // holds chunk c of row 4 g + i in x[i]
#pragma unroll
            for (int m = 2; m >= 1; m >>= 1) {
              const bool up = (lane & m) != 0;
#pragma unroll
              for (int lo = 0; lo < 4; ++lo) {
                if (lo & m) continue;
                const int hi = lo | m;
                const uint4 snd = up ? x[lo] : x[hi];
                uint4 rcv;
                rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
                rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
                rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, m);
                rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, m);
                if (up) x[lo] = rcv;
                else x[hi] = rcv;
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (drow[i] >= 0)
                *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(drow[i]) * p.c_out + c0 + 8 * c) * 2) = x[i];
          }
          continue;
        }
        for (int c0 = 0; c0 < p.c_out; c0 += 16) {
          float a[16];
          tmem_ld16(trow + static_cast<uint32_t>(c0), a);
          if (dst_row < 0) continue;
          if (MODE == kOutputStationary && p.epi == 1) {
            // first part of a split layer: fp32 partial sums
            float4* dst = reinterpret_cast<float4*>(p.acc + static_cast<int64_t>(dst_row) * p.c_out + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
            continue;
          }
          if (MODE == kOutputStationary) {
            if (p.epi == 2) {  // last part: add the earlier parts' sums
              const float4* src = reinterpret_cast<const float4*>(p.acc + static_cast<int64_t>(dst_row) * p.c_out + c0);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 q = __ldcs(src + k);
                a[4 * k] += q.x;
                a[4 * k + 1] += q.y;
                a[4 * k + 2] += q.z;
                a[4 * k + 3] += q.w;
              }
            }
            if (p.relu) {
#pragma unroll
              for (int k = 0; k < 16; ++k) a[k] = fmaxf(a[k], 0.0f);
            }
            uint4 lo, hi;
            lo.x = pack2<BF16>(a[0], a[1]);
            lo.y = pack2<BF16>(a[2], a[3]);
            lo.z = pack2<BF16>(a[4], a[5]);
            lo.w = pack2<BF16>(a[6], a[7]);
            hi.x = pack2<BF16>(a[8], a[9]);
            hi.y = pack2<BF16>(a[10], a[11]);
            hi.z = pack2<BF16>(a[12], a[13]);
            hi.w = pack2<BF16>(a[14], a[15]);
            uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(dst_row) * p.c_out + c0) * 2);
            dst[0] = lo;
            dst[1] = hi;
          } else if (MODE == kWsScatter) {
            float4* dst = reinterpret_cast<float4*>(p.acc + static_cast<int64_t>(dst_row) * p.c_out + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              atomicAdd(dst + k, make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]));
          } else {
            float4* dst = reinterpret_cast<float4*>(p.acc + static_cast<int64_t>(dst_row) * p.c_out + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
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

// W [V, c_in, c_out] -> per (offset, panel) image of c_out rows x BK channels,
// K-major, chunk-swizzled exactly as the kernel's shared-memory B tile.  With
// wt, W is a forward layer's [V, c_out, c_in] and the image is that of
// W'[v] = W[V-1-v]^T (the layer that maps output gradients to input ones).
template <int BK>
__global__ void __launch_bounds__(256) k_pack_weights(const uint16_t* __restrict__ W, uint8_t* __restrict__ img,
                                                      int V, int c_in, int c_out, int wt) {
  constexpr int ROWB = BK * 2, CPR = ROWB / 16;
  const int P = c_in / BK;
  const int64_t total = static_cast<int64_t>(V) * P * c_out * CPR;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % CPR);
    const int co = static_cast<int>((idx / CPR) % c_out);
    const int64_t vp = idx / (static_cast<int64_t>(CPR) * c_out);
    const int pnl = static_cast<int>(vp % P);
    const int v = static_cast<int>(vp / P);
    uint16_t e[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int ci = pnl * BK + c * 8 + k;
      e[k] = wt ? __ldg(W + (static_cast<int64_t>(V - 1 - v) * c_out + co) * c_in + ci)
                : __ldg(W + (static_cast<int64_t>(v) * c_in + ci) * c_out + co);
    }
    uint4 w;
    w.x = e[0] | (static_cast<uint32_t>(e[1]) << 16);
    w.y = e[2] | (static_cast<uint32_t>(e[3]) << 16);
    w.z = e[4] | (static_cast<uint32_t>(e[5]) << 16);
    w.w = e[6] | (static_cast<uint32_t>(e[7]) << 16);
    *reinterpret_cast<uint4*>(img + vp * (static_cast<int64_t>(c_out) * ROWB) + static_cast<int64_t>(co) * ROWB +
                              ((c ^ swz<BK>(co)) << 4)) = w;
  }
}

// fp32 accumulator -> output dtype (optional ReLU), 4 values per thread step.
template <bool BF16>
__global__ void __launch_bounds__(256) k_cast_out(const float4* __restrict__ acc, uint2* __restrict__ out, int64_t n4,
                                                  int relu) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = __ldg(acc + i);
    if (relu) {
      a.x = fmaxf(a.x, 0.f);
      a.y = fmaxf(a.y, 0.f);
      a.z = fmaxf(a.z, 0.f);
      a.w = fmaxf(a.w, 0.f);
    }
    out[i] = make_uint2(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w));
  }
}

// ------------------------------------------------------------ host side --
struct Plan {
  int bk;           // channels per K panel (16, 32 or 64)
  int group;        // (offset, panel) sub-blocks per pipeline stage
  int stages;
  int npw;          // producer warps per CTA (4, 8 or 16)
  int t;            // 128-row tiles per output-stationary work unit (1 or 2)
  int nbuf;         // accumulator buffers
  int ctas_per_sm;  // as shared memory, TMEM and threads allow
  size_t smem;
  int acc_cols;
  int tmem_cols;
};

int pick_bk(int c_in) { return c_in % 64 == 0 ? 64 : (c_in % 32 == 0 ? 32 : 16); }

size_t plan_smem(const Plan& pl, size_t stage_bytes) {  // stage_bytes: one stage's A and B
  return 1024 /*alignment slack*/ + 8 * kBarriers + 16 + static_cast<size_t>(pl.npw) * pl.stages * pl.group * 4 +
         pl.stages * stage_bytes;
}

// Pipeline shape.  The gathers are bound by how many cp.async instructions
// the SM's warps keep issuing: one warp sustains about 3 B/clk of 128-byte
// rows whatever its depth, and the SM's rate grows with its producer warps
// (measured up to about 13 TB/s per GPU).  Per stage the tensor core reads
// A (gathered rows) and B (a weight slice); B is re-read for every unit, so
// at C_out = 256 two tiles share it.  The plan keeps three stages, fits as
// many CTAs per SM as shared memory (about 220 KB) and TMEM (512 columns)
// allow, and gives each CTA 4 producer warps at three CTAs per SM, else 8.
// Developer overrides for measurement sweeps (environment, read per call):
// SC_DEV_BK, SC_DEV_T, SC_DEV_STAGES, SC_DEV_GROUP, SC_DEV_NPW, SC_DEV_NBUF, SC_DEV_CPS
// (an upper bound), SC_DEV_FORCECPS (launch that many CTAs per SM),
// SC_DEV_MAX_CARVEOUT (keep the largest shared-memory carveout),
// SC_DEV_NO_WEIGHT_TMA (pack W instead of reading its slices by TMA) and
// SC_DEV_VERBOSE (print each launch's plan).  None changes the result.
bool make_plan(int c_in, int c_out, bool output_stationary, Plan* pl) {
  pl->bk = pick_bk(c_in);
  if (const char* e = getenv("SC_DEV_BK")) { const int bk = atoi(e); if ((bk == 16 || bk == 32 || bk == 64) && c_in % bk == 0) pl->bk = bk; }
  int cols = 32;
  while (cols < c_out) cols <<= 1;
  pl->acc_cols = cols;
  // At C_out = 256 a stage moves twice as many weight bytes as feature
  // bytes; two tiles per unit share each weight slice (measured: a third
  // less time at 128->256 and 256->256; no gain at C_out = 128, where two
  // CTAs per SM with one tile each do better).
  pl->t = (output_stationary && pl->bk == 64 && c_out >= 256) ? 2 : 1;
  if (const char* e = getenv("SC_DEV_T")) pl->t = (atoi(e) == 2 && output_stationary && pl->bk >= 32) ? 2 : 1;
  pl->nbuf = 2 * pl->t * cols <= 512 ? 2 : 1;
  if (const char* e = getenv("SC_DEV_NBUF")) pl->nbuf = atoi(e) == 1 ? 1 : pl->nbuf;
  pl->tmem_cols = pl->nbuf * pl->t * cols;
  if (pl->tmem_cols > 512) return false;
  const size_t a = static_cast<size_t>(kRows) * pl->bk * 2 * pl->t;
  const size_t b = static_cast<size_t>(c_out) * pl->bk * 2;
  // sub-blocks per stage: stages of about 24 KB
  int g = static_cast<int>((24 * 1024) / (a + b));
  if (g < 1) g = 1;
  if (g > 4) g = 4;
  pl->group = g;
  pl->stages = 3;
  if (const char* e = getenv("SC_DEV_STAGES")) pl->stages = atoi(e);
  if (const char* e = getenv("SC_DEV_GROUP")) pl->group = atoi(e);
  pl->stages = pl->stages < 2 ? 2 : (pl->stages > kMaxStages ? kMaxStages : pl->stages);
  pl->group = pl->group < 1 ? 1 : (pl->group > 4 ? 4 : pl->group);
  const size_t stage = pl->group * (a + b);
  // a warp instruction covers whole rows, and a warp's rows lie in one tile
  const int rstep = 32 / (pl->bk * 2 / 16);
  const int max_npw = kRows * pl->t / rstep < 16 ? kRows * pl->t / rstep : 16;
  const int min_npw = pl->t == 2 ? 8 : 4;
  pl->npw = min_npw;
  pl->smem = plan_smem(*pl, stage);
  if (pl->smem > 220 * 1024) return false;
  int cps = static_cast<int>((220 * 1024) / pl->smem);
  if (cps * pl->tmem_cols > 512) cps = 512 / pl->tmem_cols;
  if (cps < 1) cps = 1;
  pl->npw = cps >= 3 ? 4 : 8;  // measured: 16 producer warps were never faster than 8
  if (const char* e = getenv("SC_DEV_NPW")) pl->npw = atoi(e);
  if (pl->npw != 4 && pl->npw != 8 && pl->npw != 16) pl->npw = 4;
  if (pl->npw > max_npw) pl->npw = max_npw;
  if (pl->npw < min_npw) pl->npw = min_npw;
  pl->smem = plan_smem(*pl, stage);
  if (pl->smem > 220 * 1024) return false;
  cps = static_cast<int>((220 * 1024) / pl->smem);
  if (cps * pl->tmem_cols > 512) cps = 512 / pl->tmem_cols;
  const int threads = (pl->npw + 6) * 32;
  if (cps * threads > 2048) cps = 2048 / threads;
  if (const char* e = getenv("SC_DEV_CPS")) { int c = atoi(e); if (c < cps) cps = c; }
  pl->ctas_per_sm = cps < 1 ? 1 : cps;
  return true;
}

template <int BK, int MODE, bool BF16, int NPW, int T, bool TT>
sc_status launch_tc(const TcParams& prm, const CUtensorMap& wmap, const Plan& pl, cudaStream_t s, const char* name) {
  auto kern = k_conv_tc<BK, MODE, BF16, NPW, T, TT>;
  constexpr int threads = (NPW + 6) * 32;
  int num_regs = 0;
  sc_status st = kernel_setup(reinterpret_cast<const void*>(kern), pl.smem, &num_regs);
  if (st) return st;
  // resident CTAs per SM: the plan's count, or fewer if registers say so
  const int regs_cta = ((num_regs + 7) / 8) * 8 * threads;
  const int fit = regs_cta > 0 ? 65536 / regs_cta : pl.ctas_per_sm;
  int cps = fit < pl.ctas_per_sm ? (fit < 1 ? 1 : fit) : pl.ctas_per_sm;
  if (const char* ev = getenv("SC_DEV_FORCECPS")) cps = atoi(ev);
  // carveout for exactly these CTAs: the remainder is L1, where the
  // producers' neighbour-index loads stay resident across a tile's offsets
  // (with the largest carveout they were re-read from L2 about 7 times)
  if (!getenv("SC_DEV_MAX_CARVEOUT")) {
    st = kernel_carveout(reinterpret_cast<const void*>(kern), cps, pl.smem);
    if (st) return st;
  }
  const int slots = device_sm_count() * cps;
  const int grid = prm.num_units < slots ? prm.num_units : slots;
  if (getenv("SC_DEV_VERBOSE")) {
    fprintf(stderr, "%s: bk %d npw %d t %d nbuf %d group %d stages %d smem %zu plan cps %d fit %d grid %d regs %d\n",
            name, BK, NPW, T, pl.nbuf, pl.group, pl.stages, pl.smem, pl.ctas_per_sm, fit, grid, num_regs);
  }
  SC_LAUNCH(name, s, kern<<<grid, threads, pl.smem, s>>>(prm, wmap));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, name);
}

template <int BK, int MODE, bool BF16, bool TT>
sc_status launch_npw(const TcParams& prm, const CUtensorMap& wm, const Plan& pl, cudaStream_t s, const char* name) {
  if constexpr (BK == 16) {
    return pl.npw == 8 ? launch_tc<BK, MODE, BF16, 8, 1, TT>(prm, wm, pl, s, name)
                       : launch_tc<BK, MODE, BF16, 4, 1, TT>(prm, wm, pl, s, name);
  } else {
    if constexpr (MODE == kOutputStationary) {
      if (pl.t == 2)
        return pl.npw == 16 ? launch_tc<BK, MODE, BF16, 16, 2, TT>(prm, wm, pl, s, name)
                            : launch_tc<BK, MODE, BF16, 8, 2, TT>(prm, wm, pl, s, name);
    }
    switch (pl.npw) {
      case 16: return launch_tc<BK, MODE, BF16, 16, 1, TT>(prm, wm, pl, s, name);
      case 8: return launch_tc<BK, MODE, BF16, 8, 1, TT>(prm, wm, pl, s, name);
      default: return launch_tc<BK, MODE, BF16, 4, 1, TT>(prm, wm, pl, s, name);
    }
  }
}

template <int MODE, bool TT>
sc_status dispatch_bk(const TcParams& prm, const CUtensorMap& wm, const Plan& pl, bool bf16, cudaStream_t s,
                      const char* name) {
  switch (pl.bk) {
    case 64:
      return bf16 ? launch_npw<64, MODE, true, TT>(prm, wm, pl, s, name)
                  : launch_npw<64, MODE, false, TT>(prm, wm, pl, s, name);
    case 32:
      return bf16 ? launch_npw<32, MODE, true, TT>(prm, wm, pl, s, name)
                  : launch_npw<32, MODE, false, TT>(prm, wm, pl, s, name);
    default:
      return bf16 ? launch_npw<16, MODE, true, TT>(prm, wm, pl, s, name)
                  : launch_npw<16, MODE, false, TT>(prm, wm, pl, s, name);
  }
}

// wm: the weights' tensor map when prm.wmode reads W by TMA (else unused)
template <int MODE>
sc_status dispatch_tc(const TcParams& prm, const Plan& pl, bool bf16, cudaStream_t s, const char* name,
                      const CUtensorMap* wm = nullptr) {
  if (prm.num_units <= 0) return SC_OK;
  static const CUtensorMap kNoMap{};
  const CUtensorMap& m = wm ? *wm : kNoMap;
  if constexpr (MODE == kOutputStationary) {
    if (prm.tnbr) return dispatch_bk<MODE, true>(prm, m, pl, bf16, s, name);
  }
  return dispatch_bk<MODE, false>(prm, m, pl, bf16, s, name);
}

sc_status pack_weights(const ConvArgs& a, int bk, uint8_t* img) {
  const int V = a.m->V;
  const int64_t chunks = static_cast<int64_t>(V) * (a.c_in / bk) * a.c_out * (bk * 2 / 16);
  int grid = static_cast<int>((chunks + 255) / 256);
  if (grid > device_sm_count() * 16) grid = device_sm_count() * 16;
  if (grid < 1) grid = 1;
  const uint16_t* W = static_cast<const uint16_t*>(a.W);
  switch (bk) {
    case 64: SC_LAUNCH("pack_weights", a.stream, k_pack_weights<64><<<grid, 256, 0, a.stream>>>(W, img, V, a.c_in, a.c_out, a.wt ? 1 : 0)); break;
    case 32: SC_LAUNCH("pack_weights", a.stream, k_pack_weights<32><<<grid, 256, 0, a.stream>>>(W, img, V, a.c_in, a.c_out, a.wt ? 1 : 0)); break;
    default: SC_LAUNCH("pack_weights", a.stream, k_pack_weights<16><<<grid, 256, 0, a.stream>>>(W, img, V, a.c_in, a.c_out, a.wt ? 1 : 0)); break;
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "pack_weights launch");
}

TcParams base_params(const ConvArgs& a, const Plan& pl, const uint8_t* img) {
  TcParams p{};
  p.feats = static_cast<const uint8_t*>(a.feats);
  p.wimg = img;
  p.out = static_cast<uint8_t*>(a.out);
  p.nbr = a.m->nbr;
  p.order = a.m->perm ? a.m->conv_order : a.m->order;
  p.perm = a.m->perm;
  p.tnbr = a.m->tnbr;
  p.present = reinterpret_cast<const uint4*>(a.m->present);
  p.in_rows = a.m->in_rows;
  p.out_rows = a.m->out_rows;
  p.offs = a.m->offs;
  p.ws_tiles = a.m->ws_tiles;
  p.n = a.m->n;
  p.num_tiles = static_cast<int>((a.m->n + kRows - 1) / kRows);
  p.num_units = (p.num_tiles + pl.t - 1) / pl.t;
  p.V = a.m->V;
  p.c_in = a.c_in;
  p.c_out = a.c_out;
  p.relu = a.relu ? 1 : 0;
  p.stages = pl.stages;
  p.group = pl.group;
  p.acc_cols = pl.acc_cols;
  p.tmem_cols = pl.tmem_cols;
  p.nbuf = pl.nbuf;
  p.status = a.m->status;
  p.epi = 0;
  p.centre_in = 1;
  return p;
}

bool fused_ok(const ConvArgs& a, Plan* pl) {
  return a.dtype != SC_F32 && a.m->V <= 128 && make_plan(a.c_in, a.c_out, true, pl);
}

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry
// point (the library does not link the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

CUtensorMapSwizzle swizzle_for(int row_bytes) {
  return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// The fused layer's weight slices read by TMA straight from W (no packed
// image): the tensor map of W and the mode (TcParams::wmode).  False when the
// shapes do not fit a TMA box (then the caller packs W as before).
// Developer override SC_DEV_NO_WEIGHT_TMA=1: always pack.
bool setup_weight_tma(const ConvArgs& a, const Plan& pl, TcParams* p, CUtensorMap* wmap) {
  if (getenv("SC_DEV_NO_WEIGHT_TMA")) return false;
  if (reinterpret_cast<uintptr_t>(a.W) % 16) return false;
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const int V = a.m->V, BK = pl.bk;
  cuuint64_t dims[2];
  cuuint64_t strides[1];
  cuuint32_t box[2];
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw;
  int mode, nb = 0;
  if (!a.wt) {
    // W [V][c_in][c_out]: rows v * c_in + ci, columns co; a slice is BK rows,
    // fetched as c_out / nb boxes of nb columns (a 32, 64 or 128-byte swizzle)
    nb = a.c_out >= 64 ? 64 : a.c_out;
    if ((nb != 16 && nb != 32 && nb != 64) || a.c_out % nb) return false;
    dims[0] = static_cast<cuuint64_t>(a.c_out);
    dims[1] = static_cast<cuuint64_t>(V) * a.c_in;
    strides[0] = static_cast<cuuint64_t>(a.c_out) * 2;
    box[0] = static_cast<cuuint32_t>(nb);
    box[1] = static_cast<cuuint32_t>(BK);
    sw = swizzle_for(nb * 2);
    mode = 1;
  } else {
    // the forward W [V][c_out][c_in] (this call's c_out rows per offset, its
    // c_in channels contiguous): one box of c_out rows x BK channels
    if (a.c_out > 256) return false;
    dims[0] = static_cast<cuuint64_t>(a.c_in);
    dims[1] = static_cast<cuuint64_t>(V) * a.c_out;
    strides[0] = static_cast<cuuint64_t>(a.c_in) * 2;
    box[0] = static_cast<cuuint32_t>(BK);
    box[1] = static_cast<cuuint32_t>(a.c_out);
    sw = swizzle_for(BK * 2);
    mode = 2;
  }
  const CUresult r = enc(wmap, a.dtype == SC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void*>(a.W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  p->wmode = mode;
  p->wnb = nb;
  return true;
}

// The output-stationary launch on an already packed weight image.
sc_status run_fused(const ConvArgs& a, const Plan& pl, const uint8_t* img) {
  TcParams prm = base_params(a, pl, img);
  return dispatch_tc<kOutputStationary>(prm, pl, a.dtype == SC_BF16, a.stream, "subm_conv_fused");
}

}  // namespace

bool fused_supported(const ConvArgs& a) {
  Plan pl;
  return fused_ok(a, &pl);
}

sc_status conv_fused(const ConvArgs& a) {
  Plan pl;
  if (!fused_ok(a, &pl))
    return set_error(SC_ERR_UNSUPPORTED, "fused kernel: f16/bf16 only, V <= 128, tile must fit shared memory");
  if (a.m->n == 0) return SC_OK;
  {
    // the weight slices straight from W by TMA: no packed image
    TcParams prm = base_params(a, pl, nullptr);
    CUtensorMap wmap;
    if (setup_weight_tma(a, pl, &prm, &wmap))
      return dispatch_tc<kOutputStationary>(prm, pl, a.dtype == SC_BF16, a.stream, "subm_conv_fused", &wmap);
  }
  const size_t img_bytes = static_cast<size_t>(a.m->V) * a.c_in * a.c_out * 2;
  void* img = nullptr;
  sc_status st = dev_alloc(&img, img_bytes, a.stream);
  if (st) return st;
  st = pack_weights(a, pl.bk, static_cast<uint8_t*>(img));
  if (!st) st = run_fused(a, pl, static_cast<const uint8_t*>(img));
  dev_free(img, a.stream);
  return st;
}

// Column splitting ("TorchSparse optimizations", section "TorchSparse++"):
// the offset loop of each output tile runs in two launches, one per part of
// the offset range, each over that part's own signature-sorted row order (a
// tile then walks fewer offsets of its part).  The first stores its fp32
// partial sums, the second adds them to its own, applies the activation and
// rounds once to the output dtype; the fp32 sums never leave fp32.
sc_status conv_fused_split(const ConvArgs& a) {
  Plan pl;
  if (!fused_ok(a, &pl))
    return set_error(SC_ERR_UNSUPPORTED, "fused kernel: f16/bf16 only, V <= 128, tile must fit shared memory");
  const KernelMap* m = a.m;
  if (m->nparts != 2)
    return set_error(SC_ERR_UNSUPPORTED, "the split layer needs a map built with SC_KMAP_SPLIT");
  if (m->n == 0) return SC_OK;
  const size_t img_bytes = static_cast<size_t>(m->V) * a.c_in * a.c_out * 2;
  const size_t acc_bytes = static_cast<size_t>(m->n) * a.c_out * sizeof(float);
  void* img = nullptr;
  void* acc = nullptr;
  sc_status st = dev_alloc(&img, img_bytes, a.stream);
  if (st) return st;
  st = dev_alloc(&acc, acc_bytes, a.stream);
  if (st) {
    dev_free(img, a.stream);
    return st;
  }
  st = pack_weights(a, pl.bk, static_cast<uint8_t*>(img));
  for (int part = 0; part < 2 && !st; ++part) {
    TcParams prm = base_params(a, pl, static_cast<const uint8_t*>(img));
    prm.perm = m->part_perm[part];
    prm.tnbr = nullptr;  // the part's own row order reads nbr
    prm.order = m->part_order[part];
    prm.present = reinterpret_cast<const uint4*>(m->part_present[part]);
    prm.acc = static_cast<float*>(acc);
    prm.epi = part == 0 ? 1 : 2;
    prm.centre_in = part == 0 ? 1 : 0;  // the centre opens part 1 of the range at index split_at - 1
    st = dispatch_tc<kOutputStationary>(prm, pl, a.dtype == SC_BF16, a.stream, "subm_conv_split");
  }
  dev_free(acc, a.stream);
  dev_free(img, a.stream);
  return st;
}

sc_status conv_weight_stationary(const ConvArgs& a) {
  Plan pl;
  if (a.dtype == SC_F32 || !make_plan(a.c_in, a.c_out, false, &pl))
    return set_error(SC_ERR_UNSUPPORTED, "weight-stationary kernel: f16/bf16 only");
  if (a.m->n == 0) return SC_OK;
  if (!a.m->host_valid) return set_error(SC_ERR_INVALID_ARG, "weight-stationary kernel needs the map's host counts");
  const size_t img_bytes = static_cast<size_t>(a.m->V) * a.c_in * a.c_out * 2;
  const size_t acc_bytes = static_cast<size_t>(a.m->n) * a.c_out * sizeof(float);
  void* img = nullptr;
  void* acc = nullptr;
  sc_status st = dev_alloc(&img, img_bytes, a.stream);
  if (st) return st;
  st = dev_alloc(&acc, acc_bytes, a.stream);
  if (st) {
    dev_free(img, a.stream);
    return st;
  }
  st = pack_weights(a, pl.bk, static_cast<uint8_t*>(img));
  TcParams prm = base_params(a, pl, static_cast<const uint8_t*>(img));
  prm.acc = static_cast<float*>(acc);
  const bool bf16 = a.dtype == SC_BF16;
  if (!st) st = dispatch_tc<kWsCentre>(prm, pl, bf16, a.stream, "subm_conv_ws_centre");
  if (!st) {
    prm.num_tiles = a.m->ws_tiles_host[a.m->V];
    prm.num_units = prm.num_tiles;
    st = dispatch_tc<kWsScatter>(prm, pl, bf16, a.stream, "subm_conv_ws_scatter");
  }
  if (!st) {
    const int64_t n4 = a.m->n * a.c_out / 4;
    int grid = static_cast<int>((n4 + 255) / 256);
    if (grid > device_sm_count() * 16) grid = device_sm_count() * 16;
    if (bf16)
      SC_LAUNCH("cast_out", a.stream, k_cast_out<true><<<grid, 256, 0, a.stream>>>(static_cast<const float4*>(acc), static_cast<uint2*>(a.out), n4, a.relu));
    else
      SC_LAUNCH("cast_out", a.stream, k_cast_out<false><<<grid, 256, 0, a.stream>>>(static_cast<const float4*>(acc), static_cast<uint2*>(a.out), n4, a.relu));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) st = set_cuda_error(e, "cast_out launch");
  }
  dev_free(acc, a.stream);
  dev_free(img, a.stream);
  return st;
}

// Id of the calling thread's current CUDA context (0 if the driver cannot
// say), through the driver entry point, so the library needs no link-time
// dependency on the driver library.  A context made after cudaDeviceReset
// gets a new id even where it reuses an old handle.
static unsigned long long current_context_id() {
  typedef int (*get_current_fn)(void**);
  typedef int (*get_id_fn)(void*, unsigned long long*);
  static get_current_fn get_current = nullptr;
  static get_id_fn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<get_current_fn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<get_id_fn>(f);
    cudaGetLastError();
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == 0 && ctx && get_id(ctx, &id) == 0) return id;
  return 0;
}

// Device address of g_noalloc_weights in the current device's context,
// looked up once per device and context (host code only holds a stand-in
// for the symbol, which is not a device address).  The cache is keyed on the
// context id as well, so a context that replaced the old one (after
// cudaDeviceReset) gets the array's address in the new context.
static sc_status noalloc_weights_ptr(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static unsigned long long ctx_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(SC_ERR_UNSUPPORTED, "device index above 63");
  // 0 when no context is current on this thread yet: the lookup below
  // makes the device's primary context current, and its id is read again
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev] || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_weights);
    if (e != cudaSuccess || !p) return set_cuda_error(e, "cudaGetSymbolAddress(g_noalloc_weights)");
    addr[dev] = p;
    ctx_of[dev] = ctx ? ctx : current_context_id();
  }
  *out = addr[dev];
  return SC_OK;
}

sc_status conv_fused_noalloc(const ConvArgs& a) {
  // set-up first, so the first call on a device always performs it
  void* img = nullptr;
  sc_status st = noalloc_weights_ptr(&img);
  if (st) return st;
  Plan pl;
  if (!fused_ok(a, &pl))
    return set_error(SC_ERR_UNSUPPORTED, "no-allocation conv: f16/bf16 only, V <= 128, tile must fit shared memory");
  const size_t img_bytes = static_cast<size_t>(a.m->V) * a.c_in * a.c_out * 2;
  if (img_bytes > kNoAllocWeightBytes)
    return set_error(SC_ERR_UNSUPPORTED,
                     "no-allocation conv: packed weights (V * c_in * c_out * 2 bytes) exceed the 4 MiB fixed buffer");
  if (a.m->n == 0) return SC_OK;
  st = pack_weights(a, pl.bk, static_cast<uint8_t*>(img));
  if (st) return st;
  return run_fused(a, pl, static_cast<const uint8_t*>(img));
}

}  // namespace sc
