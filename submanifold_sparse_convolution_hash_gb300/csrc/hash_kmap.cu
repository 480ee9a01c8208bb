// Coordinate hash table and kernel-map construction.
//
// Hash build follows "SparseConvNet: from hash table to rulebook", section 2
// (one index per unique input coordinate) with the table built on the GPU
// ("Sparse inputs and sparse convolution", section "Gather, matmul,
// scatter": rule generation moved from a CPU hash to the GPU).
//
// The map follows "Sparse inputs and sparse convolution", section "The map is
// the computation": for each output q and offset d, look up q + d; a hit p
// gives the tuple (p, q, W_d).  The centre offset is the identity at stride 1
// and is written, not searched ("TorchSparse optimizations", opening section).
// Lists are grouped by offset ("SparseConvNet: from hash table to rulebook",
// section 3).
//
// Locality order.  Rows arrive in any order, but the probe, the per-offset
// lists and the convolution's 128-row tiles work best on spatially compact
// groups of points: a compact tile touches fewer offsets and reuses the same
// neighbour rows.  For large inputs the map build therefore counting-sorts the
// points on a 20-bit bucket, the top bits of a Morton code of (batch, x, y, z)
// whose per-axis widths follow the grid extents and the largest batch id.
// Buckets are small (a few dozen points on surface data), consecutive buckets
// are neighbouring cells, and the order inside a bucket is whatever the
// atomics give; no result depends on it.  Without the order, rows are taken
// in input order.
//
// Points are taken in units of 128 positions of that order (32 when the
// kernel has more than 128 offsets), and the neighbour table is stored in
// that order too (row k belongs to input row order[k]), so a unit's
// 128 x V block is contiguous.  One kernel builds the map, one block per
// unit:
//   * probe: the block's threads split the 2x2x2 blocks that cover each
//     point's neighbourhood (8 for a 3x3x3 kernel, 27 for 5x5x5); one lookup
//     returns a block's 8 rows, which are filed under their offsets in a
//     shared-memory copy of the unit's block of the table;
//   * the table block is written with 16-byte stores;
//   * count and emit, a warp per offset: a ballot per (offset, 32 points)
//     gives the hits; one atomic per offset on that offset's cursor (a
//     warp's atomics issued together, one per lane) reserves the unit's run
//     of entries, and the (in, out) entries go to offset v's list at v * n +
//     the reserved start + rank, so a unit's entries stay together in row
//     order (the order of units inside a list is the order their atomics
//     ran); then the unit's 128-bit mask of present offsets.
// With the locality order the points' keys are read in that order (the
// order kernel stores them sorted), one coalesced load per point.
// The last block to finish turns the per-offset totals into the segment
// offsets, the weight-stationary tile prefix and |M|.  The lists live in
// fixed strides of n entries per offset; the CSR that the boundary exports is
// their compaction.

#include "sc_internal.cuh"

namespace sc {
namespace {

constexpr int kThreads = 256;    // threads per map-build block
constexpr int kLookups = 2;      // hash lookups in flight per map-build thread
constexpr int kSigBits = 20;     // signature sort: rare features in a row's key
// rows per signature-sort window: 524,288 (measured against 2^15 .. 2^20:
// the batched-LiDAR stack 3.18 ms at 2^16 against 2.96 ms, the 1M-voxel
// layer 293 against 282 us, the 2M-voxel 5x5x5 layer 3.02 against 2.99 ms)
constexpr int kSigWindowLog2 = 19;
constexpr int kWsRows = 128;     // rows per weight-stationary tile
// shared memory of a build block: 128 points x V <= 128 (or 32 x V <= 343)
// neighbour slots, the ballots and the per-offset bases
constexpr int kBuildSmemMax = 4 * (128 * 128 + 128 * 4) + 16 + 4 * 128 * 4;
constexpr int kBucketBits = 20;    // locality-order buckets
constexpr int kBuckets = 1 << kBucketBits;
constexpr int kBucketBlocks = 256;                   // blocks of the bucket scan
constexpr int kBucketChunk = kBuckets / kBucketBlocks;  // 4096 buckets per block

// Looks up block key bk; on a hit, r0/r1 hold the rows of its 8 voxels.
// Each probed entry's key and rows are loaded together (one 64-byte entry).
__device__ __forceinline__ bool lookup_block(const BlockEntry* __restrict__ table, uint32_t mask,
                                             unsigned long long bk, int4& r0, int4& r1) {
  uint32_t h = block_home(bk, mask);
  for (uint32_t probe = 0; probe <= mask; ++probe) {
    const BlockEntry* e = table + h;
    const unsigned long long k = __ldg(&e->key);
    r0 = __ldg(reinterpret_cast<const int4*>(e->rows));
    r1 = __ldg(reinterpret_cast<const int4*>(e->rows + 4));
    if (k == bk) return true;
    if (k == kEmptyKey) return false;
    h = (h + 1) & mask;
  }
  return false;
}

__device__ __forceinline__ int pick(const int4& r0, const int4& r1, int l) {
  const int4& q = l < 4 ? r0 : r1;
  switch (l & 3) {
    case 0: return q.x;
    case 1: return q.y;
    case 2: return q.z;
    default: return q.w;
  }
}

__device__ __forceinline__ bool coord_fields_ok(int4 c) {
  return static_cast<unsigned>(c.x) < 65535u && static_cast<unsigned>(c.y) < 65535u &&
         static_cast<unsigned>(c.z) < 65535u && static_cast<unsigned>(c.w) < 65535u;
}

// Insert: find or claim the entry of the voxel's block (a compare-and-swap
// of the block key against the empty key, which returns the key found), then
// CAS the voxel's row slot from -1 to its row id; a slot that is already
// taken means two rows share the coordinate.
__global__ void __launch_bounds__(256) k_hash_insert(const int4* __restrict__ coords, int64_t n,
                                                     BlockEntry* __restrict__ table, uint32_t mask,
                                                     unsigned long long* __restrict__ keys,
                                                     int* __restrict__ status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int4 c = __ldg(coords + i);
    if (!coord_fields_ok(c)) {
      keys[i] = kEmptyKey;
      atomicOr(status, kDevErrRange);
      continue;
    }
    const unsigned long long key = pack_key(c.x, c.y, c.z, c.w);
    keys[i] = key;
    {  // largest batch id, one atomic per warp
      const unsigned am = __activemask();
      const int mb = __reduce_max_sync(am, c.x);
      if ((threadIdx.x & 31) == __ffs(am) - 1 && mb > 0) atomicMax(status + 1, mb);
    }
    const unsigned long long bk = block_key(key);
    uint32_t h = block_home(bk, mask);
    int e = -1;
    for (uint32_t probe = 0; probe <= mask; ++probe) {
      // one round trip: the swap either claims an empty entry or returns the
      // key already there
      unsigned long long k = atomicCAS(&table[h].key, kEmptyKey, bk);
      if (k == kEmptyKey || k == bk) {
        e = static_cast<int>(h);
        break;
      }
      h = (h + 1) & mask;
    }
    if (e < 0) {
      atomicOr(status, kDevErrFull);
      continue;
    }
    if (atomicCAS(&table[e].rows[block_local(key)], -1, static_cast<int>(i)) != -1) atomicOr(status, kDevErrDup);
  }
}

__global__ void __launch_bounds__(256) k_hash_query(const int4* __restrict__ q, int64_t m,
                                                    const BlockEntry* __restrict__ table, uint32_t mask,
                                                    int* __restrict__ rows) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m; i += stride) {
    const int4 c = __ldg(q + i);
    int r = -1;
    if (coord_fields_ok(c)) {
      const unsigned long long key = pack_key(c.x, c.y, c.z, c.w);
      int4 r0, r1;
      if (lookup_block(table, mask, block_key(key), r0, r1)) r = pick(r0, r1, block_local(key));
    }
    rows[i] = r;
  }
}

// Bits needed to hold values 0..v.
__device__ __forceinline__ int bits_for(int v) { return v > 0 ? 32 - __clz(v) : 0; }

struct OrderBits {
  int bx, by, bz;  // widths of the x, y, z extents
};

// Locality bucket of a packed key: the top kBucketBits bits of the Morton
// code (x, y, z interleaved from the lowest bit, each axis as wide as its
// extent), with the batch id above the spatial bits.
__device__ __forceinline__ int order_bucket(unsigned long long key, const OrderBits& ob, int total_bits) {
  if (key == kEmptyKey) return 0;
  const uint32_t x = static_cast<uint32_t>((key >> 32) & 0xFFFF), y = static_cast<uint32_t>((key >> 16) & 0xFFFF),
                 z = static_cast<uint32_t>(key & 0xFFFF), b = static_cast<uint32_t>(key >> 48);
  unsigned long long code = 0;
  int pos = 0;
  const int L = max(ob.bx, max(ob.by, ob.bz));
  for (int l = 0; l < L; ++l) {
    if (l < ob.bx) code |= static_cast<unsigned long long>((x >> l) & 1u) << pos++;
    if (l < ob.by) code |= static_cast<unsigned long long>((y >> l) & 1u) << pos++;
    if (l < ob.bz) code |= static_cast<unsigned long long>((z >> l) & 1u) << pos++;
  }
  code |= static_cast<unsigned long long>(b) << pos;
  const int shift = total_bits > kBucketBits ? total_bits - kBucketBits : 0;
  return static_cast<int>((code >> shift) & (kBuckets - 1));
}

__device__ __forceinline__ int order_total_bits(const OrderBits& ob, const int* hash_status) {
  return ob.bx + ob.by + ob.bz + bits_for(__ldg(hash_status + 1));
}

__global__ void __launch_bounds__(256) k_order_count(const unsigned long long* __restrict__ keys, int64_t n,
                                                     OrderBits ob, const int* __restrict__ hash_status,
                                                     int* __restrict__ buckets) {
  const int tb = order_total_bits(ob, hash_status);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    atomicAdd(buckets + order_bucket(__ldg(keys + i), ob, tb), 1);
}

// Scan phase 1: the total of each block's chunk of buckets.
__global__ void __launch_bounds__(256) k_order_partials(const int* __restrict__ buckets, int* __restrict__ partial) {
  __shared__ int warp_sums[8];
  const int4* b = reinterpret_cast<const int4*>(buckets + blockIdx.x * kBucketChunk);
  int sum = 0;
  for (int k = threadIdx.x; k < kBucketChunk / 4; k += 256) {
    const int4 c = __ldg(b + k);
    sum += c.x + c.y + c.z + c.w;
  }
  sum = __reduce_add_sync(0xffffffffu, sum);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < 8; ++w) t += warp_sums[w];
    partial[blockIdx.x] = t;
  }
}

// Scan phase 2: exclusive prefix of the bucket counts, in place.  Each block
// adds the partials of the blocks before it, then scans its chunk in shared
// memory (16 consecutive buckets per thread).
__global__ void __launch_bounds__(256) k_order_apply(int* __restrict__ buckets, const int* __restrict__ partial) {
  __shared__ int s_c[kBucketChunk];
  __shared__ int warp_sums[8];
  __shared__ int s_base;
  constexpr int per = kBucketChunk / 256;
  int4* b = reinterpret_cast<int4*>(buckets + blockIdx.x * kBucketChunk);
  for (int k = threadIdx.x; k < kBucketChunk / 4; k += 256) reinterpret_cast<int4*>(s_c)[k] = b[k];
  if (threadIdx.x < 32) {
    int base = 0;
    for (int j = threadIdx.x; j < static_cast<int>(blockIdx.x); j += 32) base += __ldg(partial + j);
    base = __reduce_add_sync(0xffffffffu, base);
    if (threadIdx.x == 0) s_base = base;
  }
  __syncthreads();
  int c[per];
  int sum = 0;
#pragma unroll
  for (int k = 0; k < per; ++k) {
    c[k] = s_c[threadIdx.x * per + k];
    sum += c[k];
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  int before = s_base;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  int run = before + x - sum;
#pragma unroll
  for (int k = 0; k < per; ++k) {
    s_c[threadIdx.x * per + k] = run;
    run += c[k];
  }
  __syncthreads();
  for (int k = threadIdx.x; k < kBucketChunk / 4; k += 256) b[k] = reinterpret_cast<const int4*>(s_c)[k];
}

__global__ void __launch_bounds__(256) k_order_scatter(const unsigned long long* __restrict__ keys, int64_t n,
                                                       OrderBits ob, const int* __restrict__ hash_status,
                                                       int* __restrict__ cursors, int* __restrict__ order,
                                                       unsigned long long* __restrict__ skeys,
                                                       int* __restrict__ inv_order) {
  const int tb = order_total_bits(ob, hash_status);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long key = __ldg(keys + i);
    const int pos = atomicAdd(cursors + order_bucket(key, ob, tb), 1);
    order[pos] = static_cast<int>(i);
    skeys[pos] = key;  // the map build then reads keys in order, coalesced
    if (inv_order) inv_order[i] = pos;  // half probe: the table row of input row i
  }
}


// Output range [lo, hi] along one axis for an input at coordinate c: the o
// with c - r <= stride * o <= c + r inside [0, ext).  Empty when lo > hi.
__device__ __forceinline__ void out_range(int c, int r, int stride, int ext, int& lo, int& hi) {
  lo = c - r <= 0 ? 0 : (c - r + stride - 1) / stride;
  hi = min((c + r) / stride, ext - 1);
}

// Block-wide inclusive scan of one value per thread (blockDim <= 1024).
template <typename T>
__device__ __forceinline__ T block_inclusive_scan(T x, T* warp_sums, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nw ? warp_sums[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  if (warp > 0) x += warp_sums[warp - 1];
  *total = warp_sums[nw - 1];
  __syncthreads();
  return x;
}

struct BuildArgs {
  const unsigned long long* keys;  // [n] packed key of each input row
  const int* order;                // [n] or null
  const unsigned long long* skeys; // [n] keys in that order (with order)
  int64_t n;
  const BlockEntry* table;
  uint32_t mask;                   // table capacity - 1
  int V, K, ndim, dimx, dimy, dimz;  // extents of the table's grid
  int qex, qey, qez;               // extents of the queries' grid
  int stride;                      // forward: query o looks up the table points at stride * o + d
  int identity;                    // the centre list is the identity (submanifold: queries = inputs)
  int up;                          // points per unit (128; 64 when V > 64; 32 when V > 128)
  int nunits;
  int* nbr;                        // [n, V] in row order
  unsigned* present;               // [ceil(n / 128), 4] per 128-row tile (units of 128 or 64 points)
  int* in_rows;                    // [V, n] strided lists
  int* out_rows;
  int* cursors;                    // [V * kCursorStride] entries reserved so far in each offset's list
  int* status;                     // [4]: map status, hash status copy, -, done counter
  int64_t* offs;                   // [V+1]
  int* ws_tiles;                   // [V+1]
  int64_t* map_size;
  // signature sort: the offsets (centre excluded) with a neighbour, per row:
  // one word per row when V <= 32, four (a 128-bit mask) when V <= 128; or null
  unsigned* rowmask;
  // V > 32: the coarse directions (sign(dx), sign(dy), sign(dz)), 27 bits,
  // with a neighbour, per row: the signature's features; else null (the
  // features are the offsets themselves, in rowmask)
  unsigned* rowdir;
  int* sig_sel;                    // [kSigBits] features of the row signature, rarest first (with rowmask)
  const int* inv_order;            // half probe with the row order: table row of each input row; else null
  int split_at;                    // column splitting: first offset of part 1 (0: no split)
};

// Coarse direction of offset v: (sign(dx) + 1) * 9 + (sign(dy) + 1) * 3 +
// (sign(dz) + 1), in [0, 27), the centre 13 (dz = 0 in 2D).
__device__ __forceinline__ int offset_direction(int v, int K, int ndim) {
  const int r = (K - 1) / 2;
  int dx, dy, dz;
  if (ndim == 3) {
    dx = v / (K * K) - r;
    dy = (v / K) % K - r;
    dz = v % K - r;
  } else {
    dx = v / K - r;
    dy = v % K - r;
    dz = 0;
  }
  const int sx = (dx > 0) - (dx < 0) + 1, sy = (dy > 0) - (dy < 0) + 1, sz = (dz > 0) - (dz < 0) + 1;
  return sx * 9 + sy * 3 + sz;
}

// Dynamic shared memory: s_tile [up * V] ints, s_bal [V * up / 32].
// Five blocks per SM (register budget): 2560 lookups in flight per SM.
// TR: a transposed map: the queries are a layer's inputs c, the table its
// outputs o with stride * o + d = c, and the offset stored is -d (index
// V - 1 - idx(d)).
// Measured: four lookups in flight at three blocks per SM were no faster at
// 5x5x5 (1.04 ms against 1.02 ms at 2M voxels).
// UP: points per unit (128, or 32 when V > 128), a compile-time constant so
// that the count and emit loops over the unit's 32-point groups unroll and
// their shared-memory loads overlap.
// HALF: the half probe of a submanifold map (mirror symmetry: (p, q, d) is
// in the map iff (q, p, -d) is).  A unit probes only the offsets after the
// centre (lexicographically positive d) for its points and stores those
// columns and the centre; each hit p of point q at d also gives q as p's
// neighbour at -d, written straight into p's row of the table (whose
// columns before the centre were set to -1 beforehand and are written by
// nobody else), and one cursor reservation for d places both d's entry
// (p, q) and -d's entry (q, p) at the same positions of their lists.  The
// tile offset masks and row masks are then derived from the finished table
// (k_kmap_masks).
template <bool TR, int UP, bool HALF>
__global__ void __launch_bounds__(kThreads, 5) k_kmap_build(const BuildArgs a) {
  extern __shared__ int4 smem4[];
  constexpr int up = UP;
  constexpr int ngroups = UP / 32;
  const int V = a.V;
  int* s_tile = reinterpret_cast<int*>(smem4);
  unsigned* s_bal = reinterpret_cast<unsigned*>(s_tile + up * V);
  // V > 32 with the signature sort: the 128-bit offset mask of each row (in
  // the dynamic allocation only when used), word-major ([4][128]: the emit
  // phase's atomics of a warp's 32 rows fall in 32 banks), 16-byte aligned
  unsigned* s_rmask4 = reinterpret_cast<unsigned*>(
      (reinterpret_cast<uintptr_t>(s_bal + V * ngroups) + 15) & ~static_cast<uintptr_t>(15));
  __shared__ int s_last;
  __shared__ int s_row[128];
  __shared__ unsigned s_pres[4];
  __shared__ unsigned s_rmask[128];         // V <= 32: offsets per row; V > 32: directions per row
  __shared__ unsigned char s_dir[128];  // V <= 128 with rowdir: coarse direction of each offset
  // covering blocks of a neighbourhood, relative to its lowest one: block t
  // at (t & 0xFF, (t >> 8) & 0xFF, t >> 16); at most (r + 1)^3 <= 81
  __shared__ uint32_t s_trip[128];
  __shared__ int s_ntrip;

  __shared__ long long warp_sums[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kThreads / 32;
  if (threadIdx.x < 4) s_pres[threadIdx.x] = 0u;
  if (threadIdx.x < 128) s_rmask[threadIdx.x] = 0u;
  if (a.rowdir)
    for (int e = threadIdx.x; e < 128 * 4; e += kThreads) s_rmask4[e] = 0u;
  if (a.rowdir && threadIdx.x < V) s_dir[threadIdx.x] = static_cast<unsigned char>(offset_direction(threadIdx.x, a.K, a.ndim));
  for (int e = threadIdx.x; e < up * V; e += kThreads) s_tile[e] = -1;
  const int u = blockIdx.x;
  const int64_t i0 = static_cast<int64_t>(u) * up;
  const int np = static_cast<int>(min(static_cast<int64_t>(up), a.n - i0));
  const int r = (a.K - 1) / 2;
  const int rz = a.ndim == 3 ? r : 0;
  const int centre = (V - 1) / 2;
  {
    const int nb = r + 1, nbz = rz + 1;  // covering blocks per axis, at most
    if (threadIdx.x == 0) s_ntrip = nb * nb * nbz;
    if (threadIdx.x < nb * nb * nbz) {
      const int t = threadIdx.x;
      s_trip[t] = static_cast<uint32_t>(t / (nb * nbz)) | (static_cast<uint32_t>((t / nbz) % nb) << 8) |
                  (static_cast<uint32_t>(t % nbz) << 16);
    }
  }
  __syncthreads();

  // ---- probe: thread = (point p, part); parts split the covering blocks
  {
    const int p = threadIdx.x % up, part = threadIdx.x / up, nparts = kThreads / up;
    const bool live = p < np;
    const int row = live ? (a.order ? __ldg(a.order + i0 + p) : static_cast<int>(i0 + p)) : -1;
    if (part == 0 && p < up) s_row[p] = row;
    const unsigned long long ck = live ? (a.order ? __ldg(a.skeys + i0 + p) : __ldg(a.keys + row)) : kEmptyKey;
    bool valid = ck != kEmptyKey;
    const int qx = static_cast<int>((ck >> 32) & 0xFFFF), qy = static_cast<int>((ck >> 16) & 0xFFFF),
              qz = static_cast<int>(ck & 0xFFFF);
    if (valid && (qx >= a.qex || qy >= a.qey || qz >= a.qez)) {
      if (part == 0) atomicOr(a.status, kDevErrRange);
      valid = false;
    }
    // per axis: the table voxels [lo, hi] of this point's neighbourhood and
    // the offset of voxel t, d = t * mul - ctr:
    //   forward:    t in [s q - r, s q + r] (inside the table's grid), d = t - s q
    //   transposed: t with q - r <= s t <= q + r (inside it),           d = s t - q
    const int sz = a.ndim == 3 ? a.stride : 1;
    int xl, xh, yl, yh, zl, zh, cx, cy, cz;
    if (!TR) {
      cx = qx * a.stride;
      cy = qy * a.stride;
      cz = qz * sz;
      xl = max(cx - r, 0);
      xh = min(cx + r, a.dimx - 1);
      yl = max(cy - r, 0);
      yh = min(cy + r, a.dimy - 1);
      zl = max(cz - rz, 0);
      zh = min(cz + rz, a.dimz - 1);
    } else {
      cx = qx;
      cy = qy;
      cz = qz;
      out_range(qx, r, a.stride, a.dimx, xl, xh);
      out_range(qy, r, a.stride, a.dimy, yl, yh);
      out_range(qz, rz, sz, a.dimz, zl, zh);
      if (xl > xh || yl > yh || zl > zh) valid = false;  // no table point can hold one
    }
    const unsigned long long batch = ck & 0xFFFF000000000000ull;
    const int xlo = xl >> 1, xhi = xh >> 1, ylo = yl >> 1, yhi = yh >> 1, zlo = zl >> 1, zhi = zh >> 1;
    // voxel e in {0, 1} of block coordinate b has the offset d = A (2b + e) - c
    // on each axis (A = 1 forward, the stride when transposed); its index
    // contribution is (d + r) * mul, mul = (K^2, K, 1) in 3D, (K, 1, 0) in 2D
    const int ax = TR ? a.stride : 1, az = TR ? sz : 1;
    const int mx = a.ndim == 3 ? a.K * a.K : a.K, my = a.ndim == 3 ? a.K : 1, mz = a.ndim == 3 ? 1 : 0;
    const int ntrip = s_ntrip;
    // kLookups lookups in flight per thread: home entries first, then the
    // (rare) further probes of each
    for (int t0 = part; t0 < ntrip; t0 += kLookups * nparts) {
      unsigned long long bk[kLookups], kk[kLookups];
      int4 r0[kLookups], r1[kLookups];
      int bxs[kLookups], bys[kLookups], bzs[kLookups];
      bool act[kLookups];
#pragma unroll
      for (int q = 0; q < kLookups; ++q) {
        const int t = t0 + q * nparts;
        const uint32_t tr = t < ntrip ? s_trip[t] : 0u;
        bxs[q] = xlo + static_cast<int>(tr & 0xFF);
        bys[q] = ylo + static_cast<int>((tr >> 8) & 0xFF);
        bzs[q] = zlo + static_cast<int>(tr >> 16);
        act[q] = valid && t < ntrip && bxs[q] <= xhi && bys[q] <= yhi && bzs[q] <= zhi;
        if (HALF && act[q]) {
          // the block's lexicographically last voxel inside the neighbourhood
          // (the higher of its two voxels on each axis when that one is in
          // range) must lie after the centre, else the block is not probed
          const int dx0 = 2 * bxs[q] - cx, dy0 = 2 * bys[q] - cy, dz0 = 2 * bzs[q] - cz;
          const int dxm = dx0 + 1 <= r ? dx0 + 1 : dx0, dym = dy0 + 1 <= r ? dy0 + 1 : dy0,
                    dzm = dz0 + 1 <= rz ? dz0 + 1 : dz0;
          act[q] = dxm > 0 || (dxm == 0 && (dym > 0 || (dym == 0 && dzm > 0)));
        }
        bk[q] = batch | pack_key(0, 2 * bxs[q], 2 * bys[q], 2 * bzs[q]);
        if (act[q]) kk[q] = __ldg(&a.table[block_home(bk[q], a.mask)].key);
      }
      // the rows only of the entries found at home (most covering blocks of a
      // surface point are absent, and the L1 pipe bounds this kernel)
      bool hit[kLookups];
#pragma unroll
      for (int q = 0; q < kLookups; ++q) {
        hit[q] = act[q] && kk[q] == bk[q];
        if (hit[q]) {
          const BlockEntry* e = a.table + block_home(bk[q], a.mask);
          r0[q] = __ldg(reinterpret_cast<const int4*>(e->rows));
          r1[q] = __ldg(reinterpret_cast<const int4*>(e->rows + 4));
        }
      }
#pragma unroll
      for (int q = 0; q < kLookups; ++q) {
        if (!act[q]) continue;
        if (!hit[q] && kk[q] != kEmptyKey) hit[q] = lookup_block(a.table, a.mask, bk[q], r0[q], r1[q]);
        if (!hit[q]) continue;
        // per axis: which of the block's two voxels fall in the neighbourhood
        // (|d| <= r; the table holds no point outside its grid, so no other
        // bound is needed), and the index of voxel (0, 0, 0)
        const int dx0 = ax * 2 * bxs[q] - cx, dy0 = ax * 2 * bys[q] - cy, dz0 = az * 2 * bzs[q] - cz;
        const unsigned ex = (dx0 >= -r && dx0 <= r ? 1u : 0u) | (dx0 + ax >= -r && dx0 + ax <= r ? 2u : 0u);
        const unsigned ey = (dy0 >= -r && dy0 <= r ? 1u : 0u) | (dy0 + ax >= -r && dy0 + ax <= r ? 2u : 0u);
        const unsigned ez = (dz0 >= -rz && dz0 <= rz ? 1u : 0u) | (dz0 + az >= -rz && dz0 + az <= rz ? 2u : 0u);
        const int base = p * V + (dx0 + r) * mx + (dy0 + r) * my + (dz0 + rz) * mz;
        const int sx = ax * mx, sy = ax * my, sz2 = az * mz;
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          const int lx = l >> 2, ly = (l >> 1) & 1, lz = l & 1;
          const int at = base + lx * sx + ly * sy + lz * sz2;
          if ((ex >> lx) & (ey >> ly) & (ez >> lz) & 1u && (!HALF || at > p * V + centre))
            s_tile[at] = pick(r0[q], r1[q], l);
        }
      }
    }
    if (HALF && part == 0 && valid) s_tile[p * V + centre] = row;
  }
  __syncthreads();

  // ---- the unit's block of the table: contiguous, i0 * V * 4 bytes is a multiple of 128
  if (HALF) {
    // columns [centre, V) of each row; the columns before the centre are the
    // mirrored hits, written by the units that found them
    const int w = V - centre;
    for (int e = threadIdx.x; e < np * w; e += kThreads) {
      const int rr = e / w, c = centre + e - rr * w;
      __stcs(a.nbr + (i0 + rr) * V + c, s_tile[rr * V + c]);
    }
  } else {
    int* dst = a.nbr + i0 * V;
    const int items = np * V;
    const int n4 = items >> 2;
    // streaming stores (evict-first in L2): the table and lists are written
    // once here, and should not push the hash table out of L2
    for (int e = threadIdx.x; e < n4; e += kThreads) __stcs(reinterpret_cast<int4*>(dst) + e, reinterpret_cast<const int4*>(s_tile)[e]);
    for (int e = (n4 << 2) + threadIdx.x; e < items; e += kThreads) __stcs(dst + e, s_tile[e]);
  }

  // ---- count and emit, warp by warp: warp w takes offsets w, w + 8, ...
  // (up to 32 per round, lane k holding the k-th).  A ballot per 32-point
  // group gives an offset's hits; the round's atomics on the offsets'
  // cursors go out together, one per lane, and reserve each offset's run of
  // list entries; the (in, out) entries then fill the runs in row order.
  {
    const unsigned lt = (1u << lane) - 1u;
    unsigned rm[4] = {0u, 0u, 0u, 0u};  // offsets with a hit, for the rows g * 32 + lane
    int my_row[ngroups];                // input row of unit row g * 32 + lane
#pragma unroll
    for (int g = 0; g < ngroups; ++g) my_row[g] = s_row[g * 32 + lane];
    for (int vb = warp; vb < V; vb += kWarps * 32) {
      const int nk = min(32, (V - vb + kWarps - 1) / kWarps);
      int cnt_mine = 0;
      for (int k = 0; k < nk; ++k) {
        const int v = vb + kWarps * k;
        int cnt = 0;
#pragma unroll
        for (int g = 0; g < ngroups; ++g) {
          const int j = s_tile[(g * 32 + lane) * V + v];
          const unsigned b = __ballot_sync(0xffffffffu, (v != centre || !a.identity) && j >= 0);
          if (lane == 0) s_bal[v * ngroups + g] = b;
          cnt += __popc(b);
        }
        if (lane == k) cnt_mine = cnt;
      }
      int base_mine = 0;
      if (lane < nk && cnt_mine > 0) {
        const int v = vb + kWarps * lane;
        base_mine = atomicAdd(a.cursors + v * kCursorStride, cnt_mine);
        if (!HALF && v < 128 && up >= 64) atomicOr(s_pres + (v >> 5), 1u << (v & 31));
      }
      __syncwarp();
      for (int k = 0; k < nk; ++k) {
        const int v = vb + kWarps * k;
        int at0 = __shfl_sync(0xffffffffu, base_mine, k);
        const int64_t lb = static_cast<int64_t>(v) * a.n;
        unsigned bs[ngroups];
#pragma unroll
        for (int g = 0; g < ngroups; ++g) bs[g] = s_bal[v * ngroups + g];
#pragma unroll
        for (int g = 0; g < ngroups; ++g) {
          const unsigned b = bs[g];
          if ((b >> lane) & 1u) {
            const int64_t at = lb + at0 + __popc(b & lt);
            const int jn = s_tile[(g * 32 + lane) * V + v], iq = my_row[g];
            __stcs(a.in_rows + at, jn);
            __stcs(a.out_rows + at, iq);
            if (HALF) {
              // the mirrored tuple (iq, jn, -d): -d's list at the same position,
              // and iq in jn's row of the table at -d
              const int64_t atm = at + static_cast<int64_t>(V - 1 - 2 * v) * a.n;
              __stcs(a.in_rows + atm, iq);
              __stcs(a.out_rows + atm, jn);
              const int64_t pj = a.inv_order ? __ldg(a.inv_order + jn) : jn;
              a.nbr[pj * V + (V - 1 - v)] = iq;
            } else {
            if (v < 32) rm[g] |= 1u << v;
            }
            if (!HALF && a.rowdir) {  // V > 32: the row's offset and direction bits
              atomicOr(s_rmask4 + (v >> 5) * 128 + g * 32 + lane, 1u << (v & 31));
              atomicOr(s_rmask + g * 32 + lane, 1u << s_dir[v]);
            }
          }
          at0 += __popc(b);
        }
      }
    }
    if (!HALF && a.rowmask && !a.rowdir) {  // V <= 32: one word per row
#pragma unroll
      for (int g = 0; g < ngroups; ++g)
        if (rm[g]) atomicOr(s_rmask + g * 32 + lane, rm[g]);
    }
  }
  __syncthreads();
  // present offsets of the unit's 128-row tile (two 64-point units share one:
  // OR, on a zeroed mask); the half probe derives them from the table later
  if (!HALF && up == 128 && threadIdx.x < 4) a.present[static_cast<int64_t>(u) * 4 + threadIdx.x] = s_pres[threadIdx.x];
  if (!HALF && up == 64 && threadIdx.x < 4 && s_pres[threadIdx.x])
    atomicOr(a.present + static_cast<int64_t>(u >> 1) * 4 + threadIdx.x, s_pres[threadIdx.x]);
  if (!HALF && a.rowmask && !a.rowdir && threadIdx.x < np) a.rowmask[i0 + threadIdx.x] = s_rmask[threadIdx.x];
  if (!HALF && a.rowdir && threadIdx.x < np) {  // V > 32: 128-bit offset mask and direction bits per row
    const int t = threadIdx.x;
    reinterpret_cast<uint4*>(a.rowmask)[i0 + t] =
        make_uint4(s_rmask4[t], s_rmask4[128 + t], s_rmask4[256 + t], s_rmask4[384 + t]);
    a.rowdir[i0 + threadIdx.x] = s_rmask[threadIdx.x];
  }

  // ---- the last block: segment offsets, weight-stationary tile prefix, |M|
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.status + 3, 1) == a.nunits - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // per-offset totals (the cursors' final values), scanned over offsets
  long long carry = 0, carry_t = 0;
  for (int v0 = 0; v0 < V; v0 += kThreads) {
    const int v = v0 + threadIdx.x;
    // the half probe counts each pair of offsets d, -d on d's cursor
    const int vc = HALF && v < centre ? V - 1 - v : v;
    const long long cnt = v < V ? static_cast<long long>(__ldcg(a.cursors + vc * kCursorStride)) : 0;
    long long tot, tot_t;
    const long long inc = block_inclusive_scan<long long>(cnt, warp_sums, &tot);
    const long long tl = (cnt + kWsRows - 1) / kWsRows;
    const long long inc_t = block_inclusive_scan<long long>(tl, warp_sums, &tot_t);
    if (v < V) {
      a.offs[v] = carry + inc - cnt;
      a.ws_tiles[v] = static_cast<int>(carry_t + inc_t - tl);
    }
    carry += tot;
    carry_t += tot_t;
  }
  if (threadIdx.x == 0) {
    a.offs[V] = carry;
    a.ws_tiles[V] = static_cast<int>(carry_t);
    *a.map_size = (a.identity ? a.n : 0) + carry;
  }
  if (a.rowmask && a.rowdir) {
    // V > 32: a direction's count is the sum of its offsets' tuple counts
    __syncthreads();
    long long* s_dc = warp_sums;  // 27 counters (the scans above are done with it)
    if (threadIdx.x < 27) s_dc[threadIdx.x] = 0;
    __syncthreads();
    for (int v = threadIdx.x; v < V; v += kThreads)
      if (v != centre)
        atomicAdd(reinterpret_cast<unsigned long long*>(s_dc + offset_direction(v, a.K, a.ndim)),
                  static_cast<unsigned long long>(
                      __ldcg(a.cursors + (HALF && v < centre ? V - 1 - v : v) * kCursorStride)));
    __syncthreads();
  }
  if (a.rowmask && warp == 0) {
    // the kSigBits least frequent features (offsets when V <= 32, coarse
    // directions when V > 32) that occur at all, rarest first: lane f holds
    // (count, f); kSigBits rounds of a warp minimum
    const long long none = 0x7FFFFFFFFFFFFFFFll;
    const int nf = a.rowdir ? 27 : V, cf = a.rowdir ? 13 : centre;
    const int lc = HALF && lane < centre ? V - 1 - lane : lane;
    const long long c = lane < nf && lane != cf ? (a.rowdir ? warp_sums[lane]
                                                           : static_cast<long long>(__ldcg(a.cursors + lc * kCursorStride)))
                                                : 0;
    // selection 0 over every feature; with column splitting, selections 1
    // and 2 over the offsets of each part ([0, split_at) and [split_at, V))
    const int nsel = a.split_at ? 3 : 1;
    for (int sidx = 0; sidx < nsel; ++sidx) {
      const bool in_part = sidx == 0 || (sidx == 1 ? lane < a.split_at : lane >= a.split_at);
      long long key = c > 0 && in_part ? (c << 8) | lane : none;
      for (int k = 0; k < kSigBits; ++k) {
        long long mn = key;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const long long other = __shfl_xor_sync(0xffffffffu, mn, o);
          mn = other < mn ? other : mn;
        }
        // -1: no further feature occurs
        if (lane == 0) a.sig_sel[sidx * kSigBits + k] = mn == none ? -1 : static_cast<int>(mn & 255);
        if (key == mn) key = none;
      }
    }
  }
}

// The half probe's starting table: -1 in the columns before the centre of
// every row (warp per row, a row's columns written together).
__global__ void __launch_bounds__(256) k_clear_lower_half(int* __restrict__ nbr, int64_t n, int V) {
  const int lane = threadIdx.x & 31, half = (V - 1) / 2;
  const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < n; row += wstride)
    for (int c = lane; c < half; c += 32) __stcs(nbr + row * V + c, -1);
}

// Tile offset masks (present) and, with the signature sort, row masks of a
// map, derived from its finished neighbour table: after the half probe a
// row's columns before the centre arrive from other units, so its masks are
// known only once the whole table is written.  One warp per 32 rows (a
// coalesced load and a ballot per 32 offsets of a row); W mask words per row
// (1 when V <= 32, else 4).
template <int W>
__global__ void __launch_bounds__(128) k_kmap_masks(const int* __restrict__ nbr, int64_t n, int V, int K, int ndim,
                                                    unsigned* __restrict__ present, unsigned* __restrict__ rowmask,
                                                    unsigned* __restrict__ rowdir) {
  __shared__ unsigned s_p[4][4];
  __shared__ unsigned char s_dir[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int centre = (V - 1) / 2;
  if (rowdir && threadIdx.x < V) s_dir[threadIdx.x] = static_cast<unsigned char>(offset_direction(threadIdx.x, K, ndim));
  __syncthreads();
  const int64_t ntiles = (n + 127) / 128;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    unsigned m[W];
#pragma unroll
    for (int k = 0; k < W; ++k) m[k] = 0u;  // offsets of row t * 128 + warp * 32 + lane
    const int64_t r0 = t * 128 + warp * 32;
    // eight rows' loads in flight at a time
    for (int rb = 0; rb < 32; rb += 8) {
      int x[8][W];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t row = r0 + rb + i;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const int v = 32 * k + lane;
          x[i][k] = row < n && v < V ? __ldcs(nbr + row * V + v) : -1;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const unsigned b = __ballot_sync(0xffffffffu, x[i][k] >= 0 && 32 * k + lane != centre);
          if (lane == rb + i) m[k] = b;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const unsigned o = __reduce_or_sync(0xffffffffu, m[k]);
      if (lane == 0) s_p[warp][k] = o;
    }
    const int64_t row = r0 + lane;
    if (rowmask && row < n) {
      if (W == 1) rowmask[row] = m[0];
      else reinterpret_cast<uint4*>(rowmask)[row] = make_uint4(m[0], m[W > 1 ? 1 : 0], m[W > 2 ? 2 : 0], m[W > 3 ? 3 : 0]);
    }
    if (rowdir && row < n) {
      unsigned dir = 0u;
#pragma unroll
      for (int k = 0; k < W; ++k)
        for (unsigned x = m[k]; x; x &= x - 1u) dir |= 1u << s_dir[32 * k + __ffs(x) - 1];
      rowdir[row] = dir;
    }
    __syncthreads();
    if (threadIdx.x < 4)
      present[t * 4 + threadIdx.x] =
          threadIdx.x < W ? (s_p[0][threadIdx.x] | s_p[1][threadIdx.x] | s_p[2][threadIdx.x] | s_p[3][threadIdx.x]) : 0u;
    __syncthreads();
  }
}

// Signature sort, a counting sort on (window of 2^wlog2 rows, signature):
// rows keep their window (a spatially compact run of the locality order, or
// of the input order) and are grouped by which rare offsets they touch, so a
// 128-row tile spans fewer offsets.  Rows with equal keys in a warp share one
// atomic (__match_any_sync); the order inside a key is unspecified.
__device__ __forceinline__ int64_t sig_key(int64_t k, unsigned mk, const int* __restrict__ sel, int wlog2) {
  unsigned sg = 0;
#pragma unroll
  for (int b = 0; b < kSigBits; ++b) {
    const int v = __ldg(sel + b);
    if (v >= 0) sg |= ((mk >> v) & 1u) << (kSigBits - 1 - b);
  }
  return ((k >> wlog2) << kSigBits) | sg;
}

__global__ void __launch_bounds__(256) k_sig_count(const unsigned* __restrict__ rowmask, int64_t n,
                                                   const int* __restrict__ sel, int* __restrict__ buckets, int wlog2) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t nr = (n + 31) & ~int64_t(31);  // whole warps stay in the loop
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < nr; k += stride) {
    const bool live = k < n;
    const int64_t key = live ? sig_key(k, __ldg(rowmask + k), sel, wlog2) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (live && lane == __ffs(peers) - 1) atomicAdd(buckets + key, __popc(peers));
  }
}

__global__ void __launch_bounds__(256) k_sig_scatter(const unsigned* __restrict__ rowmask, const int* __restrict__ order,
                                                     int64_t n, const int* __restrict__ sel, int* __restrict__ cursors,
                                                     int* __restrict__ perm, int* __restrict__ conv_order, int wlog2) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t nr = (n + 31) & ~int64_t(31);
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < nr; k += stride) {
    const bool live = k < n;
    const int64_t key = live ? sig_key(k, __ldg(rowmask + k), sel, wlog2) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (live && lane == leader) base = atomicAdd(cursors + key, __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (live) {
      const int pos = base + __popc(peers & ((1u << lane) - 1u));
      perm[pos] = static_cast<int>(k);
      conv_order[pos] = order ? __ldg(order + k) : static_cast<int>(k);
    }
  }
}

// Present offsets of each 128-row tile of the sorted order, one warp per
// tile, the centre added: the OR of the rows' offset masks (MW = 1 word per
// row when V <= 32, 4 words when V <= 128).
template <int MW>
__global__ void __launch_bounds__(256) k_sig_present(const int* __restrict__ perm, const unsigned* __restrict__ rowmask,
                                                     int64_t n, int centre, unsigned* __restrict__ present,
                                                     unsigned pmask = 0xFFFFFFFFu, int with_centre = 1) {
  const int64_t ntiles = (n + 127) / 128;
  const int lane = threadIdx.x & 31;
  const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += wstride) {
    unsigned acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t j = t * 128 + k * 32 + lane;
      if (j < n) {
        const int64_t row = __ldg(perm + j);
        if (MW == 1) {
          acc[0] |= __ldg(rowmask + row) & pmask;  // column splitting: the part's offsets only
        } else {
          const uint4 m = __ldg(reinterpret_cast<const uint4*>(rowmask) + row);
          acc[0] |= m.x;
          acc[1] |= m.y;
          acc[2] |= m.z;
          acc[3] |= m.w;
        }
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) acc[w] = __reduce_or_sync(0xffffffffu, acc[w]);
    if (lane < 4) {
      unsigned x = lane == 0 ? acc[0] : (lane == 1 ? acc[1] : (lane == 2 ? acc[2] : acc[3]));
      if (with_centre && lane == (centre >> 5)) x |= 1u << (centre & 31);
      present[t * 4 + lane] = x;
    }
  }
}

// Rows of the table in input order: dst[order[k], :] = nbr[k, :].
__global__ void __launch_bounds__(256) k_unpermute_rows(const int* __restrict__ nbr, const int* __restrict__ order,
                                                        int64_t n, int V, int* __restrict__ dst) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t k = warp; k < n; k += stride) {
    const int64_t q = __ldg(order + k);
    for (int v = lane; v < V; v += 32) dst[q * V + v] = __ldg(nbr + k * V + v);
  }
}

// The fused layer's tile-transposed index table (SC_KMAP_TILE_TABLE):
// tnbr[(t * V + v) * 128 + r] = nbr[src, v] for the table row src at
// position t * 128 + r of the layer's row order (perm, or the identity), -1
// past the last row.  A tile's indices for one offset are then one
// contiguous 512-byte run instead of 128 loads from rows V * 4 bytes apart.
// One block per tile: the tile's table rows are staged in shared memory (a
// warp takes four rows at a time, lanes across each row's V <= 128 entries,
// all sixteen loads in flight), then the block writes them out offset by
// offset (V is odd, so the column reads fall in distinct banks).
__global__ void __launch_bounds__(256) k_tile_table(const int* __restrict__ nbr, const int* __restrict__ perm,
                                                    int64_t n, int V, int* __restrict__ tnbr) {
  extern __shared__ int s_t[];  // [128 * V]
  __shared__ int64_t s_src[128];
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 128) {
    const int64_t k = t * 128 + threadIdx.x;
    s_src[threadIdx.x] = k < n ? (perm ? static_cast<int64_t>(__ldg(perm + k)) : k) : -1;
  }
  __syncthreads();
  for (int r0 = warp * 4; r0 < 128; r0 += 32) {
    int x[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t src = s_src[r0 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = lane + 32 * j;
        x[i][j] = src >= 0 && v < V ? __ldcs(nbr + src * V + v) : -1;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = lane + 32 * j;
        if (v < V) s_t[(r0 + i) * V + v] = x[i][j];
      }
  }
  __syncthreads();
  int* dst = tnbr + t * V * 128;
  for (int e = threadIdx.x; e < V * 128; e += blockDim.x) {
    const int v = e >> 7, r = e & 127;
    dst[e] = s_t[r * V + v];
  }
}

// The strided lists (offset v at v * n) compacted into CSR order.
__global__ void __launch_bounds__(256) k_compact_lists(const int* __restrict__ src, const int64_t* __restrict__ offs,
                                                       int64_t n, int* __restrict__ dst) {
  const int v = blockIdx.y;
  const int64_t b = __ldg(offs + v), cnt = __ldg(offs + v + 1) - b;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < cnt;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[b + e] = __ldg(src + static_cast<int64_t>(v) * n + e);
}

// ------------------------------------------------------------ output sets --
// Output set of a regular (stride 1: dilating) or strided layer: an output
// wherever the kernel window covers an active input ("SparseConvNet: from
// hash table to rulebook", section 2), output o reading the input at
// stride * o + d (section 3's index relation under a stride).  Every input
// marks each output o with stride * o + d at that input (d in [-r, r], o
// inside the output grid) in a block table of the input table's layout:
// those outputs form a box, marked block by block with one atomic on the
// block entry's occupancy word.  The marked voxels are then counted per chunk
// of entries, scanned, and numbered 0 .. n_out - 1 in table order, which
// turns the table into the output set's hash table; each output's key is
// written with its number.

constexpr int kOutChunk = 256 * 8;  // table entries per counting block (8 per thread)

struct OutGrid {
  int ex, ey, ez;  // output extents
  int stride;      // on x, y (and z in 3D)
  int r, rz;       // offset radius on x, y and on z (0 in 2D)
  int sz;          // stride on z (1 in 2D: z is carried)
};

// Marks the voxels `bits` (bit 4*lx + 2*ly + lz) of output block bk: finds
// or claims its entry, then clears those bits of the entry's occupancy word
// (the second word, all ones in an empty table).  A probe run longer than
// kOutProbeLimit latches kDevErrFull: the table is too small and the host
// retries with a larger one.
constexpr uint32_t kOutProbeLimit = 256;
__device__ __forceinline__ void mark_output_block(BlockEntry* __restrict__ table, uint32_t mask, unsigned long long bk,
                                                  unsigned bits, int* __restrict__ status) {
  uint32_t h = block_home(bk, mask);
  const uint32_t limit = mask < kOutProbeLimit ? mask + 1 : kOutProbeLimit;
  for (uint32_t probe = 0; probe < limit; ++probe) {
    unsigned long long k = __ldcg(&table[h].key);
    if (k == kEmptyKey) {
      k = atomicCAS(&table[h].key, kEmptyKey, bk);
      if (k == kEmptyKey) k = bk;
    }
    if (k == bk) {
      atomicAnd(&table[h].occupancy, ~static_cast<unsigned long long>(bits));
      return;
    }
    h = (h + 1) & mask;
  }
  atomicOr(status, kDevErrFull);
}

// Voxels of block b (2b, 2b + 1) inside [lo, hi], as a 2-bit mask.
__device__ __forceinline__ unsigned pair_mask(int b, int lo, int hi) {
  return (2 * b >= lo && 2 * b <= hi ? 1u : 0u) | (2 * b + 1 >= lo && 2 * b + 1 <= hi ? 2u : 0u);
}

// Each input's outputs form a box in the output grid (the product of its
// per-axis ranges); the box is marked block by block, one atomic per block.
__global__ void __launch_bounds__(256) k_out_mark(const unsigned long long* __restrict__ keys, int64_t n,
                                                  BlockEntry* __restrict__ table, uint32_t mask, OutGrid g,
                                                  int* __restrict__ status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long key = __ldg(keys + i);
    if (key == kEmptyKey) continue;
    const unsigned long long batch = key & 0xFFFF000000000000ull;
    const int x = static_cast<int>((key >> 32) & 0xFFFF), y = static_cast<int>((key >> 16) & 0xFFFF),
              z = static_cast<int>(key & 0xFFFF);
    int xl, xh, yl, yh, zl, zh;
    out_range(x, g.r, g.stride, g.ex, xl, xh);
    out_range(y, g.r, g.stride, g.ey, yl, yh);
    out_range(z, g.rz, g.sz, g.ez, zl, zh);
    if (xl > xh || yl > yh || zl > zh) continue;
    for (int bx = xl >> 1; bx <= xh >> 1; ++bx) {
      const unsigned mx = pair_mask(bx, xl, xh);
      for (int by = yl >> 1; by <= yh >> 1; ++by) {
        const unsigned my = pair_mask(by, yl, yh);
        for (int bz = zl >> 1; bz <= zh >> 1; ++bz) {
          const unsigned mz = pair_mask(bz, zl, zh);
          unsigned bits = 0;
#pragma unroll
          for (int l = 0; l < 8; ++l)
            if (((mx >> (l >> 2)) & (my >> ((l >> 1) & 1)) & (mz >> (l & 1))) & 1u) bits |= 1u << l;
          mark_output_block(table, mask, batch | pack_key(0, 2 * bx, 2 * by, 2 * bz), bits, status);
        }
      }
    }
  }
}

// The marked voxels of an entry: the cleared low bits of its occupancy word.
__device__ __forceinline__ unsigned marked_bits(const BlockEntry& e) {
  return static_cast<unsigned>(~__ldcg(&e.occupancy)) & 0xFFu;
}

// Marked voxels of the 8 entries blockIdx.x * kOutChunk + k * 256 + threadIdx.x.
__device__ __forceinline__ int count_marked(const BlockEntry* __restrict__ table, int64_t cap) {
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kOutChunk + k * 256 + threadIdx.x;
    if (e >= cap) break;
    cnt += __popc(marked_bits(table[e]));
  }
  return cnt;
}

__global__ void __launch_bounds__(256) k_out_count(const BlockEntry* __restrict__ table, int64_t cap,
                                                   int* __restrict__ partial) {
  __shared__ int warp_sums[32];
  int tot;
  block_inclusive_scan<int>(count_marked(table, cap), warp_sums, &tot);
  if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// Exclusive prefix of the chunk counts, in place; the total into *total.
__global__ void __launch_bounds__(1024) k_out_scan(int* __restrict__ partial, int nchunks, int64_t* __restrict__ total) {
  __shared__ long long warp_sums[32];
  long long carry = 0;
  for (int c0 = 0; c0 < nchunks; c0 += 1024) {
    const int c = c0 + threadIdx.x;
    const long long v = c < nchunks ? partial[c] : 0;
    long long tot;
    const long long inc = block_inclusive_scan<long long>(v, warp_sums, &tot);
    if (c < nchunks) partial[c] = static_cast<int>(carry + inc - v);
    carry += tot;
  }
  if (threadIdx.x == 0) *total = carry;
}

// Numbers the marked slots: chunk base + the thread's exclusive prefix, then
// entry by entry in slot order; writes each number into its slot and the
// voxel key under that number.
__global__ void __launch_bounds__(256) k_out_number(BlockEntry* __restrict__ table, int64_t cap,
                                                    const int* __restrict__ partial,
                                                    unsigned long long* __restrict__ keys_out) {
  __shared__ int warp_sums[32];
  const int cnt = count_marked(table, cap);
  int tot;
  int id = __ldg(partial + blockIdx.x) + block_inclusive_scan<int>(cnt, warp_sums, &tot) - cnt;
  for (int k = 0; k < 8; ++k) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kOutChunk + k * 256 + threadIdx.x;
    if (e >= cap) break;
    const unsigned long long bk = table[e].key;
    const unsigned bits = marked_bits(table[e]);
    for (int l = 0; l < 8; ++l) {
      if (!((bits >> l) & 1u)) continue;
      table[e].rows[l] = id;
      keys_out[id] = bk | (static_cast<unsigned long long>((l >> 2) & 1) << 32) |
                     (static_cast<unsigned long long>((l >> 1) & 1) << 16) | static_cast<unsigned long long>(l & 1);
      ++id;
    }
  }
}

__global__ void __launch_bounds__(256) k_hash_coords(const unsigned long long* __restrict__ keys, int64_t n,
                                                     int4* __restrict__ coords) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long k = __ldg(keys + i);
    coords[i] = make_int4(static_cast<int>(k >> 48), static_cast<int>((k >> 32) & 0xFFFF),
                          static_cast<int>((k >> 16) & 0xFFFF), static_cast<int>(k & 0xFFFF));
  }
}

int grid_for(int64_t n, int threads) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  int64_t g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

// Points per map-build unit: 128 (one convolution tile) up to 64 offsets;
// 64 up to 128 offsets, so that a unit's neighbour slots (64 x V ints) let
// five blocks share an SM instead of three; 32 beyond.
int kmap_unit_points(int V) { return V <= 64 ? 128 : (V <= 128 ? 64 : 32); }
int kmap_order_buckets() { return kBuckets + kBucketBlocks; }
int kmap_sig_bits() { return kSigBits; }
// The signature-sort window (log2 rows): 19 by default; developer override
// SC_DEV_SIG_WINDOW_LOG2 in [12, 20] for measurement sweeps (the result is
// the same, only the row order of the tiles changes).
int kmap_sig_window_log2() {
  static int w = [] {
    const char* e = getenv("SC_DEV_SIG_WINDOW_LOG2");
    const int v = e ? atoi(e) : kSigWindowLog2;
    return v >= 12 && v <= 20 ? v : kSigWindowLog2;
  }();
  return w;
}
int64_t kmap_sig_buckets(int64_t n) {
  const int64_t win = int64_t(1) << kmap_sig_window_log2();
  return ((n + win - 1) / win) << kSigBits;
}

sc_status kmap_unpermute_nbr(const KernelMap* m, int* dst, cudaStream_t s) {
  if (m->n == 0) return SC_OK;
  SC_LAUNCH("kmap_unpermute", s,
            k_unpermute_rows<<<grid_for(m->n * 32, 256), 256, 0, s>>>(m->nbr, m->order, m->n, m->V, dst));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "kmap_unpermute launch");
}

sc_status launch_hash_insert(const int32_t* coords, int64_t n, HashTable* h, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(h->table, 0xFF, sizeof(BlockEntry) * h->capacity, s);
  if (e != cudaSuccess) return set_cuda_error(e, "hash table clear");
  e = cudaMemsetAsync(h->status, 0, sizeof(int) * 4, s);
  if (e != cudaSuccess) return set_cuda_error(e, "hash status clear");
  if (n == 0) return SC_OK;
  SC_LAUNCH("hash_insert", s,
            k_hash_insert<<<grid_for(n, 256), 256, 0, s>>>(reinterpret_cast<const int4*>(coords), n, h->table,
                                                           static_cast<uint32_t>(h->capacity - 1), h->keys,
                                                           h->status));
  e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "hash_insert launch");
}

sc_status launch_hash_query(const HashTable* h, const int32_t* q, int64_t m, int32_t* rows, cudaStream_t s) {
  if (m == 0) return SC_OK;
  SC_LAUNCH("hash_query", s,
            k_hash_query<<<grid_for(m, 256), 256, 0, s>>>(reinterpret_cast<const int4*>(q), m, h->table,
                                                          static_cast<uint32_t>(h->capacity - 1), rows));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "hash_query launch");
}

static sc_status launch_kmap_steps(const HashTable* in, const HashTable* h, KernelMap* m, cudaStream_t s) {
  const int V = m->V;
  cudaError_t e;
  if (m->n == 0) {
    e = cudaMemsetAsync(m->offs, 0, sizeof(int64_t) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->ws_tiles, 0, sizeof(int) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->map_size, 0, sizeof(int64_t), s);
    return e == cudaSuccess ? SC_OK : set_cuda_error(e, "empty kmap init");
  }
  if (m->order) {  // locality order: count, two-phase scan, scatter
    OrderBits ob;
    int b[3];
    for (int a = 0; a < 3; ++a) {
      int v = m->dims[a] - 1, c = 0;
      while (v > 0) {
        ++c;
        v >>= 1;
      }
      b[a] = c;
    }
    ob.bx = b[0];
    ob.by = b[1];
    ob.bz = b[2];
    e = cudaMemsetAsync(m->buckets, 0, sizeof(int) * kBuckets, s);
    if (e != cudaSuccess) return set_cuda_error(e, "order bucket clear");
    const int og = grid_for(m->n, 256);
    int* partial = m->buckets + kBuckets;
    SC_LAUNCH("order_count", s, k_order_count<<<og, 256, 0, s>>>(h->keys, m->n, ob, h->status, m->buckets));
    SC_LAUNCH("order_partials", s, k_order_partials<<<kBucketBlocks, 256, 0, s>>>(m->buckets, partial));
    SC_LAUNCH("order_apply", s, k_order_apply<<<kBucketBlocks, 256, 0, s>>>(m->buckets, partial));
    SC_LAUNCH("order_scatter", s,
              k_order_scatter<<<og, 256, 0, s>>>(h->keys, m->n, ob, h->status, m->buckets, m->order, m->skeys,
                                                 m->inv_order));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "locality order launch");
  }
  e = cudaMemsetAsync(m->cursors, 0, sizeof(int) * V * kCursorStride, s);
  if (e == cudaSuccess && m->up == 64)  // two units OR into each tile's mask
    e = cudaMemsetAsync(m->present, 0, sizeof(unsigned) * 4 * ((m->n + 127) / 128), s);
  if (e != cudaSuccess) return set_cuda_error(e, "kmap cursor clear");
  BuildArgs a;
  a.keys = h->keys;
  a.order = m->order;
  a.skeys = m->skeys;
  a.n = m->n;
  a.table = in->table;
  a.mask = static_cast<uint32_t>(in->capacity - 1);
  a.stride = m->stride;
  a.identity = m->identity ? 1 : 0;
  a.V = V;
  a.K = m->K;
  a.ndim = m->ndim;
  // the grids of the queries and of the table: a layer's inputs have the
  // extents dims, its outputs ceil(dims / stride) on the strided axes
  const int st = m->stride, stz = m->ndim == 3 ? st : 1;
  const int in_ext[3] = {m->dims[0], m->dims[1], m->dims[2]};
  const int out_ext[3] = {(m->dims[0] + st - 1) / st, (m->dims[1] + st - 1) / st, (m->dims[2] + stz - 1) / stz};
  const int* t_ext = m->transposed ? out_ext : in_ext;
  const int* q_ext = m->transposed ? in_ext : out_ext;
  a.dimx = t_ext[0];
  a.dimy = t_ext[1];
  a.dimz = t_ext[2];
  a.qex = q_ext[0];
  a.qey = q_ext[1];
  a.qez = q_ext[2];
  a.up = m->up;
  a.nunits = m->nunits;
  a.nbr = m->nbr;
  a.present = m->present;
  a.in_rows = m->in_rows;
  a.out_rows = m->out_rows;
  a.cursors = m->cursors;
  a.status = m->status;
  a.offs = m->offs;
  a.ws_tiles = m->ws_tiles;
  a.map_size = m->map_size;
  a.rowmask = m->rowmask;
  a.rowdir = m->rowdir;
  a.sig_sel = m->sig_sel;
  a.inv_order = m->inv_order;
  a.split_at = m->nparts == 2 ? m->split_at : 0;
  const size_t smem = sizeof(int) * (static_cast<size_t>(m->up) * V + static_cast<size_t>(V) * (m->up / 32)) +
                      (m->rowdir ? 16 + sizeof(unsigned) * 128 * 4 : 0);
  if (smem > 48 * 1024) {  // set once per device: the largest the build ever asks for
    static bool done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      const void* kerns[9] = {reinterpret_cast<const void*>(k_kmap_build<false, 128, false>),
                              reinterpret_cast<const void*>(k_kmap_build<true, 128, false>),
                              reinterpret_cast<const void*>(k_kmap_build<false, 64, false>),
                              reinterpret_cast<const void*>(k_kmap_build<true, 64, false>),
                              reinterpret_cast<const void*>(k_kmap_build<false, 32, false>),
                              reinterpret_cast<const void*>(k_kmap_build<true, 32, false>),
                              reinterpret_cast<const void*>(k_kmap_build<false, 128, true>),
                              reinterpret_cast<const void*>(k_kmap_build<false, 64, true>),
                              reinterpret_cast<const void*>(k_kmap_build<false, 32, true>)};
      e = cudaSuccess;
      for (int k = 0; k < 9 && e == cudaSuccess; ++k)
        e = cudaFuncSetAttribute(kerns[k], cudaFuncAttributeMaxDynamicSharedMemorySize, kBuildSmemMax);
      if (e != cudaSuccess) return set_cuda_error(e, "kmap_build smem attribute");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  const int V2 = (V - 1) / 2;
  if (m->half) {
    // the half probe: every column before the centre starts at -1 (absent)
    // and receives only the mirrored hits
    if (V2 > 0)
      SC_LAUNCH("kmap_clear", s, (k_clear_lower_half<<<grid_for(m->n * 32, 256), 256, 0, s>>>(m->nbr, m->n, V)));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "half-probe table clear");
    if (m->up == 128)
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 128, true><<<m->nunits, kThreads, smem, s>>>(a)));
    else if (m->up == 64)
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 64, true><<<m->nunits, kThreads, smem, s>>>(a)));
    else
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 32, true><<<m->nunits, kThreads, smem, s>>>(a)));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "kmap_build launch");
    if (V <= 128) {  // tile masks for the fused kernel, row masks for the signature sort
      const int64_t ntiles = (m->n + 127) / 128;
      int g = static_cast<int>(ntiles < static_cast<int64_t>(device_sm_count()) * 16 ? ntiles : device_sm_count() * 16);
      if (V <= 32)
        SC_LAUNCH("kmap_masks", s, (k_kmap_masks<1><<<g, 128, 0, s>>>(m->nbr, m->n, V, m->K, m->ndim, m->present,
                                                                      m->rowmask, m->rowdir)));
      else
        SC_LAUNCH("kmap_masks", s, (k_kmap_masks<4><<<g, 128, 0, s>>>(m->nbr, m->n, V, m->K, m->ndim, m->present,
                                                                      m->rowmask, m->rowdir)));
    }
  } else if (m->up == 128) {
    if (m->transposed)
      SC_LAUNCH("kmap_build", s, (k_kmap_build<true, 128, false><<<m->nunits, kThreads, smem, s>>>(a)));
    else
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 128, false><<<m->nunits, kThreads, smem, s>>>(a)));
  } else if (m->up == 64) {
    if (m->transposed)
      SC_LAUNCH("kmap_build", s, (k_kmap_build<true, 64, false><<<m->nunits, kThreads, smem, s>>>(a)));
    else
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 64, false><<<m->nunits, kThreads, smem, s>>>(a)));
  } else {
    if (m->transposed)
      SC_LAUNCH("kmap_build", s, (k_kmap_build<true, 32, false><<<m->nunits, kThreads, smem, s>>>(a)));
    else
      SC_LAUNCH("kmap_build", s, (k_kmap_build<false, 32, false><<<m->nunits, kThreads, smem, s>>>(a)));
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "kmap_build launch");
  if (!m->perm) return SC_OK;
  // signature sort of the rows for the convolution's tiles
  const int64_t nsig = kmap_sig_buckets(m->n);  // a multiple of kBucketChunk
  int* partial = m->sigbuckets + nsig;
  const int chunks = static_cast<int>(nsig / kBucketChunk);
  e = cudaMemsetAsync(m->sigbuckets, 0, sizeof(int) * nsig, s);
  if (e != cudaSuccess) return set_cuda_error(e, "signature bucket clear");
  const int g = grid_for(m->n, 256);
  // the signature's features: the offsets (V <= 32) or the coarse directions
  const unsigned* feat = m->rowdir ? m->rowdir : m->rowmask;
  const int wl2 = kmap_sig_window_log2();
  SC_LAUNCH("sig_count", s, k_sig_count<<<g, 256, 0, s>>>(feat, m->n, m->sig_sel, m->sigbuckets, wl2));
  SC_LAUNCH("sig_partials", s, k_order_partials<<<chunks, 256, 0, s>>>(m->sigbuckets, partial));
  SC_LAUNCH("sig_scan", s, k_order_apply<<<chunks, 256, 0, s>>>(m->sigbuckets, partial));
  SC_LAUNCH("sig_scatter", s,
            k_sig_scatter<<<g, 256, 0, s>>>(feat, m->order, m->n, m->sig_sel, m->sigbuckets, m->perm,
                                            m->conv_order, wl2));
  const int pg = grid_for(((m->n + 127) / 128) * 32, 256);
  if (m->rowdir)
    SC_LAUNCH("sig_present", s, k_sig_present<4><<<pg, 256, 0, s>>>(m->perm, m->rowmask, m->n, (V - 1) / 2, m->present));
  else
    SC_LAUNCH("sig_present", s, k_sig_present<1><<<pg, 256, 0, s>>>(m->perm, m->rowmask, m->n, (V - 1) / 2, m->present));
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "signature sort launch");
  // column splitting (V <= 32): each part of the offset range gets its own
  // sort, keyed by the part's rarest offsets, and tile masks of its offsets
  for (int part = 0; part < (m->nparts == 2 ? 2 : 0); ++part) {
    const int* sel = m->sig_sel + (1 + part) * kSigBits;
    const unsigned pmask = part == 0 ? ((1u << m->split_at) - 1u) : ~((1u << m->split_at) - 1u);
    e = cudaMemsetAsync(m->sigbuckets, 0, sizeof(int) * nsig, s);
    if (e != cudaSuccess) return set_cuda_error(e, "signature bucket clear");
    SC_LAUNCH("sig_count", s, k_sig_count<<<g, 256, 0, s>>>(feat, m->n, sel, m->sigbuckets, wl2));
    SC_LAUNCH("sig_partials", s, k_order_partials<<<chunks, 256, 0, s>>>(m->sigbuckets, partial));
    SC_LAUNCH("sig_scan", s, k_order_apply<<<chunks, 256, 0, s>>>(m->sigbuckets, partial));
    SC_LAUNCH("sig_scatter", s,
              k_sig_scatter<<<g, 256, 0, s>>>(feat, m->order, m->n, sel, m->sigbuckets, m->part_perm[part],
                                              m->part_order[part], wl2));
    SC_LAUNCH("sig_present", s,
              k_sig_present<1><<<pg, 256, 0, s>>>(m->part_perm[part], m->rowmask, m->n, (V - 1) / 2,
                                                  m->part_present[part], pmask, part == 0 ? 1 : 0));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "split signature sort launch");
  }
  return SC_OK;
}


// The map's kernels, then (SC_KMAP_TILE_TABLE) the fused layer's
// tile-transposed index table in its final row order.
sc_status launch_kmap_build(const HashTable* in, const HashTable* h, KernelMap* m, cudaStream_t s) {
  sc_status st = launch_kmap_steps(in, h, m, s);
  if (st || !m->tnbr || m->n == 0) return st;
  const size_t smem = sizeof(int) * 128 * static_cast<size_t>(m->V);
  if (smem > 48 * 1024) {  // set once per device: the most it asks for (V = 128)
    static bool done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k_tile_table),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 128 * 4);
      if (e != cudaSuccess) return set_cuda_error(e, "tile table smem attribute");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  const int64_t tiles = (m->n + 127) / 128;
  SC_LAUNCH("tile_table", s,
            (k_tile_table<<<static_cast<unsigned>(tiles), 256, smem, s>>>(m->nbr, m->perm, m->n, m->V, m->tnbr)));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "tile table launch");
}

sc_status launch_hash_coords(const HashTable* h, int32_t* coords, cudaStream_t s) {
  if (h->n == 0) return SC_OK;
  SC_LAUNCH("hash_coords", s,
            k_hash_coords<<<grid_for(h->n, 256), 256, 0, s>>>(h->keys, h->n, reinterpret_cast<int4*>(coords)));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "hash_coords launch");
}

sc_status launch_conv_out(const HashTable* in, int ndim, int K, int stride, const int32_t dims[3], HashTable* out,
                          void** arena_table, void** arena_keys, const sc_allocator* alloc, cudaStream_t s) {
  OutGrid g;
  g.stride = stride;
  g.r = (K - 1) / 2;
  g.rz = ndim == 3 ? g.r : 0;
  g.sz = ndim == 3 ? stride : 1;
  g.ex = (dims[0] + stride - 1) / stride;
  g.ey = (dims[1] + stride - 1) / stride;
  g.ez = ndim == 3 ? (dims[2] + stride - 1) / stride : dims[2];
  // table size: about n (K / stride)^ndim / 5 outputs on surface data (each
  // output shared by the inputs of its window), about three to a 2x2x2
  // block, at most half full; a table too small for its probe runs is
  // retried four times larger
  double per = 1.0;
  for (int a = 0; a < ndim; ++a) per *= static_cast<double>(K) / stride;
  const double blocks = static_cast<double>(in->n) * per / 15.0;
  int64_t cap = 64;
  while (static_cast<double>(cap) < 2.0 * blocks) cap <<= 1;
  const int64_t kMaxCap = int64_t(1) << 28;
  int64_t n_out = 0;
  for (;;) {
    if (cap > kMaxCap) return set_error(SC_ERR_TABLE_FULL, "output set: table would exceed 2^28 entries");
    const int nchunks = static_cast<int>((cap + kOutChunk - 1) / kOutChunk);
    const size_t tb = sizeof(BlockEntry) * static_cast<size_t>(cap);
    const size_t pb = (sizeof(int) * static_cast<size_t>(nchunks) + 255) & ~size_t(255);
    sc_status st = dev_alloc(arena_table, tb + pb + 256, s, alloc);
    if (st) return st;
    uint8_t* b = static_cast<uint8_t*>(*arena_table);
    BlockEntry* table = reinterpret_cast<BlockEntry*>(b);
    int* partial = reinterpret_cast<int*>(b + tb);
    int* status = reinterpret_cast<int*>(b + tb + pb);        // [4]: latched errors, largest batch id
    int64_t* total = reinterpret_cast<int64_t*>(status + 4);  // output count
    cudaError_t e = cudaMemsetAsync(table, 0xFF, tb, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 256, s);
    // the outputs carry the inputs' batches: copy the largest batch id
    if (e == cudaSuccess) e = cudaMemcpyAsync(status + 1, in->status + 1, sizeof(int), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return set_cuda_error(e, "output set init");
    const uint32_t mask = static_cast<uint32_t>(cap - 1);
    if (in->n > 0)
      SC_LAUNCH("out_mark", s, k_out_mark<<<grid_for(in->n, 256), 256, 0, s>>>(in->keys, in->n, table, mask, g, status));
    SC_LAUNCH("out_count", s, k_out_count<<<nchunks, 256, 0, s>>>(table, cap, partial));
    SC_LAUNCH("out_scan", s, k_out_scan<<<1, 1024, 0, s>>>(partial, nchunks, total));
    int bits = 0;
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(&bits, status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&n_out, total, sizeof(int64_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return set_cuda_error(e, "output set count");
    if (bits & kDevErrFull) {
      dev_free(*arena_table, s);
      *arena_table = nullptr;
      cap <<= 2;
      continue;
    }
    if (n_out >= (int64_t(1) << 31)) return set_error(SC_ERR_UNSUPPORTED, "output set: more than 2^31 - 1 points");
    st = dev_alloc(arena_keys, sizeof(unsigned long long) * static_cast<size_t>(n_out > 0 ? n_out : 1), s, alloc);
    if (st) return st;
    out->n = n_out;
    out->capacity = cap;
    out->table = table;
    out->status = status;
    out->keys = static_cast<unsigned long long*>(*arena_keys);
    SC_LAUNCH("out_number", s, k_out_number<<<nchunks, 256, 0, s>>>(table, cap, partial, out->keys));
    e = cudaGetLastError();
    return e == cudaSuccess ? SC_OK : set_cuda_error(e, "output set numbering");
  }
}

sc_status kmap_compact_lists(const KernelMap* m, const int* src, int* dst, int64_t total, cudaStream_t s) {
  if (total == 0) return SC_OK;
  int64_t per = (m->n + 255) / 256;
  dim3 grid(static_cast<unsigned>(per < 64 ? per : 64), static_cast<unsigned>(m->V));
  SC_LAUNCH("kmap_compact", s, k_compact_lists<<<grid, 256, 0, s>>>(src, m->offs, m->n, dst));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "kmap_compact launch");
}

}  // namespace sc
