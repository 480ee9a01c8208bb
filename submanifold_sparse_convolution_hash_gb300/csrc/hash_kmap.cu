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
// Points are taken in tiles of 32 positions of that order, and the neighbour
// table is stored in that order too (row k belongs to input row order[k]), so
// a tile's 32 x V block is contiguous.  Three kernels build the map:
//   probe  one block per tile, lane = point in every warp: the warps split
//          the 2x2x2 blocks that cover each point's neighbourhood (8 for a
//          3x3x3 kernel, 27 for 5x5x5); one lookup returns a block's 8 rows,
//          which are filed under their offsets in a shared-memory copy of the
//          tile's block of the table; a ballot per offset gives the tile's
//          hit bitmask; the block is written with coalesced 16-byte stores.
//   scan   one block per offset: exclusive prefix of the masks' popcounts
//          over tiles.  The last block to finish (a ticket counter) turns the
//          per-offset totals into the segment offsets, the weight-stationary
//          tile prefix and |M|.
//   fill   each warp takes one (tile, offset) pair: lane p holds point p's
//          neighbour, a ballot ranks the hits, and the (in, out) entries are
//          written to consecutive positions of the offset's segment, which
//          therefore follows the row order.

#include "sc_internal.cuh"

namespace sc {
namespace {

constexpr int kTile = 32;        // points per tile (one bitmask word)
constexpr int kThreads = 256;    // threads per probe / fill block
constexpr int kWsRows = 128;     // rows per weight-stationary tile
constexpr int kScanThreads = 512;  // >= the largest V (343)
constexpr int kScanPer = 8;        // tiles per scan thread per chunk
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

// Insert: find or claim the entry of the voxel's block (CAS on the block
// key), then CAS the voxel's row slot from -1 to its row id; a slot that is
// already taken means two rows share the coordinate.
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
      unsigned long long k = __ldcg(&table[h].key);
      if (k == kEmptyKey) {
        k = atomicCAS(&table[h].key, kEmptyKey, bk);
        if (k == kEmptyKey) k = bk;
      }
      if (k == bk) {
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
                                                       int* __restrict__ cursors, int* __restrict__ order) {
  const int tb = order_total_bits(ob, hash_status);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int pos = atomicAdd(cursors + order_bucket(__ldg(keys + i), ob, tb), 1);
    order[pos] = static_cast<int>(i);
  }
}


__global__ void __launch_bounds__(kThreads) k_kmap_probe(
    const unsigned long long* __restrict__ keys, const int* __restrict__ order, int64_t n,
    const BlockEntry* __restrict__ table, uint32_t mask, int V, int K, int ndim, int dimx, int dimy, int dimz,
    int* __restrict__ nbr, unsigned* __restrict__ masks, unsigned* __restrict__ present, int ntiles,
    int* __restrict__ status) {
  extern __shared__ int4 smem4[];
  int* s_tile = reinterpret_cast<int*>(smem4);  // [32 * V] the tile's block of the table
  __shared__ unsigned s_pres[4];
  constexpr int kWarps = kThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (K - 1) / 2;
  const int rz = ndim == 3 ? r : 0;
  const int centre = (V - 1) / 2;
  for (int e = threadIdx.x; e < kTile * V; e += kThreads) s_tile[e] = -1;
  if (threadIdx.x < 4) s_pres[threadIdx.x] = 0u;
  const int tile = blockIdx.x;
  const int64_t i0 = static_cast<int64_t>(tile) * kTile;
  const int np = static_cast<int>(min(static_cast<int64_t>(kTile), n - i0));
  // lane = point of the tile (every warp holds the same 32 points)
  const bool live = lane < np;
  const int row = live ? (order ? __ldg(order + i0 + lane) : static_cast<int>(i0 + lane)) : 0;
  const unsigned long long ck = live ? __ldg(keys + row) : kEmptyKey;
  bool valid = ck != kEmptyKey;
  const int x = static_cast<int>((ck >> 32) & 0xFFFF), y = static_cast<int>((ck >> 16) & 0xFFFF),
            z = static_cast<int>(ck & 0xFFFF);
  if (valid && (x >= dimx || y >= dimy || z >= dimz)) {
    if (warp == 0) atomicOr(status, kDevErrRange);
    valid = false;
  }
  const unsigned long long batch = ck & 0xFFFF000000000000ull;
  // the blocks covering the neighbourhood [x-r, x+r] x [y-r, y+r] x [z-rz, z+rz]
  const int xlo = max(x - r, 0) >> 1, xhi = min(x + r, dimx - 1) >> 1;
  const int ylo = max(y - r, 0) >> 1, yhi = min(y + r, dimy - 1) >> 1;
  const int zlo = max(z - rz, 0) >> 1, zhi = min(z + rz, dimz - 1) >> 1;
  __syncthreads();
  // warp w looks up block triples w, w + kWarps, ... and files each voxel of
  // the block that lies in the neighbourhood under its offset
  const int nb = r + 1, nbz = rz + 1;  // blocks per axis, at most
  for (int t = warp; t < nb * nb * nbz; t += kWarps) {
    const int bx = xlo + t / (nb * nbz), by = ylo + (t / nbz) % nb, bz = zlo + t % nbz;
    if (valid && bx <= xhi && by <= yhi && bz <= zhi) {
      int4 r0, r1;
      if (lookup_block(table, mask, batch | pack_key(0, 2 * bx, 2 * by, 2 * bz), r0, r1)) {
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          const int dx = 2 * bx + (l >> 2) - x, dy = 2 * by + ((l >> 1) & 1) - y, dz = 2 * bz + (l & 1) - z;
          if (dx >= -r && dx <= r && dy >= -r && dy <= r && dz >= -rz && dz <= rz) {
            const int v = ndim == 3 ? ((dx + r) * K + (dy + r)) * K + (dz + r) : (dx + r) * K + (dy + r);
            s_tile[lane * V + v] = pick(r0, r1, l);
          }
        }
      }
    }
  }
  __syncthreads();
  // per-offset hit masks of the tile; offsets present in its 128-row group
  for (int v = warp; v < V; v += kWarps) {
    const unsigned b = __ballot_sync(0xffffffffu, v != centre && s_tile[lane * V + v] >= 0);
    if (lane == 0) {
      masks[static_cast<int64_t>(v) * ntiles + tile] = b;
      if (b && v < 128) atomicOr(s_pres + (v >> 5), 1u << (v & 31));
    }
  }
  __syncthreads();
  // the tile's block of the table is contiguous: i0 * V * 4 bytes is a multiple of 128
  int* dst = nbr + i0 * V;
  const int items = np * V;
  const int n4 = items >> 2;
  for (int e = threadIdx.x; e < n4; e += kThreads) reinterpret_cast<int4*>(dst)[e] = reinterpret_cast<const int4*>(s_tile)[e];
  for (int e = (n4 << 2) + threadIdx.x; e < items; e += kThreads) dst[e] = s_tile[e];
  if (threadIdx.x < 4 && s_pres[threadIdx.x]) atomicOr(present + (tile >> 2) * 4 + threadIdx.x, s_pres[threadIdx.x]);
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

__global__ void __launch_bounds__(kScanThreads) k_kmap_scan(
    const unsigned* __restrict__ masks, int ntiles, int V, int64_t n, int* __restrict__ bases,
    int* __restrict__ totals, int64_t* __restrict__ offs, int* __restrict__ ws_tiles, int64_t* __restrict__ map_size,
    int* __restrict__ ticket) {
  __shared__ long long warp_sums[32];
  __shared__ int s_last;
  const int v = blockIdx.x;
  const unsigned* m = masks + static_cast<int64_t>(v) * ntiles;
  int* b = bases + static_cast<int64_t>(v) * ntiles;
  // each thread takes kScanPer consecutive tiles: all loads of a chunk are in
  // flight together, then one block scan of the per-thread sums
  long long carry = 0;
  for (int base = 0; base < ntiles; base += kScanThreads * kScanPer) {
    const int i0 = base + threadIdx.x * kScanPer;
    int c[kScanPer];
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) c[k] = i0 + k < ntiles ? __popc(__ldg(m + i0 + k)) : 0;
    int sum = 0;
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) sum += c[k];
    long long total;
    const long long inc = block_inclusive_scan<long long>(sum, warp_sums, &total);
    int run = static_cast<int>(carry + inc - sum);
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      if (i0 + k < ntiles) b[i0 + k] = run;
      run += c[k];
    }
    carry += total;
  }
  if (threadIdx.x == 0) {
    totals[v] = static_cast<int>(carry);
    __threadfence();
    s_last = atomicAdd(ticket, 1) == V - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // the last block: segment offsets, weight-stationary tile prefix, |M|
  __threadfence();
  const int t = threadIdx.x;
  const long long cnt = t < V ? static_cast<long long>(__ldcg(totals + t)) : 0;
  long long tot1, tot2;
  const long long inc = block_inclusive_scan<long long>(cnt, warp_sums, &tot1);
  const long long tl = (cnt + kWsRows - 1) / kWsRows;
  const long long inc2 = block_inclusive_scan<long long>(tl, warp_sums, &tot2);
  if (t < V) {
    offs[t] = inc - cnt;
    ws_tiles[t] = static_cast<int>(inc2 - tl);
  }
  if (t == 0) {
    offs[V] = tot1;
    ws_tiles[V] = static_cast<int>(tot2);
    *map_size = n + tot1;
    *ticket = 0;
  }
}

__global__ void __launch_bounds__(kThreads) k_kmap_fill(const int* __restrict__ nbr, const int* __restrict__ order,
                                                        int64_t n, int V, int ntiles,
                                                        int tiles_per_block, const int* __restrict__ bases,
                                                        const int64_t* __restrict__ offs, int* __restrict__ in_rows,
                                                        int* __restrict__ out_rows) {
  extern __shared__ int4 smem_fill[];
  int* smem_i = reinterpret_cast<int*>(smem_fill);
  int* s_nbr = smem_i;                                          // [tiles_per_block * 32 * V], 16-byte aligned
  long long* s_offs = reinterpret_cast<long long*>(s_nbr + ((tiles_per_block * kTile * V + 3) & ~3));  // [V]
  int* s_base = reinterpret_cast<int*>(s_offs + V);             // [tiles_per_block * V]
  int* s_row = s_base + tiles_per_block * V;                    // [tiles_per_block * 32]
  const int tile0 = blockIdx.x * tiles_per_block;
  const int ntl = min(tiles_per_block, ntiles - tile0);
  const int64_t i0 = static_cast<int64_t>(tile0) * kTile;
  const int np = static_cast<int>(min(static_cast<int64_t>(ntl) * kTile, n - i0));
  const int items = np * V;
  for (int p = threadIdx.x; p < np; p += kThreads) s_row[p] = order ? __ldg(order + i0 + p) : static_cast<int>(i0 + p);
  const int* src = nbr + i0 * V;
  const int n4 = items >> 2;
  for (int e = threadIdx.x; e < n4; e += kThreads)
    reinterpret_cast<int4*>(s_nbr)[e] = __ldg(reinterpret_cast<const int4*>(src) + e);
  for (int e = (n4 << 2) + threadIdx.x; e < items; e += kThreads) s_nbr[e] = __ldg(src + e);
  for (int v = threadIdx.x; v < V; v += kThreads) s_offs[v] = __ldg(offs + v);
  for (int q = threadIdx.x; q < ntl * V; q += kThreads) {
    const int tl = q / V, v = q - tl * V;
    s_base[q] = __ldg(bases + static_cast<int64_t>(v) * ntiles + tile0 + tl);
  }
  __syncthreads();
  const int centre = (V - 1) / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q = warp; q < ntl * V; q += kThreads / 32) {
    const int tl = q / V, v = q - tl * V;
    if (v == centre) continue;
    const int p = tl * kTile + lane;
    const int j = p < np ? s_nbr[p * V + v] : -1;
    const unsigned bal = __ballot_sync(0xffffffffu, j >= 0);
    if (j >= 0) {
      const long long at = s_offs[v] + s_base[q] + __popc(bal & ((1u << lane) - 1u));
      in_rows[at] = j;
      out_rows[at] = s_row[p];
    }
  }
}

int grid_for(int64_t n, int threads) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  int64_t g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

int fill_tiles_per_block(int V) {
  int t = 8000 / (kTile * (V + 1));
  return t < 1 ? 1 : (t > 8 ? 8 : t);
}

}  // namespace

int kmap_probe_tile() { return kTile; }
int kmap_order_buckets() { return kBuckets + kBucketBlocks; }

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

sc_status launch_kmap_build(const HashTable* h, KernelMap* m, cudaStream_t s) {
  const int V = m->V;
  cudaError_t e;
  if (m->n == 0) {
    e = cudaMemsetAsync(m->offs, 0, sizeof(int64_t) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->ws_tiles, 0, sizeof(int) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->map_size, 0, sizeof(int64_t), s);
    return e == cudaSuccess ? SC_OK : set_cuda_error(e, "empty kmap init");
  }
  const int tpb = fill_tiles_per_block(V);
  const size_t probe_smem = sizeof(int) * kTile * V;
  const size_t fill_smem =
      sizeof(int) * (4 + 2 * V + static_cast<size_t>(tpb) * V + static_cast<size_t>(tpb) * kTile * (V + 1));
  const uint32_t mask = static_cast<uint32_t>(h->capacity - 1);
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
              k_order_scatter<<<og, 256, 0, s>>>(h->keys, m->n, ob, h->status, m->buckets, m->order));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "locality order launch");
  }
  e = cudaMemsetAsync(m->present, 0, sizeof(unsigned) * 4 * ((m->n + 127) / 128), s);
  if (e != cudaSuccess) return set_cuda_error(e, "kmap presence clear");
  SC_LAUNCH("kmap_probe", s,
            k_kmap_probe<<<m->ntiles, kThreads, probe_smem, s>>>(h->keys, m->order, m->n, h->table, mask, V,
                                                                  m->K,
                                                                  m->ndim,
                                                                  m->dims[0], m->dims[1], m->dims[2], m->nbr,
                                                                  m->masks, m->present, m->ntiles, m->status));
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "kmap_probe launch");
  SC_LAUNCH("kmap_scan", s,
            k_kmap_scan<<<V, kScanThreads, 0, s>>>(m->masks, m->ntiles, V, m->n, m->bases, m->totals, m->offs,
                                                   m->ws_tiles, m->map_size, m->status + 2));
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "kmap_scan launch");
  const int fill_blocks = (m->ntiles + tpb - 1) / tpb;
  SC_LAUNCH("kmap_fill", s,
            k_kmap_fill<<<fill_blocks, kThreads, fill_smem, s>>>(m->nbr, m->order, m->n, V, m->ntiles, tpb, m->bases,
                                                                  m->offs,
                                                                  m->in_rows, m->out_rows));
  e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "kmap_fill launch");
}

}  // namespace sc
