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
// section 3) and, within an offset, ordered by output row.
//
// Three kernels build the map:
//   probe  one block per tile of 64 points; the block's threads take the
//          tile's (point, offset) pairs in row-major order, each thread keeps
//          eight first-slot loads in flight, and the tile's [64, V] slice of
//          the neighbour table is written with coalesced 16-byte stores.  Per
//          tile and offset it also counts hits (warp ballots).
//   scan   one block per offset: exclusive prefix of the per-tile counts.
//   fill   one block per tile: re-reads its neighbour slice and writes the
//          (in, out) list entries at their final positions, warp-ballot
//          compacted, so every list is ordered by output row.

#include "sc_internal.cuh"

namespace sc {
namespace {

constexpr int kTile = 64;       // points per probe/fill tile
constexpr int kThreads = 256;   // threads per probe/fill block
constexpr int kIlp = 8;         // outstanding first-slot probes per thread
constexpr int kWsRows = 128;    // rows per weight-stationary tile

__device__ __forceinline__ ulonglong2 load_slot(const Slot* __restrict__ t, unsigned long long i) {
  return __ldg(reinterpret_cast<const ulonglong2*>(t + i));
}

__device__ __forceinline__ int table_find(const Slot* __restrict__ table, unsigned long long mask,
                                          unsigned long long key, unsigned long long h, ulonglong2 cur) {
  for (unsigned long long probe = 0; probe <= mask; ++probe) {
    if (cur.x == key) return static_cast<int>(static_cast<unsigned>(cur.y & 0xffffffffull));
    if (cur.x == kEmptyKey) return -1;
    h = (h + 1) & mask;
    cur = load_slot(table, h);
  }
  return -1;
}

__global__ void __launch_bounds__(256) k_hash_insert(const int4* __restrict__ coords, int64_t n,
                                                     Slot* __restrict__ table, unsigned long long mask,
                                                     unsigned long long* __restrict__ keys,
                                                     int* __restrict__ status) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int4 c = __ldg(coords + i);
    if (static_cast<unsigned>(c.x) >= 65535u || static_cast<unsigned>(c.y) >= 65535u ||
        static_cast<unsigned>(c.z) >= 65535u || static_cast<unsigned>(c.w) >= 65535u) {
      keys[i] = kEmptyKey;
      atomicOr(status, kDevErrRange);
      continue;
    }
    const unsigned long long key = pack_key(c.x, c.y, c.z, c.w);
    keys[i] = key;
    unsigned long long h = hash_mix(key) & mask;
    bool placed = false;
    for (unsigned long long probe = 0; probe <= mask; ++probe) {
      const unsigned long long prev = atomicCAS(&table[h].key, kEmptyKey, key);
      if (prev == kEmptyKey) {
        table[h].val = static_cast<int>(i);
        placed = true;
        break;
      }
      if (prev == key) {
        atomicOr(status, kDevErrDup);
        placed = true;
        break;
      }
      h = (h + 1) & mask;
    }
    if (!placed) atomicOr(status, kDevErrFull);
  }
}

__global__ void __launch_bounds__(256) k_hash_query(const int4* __restrict__ q, int64_t m,
                                                    const Slot* __restrict__ table, unsigned long long mask,
                                                    int* __restrict__ rows) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m; i += stride) {
    const int4 c = __ldg(q + i);
    int r = -1;
    if (static_cast<unsigned>(c.x) < 65535u && static_cast<unsigned>(c.y) < 65535u &&
        static_cast<unsigned>(c.z) < 65535u && static_cast<unsigned>(c.w) < 65535u) {
      const unsigned long long key = pack_key(c.x, c.y, c.z, c.w);
      const unsigned long long h = hash_mix(key) & mask;
      r = table_find(table, mask, key, h, load_slot(table, h));
    }
    rows[i] = r;
  }
}

// Offsets are packed 10 bits per axis with a bias of 512.
__device__ __forceinline__ int unpack_off(int o, int axis) { return ((o >> (10 * axis)) & 1023) - 512; }

__global__ void __launch_bounds__(kThreads) k_kmap_probe(
    const unsigned long long* __restrict__ keys, int64_t n, const Slot* __restrict__ table,
    unsigned long long mask, int V, int K, int ndim, int dimx, int dimy, int dimz, int* __restrict__ nbr,
    int* __restrict__ counts, int ntiles, int* __restrict__ status) {
  extern __shared__ int4 smem4[];
  int* s_nbr = reinterpret_cast<int*>(smem4);  // [kTile * V]
  int* s_off = s_nbr + kTile * V;              // [V]
  const int tid = threadIdx.x;
  const int tile = blockIdx.x;
  const int64_t i0 = static_cast<int64_t>(tile) * kTile;
  const int np = static_cast<int>(min(static_cast<int64_t>(kTile), n - i0));
  const int r = (K - 1) / 2;
  const int centre = (V - 1) / 2;
  for (int v = tid; v < V; v += kThreads) {
    int d[3] = {0, 0, 0};
    int t = v;
    for (int k = ndim - 1; k >= 0; --k) {
      d[k] = t % K - r;
      t /= K;
    }
    s_off[v] = (d[0] + 512) | ((d[1] + 512) << 10) | ((d[2] + 512) << 20);
  }
  __syncthreads();

  const int items = np * V;
  for (int base = 0; base < items; base += kThreads * kIlp) {
    unsigned long long key[kIlp], slot[kIlp];
    ulonglong2 cur[kIlp];
    int res[kIlp];
    bool act[kIlp];
#pragma unroll
    for (int k = 0; k < kIlp; ++k) {
      const int e = base + tid + k * kThreads;
      act[k] = false;
      res[k] = -1;
      key[k] = 0;
      slot[k] = 0;
      if (e < items) {
        const int p = e / V;
        const int v = e - p * V;
        const unsigned long long ck = __ldg(keys + i0 + p);
        if (ck != kEmptyKey) {
          int x = static_cast<int>((ck >> 32) & 0xFFFF);
          int y = static_cast<int>((ck >> 16) & 0xFFFF);
          int z = static_cast<int>(ck & 0xFFFF);
          if (v == centre) {
            res[k] = static_cast<int>(i0 + p);
            if (x >= dimx || y >= dimy || z >= dimz) atomicOr(status, kDevErrRange);
          } else {
            const int o = s_off[v];
            x += unpack_off(o, 0);
            y += unpack_off(o, 1);
            z += unpack_off(o, 2);
            if (static_cast<unsigned>(x) < static_cast<unsigned>(dimx) &&
                static_cast<unsigned>(y) < static_cast<unsigned>(dimy) &&
                static_cast<unsigned>(z) < static_cast<unsigned>(dimz)) {
              key[k] = (ck & 0xFFFF000000000000ull) | pack_key(0, x, y, z);
              slot[k] = hash_mix(key[k]) & mask;
              act[k] = true;
            }
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kIlp; ++k)
      if (act[k]) cur[k] = load_slot(table, slot[k]);
#pragma unroll
    for (int k = 0; k < kIlp; ++k) {
      if (act[k]) res[k] = table_find(table, mask, key[k], slot[k], cur[k]);
      const int e = base + tid + k * kThreads;
      if (e < items) s_nbr[e] = res[k];
    }
  }
  __syncthreads();

  // The tile's slice of nbr is contiguous: i0*V*4 bytes is a multiple of 256.
  int* dst = nbr + i0 * V;
  const int n4 = items >> 2;
  for (int e = tid; e < n4; e += kThreads)
    reinterpret_cast<int4*>(dst)[e] = reinterpret_cast<const int4*>(s_nbr)[e];
  for (int e = (n4 << 2) + tid; e < items; e += kThreads) dst[e] = s_nbr[e];

  const int warp = tid >> 5, lane = tid & 31;
  for (int v = warp; v < V; v += kThreads / 32) {
    int cnt = 0;
    if (v != centre) {
      for (int p0 = 0; p0 < np; p0 += 32) {
        const int p = p0 + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, p < np && s_nbr[p * V + v] >= 0));
      }
    }
    if (lane == 0) counts[static_cast<int64_t>(v) * ntiles + tile] = cnt;
  }
}

// Exclusive prefix of counts[v, 0:ntiles] in place; totals[v] = sum.
__global__ void __launch_bounds__(1024) k_kmap_scan(int* __restrict__ counts, int ntiles, int* __restrict__ totals) {
  __shared__ int warp_sums[32];
  const int v = blockIdx.x;
  int* c = counts + static_cast<int64_t>(v) * ntiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < ntiles; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int x = i < ntiles ? c[i] : 0;
    int y = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += t;
    }
    if (lane == 31) warp_sums[warp] = y;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    if (i < ntiles) c[i] = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + y - x;
    carry += warp_sums[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) totals[v] = carry;
}

__global__ void __launch_bounds__(kThreads) k_kmap_fill(
    const int* __restrict__ nbr, int64_t n, int V, const int* __restrict__ bases, const int* __restrict__ totals,
    int ntiles, int64_t* __restrict__ offs, int* __restrict__ ws_tiles, int64_t* __restrict__ map_size,
    int* __restrict__ in_rows, int* __restrict__ out_rows) {
  extern __shared__ int4 smem4[];
  int* s_nbr = reinterpret_cast<int*>(smem4);                               // [kTile * V]
  long long* s_offs = reinterpret_cast<long long*>(s_nbr + ((kTile * V + 1) & ~1));  // [V+1]
  const int tid = threadIdx.x;
  const int tile = blockIdx.x;
  const int64_t i0 = static_cast<int64_t>(tile) * kTile;
  const int np = static_cast<int>(min(static_cast<int64_t>(kTile), n - i0));
  const int centre = (V - 1) / 2;
  const int items = np * V;
  const int* src = nbr + i0 * V;
  const int n4 = items >> 2;
  for (int e = tid; e < n4; e += kThreads)
    reinterpret_cast<int4*>(s_nbr)[e] = __ldg(reinterpret_cast<const int4*>(src) + e);
  for (int e = (n4 << 2) + tid; e < items; e += kThreads) s_nbr[e] = __ldg(src + e);
  if (tid == 0) {
    long long acc = 0;
    for (int v = 0; v < V; ++v) {
      s_offs[v] = acc;
      acc += totals[v];
    }
    s_offs[V] = acc;
  }
  __syncthreads();
  if (tile == 0) {
    for (int v = tid; v <= V; v += kThreads) offs[v] = s_offs[v];
    if (tid == 0) {
      *map_size = n + s_offs[V];
      int t = 0;
      for (int v = 0; v < V; ++v) {
        ws_tiles[v] = t;
        t += (totals[v] + kWsRows - 1) / kWsRows;
      }
      ws_tiles[V] = t;
    }
  }
  const int warp = tid >> 5, lane = tid & 31;
  for (int v = warp; v < V; v += kThreads / 32) {
    if (v == centre) continue;
    long long pos = s_offs[v] + bases[static_cast<int64_t>(v) * ntiles + tile];
    for (int p0 = 0; p0 < np; p0 += 32) {
      const int p = p0 + lane;
      const int j = p < np ? s_nbr[p * V + v] : -1;
      const unsigned b = __ballot_sync(0xffffffffu, j >= 0);
      if (j >= 0) {
        const long long at = pos + __popc(b & ((1u << lane) - 1u));
        in_rows[at] = j;
        out_rows[at] = static_cast<int>(i0 + p);
      }
      pos += __popc(b);
    }
  }
}

int grid_for(int64_t n, int threads) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  int64_t g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

int kmap_probe_tile() { return kTile; }

sc_status launch_hash_insert(const int32_t* coords, int64_t n, HashTable* h, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(h->table, 0xFF, sizeof(Slot) * h->capacity, s);
  if (e != cudaSuccess) return set_cuda_error(e, "hash table clear");
  e = cudaMemsetAsync(h->status, 0, sizeof(int), s);
  if (e != cudaSuccess) return set_cuda_error(e, "hash status clear");
  if (n == 0) return SC_OK;
  SC_LAUNCH("hash_insert", s,
            k_hash_insert<<<grid_for(n, 256), 256, 0, s>>>(reinterpret_cast<const int4*>(coords), n, h->table,
                                                           static_cast<unsigned long long>(h->capacity - 1),
                                                           h->keys, h->status));
  e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "hash_insert launch");
}

sc_status launch_hash_query(const HashTable* h, const int32_t* q, int64_t m, int32_t* rows, cudaStream_t s) {
  if (m == 0) return SC_OK;
  SC_LAUNCH("hash_query", s,
            k_hash_query<<<grid_for(m, 256), 256, 0, s>>>(reinterpret_cast<const int4*>(q), m, h->table,
                                                          static_cast<unsigned long long>(h->capacity - 1),
                                                          rows));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "hash_query launch");
}

sc_status launch_kmap_build(const HashTable* h, KernelMap* m, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(m->status, 0, sizeof(int), s);
  if (e != cudaSuccess) return set_cuda_error(e, "kmap status clear");
  const int V = m->V;
  if (m->n == 0) {
    e = cudaMemsetAsync(m->offs, 0, sizeof(int64_t) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->ws_tiles, 0, sizeof(int) * (V + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->map_size, 0, sizeof(int64_t), s);
    return e == cudaSuccess ? SC_OK : set_cuda_error(e, "empty kmap init");
  }
  const size_t probe_smem = sizeof(int) * (static_cast<size_t>(kTile) * V + V);
  const size_t fill_smem = sizeof(int) * ((static_cast<size_t>(kTile) * V + 1) & ~static_cast<size_t>(1)) +
                           sizeof(long long) * (V + 1);
  static bool attrs_set = false;
  if (!attrs_set) {
    const int max_smem = 200 * 1024;
    cudaFuncSetAttribute(k_kmap_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    cudaFuncSetAttribute(k_kmap_fill, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    attrs_set = true;
  }
  const unsigned long long mask = static_cast<unsigned long long>(h->capacity - 1);
  SC_LAUNCH("kmap_probe", s,
            k_kmap_probe<<<m->ntiles, kThreads, probe_smem, s>>>(h->keys, m->n, h->table, mask, V, m->K, m->ndim,
                                                                  m->dims[0], m->dims[1], m->dims[2], m->nbr,
                                                                  m->counts, m->ntiles, m->status));
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "kmap_probe launch");
  int scan_threads = 1024;
  if (m->ntiles <= 256) scan_threads = 256;
  SC_LAUNCH("kmap_scan", s, k_kmap_scan<<<V, scan_threads, 0, s>>>(m->counts, m->ntiles, m->totals));
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e, "kmap_scan launch");
  SC_LAUNCH("kmap_fill", s,
            k_kmap_fill<<<m->ntiles, kThreads, fill_smem, s>>>(m->nbr, m->n, V, m->counts, m->totals, m->ntiles,
                                                                m->offs, m->ws_tiles, m->map_size, m->in_rows,
                                                                m->out_rows));
  e = cudaGetLastError();
  return e == cudaSuccess ? SC_OK : set_cuda_error(e, "kmap_fill launch");
}

}  // namespace sc
