// Internal declarations shared by the libsc translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "sc.h"

namespace sc {

// ---------------------------------------------------------------- status --
// Bits latched by kernels in a device status word.
enum : int {
  kDevErrRange = 1,    // coordinate outside its field / outside dims
  kDevErrDup = 2,      // duplicate coordinate at insert
  kDevErrFull = 4,     // insert probed every slot without finding room
  kDevErrTimeout = 8,  // a bounded mbarrier wait gave up
};

// ------------------------------------------------------------ hash table --
// 64-bit key: batch in bits 48..63, x in 32..47, y in 16..31, z in 0..15.
// Every field is < 65535, so the all-ones word never occurs as a key and
// marks an empty slot.
constexpr unsigned long long kEmptyKey = ~0ull;

__host__ __device__ __forceinline__ unsigned long long pack_key(uint32_t b, uint32_t x, uint32_t y,
                                                                uint32_t z) {
  return (static_cast<unsigned long long>(b) << 48) | (static_cast<unsigned long long>(x) << 32) |
         (static_cast<unsigned long long>(y) << 16) | static_cast<unsigned long long>(z);
}

// The table holds one entry per occupied 2x2x2 block of voxels: the block's
// packed key (the voxel key with the low bit of x, y and z cleared) and the
// row ids of its eight voxels (-1 where absent).  A voxel's position in its
// block is 4*(x&1) + 2*(y&1) + (z&1).  64-byte entries, two per cache line.
// Open addressing with linear probing over entries, home entry = Fibonacci
// (multiplicative) hash of the block key.  A point's 3x3x3 neighbourhood
// spans exactly 8 blocks and its 5x5x5 neighbourhood 27, so a few lookups
// return every neighbour, present or absent.
struct __align__(64) BlockEntry {
  unsigned long long key;
  unsigned long long occupancy;  // output-set construction only: a cleared bit l marks voxel l
  int rows[8];
  int pad1[4];
};

constexpr unsigned long long kBlockLowBits = 0x0000000100010001ull;

__host__ __device__ __forceinline__ unsigned long long block_key(unsigned long long key) {
  return key & ~kBlockLowBits;
}
__host__ __device__ __forceinline__ int block_local(unsigned long long key) {
  return static_cast<int>(((key >> 30) & 4u) | ((key >> 15) & 2u) | (key & 1u));
}
__host__ __device__ __forceinline__ uint32_t block_home(unsigned long long bkey, uint32_t mask) {
  return static_cast<uint32_t>((bkey * 0x9E3779B97F4A7C15ull) >> 32) & mask;
}

// ------------------------------------------------------------- handles --
struct HashTable {
  int64_t n = 0;
  int64_t capacity = 0;              // block entries, a power of two
  BlockEntry* table = nullptr;       // [capacity]
  unsigned long long* keys = nullptr;  // [n]  packed key of each row (kEmptyKey if invalid)
  int* status = nullptr;             // [4]: latched errors, largest batch id
};

struct ConvChoice {
  int c_in, c_out, dtype;
  unsigned variant;
};

struct KernelMap {
  int64_t n = 0;                     // rows of the map (output points)
  int64_t n_in = 0;                  // rows of the input (= n for a submanifold map)
  int stride = 1;                    // output o reads the inputs at stride * o + d
  bool identity = true;              // submanifold: outputs = inputs, the centre list is the identity
  bool transposed = false;           // rows = a layer's inputs, neighbours = its outputs at mirrored offsets
  int ndim = 3, K = 3, V = 27;
  int dims[3] = {1, 1, 1};
  int up = 128;                      // points per map-build unit (128; 64 when V > 64; 32 when V > 128)
  int nunits = 0;                    // map-build units
  bool half = false;                 // built by the half probe (mirror symmetry)
  int* order = nullptr;              // [n] input rows in locality order, or null: input order
  int* inv_order = nullptr;          // half probe with the order: [n] table row of each input row
  unsigned long long* skeys = nullptr;  // [n] packed keys in locality order (with order)
  int* buckets = nullptr;            // counting-sort buckets of that order (+ scan partials)
  int* nbr = nullptr;                // [n, V], rows in the row order (position k = input row order[k])
  int64_t* offs = nullptr;           // [V+1]
  int* in_rows = nullptr;            // [V, n]: offset v's list at v * n, offs[v+1] - offs[v] entries
  int* out_rows = nullptr;
  unsigned* present = nullptr;       // [ceil(n/128), 4] offsets (< 128) with a hit in each 128-row tile of the row order
  int* cursors = nullptr;            // [V * kCursorStride] list entries reserved per offset during the build
  // signature sort (V <= 128): the convolution walks rows in a second order
  unsigned* rowmask = nullptr;       // [n] (V <= 32) or [n, 4] (V <= 128) offsets with a neighbour, per row of the table
  unsigned* rowdir = nullptr;        // V > 32: [n] coarse directions with a neighbour, per row; else null
  int* sig_sel = nullptr;            // [16 (x 3 when split)] signature features (offsets or directions), rarest first
  int* sigbuckets = nullptr;         // counting-sort buckets (+ scan partials)
  int* perm = nullptr;               // [n] sorted position -> table row, or null: no sort
  int* conv_order = nullptr;         // [n] sorted position -> input row
  // SC_KMAP_TILE_TABLE: the fused layer's neighbour indices in its row order
  // (perm, or the table's own), transposed within each 128-row tile,
  // [ceil(n/128)][V][128], -1 past the last row; null: the layer reads nbr
  int* tnbr = nullptr;
  // column splitting (V <= 32): offsets [0, split_at) form part 0 (the
  // centre is the last of them), [split_at, V) part 1; each part has its own
  // signature sort of the rows and tile masks restricted to its offsets
  int nparts = 1;
  int split_at = 0;
  int* part_perm[2] = {nullptr, nullptr};
  int* part_order[2] = {nullptr, nullptr};
  unsigned* part_present[2] = {nullptr, nullptr};
  int* ws_tiles = nullptr;           // [V+1] prefix of ceil(count/128) per offset
  int64_t* map_size = nullptr;       // device: n + offs[V]
  int* status = nullptr;             // [4]: map status, copy of the hash status, scan ticket
  // host mirrors, valid once synchronised
  bool host_valid = false;
  std::vector<int64_t> offs_host;    // [V+1]
  std::vector<int> ws_tiles_host;    // [V+1]
  int64_t map_size_host = -1;
  std::vector<ConvChoice> tuned;
};

// The map build's per-offset list cursors sit one per 128-byte line: every
// build block adds to each of them, and atomics on one line serialise.
constexpr int kCursorStride = 32;

// Size of the fixed packed-weight buffer behind sc_subm_conv_fwd_noalloc.
constexpr size_t kNoAllocWeightBytes = size_t(4) << 20;

// ------------------------------------------------------------ launching --
// Launch bookkeeping shared by every translation unit: counts launches and,
// while profiling is on, brackets each launch with CUDA events.
int prof_begin(const char* name, cudaStream_t s);
void prof_end(int token, cudaStream_t s);

// Records a failing CUDA call's text for sc_last_error().
sc_status set_cuda_error(cudaError_t e, const char* where);
sc_status set_error(sc_status s, const char* msg);

int device_sm_count();

// Prepares a kernel for a launch with `smem` bytes of dynamic shared memory:
// raises its shared-memory limit (and asks for the largest carveout) the
// first time a device needs that much, and reports its registers per
// thread.  Cached per device and kernel, so a launch costs no attribute
// calls once warm.
sc_status kernel_setup(const void* kern, size_t smem, int* num_regs);
// Sets a kernel's shared-memory carveout to what `ctas_per_sm` CTAs of
// `smem` bytes need (the rest of the SM's L1/shared array stays L1, which
// holds the neighbour-index loads); cached, so set only when it changes.
sc_status kernel_carveout(const void* kern, int ctas_per_sm, size_t smem);

// kernels: hash + map (hash_kmap.cu)
sc_status launch_hash_insert(const int32_t* coords, int64_t n, HashTable* h, cudaStream_t s);
sc_status launch_hash_query(const HashTable* h, const int32_t* q, int64_t m, int32_t* rows,
                            cudaStream_t s);
// Map of the points of `out` against the table of `in` (out == in for a submanifold map).
sc_status launch_kmap_build(const HashTable* in, const HashTable* out, KernelMap* m, cudaStream_t s);
// Output set of a regular / strided layer as a new hash table `out` (its table
// in *arena_table, its keys in *arena_keys); synchronises once to size it.
sc_status launch_conv_out(const HashTable* in, int ndim, int K, int stride, const int32_t dims[3], HashTable* out,
                          void** arena_table, void** arena_keys, const sc_allocator* alloc, cudaStream_t s);
sc_status launch_hash_coords(const HashTable* h, int32_t* coords, cudaStream_t s);
int kmap_unit_points(int V);
sc_status kmap_compact_lists(const KernelMap* m, const int* src, int* dst, int64_t total, cudaStream_t s);
int kmap_order_buckets();
int kmap_sig_bits();
int64_t kmap_sig_buckets(int64_t n);

// kernels: convolution (conv_tc.cu, conv_simt.cu)
struct ConvArgs {
  const KernelMap* m;
  const void* feats;
  const void* W;
  void* out;
  int c_in, c_out;
  sc_dtype dtype;
  bool relu;
  cudaStream_t stream;
  // W holds a forward layer's weights [V, c_out, c_in] and the layer applied
  // is its input gradient: W'[v] = W[V-1-v]^T (mirrored offset, transposed)
  bool wt = false;
};
sc_status conv_bwd_weight(const KernelMap* m, const void* feats, const void* gout, void* dW, int c_in, int c_out,
                          sc_dtype dtype, cudaStream_t s);
sc_status conv_fused(const ConvArgs& a);
sc_status conv_fused_split(const ConvArgs& a);
sc_status conv_weight_stationary(const ConvArgs& a);
sc_status conv_simt(const ConvArgs& a);
// nbr rows in input order (undoing the row order) into a device buffer
sc_status kmap_unpermute_nbr(const KernelMap* m, int* dst, cudaStream_t s);
bool fused_supported(const ConvArgs& a);
sc_status conv_fused_noalloc(const ConvArgs& a);

// stream-ordered allocation helpers: `with` (if not null) is the caller's
// allocator of a build call, else the process-wide setting is used; a buffer
// goes back to whichever allocator made it
sc_status dev_alloc(void** p, size_t bytes, cudaStream_t s, const sc_allocator* with = nullptr);
void dev_free(void* p, cudaStream_t s);

}  // namespace sc

#define SC_LAUNCH(name, stream, ...)                   \
  do {                                                 \
    int _tok = ::sc::prof_begin(name, stream);         \
    __VA_ARGS__;                                       \
    ::sc::prof_end(_tok, stream);                      \
  } while (0)
