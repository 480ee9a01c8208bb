// CPU oracle for the submanifold sparse convolution layer.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / reference legs of bench.py may load or call this code.  It
// shares nothing with the CUDA library: no headers, no helpers, no tables.
//
// It is the plain definition of the layer, written out:
//
//   * Sparse representation: a coordinate list and a feature list, row i of
//     one belonging to row i of the other ("SparseConvNet: from hash table to
//     rulebook", section 1).
//   * Submanifold output set: an output exists exactly where an input exists,
//     P_out = P_in ("Sparse inputs and sparse convolution", section "The fix";
//     exam sheet "Sparse convolution for point clouds", definition).
//   * Kernel map: for every output q and every offset d, look up the input at
//     coordinate q + d in a hash table on coordinates; a hit p adds the tuple
//     (p, q, W_d) ("Sparse inputs and sparse convolution", section "The map is
//     the computation").  Sign convention: input P sits at output Q shifted by
//     the offset, P = Q + d (same page, section "Follow the boxed point"; exam
//     sheet, "The map and the update rule").
//   * Update rule: f_out(Q) += f_in(P) x W_d for every tuple (exam sheet, "The
//     map and the update rule").  Accumulated here in fp64.
//   * Backward (the layer is linear in f and in W): the gradients of a loss
//     with respect to f and W follow from the same tuples, written out below
//     as their plain definitions.
//   * Regular and strided layers (the other output definition of
//     "SparseConvNet: from hash table to rulebook", section 2): an output
//     exists wherever the kernel window covers at least one active input, so
//     the active set grows; with a stride s the output grid is coarser and
//     output o reads the input at s * o + d through W_d (section 3's index
//     relation between input, output, offset and stride).
//
// Offsets are indexed lexicographically with the first spatial axis slowest:
// idx(d) = sum_k (d_k + r) * K^(ndim-1-k), r = (K-1)/2.  In 2D the offsets act
// on (x, y) only and z is carried unchanged.
//
// Parity pins: every function here is pinned by tests under tests/ against the
// pages' worked examples, brute force over point pairs, and an fp64 dense
// convolution from a library routine.  Nothing here is "parity unpinned".

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <unordered_map>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// Status codes returned to the Python wrapper.
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_OUT_OF_RANGE = 2, OR_DUPLICATE = 3 };

// The oracle's own coordinate key: four 16-bit fields, batch highest.
inline uint64_t pack_key(int64_t b, int64_t x, int64_t y, int64_t z) {
  return (uint64_t(b) << 48) | (uint64_t(x) << 32) | (uint64_t(y) << 16) | uint64_t(z);
}

struct Problem {
  const int32_t* coords;  // [n, 4] = (batch, x, y, z)
  int64_t n;
  int ndim;                // 2 or 3
  int K;                   // odd kernel size
  int32_t dims[3];         // spatial extents
  int volume;              // K^ndim
  std::unordered_map<uint64_t, int32_t> table;
};

int check_args(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims) {
  if (n < 0 || (n > 0 && !coords) || !dims) return OR_BAD_ARG;
  if (ndim != 2 && ndim != 3) return OR_BAD_ARG;
  if (K < 1 || (K % 2) == 0) return OR_BAD_ARG;
  for (int a = 0; a < 3; ++a)
    if (dims[a] < 1 || dims[a] > 65535) return OR_BAD_ARG;
  return OR_OK;
}

// Step 1: put every coordinate into a hash table, row id as the value.
int build_table(Problem& P) {
  P.table.clear();
  P.table.reserve(size_t(P.n) * 2 + 1);
  for (int64_t i = 0; i < P.n; ++i) {
    const int32_t* c = P.coords + 4 * i;
    if (c[0] < 0 || c[0] >= 65535) return OR_OUT_OF_RANGE;
    for (int a = 0; a < 3; ++a)
      if (c[1 + a] < 0 || c[1 + a] >= P.dims[a]) return OR_OUT_OF_RANGE;
    auto ins = P.table.emplace(pack_key(c[0], c[1], c[2], c[3]), int32_t(i));
    if (!ins.second) return OR_DUPLICATE;
  }
  return OR_OK;
}

// The spatial offset with lexicographic index idx (first axis slowest).
void offset_of(int idx, int ndim, int K, int d[3]) {
  const int r = (K - 1) / 2;
  d[0] = d[1] = d[2] = 0;
  for (int k = ndim - 1; k >= 0; --k) {
    d[k] = idx % K - r;
    idx /= K;
  }
}

// Step 2: the input row at coordinate c_q + d, or -1 if none is active there
// (outside the grid counts as absent: zero padding).
int32_t neighbour(const Problem& P, int64_t q, const int d[3]) {
  const int32_t* c = P.coords + 4 * q;
  int64_t x = int64_t(c[1]) + d[0];
  int64_t y = int64_t(c[2]) + d[1];
  int64_t z = int64_t(c[3]) + d[2];
  if (x < 0 || x >= P.dims[0] || y < 0 || y >= P.dims[1] || z < 0 || z >= P.dims[2]) return -1;
  auto it = P.table.find(pack_key(c[0], x, y, z));
  return it == P.table.end() ? -1 : it->second;
}

int setup(Problem& P, const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims) {
  int st = check_args(coords, n, ndim, K, dims);
  if (st) return st;
  P.coords = coords;
  P.n = n;
  P.ndim = ndim;
  P.K = K;
  for (int a = 0; a < 3; ++a) P.dims[a] = dims[a];
  P.volume = 1;
  for (int a = 0; a < ndim; ++a) P.volume *= K;
  return build_table(P);
}

int threads_to_use(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

// Output features of the listed rows against a built table (step 2's
// lookups and step 3's accumulation; see oracle_subm_conv).
int conv_rows(const Problem& P, const double* feats, const double* W, int c_in, int c_out, int relu,
              const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  const int64_t n = P.n;
  const int ndim = P.ndim, K = P.K;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  for (int64_t k = 0; k < nrows; ++k)
    if (rows && (rows[k] < 0 || rows[k] >= n)) return OR_BAD_ARG;
  const int nt = threads_to_use(nthreads);
  // small chunks: a sample of a few hundred rows per thread still spreads
  // evenly over the threads (rows are independent; the result is the same)
#pragma omp parallel for schedule(dynamic, 4) num_threads(nt)
  for (int64_t k = 0; k < nrows; ++k) {
    const int64_t q = rows ? rows[k] : k;
    double* acc = out + k * c_out;
    for (int co = 0; co < c_out; ++co) acc[co] = 0.0;
    for (int v = 0; v < V; ++v) {
      const int32_t p = neighbour(P, q, &offs[3 * v]);
      if (p < 0) continue;
      const double* f = feats + int64_t(p) * c_in;
      const double* w = W + int64_t(v) * c_in * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double a = f[ci];
        const double* wrow = w + int64_t(ci) * c_out;
        for (int co = 0; co < c_out; ++co) acc[co] += a * wrow[co];
      }
    }
    if (relu)
      for (int co = 0; co < c_out; ++co) acc[co] = acc[co] > 0.0 ? acc[co] : 0.0;
  }
  return OR_OK;
}

}  // namespace

extern "C" {

// Neighbour table: nbr[q * V + idx(d)] = row of the input at c_q + d, or -1.
// Built by the double loop over outputs and offsets.
int oracle_kmap(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims,
                int32_t* nbr, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t q = 0; q < n; ++q)
    for (int v = 0; v < V; ++v) nbr[q * V + v] = neighbour(P, q, &offs[3 * v]);
  return OR_OK;
}

// Output features for the listed output rows (all rows if rows == NULL):
// out[k, :] = sum over offsets d with an input p at c_q + d of f[p, :] W[d],
// q = rows[k], accumulated in fp64, then max(., 0) if relu != 0.
// feats [n, c_in], W [V, c_in, c_out], out [nrows, c_out], all fp64.
int oracle_subm_conv(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims,
                     const double* feats, const double* W, int c_in, int c_out, int relu,
                     const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (c_in < 1 || c_out < 1 || !W || (n > 0 && !feats) || !out) return OR_BAD_ARG;
  if (!rows) nrows = n;
  return conv_rows(P, feats, W, c_in, c_out, relu, rows, nrows, out, nthreads);
}

// Gradient with respect to the input features of the layer above (without
// its ReLU): the layer is linear in f, out[q] = sum_d f[p(q,d)] W_d with
// p(q,d) the row at c_q + d, so d loss / d f[p] = sum over the pairs (q, d)
// with c_p = c_q + d of gout[q] W_d^T.  For each input row p and offset d the
// output row is the one at c_p - d.  gout [n, c_out], W [V, c_in, c_out],
// gin [nrows, c_in] for the listed input rows (all rows if rows == NULL), fp64.
int oracle_subm_conv_bwd_data(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims,
                              const double* gout, const double* W, int c_in, int c_out, const int64_t* rows,
                              int64_t nrows, double* gin, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (c_in < 1 || c_out < 1 || !W || (n > 0 && (!gout || !gin))) return OR_BAD_ARG;
  if (!rows) nrows = n;
  for (int64_t k = 0; k < nrows; ++k)
    if (rows && (rows[k] < 0 || rows[k] >= n)) return OR_BAD_ARG;
  const int V = P.volume;
  std::vector<int> neg(size_t(V) * 3);
  for (int v = 0; v < V; ++v) {
    offset_of(v, ndim, K, &neg[3 * v]);
    for (int a = 0; a < 3; ++a) neg[3 * v + a] = -neg[3 * v + a];
  }
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(dynamic, 64) num_threads(nt)
  for (int64_t k = 0; k < nrows; ++k) {
    const int64_t p = rows ? rows[k] : k;
    double* acc = gin + k * c_in;
    for (int ci = 0; ci < c_in; ++ci) acc[ci] = 0.0;
    for (int v = 0; v < V; ++v) {
      const int32_t q = neighbour(P, p, &neg[3 * v]);  // the output at c_p - d
      if (q < 0) continue;
      const double* g = gout + int64_t(q) * c_out;
      const double* w = W + int64_t(v) * c_in * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double* wrow = w + int64_t(ci) * c_out;
        double sum = 0.0;
        for (int co = 0; co < c_out; ++co) sum += wrow[co] * g[co];
        acc[ci] += sum;
      }
    }
  }
  return OR_OK;
}

// Gradient with respect to the weights: d loss / d W_d = sum over the pairs
// (q, d) with an input p at c_q + d of f[p]^T gout[q].  feats [n, c_in],
// gout [n, c_out], dW [V, c_in, c_out], fp64; one offset per thread.
int oracle_subm_conv_bwd_weight(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims,
                                const double* feats, const double* gout, int c_in, int c_out, double* dW,
                                int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (c_in < 1 || c_out < 1 || !dW || (n > 0 && (!feats || !gout))) return OR_BAD_ARG;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int v = 0; v < V; ++v) {
    double* acc = dW + int64_t(v) * c_in * c_out;
    for (int64_t e = 0; e < int64_t(c_in) * c_out; ++e) acc[e] = 0.0;
    for (int64_t q = 0; q < n; ++q) {
      const int32_t p = neighbour(P, q, &offs[3 * v]);
      if (p < 0) continue;
      const double* f = feats + int64_t(p) * c_in;
      const double* g = gout + q * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double a = f[ci];
        double* row = acc + int64_t(ci) * c_out;
        for (int co = 0; co < c_out; ++co) row[co] += a * g[co];
      }
    }
  }
  return OR_OK;
}

// Step 1 alone (the coordinate hash table), for timing the oracle's phases.
int oracle_hash_only(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims) {
  Problem P;
  return setup(P, coords, n, ndim, K, dims);
}

// Number of threads the OpenMP runtime would use by default.
int oracle_max_threads(void) { return threads_to_use(0); }

// The coordinate table (step 1) built once and kept, and layer outputs of
// listed rows computed against it: lets a caller time the table and the rows
// apart.  coords must stay alive and unchanged while the table lives.
void* oracle_table_build(const int32_t* coords, int64_t n, int ndim, int K, const int32_t* dims, int* status) {
  Problem* P = new Problem;
  const int st = setup(*P, coords, n, ndim, K, dims);
  if (status) *status = st;
  if (st) {
    delete P;
    return nullptr;
  }
  return P;
}

int oracle_table_subm_conv(const void* table, const double* feats, const double* W, int c_in, int c_out, int relu,
                           const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  if (!table) return OR_BAD_ARG;
  const Problem& P = *static_cast<const Problem*>(table);
  if (c_in < 1 || c_out < 1 || !W || (P.n > 0 && !feats) || !out) return OR_BAD_ARG;
  if (!rows) nrows = P.n;
  return conv_rows(P, feats, W, c_in, c_out, relu, rows, nrows, out, nthreads);
}

void oracle_table_free(void* table) { delete static_cast<Problem*>(table); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Regular (stride 1: dilating) and strided sparse convolution.
//
// Output grid: extents ceil(dims / s) along the strided axes (x, y, and z in
// 3D; in 2D z is carried unchanged, like the offsets).  Output o is active iff
// some offset d puts an active input at s * o + d; the layer is
// out[o] = sum over those d of f[input at s * o + d] W_d.  At s = 1 the output
// set is the input set dilated by the kernel window.
// ---------------------------------------------------------------------------

namespace {

int out_extent(int dim, int s) { return (dim + s - 1) / s; }

// The input row at coordinate (b, x, y, z), or -1 (outside the grid: absent).
int32_t input_at(const Problem& P, int64_t b, int64_t x, int64_t y, int64_t z) {
  if (x < 0 || x >= P.dims[0] || y < 0 || y >= P.dims[1] || z < 0 || z >= P.dims[2]) return -1;
  auto it = P.table.find(pack_key(b, x, y, z));
  return it == P.table.end() ? -1 : it->second;
}

// The input row that output coordinate c_o reads through offset d.
int32_t strided_neighbour(const Problem& P, const int32_t* c_o, int stride, const int d[3]) {
  const int64_t sz = P.ndim == 3 ? stride : 1;
  return input_at(P, c_o[0], int64_t(c_o[1]) * stride + d[0], int64_t(c_o[2]) * stride + d[1],
                  int64_t(c_o[3]) * sz + d[2]);
}

int check_out_coords(const Problem& P, const int32_t* out_coords, int64_t n_out, int stride) {
  if (n_out < 0 || (n_out > 0 && !out_coords)) return OR_BAD_ARG;
  for (int64_t q = 0; q < n_out; ++q) {
    const int32_t* c = out_coords + 4 * q;
    if (c[1] < 0 || c[1] >= out_extent(P.dims[0], stride) || c[2] < 0 || c[2] >= out_extent(P.dims[1], stride))
      return OR_OUT_OF_RANGE;
    const int zext = P.ndim == 3 ? out_extent(P.dims[2], stride) : P.dims[2];
    if (c[3] < 0 || c[3] >= zext || c[0] < 0) return OR_OUT_OF_RANGE;
  }
  return OR_OK;
}

}  // namespace

extern "C" {

// Output set of a regular / strided layer, sorted by (batch, x, y, z):
// every o with an active input at s * o + d for some offset d.  Writes up to
// `cap` rows of out_coords and the count to *n_out (OR_BAD_ARG if cap is too
// small; *n_out still holds the count).
int oracle_conv_out_coords(const int32_t* coords, int64_t n, int ndim, int K, int stride, const int32_t* dims,
                           int32_t* out_coords, int64_t cap, int64_t* n_out) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (stride < 1 || !n_out) return OR_BAD_ARG;
  const int V = P.volume;
  const int64_t sz = ndim == 3 ? stride : 1;
  const int ext[3] = {out_extent(dims[0], stride), out_extent(dims[1], stride),
                      ndim == 3 ? out_extent(dims[2], stride) : dims[2]};
  std::vector<uint64_t> keys;
  {
    std::unordered_map<uint64_t, int> seen;
    for (int64_t i = 0; i < n; ++i) {
      const int32_t* c = coords + 4 * i;
      for (int v = 0; v < V; ++v) {
        int d[3];
        offset_of(v, ndim, K, d);
        // o with s * o + d = c_i, where it is a whole grid point inside the output grid
        const int64_t px = int64_t(c[1]) - d[0], py = int64_t(c[2]) - d[1], pz = int64_t(c[3]) - d[2];
        if (px % stride || py % stride || pz % sz) continue;
        const int64_t o[3] = {px / stride, py / stride, pz / sz};
        if (o[0] < 0 || o[0] >= ext[0] || o[1] < 0 || o[1] >= ext[1] || o[2] < 0 || o[2] >= ext[2]) continue;
        const uint64_t key = pack_key(c[0], o[0], o[1], o[2]);
        if (seen.emplace(key, 1).second) keys.push_back(key);
      }
    }
  }
  std::sort(keys.begin(), keys.end());
  *n_out = int64_t(keys.size());
  if (int64_t(keys.size()) > cap || (cap > 0 && !out_coords)) return OR_BAD_ARG;
  for (size_t q = 0; q < keys.size(); ++q) {
    out_coords[4 * q + 0] = int32_t(keys[q] >> 48);
    out_coords[4 * q + 1] = int32_t((keys[q] >> 32) & 0xFFFF);
    out_coords[4 * q + 2] = int32_t((keys[q] >> 16) & 0xFFFF);
    out_coords[4 * q + 3] = int32_t(keys[q] & 0xFFFF);
  }
  return OR_OK;
}

// Neighbour table of a regular / strided layer: nbr[q * V + idx(d)] = row of
// the input at s * c_q + d (c_q = out_coords row q), or -1.
int oracle_conv_kmap(const int32_t* coords, int64_t n, const int32_t* out_coords, int64_t n_out, int ndim, int K,
                     int stride, const int32_t* dims, int32_t* nbr, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (stride < 1 || (n_out > 0 && !nbr)) return OR_BAD_ARG;
  st = check_out_coords(P, out_coords, n_out, stride);
  if (st) return st;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t q = 0; q < n_out; ++q)
    for (int v = 0; v < V; ++v) nbr[q * V + v] = strided_neighbour(P, out_coords + 4 * q, stride, &offs[3 * v]);
  return OR_OK;
}

// Output features of a regular / strided layer for every output row:
// out[q, :] = sum over offsets d with an input p at s * c_q + d of f[p, :] W_d,
// fp64, then max(., 0) if relu != 0.  feats [n, c_in], W [V, c_in, c_out],
// out [n_out, c_out].
int oracle_conv(const int32_t* coords, int64_t n, const int32_t* out_coords, int64_t n_out, int ndim, int K,
                int stride, const int32_t* dims, const double* feats, const double* W, int c_in, int c_out, int relu,
                double* out, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (stride < 1 || c_in < 1 || c_out < 1 || !W || (n > 0 && !feats) || (n_out > 0 && !out)) return OR_BAD_ARG;
  st = check_out_coords(P, out_coords, n_out, stride);
  if (st) return st;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(dynamic, 64) num_threads(nt)
  for (int64_t q = 0; q < n_out; ++q) {
    double* acc = out + q * c_out;
    for (int co = 0; co < c_out; ++co) acc[co] = 0.0;
    for (int v = 0; v < V; ++v) {
      const int32_t p = strided_neighbour(P, out_coords + 4 * q, stride, &offs[3 * v]);
      if (p < 0) continue;
      const double* f = feats + int64_t(p) * c_in;
      const double* w = W + int64_t(v) * c_in * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double a = f[ci];
        const double* wrow = w + int64_t(ci) * c_out;
        for (int co = 0; co < c_out; ++co) acc[co] += a * wrow[co];
      }
    }
    if (relu)
      for (int co = 0; co < c_out; ++co) acc[co] = acc[co] > 0.0 ? acc[co] : 0.0;
  }
  return OR_OK;
}

// Weight gradient of a regular / strided layer: d loss / d W_d = sum over the
// output rows q with an input p at s * c_q + d of f[p]^T gout[q].
// feats [n, c_in], gout [n_out, c_out], dW [V, c_in, c_out], fp64.
int oracle_conv_bwd_weight(const int32_t* coords, int64_t n, const int32_t* out_coords, int64_t n_out, int ndim,
                           int K, int stride, const int32_t* dims, const double* feats, const double* gout, int c_in,
                           int c_out, double* dW, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (stride < 1 || c_in < 1 || c_out < 1 || !dW || (n > 0 && !feats) || (n_out > 0 && !gout)) return OR_BAD_ARG;
  st = check_out_coords(P, out_coords, n_out, stride);
  if (st) return st;
  const int V = P.volume;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int v = 0; v < V; ++v) {
    double* acc = dW + int64_t(v) * c_in * c_out;
    for (int64_t e = 0; e < int64_t(c_in) * c_out; ++e) acc[e] = 0.0;
    for (int64_t q = 0; q < n_out; ++q) {
      const int32_t p = strided_neighbour(P, out_coords + 4 * q, stride, &offs[3 * v]);
      if (p < 0) continue;
      const double* f = feats + int64_t(p) * c_in;
      const double* g = gout + q * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double a = f[ci];
        double* row = acc + int64_t(ci) * c_out;
        for (int co = 0; co < c_out; ++co) row[co] += a * g[co];
      }
    }
  }
  return OR_OK;
}

}  // extern "C"

namespace {

// The output row at coordinate (b, x, y, z) of an output set, or -1.
int32_t output_at(const std::unordered_map<uint64_t, int32_t>& out_table, int64_t b, int64_t x, int64_t y, int64_t z) {
  if (x < 0 || y < 0 || z < 0) return -1;
  auto it = out_table.find(pack_key(b, x, y, z));
  return it == out_table.end() ? -1 : it->second;
}

}  // namespace

extern "C" {

// Input gradient of a regular / strided layer (linear in f): d loss / d f[p]
// = sum over the offsets d and outputs q with stride * c_q + d = c_p of
// gout[q] W_d^T.  For each input p and offset d the output is the one at
// (c_p - d) / stride, where that is a whole grid point of the output set.
// gout [n_out, c_out], W [V, c_in, c_out], gin [n, c_in], fp64.
int oracle_conv_bwd_data(const int32_t* coords, int64_t n, const int32_t* out_coords, int64_t n_out, int ndim, int K,
                         int stride, const int32_t* dims, const double* gout, const double* W, int c_in, int c_out,
                         double* gin, int nthreads) {
  Problem P;
  int st = setup(P, coords, n, ndim, K, dims);
  if (st) return st;
  if (stride < 1 || c_in < 1 || c_out < 1 || !W || (n > 0 && !gin) || (n_out > 0 && !gout)) return OR_BAD_ARG;
  st = check_out_coords(P, out_coords, n_out, stride);
  if (st) return st;
  std::unordered_map<uint64_t, int32_t> out_table;
  out_table.reserve(size_t(n_out) * 2 + 1);
  for (int64_t q = 0; q < n_out; ++q) {
    const int32_t* c = out_coords + 4 * q;
    if (!out_table.emplace(pack_key(c[0], c[1], c[2], c[3]), int32_t(q)).second) return OR_DUPLICATE;
  }
  const int V = P.volume;
  const int64_t sz = ndim == 3 ? stride : 1;
  std::vector<int> offs(size_t(V) * 3);
  for (int v = 0; v < V; ++v) offset_of(v, ndim, K, &offs[3 * v]);
  const int nt = threads_to_use(nthreads);
#pragma omp parallel for schedule(dynamic, 64) num_threads(nt)
  for (int64_t p = 0; p < n; ++p) {
    const int32_t* c = coords + 4 * p;
    double* acc = gin + p * c_in;
    for (int ci = 0; ci < c_in; ++ci) acc[ci] = 0.0;
    for (int v = 0; v < V; ++v) {
      const int* d = &offs[3 * v];
      const int64_t px = int64_t(c[1]) - d[0], py = int64_t(c[2]) - d[1], pz = int64_t(c[3]) - d[2];
      if (px % stride || py % stride || pz % sz) continue;
      const int32_t q = output_at(out_table, c[0], px / stride, py / stride, pz / sz);
      if (q < 0) continue;
      const double* g = gout + int64_t(q) * c_out;
      const double* w = W + int64_t(v) * c_in * c_out;
      for (int ci = 0; ci < c_in; ++ci) {
        const double* wrow = w + int64_t(ci) * c_out;
        double sum = 0.0;
        for (int co = 0; co < c_out; ++co) sum += wrow[co] * g[co];
        acc[ci] += sum;
      }
    }
  }
  return OR_OK;
}

}  // extern "C"
