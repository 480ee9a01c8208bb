// C ABI of libsc (declared in include/sc.h): argument checks, handle
// ownership, stream-ordered allocation, variant choice, launch bookkeeping.
// Every step of the layer runs in this library's kernels; there is no host
// or CPU path for any of them.

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <unordered_map>
#include <string>
#include <vector>

#include "sc_internal.cuh"

// The opaque handle types of sc.h.
struct sc_hash_s {
  sc::HashTable t;
  void* arena = nullptr;   // one device allocation: table, keys, status (an output set: table, status)
  void* arena2 = nullptr;  // an output set's keys (sized once its count is known), or null
};
struct sc_kmap_s {
  sc::KernelMap k;
  void* arena = nullptr;  // one device allocation holding every buffer of k
  // the build call's allocator (if one was given) and stream, for the
  // buffers made later (the exported forms behind sc_kmap_view)
  bool has_alloc = false;
  sc_allocator alloc{};
  cudaStream_t stream = nullptr;
  // sc_kmap_view: rows in input order (k.nbr itself without the locality
  // order) and the compacted lists, materialised on first use
  bool view_ready = false;
  void* view_arena = nullptr;
  const int32_t* view_nbr = nullptr;
  const int32_t* view_in = nullptr;
  const int32_t* view_out = nullptr;
};

namespace sc {

// --------------------------------------------------------------- errors --
namespace {
thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};
}  // namespace

sc_status set_error(sc_status s, const char* msg) {
  g_last_error = msg ? msg : "";
  return s;
}

sc_status set_cuda_error(cudaError_t e, const char* where) {
  std::string m = where ? where : "";
  m += ": ";
  m += cudaGetErrorString(e);
  g_last_error = m;
  return e == cudaErrorMemoryAllocation ? SC_ERR_OOM : SC_ERR_CUDA;
}

// ---------------------------------------------------------- bookkeeping --
namespace {
struct Pending {
  int id;
  cudaEvent_t a, b;
};
struct Profiler {
  std::mutex mu;
  bool on = false;
  std::string only;  // bracket only kernels whose name starts with this ("" = all)
  std::vector<std::string> names;
  std::vector<int64_t> launches;
  std::vector<double> ms;
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
Profiler& prof() {
  static Profiler* p = new Profiler();  // never destroyed: safe at process exit
  return *p;
}
}  // namespace

int prof_begin(const char* name, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  Profiler& P = prof();
  if (!P.on) return -1;
  std::lock_guard<std::mutex> lk(P.mu);
  if (!P.only.empty() && std::strncmp(name, P.only.c_str(), P.only.size()) != 0) return -1;
  int id = -1;
  for (size_t i = 0; i < P.names.size(); ++i)
    if (P.names[i] == name) id = static_cast<int>(i);
  if (id < 0) {
    P.names.emplace_back(name);
    P.launches.push_back(0);
    P.ms.push_back(0.0);
    id = static_cast<int>(P.names.size() - 1);
  }
  Pending pd{id, P.take(), nullptr};
  cudaEventRecord(pd.a, s);
  P.pending.push_back(pd);
  return static_cast<int>(P.pending.size() - 1);
}

void prof_end(int token, cudaStream_t s) {
  if (token < 0) return;
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  if (token >= static_cast<int>(P.pending.size())) return;
  P.pending[token].b = P.take();
  cudaEventRecord(P.pending[token].b, s);
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cache[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = v > 0 ? v : 1;
  }
  return cache[dev];
}

sc_status kernel_setup(const void* kern, size_t smem, int* num_regs) {
  struct Entry {
    size_t smem = 0;
    int regs = 0;
  };
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, Entry> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find({dev, kern});
  if (it == cache.end()) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return set_cuda_error(e, "kernel attribute query");
    // the kernels live in shared memory: the largest carveout (occupancy
    // planning assumes it)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return set_cuda_error(e, "kernel carveout attribute");
    Entry en;
    en.regs = fa.numRegs;
    it = cache.emplace(std::make_pair(dev, kern), en).first;
  }
  if (smem > it->second.smem) {
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return set_cuda_error(e, "kernel shared-memory attribute");
    }
    it->second.smem = smem;
  }
  if (num_regs) *num_regs = it->second.regs;
  return SC_OK;
}

sc_status kernel_carveout(const void* kern, int ctas_per_sm, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> last;
  static int max_smem[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  int per_sm = dev >= 0 && dev < 64 ? max_smem[dev] : 0;
  if (!per_sm) {
    e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess || per_sm <= 0) return set_cuda_error(e, "shared memory per SM query");
    if (dev >= 0 && dev < 64) max_smem[dev] = per_sm;
  }
  // the CTAs' dynamic shared memory plus the 1 KB the system reserves per CTA
  const double need = static_cast<double>(ctas_per_sm) * static_cast<double>(smem + 1024);
  int pct = static_cast<int>((need * 100.0 + per_sm - 1) / per_sm);
  if (pct > 100) pct = 100;
  if (pct < 1) pct = 1;
  auto it = last.find({dev, kern});
  if (it != last.end() && it->second == pct) return SC_OK;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, pct);
  if (e != cudaSuccess) return set_cuda_error(e, "kernel carveout attribute");
  last[{dev, kern}] = pct;
  return SC_OK;
}

// The device's default stream-ordered pool keeps freed blocks for reuse
// (release threshold = unlimited) instead of trimming them at every
// synchronisation; set once per device on first use.
void keep_pool_memory() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || done[dev]) return;
  cudaMemPool_t pool;
  if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
  }
  done[dev] = true;
}

namespace {
// The caller's allocator (sc_set_allocator), if any, and the allocator that
// made each live buffer it handed out, so a buffer goes back to its own
// allocator whatever is set when it is freed.
struct Allocator {
  sc_alloc_fn alloc = nullptr;
  sc_free_fn free = nullptr;
  void* ctx = nullptr;
};
std::mutex g_alloc_mu;
Allocator g_alloc;
std::unordered_map<void*, Allocator> g_alloc_owner;
}  // namespace

sc_status dev_alloc(void** p, size_t bytes, cudaStream_t s, const sc_allocator* with) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  Allocator a;
  if (with && with->alloc) {
    a.alloc = with->alloc;
    a.free = with->free;
    a.ctx = with->ctx;
  } else {
    std::lock_guard<std::mutex> lk(g_alloc_mu);
    a = g_alloc;
  }
  if (a.alloc) {
    void* q = a.alloc(bytes, reinterpret_cast<sc_stream>(s), a.ctx);
    if (!q) return set_error(SC_ERR_OOM, "the caller's allocator returned NULL");
    if (reinterpret_cast<uintptr_t>(q) % 256) {
      a.free(q, reinterpret_cast<sc_stream>(s), a.ctx);
      return set_error(SC_ERR_INVALID_ARG, "the caller's allocator returned memory that is not 256-byte aligned");
    }
    std::lock_guard<std::mutex> lk(g_alloc_mu);
    g_alloc_owner[q] = a;
    *p = q;
    return SC_OK;
  }
  keep_pool_memory();
  cudaError_t e = cudaMallocAsync(p, bytes, s);
  if (e != cudaSuccess) {
    *p = nullptr;
    return set_cuda_error(e, "cudaMallocAsync");
  }
  return SC_OK;
}

void dev_free(void* p, cudaStream_t s) {
  if (!p) return;
  Allocator a;
  bool caller = false;
  {
    std::lock_guard<std::mutex> lk(g_alloc_mu);
    auto it = g_alloc_owner.find(p);
    if (it != g_alloc_owner.end()) {
      a = it->second;
      g_alloc_owner.erase(it);
      caller = true;
    }
  }
  if (caller) a.free(p, reinterpret_cast<sc_stream>(s), a.ctx);
  else cudaFreeAsync(p, s);
}

namespace {

// A device (or managed) pointer with the given alignment; host memory is
// refused: the library has no host path.
sc_status check_dev_ptr(const void* p, size_t align, const char* what) {
  if (!p) return set_error(SC_ERR_INVALID_ARG, (std::string(what) + " is NULL").c_str());
  if (reinterpret_cast<uintptr_t>(p) % align)
    return set_error(SC_ERR_INVALID_ARG, (std::string(what) + " is not 16-byte aligned").c_str());
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(SC_ERR_INVALID_ARG, (std::string(what) + " is not a CUDA pointer").c_str());
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return set_error(SC_ERR_INVALID_ARG, (std::string(what) + " is not device memory").c_str());
  return SC_OK;
}

sc_status status_from_bits(int bits) {
  if (bits & kDevErrDup) return set_error(SC_ERR_DUPLICATE_COORD, "duplicate coordinate");
  if (bits & kDevErrRange) return set_error(SC_ERR_OUT_OF_RANGE, "coordinate out of range");
  if (bits & kDevErrFull) return set_error(SC_ERR_TABLE_FULL, "hash table full");
  if (bits & kDevErrTimeout) return set_error(SC_ERR_TIMEOUT, "device-side wait timed out");
  return SC_OK;
}

// Reads the map's status words, segment offsets and weight-stationary tile
// prefix into host mirrors; synchronises the stream.
sc_status sync_host(KernelMap* m, cudaStream_t s) {
  int bits[2] = {0, 0};
  m->offs_host.assign(m->V + 1, 0);
  m->ws_tiles_host.assign(m->V + 1, 0);
  int64_t ms = 0;
  cudaError_t e = cudaMemcpyAsync(bits, m->status, 2 * sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(m->offs_host.data(), m->offs, sizeof(int64_t) * (m->V + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(m->ws_tiles_host.data(), m->ws_tiles, sizeof(int) * (m->V + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&ms, m->map_size, sizeof(int64_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_cuda_error(e, "kmap synchronise");
  m->map_size_host = ms;
  m->host_valid = true;
  return status_from_bits(bits[0] | bits[1]);
}

bool valid_dtype(int d) { return d == SC_F32 || d == SC_F16 || d == SC_BF16; }
size_t dtype_bytes(sc_dtype d) { return d == SC_F32 ? 4 : 2; }

sc_status check_conv_args(sc_kmap m, const void* feats, const void* W, const void* out, int c_in, int c_out,
                          sc_dtype dtype) {
  if (!m) return set_error(SC_ERR_INVALID_ARG, "kmap handle is NULL");
  if (!valid_dtype(dtype)) return set_error(SC_ERR_INVALID_ARG, "unknown dtype");
  if (c_in < 16 || c_out < 16 || c_in > 256 || c_out > 256 || c_in % 16 || c_out % 16)
    return set_error(SC_ERR_UNSUPPORTED, "c_in and c_out must be multiples of 16 in [16, 256]");
  sc_status st = check_dev_ptr(W, 16, "W");
  if (st) return st;
  if (m->k.n == 0) return SC_OK;
  if ((st = check_dev_ptr(feats, 16, "feats"))) return st;
  if ((st = check_dev_ptr(out, 16, "out"))) return st;
  const size_t eb = dtype_bytes(dtype);
  const uintptr_t f0 = reinterpret_cast<uintptr_t>(feats), f1 = f0 + m->k.n_in * c_in * eb;
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + m->k.n * c_out * eb;
  if (f0 < o1 && o0 < f1) return set_error(SC_ERR_INVALID_ARG, "out overlaps feats");
  return SC_OK;
}

unsigned default_variant(KernelMap* m, const ConvArgs& a) {
  if (a.dtype == SC_F32) return SC_VARIANT_SIMT;
  if (!m->identity) return fused_supported(a) ? SC_VARIANT_FUSED : SC_VARIANT_SIMT;
  for (const ConvChoice& c : m->tuned)
    if (c.c_in == a.c_in && c.c_out == a.c_out && c.dtype == a.dtype) return c.variant;
  return fused_supported(a) ? SC_VARIANT_FUSED : SC_VARIANT_WS;
}

sc_status run_variant(KernelMap* m, const ConvArgs& a, unsigned variant) {
  if (a.dtype == SC_F32 && variant != SC_VARIANT_SIMT)
    return set_error(SC_ERR_UNSUPPORTED, "fp32 layers run on the CUDA-core kernel only");
  switch (variant) {
    case SC_VARIANT_FUSED:
      return conv_fused(a);
    case SC_VARIANT_WS:
      if (!m->identity)
        return set_error(SC_ERR_UNSUPPORTED, "the weight-stationary kernel needs a submanifold map");
      if (!m->host_valid) {
        sc_status st = sync_host(m, a.stream);
        if (st) return st;
      }
      return conv_weight_stationary(a);
    case SC_VARIANT_SIMT:
      return conv_simt(a);
    case SC_VARIANT_SPLIT:
      return conv_fused_split(a);
  }
  return set_error(SC_ERR_INVALID_ARG, "more than one variant flag");
}

}  // namespace
}  // namespace sc

using namespace sc;

extern "C" {

const char* sc_status_str(sc_status s) {
  switch (s) {
    case SC_OK: return "ok";
    case SC_ERR_INVALID_ARG: return "invalid argument";
    case SC_ERR_OUT_OF_RANGE: return "coordinate out of range";
    case SC_ERR_DUPLICATE_COORD: return "duplicate coordinate";
    case SC_ERR_TABLE_FULL: return "hash table full";
    case SC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SC_ERR_CUDA: return "CUDA error";
    case SC_ERR_OOM: return "out of device memory";
    case SC_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

sc_status sc_set_allocator(sc_alloc_fn alloc, sc_free_fn free_fn, void* ctx) {
  if ((alloc == nullptr) != (free_fn == nullptr))
    return set_error(SC_ERR_INVALID_ARG, "set both alloc and free, or neither");
  std::lock_guard<std::mutex> lk(g_alloc_mu);
  g_alloc.alloc = alloc;
  g_alloc.free = free_fn;
  g_alloc.ctx = ctx;
  return SC_OK;
}

const char* sc_last_error(void) { return g_last_error.c_str(); }

int64_t sc_launch_count(void) { return g_launches.load(); }

void sc_profile_enable(int on) { prof().on = on != 0; }

void sc_profile_only(const char* name_prefix) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  P.only = name_prefix ? name_prefix : "";
}

sc_status sc_profile_collect(void) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  for (Pending& pd : P.pending) {
    if (pd.b) {
      cudaError_t e = cudaEventSynchronize(pd.b);
      if (e != cudaSuccess) return set_cuda_error(e, "profile event");
      float ms = 0.f;
      cudaEventElapsedTime(&ms, pd.a, pd.b);
      P.ms[pd.id] += ms;
      P.launches[pd.id] += 1;
      P.pool.push_back(pd.b);
    }
    P.pool.push_back(pd.a);
  }
  P.pending.clear();
  return SC_OK;
}

void sc_profile_reset(void) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  for (size_t i = 0; i < P.ms.size(); ++i) {
    P.ms[i] = 0.0;
    P.launches[i] = 0;
  }
}

sc_status sc_profile_get(int index, const char** name, int64_t* launches, double* total_ms) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  if (index < 0 || index >= static_cast<int>(P.names.size())) return SC_ERR_INVALID_ARG;
  if (name) *name = P.names[index].c_str();
  if (launches) *launches = P.launches[index];
  if (total_ms) *total_ms = P.ms[index];
  return SC_OK;
}

// ------------------------------------------------------------------ hash --
sc_status sc_hash_build(const int32_t* d_coords, int64_t n, const sc_allocator* alloc, sc_stream stream, sc_hash* out) {
  if (!out) return set_error(SC_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n < 0 || n >= (int64_t(1) << 31)) return set_error(SC_ERR_INVALID_ARG, "n must be in [0, 2^31)");
  if (alloc && (alloc->alloc == nullptr) != (alloc->free == nullptr))
    return set_error(SC_ERR_INVALID_ARG, "an sc_allocator needs both alloc and free, or neither");
  if (n > 0) {
    sc_status st = check_dev_ptr(d_coords, 16, "coords");
    if (st) return st;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  sc_hash h = new sc_hash_s();
  HashTable& t = h->t;
  t.n = n;
  // one entry per occupied 2x2x2 block, at most n of them: 2n entries while
  // the table stays within 256 MB, n beyond that (surface data fills a block
  // with several points, so the load stays well below 1/2 either way;
  // measured: a table of 1.25 n entries made the map build's lookups 9 %
  // slower at 100k voxels)
  int64_t cap = 16;
  const int64_t want = 2 * n * static_cast<int64_t>(sizeof(BlockEntry)) <= (int64_t(256) << 20) ? 2 * n : n;
  while (cap < want) cap <<= 1;
  // developer override for testing the full-table path: SC_DEV_HASH_CAPACITY
  // entries (rounded up to a power of two, at least 16)
  if (const char* ev = getenv("SC_DEV_HASH_CAPACITY")) {
    const long long c = atoll(ev);
    if (c > 0) {
      cap = 16;
      while (cap < c) cap <<= 1;
    }
  }
  t.capacity = cap;
  const size_t tb = sizeof(BlockEntry) * static_cast<size_t>(cap);
  const size_t kb = (sizeof(unsigned long long) * static_cast<size_t>(n > 0 ? n : 1) + 255) & ~size_t(255);
  sc_status st = dev_alloc(&h->arena, tb + kb + 256, s, alloc);
  if (!st) {
    uint8_t* b = static_cast<uint8_t*>(h->arena);
    t.table = reinterpret_cast<BlockEntry*>(b);
    t.keys = reinterpret_cast<unsigned long long*>(b + tb);
    t.status = reinterpret_cast<int*>(b + tb + kb);
  }
  if (!st) st = launch_hash_insert(d_coords, n, &t, s);
  if (st) {
    sc_hash_destroy(h, stream);
    return st;
  }
  *out = h;
  return SC_OK;
}

sc_status sc_hash_query(sc_hash h, const int32_t* d_query, int64_t m, int32_t* d_rows, sc_stream stream) {
  if (!h || m < 0) return set_error(SC_ERR_INVALID_ARG, "bad hash handle or size");
  if (m == 0) return SC_OK;
  sc_status st = check_dev_ptr(d_query, 16, "query");
  if (!st) st = check_dev_ptr(d_rows, 4, "rows");
  if (st) return st;
  return launch_hash_query(&h->t, d_query, m, d_rows, reinterpret_cast<cudaStream_t>(stream));
}

sc_status sc_hash_info(sc_hash h, int64_t* n, int64_t* capacity) {
  if (!h) return set_error(SC_ERR_INVALID_ARG, "hash handle is NULL");
  if (n) *n = h->t.n;
  if (capacity) *capacity = h->t.capacity;
  return SC_OK;
}

sc_status sc_hash_check(sc_hash h, sc_stream stream) {
  if (!h) return set_error(SC_ERR_INVALID_ARG, "hash handle is NULL");
  int bits = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&bits, h->t.status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_cuda_error(e, "hash check");
  return status_from_bits(bits);
}

sc_status sc_hash_destroy(sc_hash h, sc_stream stream) {
  if (!h) return SC_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dev_free(h->arena, s);
  dev_free(h->arena2, s);
  delete h;
  return SC_OK;
}

sc_status sc_hash_build_conv_out(sc_hash in, int ndim, int K, int stride, const int32_t dims[3],
                                 const sc_allocator* alloc, sc_stream stream, sc_hash* out) {
  if (!out) return set_error(SC_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!in) return set_error(SC_ERR_INVALID_ARG, "hash handle is NULL");
  if (ndim != 2 && ndim != 3) return set_error(SC_ERR_INVALID_ARG, "ndim must be 2 or 3");
  if (K < 1 || K % 2 == 0 || K > 7) return set_error(SC_ERR_INVALID_ARG, "K must be odd and in [1, 7]");
  if (stride < 1 || stride > 64) return set_error(SC_ERR_INVALID_ARG, "stride must be in [1, 64]");
  if (!dims) return set_error(SC_ERR_INVALID_ARG, "dims is NULL");
  for (int a = 0; a < 3; ++a)
    if (dims[a] < 1 || dims[a] > 65535) return set_error(SC_ERR_INVALID_ARG, "dims must be in [1, 65535]");
  if (alloc && (alloc->alloc == nullptr) != (alloc->free == nullptr))
    return set_error(SC_ERR_INVALID_ARG, "an sc_allocator needs both alloc and free, or neither");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the inputs must be valid points inside dims before their outputs are derived
  sc_status st = sc_hash_check(in, stream);
  if (st) return st;
  sc_hash h = new sc_hash_s();
  st = launch_conv_out(&in->t, ndim, K, stride, dims, &h->t, &h->arena, &h->arena2, alloc, s);
  if (st) {
    sc_hash_destroy(h, stream);
    return st;
  }
  *out = h;
  return SC_OK;
}

sc_status sc_hash_coords(sc_hash h, int32_t* d_coords, sc_stream stream) {
  if (!h) return set_error(SC_ERR_INVALID_ARG, "hash handle is NULL");
  if (h->t.n == 0) return SC_OK;
  sc_status st = check_dev_ptr(d_coords, 16, "coords");
  if (st) return st;
  return launch_hash_coords(&h->t, d_coords, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------- map --
sc_status sc_kmap_destroy(sc_kmap m, sc_stream stream) {
  if (!m) return SC_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dev_free(m->view_arena, s);
  dev_free(m->arena, s);
  delete m;
  return SC_OK;
}

// Inputs at least this large get a locality order by default.
constexpr int64_t kOrderMinPoints = 262144;
// ... and a signature sort of the convolution's rows (V <= 128).
constexpr int64_t kSortMinPoints = 262144;

namespace {

// The map of the points of `ho` against the table of `hi`: a submanifold map
// when ho == hi and stride == 1 (the centre list is the identity), else the
// map of a regular / strided layer.
sc_status kmap_build_impl(sc_hash hi, sc_hash ho, int ndim, int K, int stride, const int32_t dims[3],
                          unsigned flags, const sc_allocator* alloc, sc_stream stream, sc_kmap* out) {
  if (!out) return set_error(SC_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!hi || !ho) return set_error(SC_ERR_INVALID_ARG, "hash handle is NULL");
  if (stride < 1 || stride > 64) return set_error(SC_ERR_INVALID_ARG, "stride must be in [1, 64]");
  const bool identity = hi == ho && stride == 1;
  const bool transposed = (flags & SC_KMAP_TRANSPOSE) != 0;
  if (transposed && identity) return set_error(SC_ERR_INVALID_ARG, "SC_KMAP_TRANSPOSE is for regular / strided maps");
  // rows: the queries (outputs; a transposed map's are the inputs); table: the other set
  sc_hash h = transposed ? hi : ho;
  sc_hash ht = transposed ? ho : hi;
  if (ndim != 2 && ndim != 3) return set_error(SC_ERR_INVALID_ARG, "ndim must be 2 or 3");
  if (K < 1 || K % 2 == 0) return set_error(SC_ERR_INVALID_ARG, "K must be odd and >= 1");
  int V = 1;
  for (int a = 0; a < ndim; ++a) {
    V *= K;
    if (V > 343) return set_error(SC_ERR_UNSUPPORTED, "K^ndim must be <= 343");
  }
  if (!dims) return set_error(SC_ERR_INVALID_ARG, "dims is NULL");
  for (int a = 0; a < 3; ++a)
    if (dims[a] < 1 || dims[a] > 65535) return set_error(SC_ERR_INVALID_ARG, "dims must be in [1, 65535]");
  if (flags & ~(SC_KMAP_NO_SYNC | SC_KMAP_ORDER | SC_KMAP_NO_ORDER | SC_KMAP_SORT | SC_KMAP_NO_SORT | SC_KMAP_TRANSPOSE |
                SC_KMAP_HALF | SC_KMAP_SPLIT | SC_KMAP_TILE_TABLE))
    return set_error(SC_ERR_INVALID_ARG, "unknown kmap flag");
  if ((flags & SC_KMAP_TILE_TABLE) && (V > 128 || (flags & SC_KMAP_SPLIT)))
    return set_error(SC_ERR_UNSUPPORTED, "SC_KMAP_TILE_TABLE: K^ndim <= 128, and not with SC_KMAP_SPLIT");
  if ((flags & SC_KMAP_HALF) && !identity)
    return set_error(SC_ERR_UNSUPPORTED, "SC_KMAP_HALF builds submanifold maps only");
  if ((flags & SC_KMAP_ORDER) && (flags & SC_KMAP_NO_ORDER))
    return set_error(SC_ERR_INVALID_ARG, "SC_KMAP_ORDER and SC_KMAP_NO_ORDER together");
  if ((flags & SC_KMAP_SORT) && (flags & SC_KMAP_NO_SORT))
    return set_error(SC_ERR_INVALID_ARG, "SC_KMAP_SORT and SC_KMAP_NO_SORT together");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((flags & SC_KMAP_SPLIT) && (!identity || V > 32))
    return set_error(SC_ERR_UNSUPPORTED, "SC_KMAP_SPLIT: submanifold maps with K^ndim <= 32 only");
  if ((flags & SC_KMAP_SPLIT) && (flags & SC_KMAP_NO_SORT))
    return set_error(SC_ERR_INVALID_ARG, "SC_KMAP_SPLIT needs the signature sort (not SC_KMAP_NO_SORT)");
  sc_kmap m = new sc_kmap_s();
  KernelMap& k = m->k;
  k.n = h->t.n;
  k.n_in = ht->t.n;
  k.stride = stride;
  k.identity = identity;
  k.transposed = transposed;
  k.ndim = ndim;
  k.K = K;
  k.V = V;
  for (int a = 0; a < 3; ++a) k.dims[a] = dims[a];
  k.half = (flags & SC_KMAP_HALF) != 0;
  if ((flags & SC_KMAP_SPLIT) && k.n > 0) {
    k.nparts = 2;
    k.split_at = (V - 1) / 2 + 1;  // part 0: offsets up to and including the centre
  }
  k.up = kmap_unit_points(V);
  k.nunits = static_cast<int>((k.n + k.up - 1) / k.up);
  const bool ordered = (flags & SC_KMAP_ORDER) || (!(flags & SC_KMAP_NO_ORDER) && k.n >= kOrderMinPoints);
  // the signature sort keeps a mask of up to 128 offsets per row (V <= 128)
  // column splitting (SC_KMAP_SPLIT): submanifold maps with V <= 32; it
  // brings the signature sort with it
  const bool split = (flags & SC_KMAP_SPLIT) != 0;
  // by default at kSortMinPoints rows and more; for a regular / strided map
  // only when V > 32 (measured at 2M voxels 5x5x5, stride 2: the step 5.60 ->
  // 4.51 ms; at 1M voxels 3x3x3 the layer gained 40 us and the step lost)
  const bool sort_default = k.n >= kSortMinPoints && (identity || V > 32);
  const bool sorted = V <= 128 && k.n > 0 &&
                      (split || (flags & SC_KMAP_SORT) || (!(flags & SC_KMAP_NO_SORT) && sort_default));
  const size_t mask_words = V <= 32 ? 1 : 4;
  const bool tile_table = (flags & SC_KMAP_TILE_TABLE) && k.n > 0;
  const size_t tiles = static_cast<size_t>((k.n + 127) / 128);
  const size_t nsig = sorted ? static_cast<size_t>(kmap_sig_buckets(k.n)) : 0;
  // every buffer of the map carved from one allocation, each 256-byte aligned
  const size_t n = static_cast<size_t>(k.n);
  struct Part {
    void** dst;
    size_t bytes;
  } parts[] = {
      {reinterpret_cast<void**>(&k.nbr), sizeof(int) * n * V},
      {reinterpret_cast<void**>(&k.in_rows), sizeof(int) * n * V},
      {reinterpret_cast<void**>(&k.out_rows), sizeof(int) * n * V},
      {reinterpret_cast<void**>(&k.cursors), sizeof(int) * V * kCursorStride},
      {reinterpret_cast<void**>(&k.present), sizeof(unsigned) * 4 * ((n + 127) / 128)},
      {reinterpret_cast<void**>(&k.offs), sizeof(int64_t) * (V + 1)},
      {reinterpret_cast<void**>(&k.ws_tiles), sizeof(int) * (V + 1)},
      {reinterpret_cast<void**>(&k.map_size), sizeof(int64_t)},
      {reinterpret_cast<void**>(&k.status), sizeof(int) * 4},
      {reinterpret_cast<void**>(&k.order), ordered && k.n > 0 ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.skeys), ordered && k.n > 0 ? sizeof(unsigned long long) * n : 0},
      {reinterpret_cast<void**>(&k.inv_order), ordered && k.half && k.n > 0 ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.buckets), ordered && k.n > 0 ? sizeof(int) * kmap_order_buckets() : 0},
      {reinterpret_cast<void**>(&k.rowmask), sorted ? sizeof(unsigned) * n * mask_words : 0},
      {reinterpret_cast<void**>(&k.rowdir), sorted && V > 32 ? sizeof(unsigned) * n : 0},
      {reinterpret_cast<void**>(&k.sig_sel), sorted ? sizeof(int) * kmap_sig_bits() * (split ? 3 : 1) : 0},
      {reinterpret_cast<void**>(&k.part_perm[0]), sorted && split ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.part_perm[1]), sorted && split ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.part_order[0]), sorted && split ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.part_order[1]), sorted && split ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.part_present[0]), sorted && split ? sizeof(unsigned) * 4 * ((n + 127) / 128) : 0},
      {reinterpret_cast<void**>(&k.part_present[1]), sorted && split ? sizeof(unsigned) * 4 * ((n + 127) / 128) : 0},
      {reinterpret_cast<void**>(&k.sigbuckets), sorted ? sizeof(int) * (nsig + nsig / 4096 + 1) : 0},
      {reinterpret_cast<void**>(&k.perm), sorted ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.conv_order), sorted ? sizeof(int) * n : 0},
      {reinterpret_cast<void**>(&k.tnbr), tile_table ? sizeof(int) * tiles * 128 * V : 0},
  };
  size_t total = 0;
  for (const Part& pt : parts) total += (pt.bytes + 255) & ~size_t(255);
  if (alloc && (alloc->alloc == nullptr) != (alloc->free == nullptr)) {
    delete m;
    return set_error(SC_ERR_INVALID_ARG, "an sc_allocator needs both alloc and free, or neither");
  }
  m->stream = s;
  if (alloc && alloc->alloc) {
    m->has_alloc = true;
    m->alloc = *alloc;
  }
  sc_status st = dev_alloc(&m->arena, total, s, m->has_alloc ? &m->alloc : nullptr);
  if (!st) {
    uint8_t* base = static_cast<uint8_t*>(m->arena);
    for (const Part& pt : parts) {
      *pt.dst = pt.bytes ? base : nullptr;
      base += (pt.bytes + 255) & ~size_t(255);
    }
  }
  // status[1] carries the hash's latched insert status from here on
  if (!st) {
    cudaError_t e = cudaMemsetAsync(k.status, 0, sizeof(int) * 4, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(k.status + 1, hi->t.status, sizeof(int), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) st = set_cuda_error(e, "kmap status init");
  }
  if (!st) st = launch_kmap_build(&ht->t, &h->t, &k, s);
  if (!st && !(flags & SC_KMAP_NO_SYNC)) st = sync_host(&k, s);
  if (st) {
    sc_kmap_destroy(m, stream);
    return st;
  }
  *out = m;
  return SC_OK;
}

}  // namespace

sc_status sc_kmap_build(sc_hash h, int ndim, int K, const int32_t dims[3], unsigned flags, const sc_allocator* alloc,
                        sc_stream stream, sc_kmap* out) {
  return kmap_build_impl(h, h, ndim, K, 1, dims, flags, alloc, stream, out);
}

sc_status sc_kmap_build_conv(sc_hash in, sc_hash out_set, int ndim, int K, int stride, const int32_t dims[3],
                             unsigned flags, const sc_allocator* alloc, sc_stream stream, sc_kmap* out) {
  return kmap_build_impl(in, out_set, ndim, K, stride, dims, flags, alloc, stream, out);
}

sc_status sc_kmap_info(sc_kmap m, int64_t* n, int32_t* volume, int64_t* map_size, sc_stream stream) {
  if (!m) return set_error(SC_ERR_INVALID_ARG, "kmap handle is NULL");
  if (n) *n = m->k.n;
  if (volume) *volume = m->k.V;
  if (map_size) {
    if (!m->k.host_valid) {
      sc_status st = sync_host(&m->k, reinterpret_cast<cudaStream_t>(stream));
      if (st) return st;
    }
    *map_size = m->k.map_size_host;
  }
  return SC_OK;
}

sc_status sc_kmap_check(sc_kmap m, sc_stream stream) {
  if (!m) return set_error(SC_ERR_INVALID_ARG, "kmap handle is NULL");
  // the status words only (the map's and the hash's copy): one small read
  int bits[2] = {0, 0};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(bits, m->k.status, 2 * sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_cuda_error(e, "kmap check");
  return status_from_bits(bits[0] | bits[1]);
}

sc_status sc_kmap_export(sc_kmap m, int32_t* nbr, int64_t* offs, int32_t* in_rows, int32_t* out_rows,
                         sc_stream stream) {
  if (!m) return set_error(SC_ERR_INVALID_ARG, "kmap handle is NULL");
  KernelMap& k = m->k;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((in_rows || out_rows) && !k.host_valid) {
    sc_status st = sync_host(&k, s);
    if (st) return st;
  }
  cudaError_t e = cudaSuccess;
  if (nbr && k.n) {
    if (!k.order) {
      e = cudaMemcpyAsync(nbr, k.nbr, sizeof(int) * k.n * k.V, cudaMemcpyDefault, s);
    } else {  // the table is stored in the locality order: put rows back in input order
      int* tmp = nullptr;
      sc_status st = dev_alloc(reinterpret_cast<void**>(&tmp), sizeof(int) * k.n * k.V, s);
      if (!st) st = kmap_unpermute_nbr(&k, tmp, s);
      if (!st) e = cudaMemcpyAsync(nbr, tmp, sizeof(int) * k.n * k.V, cudaMemcpyDefault, s);
      dev_free(tmp, s);
      if (st) return st;
    }
  }
  if (e == cudaSuccess && offs) e = cudaMemcpyAsync(offs, k.offs, sizeof(int64_t) * (k.V + 1), cudaMemcpyDefault, s);
  const int64_t L = k.host_valid ? k.offs_host[k.V] : 0;
  if (e != cudaSuccess) return set_cuda_error(e, "kmap export");
  // the lists are stored in strides of n per offset: compact them into CSR
  for (int which = 0; which < 2 && L; ++which) {
    int32_t* dst = which == 0 ? in_rows : out_rows;
    if (!dst) continue;
    int* tmp = nullptr;
    sc_status st = dev_alloc(reinterpret_cast<void**>(&tmp), sizeof(int) * L, s);
    if (!st) st = kmap_compact_lists(&k, which == 0 ? k.in_rows : k.out_rows, tmp, L, s);
    if (!st) {
      e = cudaMemcpyAsync(dst, tmp, sizeof(int) * L, cudaMemcpyDefault, s);
      if (e != cudaSuccess) st = set_cuda_error(e, "kmap export");
    }
    dev_free(tmp, s);
    if (st) return st;
  }
  return SC_OK;
}

sc_status sc_kmap_view(sc_kmap m, const int32_t** d_nbr, const int64_t** d_offs, const int32_t** d_in,
                       const int32_t** d_out, int64_t* map_size) {
  if (!m) return set_error(SC_ERR_INVALID_ARG, "kmap handle is NULL");
  KernelMap& k = m->k;
  cudaStream_t s = m->stream;
  if (!m->view_ready) {
    // the latched status and the segment offsets on the host
    sc_status st = k.host_valid ? sc_kmap_check(m, reinterpret_cast<sc_stream>(s)) : sync_host(&k, s);
    if (st) return st;
    const int64_t L = k.offs_host[k.V];
    const size_t nb = k.order ? sizeof(int) * static_cast<size_t>(k.n) * k.V : 0;
    const size_t nb_al = (nb + 255) & ~size_t(255);
    const size_t lb = (sizeof(int) * static_cast<size_t>(L) + 255) & ~size_t(255);
    if (nb + 2 * lb > 0) {
      st = dev_alloc(&m->view_arena, nb_al + 2 * lb, s, m->has_alloc ? &m->alloc : nullptr);
      if (st) return st;
    }
    uint8_t* base = static_cast<uint8_t*>(m->view_arena);
    int* vn = k.order ? reinterpret_cast<int*>(base) : k.nbr;
    int* vi = L ? reinterpret_cast<int*>(base + nb_al) : nullptr;
    int* vo = L ? reinterpret_cast<int*>(base + nb_al + lb) : nullptr;
    if (k.order && k.n) st = kmap_unpermute_nbr(&k, vn, s);
    if (!st && L) st = kmap_compact_lists(&k, k.in_rows, vi, L, s);
    if (!st && L) st = kmap_compact_lists(&k, k.out_rows, vo, L, s);
    if (!st) {
      cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) st = set_cuda_error(e, "kmap view");
    }
    if (st) {
      dev_free(m->view_arena, s);
      m->view_arena = nullptr;
      return st;
    }
    m->view_nbr = vn;
    m->view_in = vi;
    m->view_out = vo;
    m->view_ready = true;
  }
  if (d_nbr) *d_nbr = m->view_nbr;
  if (d_offs) *d_offs = k.offs;
  if (d_in) *d_in = m->view_in;
  if (d_out) *d_out = m->view_out;
  if (map_size) *map_size = k.map_size_host;
  return SC_OK;
}

// ----------------------------------------------------------- convolution --
sc_status sc_subm_conv_fwd(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in, int c_out,
                           sc_dtype dtype, unsigned flags, sc_stream stream) {
  sc_status st = check_conv_args(m, d_feats, d_W, d_out, c_in, c_out, dtype);
  if (st) return st;
  if (flags & ~(SC_RELU | SC_VARIANT_MASK)) return set_error(SC_ERR_INVALID_ARG, "unknown conv flag");
  ConvArgs a{&m->k, d_feats, d_W, d_out, c_in, c_out, dtype, (flags & SC_RELU) != 0,
             reinterpret_cast<cudaStream_t>(stream)};
  unsigned variant = flags & SC_VARIANT_MASK;
  if (!variant) variant = default_variant(&m->k, a);
  return run_variant(&m->k, a, variant);
}

sc_status sc_subm_conv_bwd_data(sc_kmap m, const void* d_gout, const void* d_W, void* d_gin, int c_in, int c_out,
                                sc_dtype dtype, unsigned flags, sc_stream stream) {
  if (m && !m->k.identity && !m->k.transposed)
    return set_error(SC_ERR_UNSUPPORTED,
                     "input gradient of a regular or strided layer: pass its transposed map (SC_KMAP_TRANSPOSE)");
  // the input gradient is a submanifold layer with c_out -> c_in channels
  sc_status st = check_conv_args(m, d_gout, d_W, d_gin, c_out, c_in, dtype);
  if (st) return st;
  if (flags & ~SC_VARIANT_MASK) return set_error(SC_ERR_INVALID_ARG, "bwd_data takes an SC_VARIANT_* flag only");
  ConvArgs a{&m->k, d_gout, d_W, d_gin, c_out, c_in, dtype, false, reinterpret_cast<cudaStream_t>(stream)};
  a.wt = true;
  unsigned variant = flags & SC_VARIANT_MASK;
  if (!variant) variant = default_variant(&m->k, a);
  return run_variant(&m->k, a, variant);
}

sc_status sc_subm_conv_bwd_weight(sc_kmap m, const void* d_feats, const void* d_gout, void* d_dW, int c_in,
                                  int c_out, sc_dtype dtype, unsigned flags, sc_stream stream) {
  sc_status st = check_conv_args(m, d_feats, d_dW, d_gout, c_in, c_out, dtype);
  if (st) return st;
  if (flags) return set_error(SC_ERR_INVALID_ARG, "bwd_weight takes no flags");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!m->k.host_valid) {
    st = sync_host(&m->k, s);
    if (st) return st;
  }
  return conv_bwd_weight(&m->k, d_feats, d_gout, d_dW, c_in, c_out, dtype, s);
}

sc_status sc_subm_conv_fwd_noalloc(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in,
                                   int c_out, sc_dtype dtype, unsigned flags, sc_stream stream) {
  sc_status st = check_conv_args(m, d_feats, d_W, d_out, c_in, c_out, dtype);
  if (st) return st;
  if (flags & ~SC_RELU) return set_error(SC_ERR_INVALID_ARG, "the no-allocation conv takes SC_RELU only");
  ConvArgs a{&m->k, d_feats, d_W, d_out, c_in, c_out, dtype, (flags & SC_RELU) != 0,
             reinterpret_cast<cudaStream_t>(stream)};
  return conv_fused_noalloc(a);
}

sc_status sc_subm_conv_tune(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in, int c_out,
                            sc_dtype dtype, unsigned flags, int reps, sc_stream stream, unsigned* chosen) {
  sc_status st = check_conv_args(m, d_feats, d_W, d_out, c_in, c_out, dtype);
  if (st) return st;
  if (flags & ~SC_RELU) return set_error(SC_ERR_INVALID_ARG, "tune takes SC_RELU only");
  if (reps < 1) reps = 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ConvArgs a{&m->k, d_feats, d_W, d_out, c_in, c_out, dtype, (flags & SC_RELU) != 0, s};
  std::vector<unsigned> cands;
  if (dtype == SC_F32) {
    cands.push_back(SC_VARIANT_SIMT);
  } else {
    if (fused_supported(a)) cands.push_back(SC_VARIANT_FUSED);
    if (fused_supported(a) && m->k.nparts == 2) cands.push_back(SC_VARIANT_SPLIT);
    if (m->k.identity) cands.push_back(SC_VARIANT_WS);
    if (cands.empty()) return set_error(SC_ERR_UNSUPPORTED, "no tensor-core variant for this layer");
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  unsigned best = cands[0];
  float best_ms = 1e30f;
  for (unsigned v : cands) {
    st = run_variant(&m->k, a, v);  // warm-up
    if (st) break;
    cudaEventRecord(e0, s);
    for (int r = 0; r < reps && !st; ++r) st = run_variant(&m->k, a, v);
    cudaEventRecord(e1, s);
    if (st) break;
    cudaError_t e = cudaEventSynchronize(e1);
    if (e != cudaSuccess) {
      st = set_cuda_error(e, "tune timing");
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (ms < best_ms) {
      best_ms = ms;
      best = v;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st) return st;
  bool found = false;
  for (ConvChoice& c : m->k.tuned)
    if (c.c_in == c_in && c.c_out == c_out && c.dtype == dtype) {
      c.variant = best;
      found = true;
    }
  if (!found) m->k.tuned.push_back({c_in, c_out, static_cast<int>(dtype), best});
  if (chosen) *chosen = best;
  // leave d_out holding the chosen variant's result
  return run_variant(&m->k, a, best);
}

}  // extern "C"
