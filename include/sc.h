/*
 * sc.h -- C ABI of libsc: submanifold sparse convolution on one GPU
 * (sm_103a).  Plain pointers and sizes only; no C++ or framework types.
 *
 * The layer (after "Sparse inputs and sparse convolution", sections "The fix"
 * and "The map is the computation", and the exam sheet "Sparse convolution
 * for point clouds", sections "Submanifold sparse convolution" and "The map
 * and the update rule"):
 *
 *   points   coords[i] = (batch, x, y, z), features feats[i, 0:C_in]
 *   offsets  d in [-r, r]^ndim, r = (K-1)/2, K odd, stride 1
 *   map      M = {(p, q, d) : coords[p] = coords[q] + d}       (P = Q + d)
 *   layer    out[q, :] = sum_{(p, q, d) in M} feats[p, :] @ W[d]
 *
 * The output point set equals the input point set (P_out = P_in): out has the
 * same N rows, in the same order, as feats.
 *
 * Offset index: lexicographic over (dx, dy[, dz]) with the first axis
 * slowest, idx = sum_k (d_k + r) * K^(ndim-1-k); the centre offset is
 * (V-1)/2 and the mirror of idx is V-1-idx, V = K^ndim.  In 2D (ndim = 2)
 * offsets move x and y only; z is carried unchanged as part of the key.
 *
 * Pointers.  Arguments named d_* are device pointers (cudaMalloc'd or
 * equivalent); the library never dereferences them on the host.  Arguments of
 * sc_kmap_export may be device or host pointers (UVA).  All calls are
 * asynchronous on the given stream unless stated.  Errors in the arguments
 * are returned synchronously; no call aborts, throws or traps.
 *
 * Memory.  Handles own their device buffers, allocated on the stream passed
 * at build time from the allocator passed to the build call (NULL: the
 * process-wide one, see sc_set_allocator; by default CUDA's stream-ordered
 * pool) and released stream-ordered on the stream passed to *_destroy, each
 * buffer to the allocator that made it.  The caller owns coords, feats, W and
 * out.
 */
#ifndef SC_H_
#define SC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* sc_stream;

typedef enum {
  SC_OK = 0,
  SC_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment, K, ndim, dims */
  SC_ERR_OUT_OF_RANGE = 2,    /* a coordinate outside [0, dims) or batch outside [0, 65535) */
  SC_ERR_DUPLICATE_COORD = 3, /* two rows share one (batch, x, y, z) */
  SC_ERR_TABLE_FULL = 4,      /* hash insert gave up after probing every slot */
  SC_ERR_UNSUPPORTED = 5,     /* channel counts or dtype the kernels do not cover */
  SC_ERR_CUDA = 6,            /* a CUDA runtime call failed; see sc_last_error() */
  SC_ERR_OOM = 7,             /* device allocation failed */
  SC_ERR_TIMEOUT = 8          /* a bounded device-side wait gave up (kernel bug) */
} sc_status;

typedef enum { SC_F32 = 0, SC_F16 = 1, SC_BF16 = 2 } sc_dtype;

/* flags for sc_subm_conv_fwd / sc_subm_conv_tune */
#define SC_RELU 0x1u            /* max(out, 0) before the cast to the output dtype */
#define SC_VARIANT_FUSED 0x10u  /* force the output-stationary tcgen05 kernel */
#define SC_VARIANT_WS 0x20u     /* force the weight-stationary gather/GEMM/scatter kernels */
#define SC_VARIANT_SIMT 0x40u   /* force the CUDA-core kernel (the only one for SC_F32) */
#define SC_VARIANT_SPLIT 0x80u  /* force the fused kernel with column splitting (a map built with SC_KMAP_SPLIT) */
#define SC_VARIANT_MASK 0xF0u

/* flags for sc_kmap_build */
#define SC_KMAP_NO_SYNC 0x100u  /* do not synchronise; check errors later with sc_kmap_check */
#define SC_KMAP_ORDER 0x200u    /* always compute the locality order (default: n >= 262144) */
#define SC_KMAP_NO_ORDER 0x400u /* never compute it: tiles follow the input row order */
#define SC_KMAP_SORT 0x800u     /* always sort the convolution's rows by signature (default: n >= 262144, V <= 128) */
#define SC_KMAP_NO_SORT 0x1000u /* never sort them */
#define SC_KMAP_TRANSPOSE 0x2000u /* sc_kmap_build_conv: the transposed map (rows = the layer's inputs) */
#define SC_KMAP_HALF 0x4000u    /* sc_kmap_build: half probe by mirror symmetry (same map, another build) */
#define SC_KMAP_SPLIT 0x8000u   /* sc_kmap_build, K^ndim <= 32: row orders for column splitting (see below) */
#define SC_KMAP_TILE_TABLE 0x10000u /* K^ndim <= 128: also the fused layer's tile-transposed index table (see below) */

typedef struct sc_hash_s* sc_hash;
typedef struct sc_kmap_s* sc_kmap;

/*
 * A caller's device-memory allocator (see "Device memory" below).
 * alloc(bytes, stream, ctx) returns device memory of at least `bytes`,
 * 256-byte aligned, usable in stream order on `stream`, or NULL (the call
 * then fails with SC_ERR_OOM); free(ptr, stream, ctx) releases it after the
 * work queued on `stream`.  The callbacks run on the calling host thread and
 * must not call back into the library.
 */
typedef void* (*sc_alloc_fn)(size_t bytes, sc_stream stream, void* ctx);
typedef void (*sc_free_fn)(void* ptr, sc_stream stream, void* ctx);
typedef struct {
  sc_alloc_fn alloc;
  sc_free_fn free;
  void* ctx;
} sc_allocator;

/* ---------------------------------------------------------------- hash -- */

/*
 * Coordinate hash table: key (batch, x, y, z) -> row id i.
 * After "SparseConvNet: from hash table to rulebook", section 2 (each unique
 * input coordinate gets an incremental index) and "Sparse inputs and sparse
 * convolution", section "Gather, matmul, scatter" (the map is built on the
 * GPU, not copied from a CPU hash).
 *
 * d_coords  int32 [n, 4] row-major (batch, x, y, z), 16-byte aligned.
 *           batch in [0, 65535), x, y, z in [0, 65535).
 * n         number of points, 0 <= n < 2^31.
 * alloc     the allocator of the handle's buffers, or NULL (the process-wide
 *           one).  The struct is copied; its callbacks and ctx must stay
 *           valid until the handle is destroyed.
 * out       receives the handle.
 *
 * Keys are packed into 64 bits (16 bits per field, batch highest).  The
 * table is open addressing with linear probing over entries of one 2x2x2
 * block of voxels each: the block's key (the voxel key with the low bit of x,
 * y, z cleared) and the rows of its 8 voxels.  Capacity = next power of two
 * >= 2n entries (>= n when that would exceed 256 MB).  Asynchronous: a
 * duplicate or out-of-range coordinate is latched in the handle and reported
 * by sc_hash_check, sc_kmap_build or sc_kmap_check.
 */
sc_status sc_hash_build(const int32_t* d_coords, int64_t n, const sc_allocator* alloc, sc_stream stream,
                        sc_hash* out);

/* Row id of each query coordinate, -1 where it is not in the table.
 * d_query int32 [m, 4] (16-byte aligned), d_rows int32 [m]. Asynchronous. */
sc_status sc_hash_query(sc_hash h, const int32_t* d_query, int64_t m, int32_t* d_rows, sc_stream stream);

/* Number of points and table capacity in block entries (host values, no
 * synchronisation). */
sc_status sc_hash_info(sc_hash h, int64_t* n, int64_t* capacity);

/* Synchronises the stream and returns the latched insert status. */
sc_status sc_hash_check(sc_hash h, sc_stream stream);

/* Releases the handle's buffers stream-ordered on `stream`. */
sc_status sc_hash_destroy(sc_hash h, sc_stream stream);

/*
 * Output set of a regular (stride 1) or strided sparse convolution layer, as
 * a new hash handle over the output points.  "SparseConvNet: from hash table
 * to rulebook", section 2, gives the regular output definition: an output is
 * computed wherever the kernel window covers at least one active input, so
 * the active set grows (at stride 1, by the window: "Sparse inputs and sparse
 * convolution", section "What a dense convolution does to empty space");
 * section 3 relates input, output and offset under a stride.  Here output o
 * reads the input at stride * o + d, d in [-(K-1)/2, (K-1)/2]^ndim, and o is
 * an output iff one of those inputs is active.
 *
 * in       the input points' hash.
 * ndim     2 or 3; in 2D the offsets and the stride act on (x, y) and z is
 *          carried unchanged.
 * K        odd, in [1, 7].
 * stride   in [1, 64].
 * dims     the input grid's extents (x, y, z); the outputs lie on the grid
 *          of extents ceil(dims / stride) on the strided axes.
 * out      receives the output set: n = its point count (sc_hash_info),
 *          row ids 0 .. n - 1 in an unspecified order (their coordinates:
 *          sc_hash_coords).  It serves as the input hash of the next layer
 *          and as the output set of sc_kmap_build_conv.  The caller destroys
 *          it with sc_hash_destroy.
 *
 * Synchronises the stream (twice: the input hash's status, then the output
 * count).  Errors: the input hash's latched errors; SC_ERR_TABLE_FULL if the
 * output table would exceed 2^28 entries.  Device memory is allocated
 * stream-ordered on `stream` and owned by the handle.
 */
sc_status sc_hash_build_conv_out(sc_hash in, int ndim, int K, int stride, const int32_t dims[3],
                                 const sc_allocator* alloc, sc_stream stream, sc_hash* out);

/* Coordinates of every row of the hash: d_coords int32 [n, 4] = (batch, x,
 * y, z), device memory, 16-byte aligned, written asynchronously. */
sc_status sc_hash_coords(sc_hash h, int32_t* d_coords, sc_stream stream);

/* ---------------------------------------------------------- kernel map -- */

/*
 * Kernel map (rulebook) for a K^ndim submanifold convolution.
 * After "Sparse inputs and sparse convolution", section "The map is the
 * computation" (for each output q and offset d, look up q + d in the hash);
 * "TorchSparse optimizations", opening section (the centre offset maps every
 * point to itself at stride 1 and is not searched); "SparseConvNet: from hash
 * table to rulebook", section 3 (the rulebook is grouped by weight offset).
 *
 * ndim      2 or 3.
 * K         odd, K >= 1, with V = K^ndim <= 343 (K <= 7 in 3D, K <= 17 in 2D).
 * dims      spatial extents (x, y, z), each in [1, 65535]; every point must
 *           lie inside; neighbours outside are absent (zero padding).
 * flags     0, SC_KMAP_NO_SYNC, at most one of SC_KMAP_ORDER /
 *           SC_KMAP_NO_ORDER, at most one of SC_KMAP_SORT /
 *           SC_KMAP_NO_SORT, SC_KMAP_HALF (build by the half probe: the
 *           offsets after the centre are looked up and each hit is mirrored
 *           by symmetry, "Sparse inputs and sparse convolution", section "A
 *           symmetry you can check"; the same map), SC_KMAP_SPLIT (below),
 *           SC_KMAP_TILE_TABLE (below).
 *
 * Locality order: for n >= 262144 (or with SC_KMAP_ORDER) the build first
 * sorts the points into spatially compact groups (a counting sort on the top
 * 20 bits of a Morton code of (batch, x, y, z)); the convolution's 128-row
 * tiles are runs of that order, so they touch fewer offsets and reuse
 * neighbour rows.  It changes no result: outputs still land on their own
 * rows and nbr stays in input row order.
 *
 * Signature sort (V <= 128; for n >= 262144 or with SC_KMAP_SORT): inside
 * windows of 524288 consecutive rows of that order, the convolution's rows
 * are counting-sorted by a 20-bit signature, which of the 20 least frequent
 * features (over the whole map) the row has a neighbour under.  The
 * features are the offsets when V <= 32, else the 26 coarse directions
 * (sign(dx), sign(dy), sign(dz)), a feature's frequency being the tuple
 * count of its offsets.  Rows that touch the same rare features then share
 * 128-row tiles, and a tile walks fewer offsets (the bitmask reordering of
 * "TorchSparse optimizations", section "TorchSparse++").  It too changes no
 * result.
 *
 * Column splitting (SC_KMAP_SPLIT, V <= 32; implies the signature sort): the
 * offset range is cut at the centre into part 0 (offsets up to and including
 * the centre) and part 1 (the rest), and each part gets a row order of its
 * own, sorted by the signature of its own offsets, with tile masks of its
 * offsets only ("TorchSparse optimizations", section "TorchSparse++": the
 * column split that lets each part's tiles walk fewer offsets).  The layer
 * then uses them when run with SC_VARIANT_SPLIT (or when sc_subm_conv_tune
 * measured that variant fastest): two launches, the first storing fp32
 * partial sums, the second adding its own to them and rounding once.  The map
 * itself is unchanged.
 *
 * Tile table (SC_KMAP_TILE_TABLE, V <= 128, not with SC_KMAP_SPLIT): the
 * build also writes the fused layer's neighbour indices in that layer's row
 * order, transposed within each 128-row tile ([ceil(n/128)][V][128] int32,
 * 4 n V more bytes held by the handle), so that a tile's indices for one
 * offset are one contiguous 512-byte run.  Every fused layer (and input
 * gradient) on the map then reads them there instead of nbr.  Results are
 * unchanged.  It costs one pass over nbr after the build and pays when the
 * map serves several layers: on a batch of four 120k-point LiDAR scans
 * (3x3x3) eight layers 32 -> 256 took 2.37 ms instead of 2.65 ms for a 34 us
 * pass, while a single layer does not recover it (1M voxels 3x3x3: the layer
 * 25 us faster, the pass 60 us; 2M voxels 5x5x5: 100 us and 388 us).
 *
 * Products, owned by the handle:
 *   nbr      int32 [n, V]: nbr[q*V + idx(d)] = row p with coords[p] =
 *            coords[q] + d, or -1.  Column (V-1)/2 is the identity.
 *   offs     int64 [V+1]: per-offset segments of the (in, out) lists.  The
 *            centre segment is empty: its tuples are (i, i) for every i.
 *   in/out   int32 [offs[V]]: list entries (p, q).  The order of the
 *            entries inside a segment is not part of the result and may
 *            differ between builds (runs of up to 128 consecutive rows stay
 *            together, in row order).
 *   map size |M| = n + offs[V] tuples, centre included.
 *
 * Without SC_KMAP_NO_SYNC the call synchronises the stream once and returns
 * the hash's latched errors and its own (SC_ERR_OUT_OF_RANGE when a point
 * lies outside dims).  With it the call is fully asynchronous and errors
 * surface in sc_kmap_check.
 */
sc_status sc_kmap_build(sc_hash h, int ndim, int K, const int32_t dims[3], unsigned flags,
                        const sc_allocator* alloc, sc_stream stream, sc_kmap* out);

/*
 * Kernel map of a regular / strided layer: the rows are the points of
 * `out_set` (from sc_hash_build_conv_out with the same ndim, K, stride and
 * dims), and nbr[q*V + idx(d)] is the row p of `in` with coords[p] = stride *
 * coords[q] + d, or -1 (absent neighbours and the grid's edges: zero
 * padding).  The tuples (p, q, d) follow "SparseConvNet: from hash table to
 * rulebook", section 3 (rulebook grouped by offset).  Unlike a submanifold
 * map the centre offset is searched like the others and has its own list
 * segment; |M| = offs[V].  The map keeps neither hash: both stay owned by
 * the caller.  Flags as for sc_kmap_build (SC_KMAP_TILE_TABLE included)
 * except SC_KMAP_HALF and SC_KMAP_SPLIT (SC_ERR_UNSUPPORTED: submanifold maps
 * only); the locality
 * order and the signature sort apply to the map's rows (the outputs, or the
 * inputs of a transposed map) as for a submanifold map, except that the sort
 * is on by default only when V > 32 as well.
 *
 * sc_subm_conv_fwd and sc_subm_conv_bwd_weight take such a map: feats then
 * has the input's n_in rows and out / gout the map's n rows.  The
 * weight-stationary variant returns SC_ERR_UNSUPPORTED for it.
 *
 * With SC_KMAP_TRANSPOSE the map is transposed: its rows are the points of
 * `in` (the layer's inputs) and nbr[p*V + idx(-d)] is the row q of `out_set`
 * with stride * coords[q] + d = coords[p], or -1 (the outputs whose windows
 * contain p, at the mirrored offset).  sc_subm_conv_bwd_data takes the
 * transposed map of a layer, with d_gout [n_out, c_out] and d_gin [n, c_in]:
 * gin[p] = sum over those (q, d) of gout[q] @ W[idx(d)]^T, the layer's input
 * gradient, on the same kernels as the submanifold one.  A forward map
 * returns SC_ERR_UNSUPPORTED there.
 */
sc_status sc_kmap_build_conv(sc_hash in, sc_hash out_set, int ndim, int K, int stride, const int32_t dims[3],
                             unsigned flags, const sc_allocator* alloc, sc_stream stream, sc_kmap* out);

/* n, V and |M| (centre included).  Synchronises the stream when |M| is not
 * yet known on the host. */
sc_status sc_kmap_info(sc_kmap m, int64_t* n, int32_t* volume, int64_t* map_size, sc_stream stream);

/* Synchronises the stream and returns the latched hash and map status (it
 * reads the two status words only). */
sc_status sc_kmap_check(sc_kmap m, sc_stream stream);

/*
 * Copies the products into caller buffers (device or host pointers; any may
 * be NULL to skip): nbr int32 [n*V], offs int64 [V+1], in_rows and out_rows
 * int32 [offs[V]].  Asynchronous for device destinations.
 */
sc_status sc_kmap_export(sc_kmap m, int32_t* nbr, int64_t* offs, int32_t* in_rows, int32_t* out_rows,
                         sc_stream stream);

/*
 * Borrowed device pointers to the products (the rulebook grouped by weight
 * offset, "SparseConvNet: from hash table to rulebook", section 3; the map as
 * the computation, "Sparse inputs and sparse convolution", section "The map
 * is the computation"), in the layout sc_kmap_export writes:
 *   *d_nbr   int32 [n, V], rows in input row order (nbr[q*V + idx(d)]);
 *   *d_offs  int64 [V+1], the segments of the lists;
 *   *d_in, *d_out  int32 [offs[V]], the list entries (p, q) by segment;
 *   *map_size      |M| (host value).
 * Any output may be NULL to skip it.  The pointers stay valid, and their
 * contents unchanged, until the handle is destroyed; the caller must not
 * write through them.  The first call materialises the forms the handle does
 * not keep internally (rows back in input order when the locality order is
 * on; the lists compacted from their fixed per-offset strides) into buffers
 * the handle owns, from the handle's allocator, on the stream the map was
 * built on, and synchronises that stream (which must still exist); later
 * calls return the same pointers without device work.  Errors: the map's
 * latched status (as sc_kmap_check), SC_ERR_OOM, SC_ERR_CUDA.
 */
sc_status sc_kmap_view(sc_kmap m, const int32_t** d_nbr, const int64_t** d_offs, const int32_t** d_in,
                       const int32_t** d_out, int64_t* map_size);

/* Releases the handle's buffers stream-ordered on `stream`. */
sc_status sc_kmap_destroy(sc_kmap m, sc_stream stream);

/* ---------------------------------------------------------- convolution -- */

/*
 * One submanifold convolution layer on a built map:
 *   out[q, :] = act( sum_{(p, q, d) in M} feats[p, :] @ W[d] )
 * with fp32 accumulation and one rounding to the output dtype; act is
 * max(., 0) with SC_RELU, else the identity.  Update rule after the exam
 * sheet "Sparse convolution for point clouds", section "The map and the
 * update rule", and "Sparse inputs and sparse convolution", section "The map
 * is the computation".
 *
 * d_feats  [n, c_in] row-major, dtype; 16-byte aligned.
 * d_W      [V, c_in, c_out] row-major, dtype (W[idx(d)] is the c_in x c_out
 *          matrix of offset d); 16-byte aligned.
 * d_out    [n, c_out] row-major, dtype; 16-byte aligned; must not alias
 *          d_feats.  Every row is written exactly once.
 * c_in, c_out  multiples of 16 in [16, 256].
 * dtype    SC_F16 / SC_BF16 (tensor-core kernels) or SC_F32 (CUDA cores).
 * flags    SC_RELU, optionally one SC_VARIANT_* to force a kernel family.
 *
 * The fused kernel covers V <= 128; larger kernels use the weight-stationary
 * one.  SC_VARIANT_SPLIT (a map built with SC_KMAP_SPLIT) runs the fused
 * kernel with column splitting and an fp32 partial-sum buffer [n, c_out]
 * allocated for the call.  Variant: forced by flags, else the one sc_subm_conv_tune measured fastest
 * for (c_in, c_out, dtype) on this map, else the fused output-stationary
 * kernel (f16/bf16) or the CUDA-core kernel (f32).  The fused kernel reads
 * each weight slice by TMA straight from d_W (which must then be 16-byte
 * aligned; otherwise, and for output widths that fit no TMA box such as 48
 * or 80 channels, it repacks W into a temporary first) and allocates
 * nothing.  Temporary device memory of the other variants (packed weights,
 * the fp32 accumulator of the weight-stationary variant) is allocated and
 * freed stream-ordered on `stream`.
 */
sc_status sc_subm_conv_fwd(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in,
                           int c_out, sc_dtype dtype, unsigned flags, sc_stream stream);

/*
 * Times every variant that supports (c_in, c_out, dtype) on this map with
 * CUDA events (`reps` runs each after one warm-up; synchronises), caches the
 * fastest in the handle for sc_subm_conv_fwd, and stores its SC_VARIANT_*
 * flag in *chosen.  d_out receives the last variant's result.
 */
sc_status sc_subm_conv_tune(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in,
                            int c_out, sc_dtype dtype, unsigned flags, int reps, sc_stream stream,
                            unsigned* chosen);

/*
 * Backward pass of a layer computed by sc_subm_conv_fwd without SC_RELU (for
 * a ReLU layer, mask d_gout by the forward output first).  The layer is
 * linear in feats and in W, so both gradients come from the same map:
 *
 * sc_subm_conv_bwd_data: d_gin[p, :] = sum over the tuples (p, q, d) of
 *   d_gout[q, :] @ W[d]^T.  The tuple (p, q, d) of the forward map is the
 *   tuple (q, p, -d) of the same map (mirror symmetry), so this is a
 *   submanifold layer from c_out to c_in channels with weights
 *   W'[idx(d)] = W[idx(-d)]^T, and it runs on the forward kernels: the fused
 *   kernel reads each slice W[idx(-d)]^T by TMA straight from d_W (16-byte
 *   aligned, c_in at most 256), with no temporary; otherwise,
 *   and in the weight-stationary variant, the weight packing transposes and
 *   mirrors W into a temporary.
 *   d_gout [n, c_out], d_W [V, c_in, c_out] (the forward layer's weights),
 *   d_gin [n, c_in]; c_in and c_out are the forward layer's.  flags: 0 or one
 *   SC_VARIANT_*.
 *
 * sc_subm_conv_bwd_weight: d_dW[d] = sum over the tuples (p, q, d) of
 *   d_feats[p, :]^T d_gout[q, :], accumulated in fp32 from the map's
 *   per-offset lists (the identity for the centre) and rounded once to dtype.
 *   d_feats [n, c_in], d_gout [n, c_out], d_dW [V, c_in, c_out].  flags: 0.
 *   Synchronises once if the map's host counts are not yet known.
 *
 * The source pages show the forward layer only; these follow from it by
 * differentiation.  Argument rules as for sc_subm_conv_fwd.
 */
sc_status sc_subm_conv_bwd_data(sc_kmap m, const void* d_gout, const void* d_W, void* d_gin, int c_in, int c_out,
                                sc_dtype dtype, unsigned flags, sc_stream stream);
sc_status sc_subm_conv_bwd_weight(sc_kmap m, const void* d_feats, const void* d_gout, void* d_dW, int c_in,
                                  int c_out, sc_dtype dtype, unsigned flags, sc_stream stream);

/*
 * The layer of sc_subm_conv_fwd, computed by its fused tensor-core kernel,
 * without allocating any memory.  The source pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc (or any
 * allocator) at this point, such as programs that plan all device memory up
 * front and hand kernels fixed buffers, runtimes that own every allocation
 * themselves, or latency-critical code where an allocation that may block or
 * fail is not acceptable.
 *
 * This entry point always repacks the weights into the fused kernel's
 * shared-memory layout (rather than reading W by TMA as sc_subm_conv_fwd
 * does), into one fixed 4 MiB device array inside the library, present on
 * every GPU that loads the library until the process exits.  The caller still
 * passes every input and output.
 *
 * Limits: f16/bf16 only; V <= 128; V * c_in * c_out * 2 bytes <= 4 MiB
 * (4,194,304), else SC_ERR_UNSUPPORTED with a message in sc_last_error().
 * flags: 0 or SC_RELU.  Other arguments as for sc_subm_conv_fwd.
 *
 * The first call on each device looks up the array's device address with
 * cudaGetSymbolAddress while that device is current; make that first call
 * before any stream capture.  The address is cached per device and per CUDA
 * context: a call made after the device's context was replaced (for example
 * after cudaDeviceReset) looks it up again, so it too should come before any
 * capture.  Every call reuses the one array and overwrites
 * all of the packed weights it uses, so nothing carries over between calls
 * except stale bytes that are never read.  Calls whose GPU work overlaps (on
 * different streams, or from different threads) race on the array: order
 * them on one stream or synchronise between them.
 */
sc_status sc_subm_conv_fwd_noalloc(sc_kmap m, const void* d_feats, const void* d_W, void* d_out, int c_in,
                                   int c_out, sc_dtype dtype, unsigned flags, sc_stream stream);

/* ------------------------------------------------------- device memory -- */

/*
 * Where the library's device memory comes from: the buffers a hash or map
 * handle owns and the temporaries of a call (packed weights, accumulators).
 * By default CUDA's stream-ordered pool (cudaMallocAsync / cudaFreeAsync on
 * the call's stream; the pool keeps freed blocks for reuse).  With
 * sc_set_allocator the library asks the caller's allocator instead, so an
 * application can keep all device memory in one pool (the Python binding
 * offers PyTorch's caching allocator).  A build call (sc_hash_build,
 * sc_hash_build_conv_out, sc_kmap_build, sc_kmap_build_conv) given a non-NULL
 * sc_allocator uses that one for the handle it makes, whatever the
 * process-wide setting is; the handle keeps a copy for the buffers it
 * allocates later (sc_kmap_view).  The source pages have no counterpart.
 *
 * alloc(bytes, stream, ctx) returns device memory of at least `bytes`,
 * 256-byte aligned, usable in stream order on `stream` (the stream of the
 * call that allocates), or NULL (the call then fails with SC_ERR_OOM).
 * free(ptr, stream, ctx) releases it; `stream` is the stream of the call
 * that frees (a handle's destroy, or the allocating call for temporaries),
 * after whose queued work the memory may be reused.  A buffer goes back to
 * the allocator that made it, whatever is set when it is freed.  Pass
 * NULL, NULL to return to the stream-ordered pool; both or neither must be
 * set (else SC_ERR_INVALID_ARG).  The setting is global to the process and
 * thread-safe; the callbacks run on the thread of the library call and must
 * not call back into the library.  sc_subm_conv_fwd_noalloc allocates
 * nothing either way.
 */
sc_status sc_set_allocator(sc_alloc_fn alloc, sc_free_fn free_fn, void* ctx);

/* ---------------------------------------------------------- diagnostics -- */

const char* sc_status_str(sc_status s);

/* Text of the last error raised on the calling host thread ("" if none). */
const char* sc_last_error(void);

/* Total number of kernels this library has launched in this process. */
int64_t sc_launch_count(void);

/*
 * Per-kernel device timing.  While enabled, every launch is bracketed with a
 * pair of CUDA events on its stream.  sc_profile_collect synchronises those
 * events and folds them into per-kernel totals; sc_profile_get reads entry
 * `index` (0-based; returns SC_ERR_INVALID_ARG past the end).
 */
void sc_profile_enable(int on);
/* Restrict the bracketing to kernels whose profile name starts with
 * `name_prefix` (for example "subm_conv"), so that timing one kernel adds no
 * events around the others.  NULL or "" restores all kernels.  The string is
 * copied. */
void sc_profile_only(const char* name_prefix);
sc_status sc_profile_collect(void);
void sc_profile_reset(void);
sc_status sc_profile_get(int index, const char** name, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* SC_H_ */
