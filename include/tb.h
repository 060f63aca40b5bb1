/*
 * tb.h -- batched generated-topology passes for sparse voxel grids (GB300).
 *
 * C ABI of libtb.so.  The operations are the ones fVDB issue #755
 * ("Generated-topology grid construction dominates per-iteration
 * ConvolutionPlan cost", Suggested direction) asks for and fVDB PR #757
 * ("Batched leaf-mask topology construction for generated conv grids",
 * Summary items 1-2) describes: build the refined, coarsened or box-dilated
 * topology of every member of a grid batch in one batched pass instead of one
 * member at a time.
 *
 * Data model.  A batch holds B grids.  Each grid is a set of 8^3 leaves; a
 * leaf is an int32 origin (a multiple of 8 on each axis) and a 512-bit
 * active mask stored as eight little-endian 64-bit words: voxel
 * (origin + (lx, ly, lz)) is bit 8*ly + lz of word lx.  Leaves of a grid are
 * stored in canonical node order (PR #757, Summary item 1, sort bullet): by
 * root tile floor(v/4096) compared as signed integers, then by the x-major
 * child offset inside the 4096^3 upper node (floor(v/128) mod 32), then by the
 * x-major child offset inside the 128^3 lower node (floor(v/8) mod 16); x is
 * the most significant axis at every level.  Grids follow in input order.
 *
 * Outputs of every producing call (PR #757, Summary item 1, writer bullet):
 * per-grid leaf offsets, per-leaf voxel offsets (0-based within the grid),
 * per-leaf word popcount prefix, per-leaf and per-grid bounding boxes,
 * per-grid voxel and node counts, and lower/upper node lists with parent
 * linkage.  All arrays live in device memory owned by the batch.
 *
 * Conventions shared by every call:
 *  - Streams.  All device work is enqueued on `stream` (NULL = legacy default
 *    stream) of the current CUDA device.  A producing call blocks the host
 *    once, on the readback of the per-grid counts (PR #757, Summary item 1,
 *    readback bullet); for tb_from_ijk and tb_from_leaves the pass kernel
 *    reads the input's coordinate range itself and sizes the sort key on the
 *    device.  Outputs are ready in stream order when the call returns.
 *  - Memory.  `alloc` may be NULL: memory then comes from cudaMallocAsync on
 *    the device's default memory pool.  Otherwise every device allocation
 *    (outputs and per-call scratch) goes through alloc->alloc / alloc->free,
 *    which receive `stream`; the batch keeps a copy of the allocator and frees
 *    its memory through it.  A call whose shape (source kind, grid count,
 *    source count, ops) repeats an earlier call on the same thread allocates
 *    its outputs before the count readback, with room for that call's counts
 *    plus about an eighth, and queues its writers behind the pass kernel; the
 *    batch's arrays may then be larger than its counts (the view reports the
 *    counts).  Outputs that outgrow the room are written again at their exact
 *    size within the same call.
 *  - Ownership.  Inputs are borrowed, read only, and may be freed once the
 *    call returns.  On TB_OK, *out is a new batch the caller releases with
 *    tb_batch_free.  On any error *out is set to NULL and nothing is leaked.
 *  - Errors.  Every call returns a tb_status; tb_last_error() gives a message
 *    for the calling thread's most recent failure.
 */
#ifndef TB_H_
#define TB_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define TB_API __attribute__((visibility("default")))
#else
#define TB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tb_stream; /* identical to cudaStream_t */

typedef enum {
  TB_OK = 0,
  TB_ERR_INVALID_ARG = 1,     /* bad pointer, size, factor, box or offsets          */
  TB_ERR_OOM = 2,             /* the allocator returned NULL                         */
  TB_ERR_CUDA = 3,            /* a CUDA runtime call failed                          */
  TB_ERR_COORD_OVERFLOW = 4,  /* an output coordinate would leave int32              */
  TB_ERR_NOT_CANONICAL = 5,   /* tb_validate found an order/mask/offset violation    */
  TB_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up (result invalid) */
  TB_ERR_TOO_LARGE = 7,       /* sizes beyond the library's documented limits        */
  TB_ERR_INTERNAL = 8         /* an internal bound of the library was exceeded (bug) */
} tb_status;

typedef struct tb_allocator {
  void* (*alloc)(void* ctx, size_t bytes, tb_stream stream); /* NULL on failure */
  void (*free)(void* ctx, void* ptr, tb_stream stream);
  void* ctx;
} tb_allocator;

typedef enum { TB_OP_REFINE = 0, TB_OP_COARSEN = 1, TB_OP_BOX_DILATE = 2 } tb_op_kind;

/* One pass of a chain.  REFINE / COARSEN use `factor` (2, 4 or 8); BOX_DILATE
 * uses lo[a] in [-7, 0] and hi[a] in [0, 7] per axis a (x, y, z). */
typedef struct tb_op {
  int32_t kind;
  int32_t factor;
  int32_t lo[3];
  int32_t hi[3];
} tb_op;

typedef struct tb_batch tb_batch; /* opaque; owns its device arrays */

/* Read-only view of a batch.  Device pointers are NULL when their array is
 * empty.  Shapes use B = num_grids, L = num_leaves, NL = num_lowers,
 * NU = num_uppers; all arrays are C-contiguous. */
typedef struct tb_batch_view {
  int32_t num_grids;
  int32_t device;
  int64_t num_leaves;
  int64_t num_lowers;
  int64_t num_uppers;
  const int64_t* leaf_offsets_host;  /* [B+1] host copy, owned by the batch      */
  int32_t bbox[6];                   /* whole-batch voxel bbox (min xyz, max xyz) */
  const int64_t* leaf_offsets;       /* [B+1] first leaf of each grid             */
  const int32_t* origins;            /* [L,3] leaf origins                         */
  const uint64_t* masks;             /* [L,8] active masks                         */
  const int64_t* voxel_offset;       /* [L] voxels in earlier leaves of the grid  */
  const uint64_t* word_prefix;       /* [L] 7 x 9-bit fields: field k-1 = voxels
                                        in words 0..k-1, k = 1..7                  */
  const int32_t* leaf_bbox;          /* [L,6] inclusive voxel bbox of each leaf   */
  const int32_t* leaf_grid;          /* [L] grid index of each leaf               */
  const int32_t* leaf_parent;        /* [L] index of the leaf's lower node within
                                        its grid                                   */
  const int64_t* voxel_counts;       /* [B] active voxels per grid                */
  const int32_t* grid_bbox;          /* [B,6]; empty grid: INT32_MAX x3, INT32_MIN x3 */
  const int32_t* node_counts;        /* [B,3] upper nodes (= root tiles), lower
                                        nodes, leaves                              */
  const int64_t* lower_offsets;      /* [B+1] first lower node of each grid       */
  const int64_t* upper_offsets;      /* [B+1] first upper node of each grid       */
  const int32_t* lower_origins;      /* [NL,3] lower-node origins (multiples of 128) */
  const int32_t* lower_parent;       /* [NL] index of the upper node within the grid */
  const int32_t* upper_origins;      /* [NU,3] upper-node origins (multiples of 4096) */
  /* statistics of the pass that produced the batch */
  int64_t build_slots;               /* candidate leaves emitted and sorted       */
  int64_t build_source_leaves;       /* leaves (or voxels) the pass read          */
  int32_t build_key_bits;            /* width of the compressed sort key          */
  int32_t build_digit_passes;        /* 8-bit radix passes run                    */
  int64_t num_voxels;                /* active voxels of the whole batch (host)   */
  int32_t build_member_ctas;         /* CTAs per member of the pass's member launch,
                                        0: the whole-grid kernel (tb_set_launch_mode) */
  int32_t reserved;
} tb_batch_view;

/* Per-kernel timing record (see tb_profile_enable). */
typedef struct tb_kernel_stat {
  const char* name;     /* static kernel name                                   */
  int64_t launches;
  double total_ms;      /* sum of CUDA-event durations on the launching stream  */
} tb_kernel_stat;

/* Batch from a jagged list of voxel coordinates: the ijk front end that fVDB
 * PR #757 (Follow-ups paragraph) names for BuildGridFromIjk.
 *   ijk      [num_voxels, 3] int32, host or device memory; duplicates allowed,
 *            any order.
 *   offsets  [num_grids + 1] int64, host or device memory; offsets[0] == 0,
 *            non-decreasing, offsets[num_grids] == num_voxels.  Grid g holds
 *            ijk[offsets[g] .. offsets[g+1]).  Empty grids are allowed.
 * Limits: num_grids <= 2^24, num_voxels < 2^30.  Violations of the offsets
 * contract return TB_ERR_INVALID_ARG (checked on the device). */
TB_API tb_status tb_from_ijk(const int32_t* ijk, const int64_t* offsets, int32_t num_grids,
                      int64_t num_voxels, const tb_allocator* alloc, tb_stream stream,
                      tb_batch** out);

/* Batch from a jagged list of leaves in any order.  Leaves with equal origin
 * in one grid are merged by OR-ing their masks; all-zero masks are dropped.
 *   origins  [num_leaves, 3] int32 (multiples of 8), masks [num_leaves, 8]
 *            uint64, leaf_offsets [num_grids + 1] int64; host or device memory.
 * Limits: num_grids <= 2^24, num_leaves < 2^27. */
TB_API tb_status tb_from_leaves(const int32_t* origins, const uint64_t* masks, const int64_t* leaf_offsets,
                         int32_t num_grids, int64_t num_leaves, const tb_allocator* alloc,
                         tb_stream stream, tb_batch** out);

/* Refinement (PR #757 Summary item 1; conv_transpose_grid k2s2 for factor 2):
 * every voxel v becomes the factor^3 voxels factor*v + [0, factor)^3.
 * factor in {2, 4, 8}.  The pages chain x2 passes for 4 and 8 (Summary item
 * 1, multi-pass paragraph); here one pass emits the factor^3 children
 * directly, with the same result. */
TB_API tb_status tb_refine(const tb_batch* in, int32_t factor, const tb_allocator* alloc, tb_stream stream,
                    tb_batch** out);

/* Coarsening (PR #757 Summary item 1; conv_grid k2s2 for factor 2): voxel V is
 * active iff some v with floor(v / factor) == V is active.  factor in
 * {2, 4, 8}, one pass for any factor as for tb_refine. */
TB_API tb_status tb_coarsen(const tb_batch* in, int32_t factor, const tb_allocator* alloc, tb_stream stream,
                     tb_batch** out);

/* Box dilation (PR #757 Summary item 2): the Minkowski sum of each grid with
 * the box [lo, hi], per axis lo in [-7, 0] and hi in [0, 7]; one pass, at most
 * 27 target leaves per source leaf.  [-1,1]^3 is conv_grid k3s1; {-1,0}^3
 * and {0,1}^3 are the two PadGrid octants.  The stride-1 topology of a
 * uniform kernel of size K (2 <= K <= 15; the PR's tests use K in 2..5) is
 * the box [-floor((K-1)/2), ceil((K-1)/2)]^3 -- for even K the extra offset
 * is on the positive side, a reading the pages leave open -- and the
 * integer-radius dilation by r (r <= 7) is [-r, r]^3.  Other bounds return
 * TB_ERR_INVALID_ARG. */
TB_API tb_status tb_box_dilate(const tb_batch* in, const int32_t lo[3], const int32_t hi[3],
                        const tb_allocator* alloc, tb_stream stream, tb_batch** out);

/* The box of the stride-1 topology of a uniform kernel of size K (the rule
 * above, written once): lo[a] = -floor((K-1)/2), hi[a] = ceil((K-1)/2) on
 * every axis for conv_grid; with transpose != 0 the mirror image [-hi, -lo]
 * for conv_transpose_grid.  Host only, no device work.  TB_ERR_INVALID_ARG
 * for K outside 1..15 or NULL lo/hi (left unwritten). */
TB_API tb_status tb_stride1_box(int32_t kernel_size, int32_t transpose, int32_t lo[3], int32_t hi[3]);

/* Masked refinement (fVDB PR #757 test plan: masked refine; Summary item 1:
 * masked subdivision prunes upstream, then refines): the refinement by
 * `factor` (2, 4 or 8) of the voxels of `in` whose flag is non-zero.
 *   voxel_mask  one byte per active voxel of `in`, host or device memory, in
 *               the batch's voxel order: grid by grid, leaf by leaf, and within
 *               a leaf by ascending bit index n = 64 x + 8 y + z; so voxel
 *               (leaf i, rank r among its set bits) of grid g is flag
 *               sum(voxel_counts[0..g)) + voxel_offset[i] + r.  Borrowed;
 *               must stay valid until the call returns.  May be NULL when the
 *               batch has no voxels.
 * The prune is one kernel before the refinement's pass kernel; the result
 * equals tb_refine of the batch of the flagged voxels.  Errors as tb_refine;
 * TB_ERR_INVALID_ARG for a NULL voxel_mask over a non-empty batch. */
TB_API tb_status tb_refine_masked(const tb_batch* in, const uint8_t* voxel_mask, int32_t factor,
                                  const tb_allocator* alloc, tb_stream stream, tb_batch** out);

/* Kernel map of a sparse convolution from batch `in` to batch `out` (the
 * ConvolutionPlan step after topology generation: issue #755 times the k3s1
 * same-topology map and the k2s2 transpose map).  For every active voxel p of
 * `out` (row j = p's index in the batch's voxel order, see tb_refine_masked)
 * and every offset d of the box [lo, hi] (-7 <= lo <= hi <= 7 per axis;
 * column k enumerates the offsets x-major: k = ((dx-lo0) ny + (dy-lo1)) nz +
 * (dz-lo2)), map[j * K + k] is the index, in the voxel order of `in`, of the
 * input voxel that p reads through d, or -1:
 *   stride 1, transposed == 0: p + d
 *   stride 2, transposed == 0: 2 p + d      (e.g. conv_grid k2s2, box [0,1])
 *   stride 1, transposed != 0: p - d
 *   stride 2, transposed != 0: (p - d) / 2 where p - d is even on every axis
 *                              (conv_transpose_grid k2s2: box [0,1]; k3s2:
 *                              box [-1,1])
 * looked up in the same grid of `in` (both batches have B grids).  K is the
 * box volume; map is device memory of at least map_len >= V_out * K int32
 * entries (V_out = the voxels of `out`), written in stream order, no host
 * synchronization.  Errors: TB_ERR_INVALID_ARG for mismatched batches, bounds,
 * stride, or a short map; TB_ERR_TOO_LARGE for 2^31 or more input voxels. */
TB_API tb_status tb_kernel_map(const tb_batch* in, const tb_batch* out, const int32_t lo[3], const int32_t hi[3],
                               int32_t stride, int32_t transposed, int32_t* map, int64_t map_len, tb_stream stream);

/* Chain of ops applied in order, intermediate results kept on the device
 * (PR #757 Summary items 1-2: multi-pass factors and the k3s2 transpose =
 * refine x2 then the {-1,0}^3 pad).  Consecutive ops are fused into one pass
 * where that pass computes their composition exactly: refinements (or
 * coarsenings) whose factors multiply to at most 8, box dilations whose
 * summed bounds stay within [-7, 7], and refinement by 2 followed by a box
 * within [-1, 1]^3 (so k3s2 is one pass).  The result is the same either way:
 * each op maps voxels to unions of voxels.  n_ops == 0 copies the batch. */
TB_API tb_status tb_chain(const tb_batch* in, const tb_op* ops, int32_t n_ops, const tb_allocator* alloc,
                   tb_stream stream, tb_batch** out);

/* Several chains over the same input in one call: chain c applies
 * chain_lengths[c] ops taken in order from `ops` (the chains' ops are
 * concatenated); outs[c] receives its result (a copy of the input when its
 * length is 0).  All chains run in one launch -- the cooperative whole-grid
 * kernel, phase by phase, or a member launch (tb_set_launch_mode) -- so
 * they share the launch, the readback and the call's host overhead --
 * the batching of PR #757 (Summary) extended from batch members to the
 * several topologies a convolution plan derives from one grid.  Results equal
 * those of separate tb_chain calls.  On error every outs[c] is NULL.
 * Limit: n_chains <= 1024. */
TB_API tb_status tb_multi(const tb_batch* in, const tb_op* ops, const int32_t* chain_lengths, int32_t n_chains,
                          const tb_allocator* alloc, tb_stream stream, tb_batch** outs);

/* Checks the canonical-batch invariants on the device: origins multiples of
 * 8, masks non-zero, leaf_grid consistent with leaf_offsets, leaves strictly
 * increasing in canonical order within each grid.  Blocks once.  Returns
 * TB_OK or TB_ERR_NOT_CANONICAL. */
TB_API tb_status tb_validate(const tb_batch* batch, tb_stream stream);

/* Fills *view.  No device work. */
TB_API tb_status tb_batch_get_view(const tb_batch* batch, tb_batch_view* view);

/* Copies leaf records into caller buffers (host or device memory; any may be
 * NULL to skip): origins [L,3] int32, masks [L,8] uint64, voxel_offset [L]
 * int64, leaf_offsets [B+1] int64.  Enqueued on `stream`; the caller
 * synchronizes before reading host buffers. */
TB_API tb_status tb_batch_export(const tb_batch* batch, int32_t* origins, uint64_t* masks,
                          int64_t* voxel_offset, int64_t* leaf_offsets, tb_stream stream);

/* The same for n batches at once: origins[i], masks[i], voxel_offset[i],
 * leaf_offsets[i] receive batch i's arrays (each of the four lists, and each
 * entry, may be NULL to skip).  Arrays of 1 MiB or more are copied by the
 * copy engines (no SM time, so an export overlaps kernels on other
 * streams); smaller ones whose destination the device can write -- device
 * memory, or pinned host memory through its mapped address -- by one copy
 * kernel for all of them (up to 64 per launch); the rest by plain copies.
 * Enqueued on `stream`; the caller synchronizes before reading host
 * buffers. */
TB_API tb_status tb_batch_export_many(const tb_batch* const* batches, int32_t n, int32_t* const* origins,
                                      uint64_t* const* masks, int64_t* const* voxel_offset,
                                      int64_t* const* leaf_offsets, tb_stream stream);


/* Releases the batch's memory (stream-ordered on `stream`).  NULL is a no-op. */
TB_API tb_status tb_batch_free(tb_batch* batch, tb_stream stream);

/* Message for the calling thread's most recent failure ("" if none). */
TB_API const char* tb_last_error(void);

/* Static name of a status code. */
TB_API const char* tb_status_string(tb_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
TB_API int32_t tb_version(void);

/* Output buffers of tb_refine_static, all device memory owned by the caller.
 * Per-grid arrays hold num_grids (+1) rows; per-leaf arrays leaf_capacity
 * rows, lower-node arrays lower_capacity rows, upper_origins upper_capacity
 * rows.  Shapes and meanings match the arrays of tb_batch_view. */
typedef struct tb_out_buffers {
  int64_t leaf_capacity;
  int64_t lower_capacity;
  int64_t upper_capacity;
  int64_t* leaf_offsets;   /* [B+1] */
  int64_t* lower_offsets;  /* [B+1] */
  int64_t* upper_offsets;  /* [B+1] */
  int64_t* voxel_counts;   /* [B]   */
  int32_t* grid_bbox;      /* [B,6] */
  int32_t* node_counts;    /* [B,3] */
  int32_t* origins;        /* [leaf_capacity,3] */
  uint64_t* masks;         /* [leaf_capacity,8] */
  int64_t* voxel_offset;   /* [leaf_capacity]   */
  uint64_t* word_prefix;   /* [leaf_capacity]   */
  int32_t* leaf_bbox;      /* [leaf_capacity,6] */
  int32_t* leaf_grid;      /* [leaf_capacity]   */
  int32_t* leaf_parent;    /* [leaf_capacity]   */
  int32_t* lower_origins;  /* [lower_capacity,3] */
  int32_t* lower_parent;   /* [lower_capacity]   */
  int32_t* upper_origins;  /* [upper_capacity,3] */
} tb_out_buffers;

/* Refinement by 2 that allocates nothing.  The paper has no counterpart: this
 * is for callers that cannot call cudaMalloc -- applications that reserve all
 * device memory in their own arena, or code running where the CUDA allocator
 * must not be entered (a deadline-bound loop, a callback of the caller's own
 * allocator).  The result equals tb_refine(batch, 2) on the same leaves.
 *   origins [num_leaves,3], masks [num_leaves,8] (16-byte aligned),
 *   leaf_offsets [num_grids+1]: the input leaves in device memory, any order
 *   (duplicates merge); out: caller-owned output buffers (see tb_out_buffers);
 *   out_counts: optional host int64[3] receiving the output's leaf, lower-node
 *   and upper-node totals (also written when the capacity check fails).
 * Every input and output pointer must be device memory (or managed memory):
 * a host pointer returns TB_ERR_INVALID_ARG before any launch.
 * Scratch is one static device array of 32 MiB that every GPU loading the
 * library holds until the process exits; about 52 bytes per candidate leaf
 * (8 per input leaf) plus per-grid control, so inputs of up to roughly 75k
 * leaves fit.  An input that cannot fit (more than 80,659 leaves) returns
 * TB_ERR_TOO_LARGE before any launch; one whose key layout needs more room,
 * or outputs beyond the given capacities, return TB_ERR_TOO_LARGE before
 * anything is written.  Each call looks up the array's device address on the
 * current device (cudaGetSymbolAddress); the first lookup on a device can
 * load the library's device code, so make the first call before any stream
 * capture.  Calls share the array and its contents persist: each call clears
 * its control region first, and calls that overlap on the GPU race.  Blocks
 * twice (range readback, count readback) into host stack memory. */
TB_API tb_status tb_refine_static(const int32_t* origins, const uint64_t* masks, const int64_t* leaf_offsets,
                                  int32_t num_grids, int64_t num_leaves, const tb_out_buffers* out,
                                  int64_t* out_counts, tb_stream stream);

/* Self-test of failure detection without a GPU fault: one thread waits, with
 * the same bounded spin as the pass kernel's grid barrier, for a device flag
 * that is preset (set_flag != 0) or that nothing ever sets; after spin_limit
 * polls (>= 1; about 100 ns each past the first 256) the wait gives up.
 * Returns TB_OK when the flag was seen, TB_ERR_DEVICE_TIMEOUT when the wait
 * ran out; either way the context stays usable.  Blocks once. */
TB_API tb_status tb_selftest_wait(int32_t set_flag, int32_t spin_limit, tb_stream stream);

/* Kernel timing for profiling (library extension, no counterpart on the
 * pages).  With `on` >= 1 on the calling thread, every kernel the library
 * launches is bracketed by two CUDA events on its stream; with `on` >= 2 the
 * pass kernel also stamps the GPU global timer at each of its phase
 * boundaries (records named "phase_*", one per stage of a call: the span from
 * the end of the previous phase to the latest end of this one over the stage's
 * chains, which run the phase side by side).  tb_profile_read waits for the
 * recorded events, writes up to `max` records (aggregated by name) and clears
 * them; it returns the number of distinct records (which may exceed `max`). */
TB_API tb_status tb_profile_enable(int32_t on);
TB_API int32_t tb_profile_read(tb_kernel_stat* stats, int32_t max);

/* Launch shape of the pass kernel (library extension: the pages prescribe
 * none).  mode 0 (default): a member launch -- one cluster of 1 to 8 CTAs per
 * grid of every chain, each running its grid's passes as a batch of one grid,
 * the call's counts gathered by the last cluster to finish -- when every grid
 * is small (at most 16384 candidate leaves or input voxels per CTA of its
 * cluster, and at most 4096 grids), else the cooperative whole-grid kernel;
 * 1: always the whole-grid kernel; 2: a member launch for every non-empty
 * input.  Both give identical outputs.  Process-wide; returns the previous
 * mode, or -1 (mode unchanged) for a mode outside 0..2. */
TB_API int32_t tb_set_launch_mode(int32_t mode);

/* How the whole-grid kernel puts a pass's output leaves in canonical order
 * (library extension; PR #757, Summary item 1, names the canonical NanoVDB
 * node order, which both ways produce).  mode 0 (default): where the pass's
 * output can hold at most 16384 lower nodes (a bound from the source's lower
 * nodes, or its voxel / leaf count for a front end), the node path: every
 * target leaf sets its bit in its lower node's 4096-bit child mask, the few
 * lower nodes are ranked by canonical key and every leaf's index is its
 * node's leaf base plus the set bits before it -- no radix sort; elsewhere
 * the radix sort and head-flag scan.  mode 1: always the radix sort.  Both
 * give identical outputs.  Process-wide; returns the previous mode, or -1
 * (mode unchanged) for a mode outside 0..1. */
TB_API int32_t tb_set_node_mode(int32_t mode);

/* Which kernel writes tb_kernel_map (library extension: the pages prescribe
 * none).  mode 0 (default): picked from the box and the output's size -- the
 * staged form (the candidate input leaves' mask words staged in shared
 * memory: batches of 4 to 16 output leaves per warp where an output leaf's
 * reach spans at most 2 input leaves per axis and the box has at most 32
 * columns, else one leaf per warp) where the reach spans at most 3 input
 * leaves per axis and the output has at least 32 leaves per SM; the
 * tabulated form (a table of the
 * input voxel index of every voxel in an output leaf's reach, one leaf per
 * warp) for fewer leaves where the reach is small; else the per-entry form.
 * mode 1: staged; 2: staged after a candidate look-up pass of its own; 3:
 * tabulated; 4: per entry -- each where the box allows it, else per entry.
 * All give identical maps.  Process-wide; returns the previous mode, or -1
 * (mode unchanged) for a mode outside 0..4. */
TB_API int32_t tb_set_kmap_mode(int32_t mode);

/* Number of kernels this thread has launched through the library so far. */
TB_API int64_t tb_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TB_H_ */
