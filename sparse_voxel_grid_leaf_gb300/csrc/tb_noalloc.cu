// tb_refine_static: refinement by 2 for callers that cannot allocate device
// memory.  The paper has no counterpart; this is a library extension.
//
// Who needs it: applications that reserve all device memory up front in
// their own arena (so a library cudaMalloc would fail or fragment their pool),
// and code that runs where calling the CUDA allocator is not allowed, such as
// a deadline-bound loop or a callback of the application's own allocator,
// where re-entering the allocator could deadlock.  Such a caller passes the
// input leaves and every output buffer; the pass's scratch (sort slots, key
// buffers, look-back status words, counters) lives in one file-scope device
// array of kStaticScratchBytes that every GPU loading this library holds
// until the process exits.
//
// The same emission, sort, dedup and writer kernels as tb_refine run on
// pointers into that array.  Each call looks up the array's device address on
// the current device with cudaGetSymbolAddress (the array's name in host code
// is only a host-side stand-in, and a device reset between calls can move the
// array); the first lookup on a device can load the library's device code, so
// make the first call before any stream capture.  Every call reuses the
// array, whose contents persist between calls: the control region is cleared
// at the start of each call, and calls that overlap on the GPU (other
// streams, other threads) race on it.
#include <algorithm>
#include <cstring>

#include "../../include/tb.h"
#include "tb_common.cuh"
#include "tb_launch.h"
#include "tb_layout.h"

using namespace tb;

namespace {

constexpr size_t kStaticScratchBytes = 32ull << 20;  // 32 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

tb_status static_fail(tb_status st, const char* msg) {
  set_error_message(msg);
  return st;
}

// Device address of the scratch array on the current device, looked up on
// every call (never cached: after a device reset the module is loaded again
// and the array can sit elsewhere).
tb_status scratch_address(char** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    return static_fail(TB_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
  }
  *out = (char*)p;
  return TB_OK;
}

// Bytes of the scratch carve that grow with the candidate slots alone: two
// key and two value buffers of the digit passes, the run starts and the
// per-leaf arrays of the last pass (see the carve in tb_refine_static).
constexpr size_t kSlotBytes = 8 + 8 + 4 + 4 + 4 + 4 + 4 + 8 + 4 + 4;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

#define TB_STATIC_CUDA(expr)                                   \
  do {                                                         \
    if ((expr) != cudaSuccess) return static_fail(TB_ERR_CUDA, #expr " failed"); \
  } while (0)

int blocks_of(long long work, long long per, long long cap) {
  long long n = (work + per - 1) / per;
  if (n < 1) n = 1;
  if (n > cap) n = cap;
  return (int)n;
}

}  // namespace

extern "C" {

tb_status tb_refine_static(const int32_t* origins, const uint64_t* masks, const int64_t* leaf_offsets,
                           int32_t num_grids, int64_t num_leaves, const tb_out_buffers* out, int64_t* out_counts,
                           tb_stream stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  const int32_t B = num_grids;
  const long long L = num_leaves;
  if (!out || !leaf_offsets || B < 0 || L < 0 || (L > 0 && (!origins || !masks)))
    return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: bad pointer or negative size");
  if (B == 0 && L != 0) return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: leaves without grids");
  if (((uintptr_t)masks & 15) != 0) return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: masks must be 16-byte aligned");
  if (L >= (1ll << (32 - pass_code_bits(kRefine, 2)))) return static_fail(TB_ERR_TOO_LARGE, "tb_refine_static: too many input leaves");
  // up to 8 candidate slots per input leaf, each needing kSlotBytes of scratch
  if ((unsigned long long)L * 8ull * kSlotBytes > kStaticScratchBytes)
    return static_fail(TB_ERR_TOO_LARGE, "tb_refine_static: input needs more than the 32 MiB static scratch");
  // every pointer the kernels touch must be device memory
  if (!device_accessible(leaf_offsets) || (L > 0 && (!device_accessible(origins) || !device_accessible(masks))))
    return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: inputs must be device memory");
  {
    const void* outs[] = {out->leaf_offsets, out->lower_offsets, out->upper_offsets, out->voxel_counts,
                          out->grid_bbox,    out->node_counts,   out->origins,       out->masks,
                          out->voxel_offset, out->word_prefix,   out->leaf_bbox,     out->leaf_grid,
                          out->leaf_parent,  out->lower_origins, out->lower_parent,  out->upper_origins};
    for (const void* p : outs)
      if (p && !device_accessible(p))
        return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: output buffers must be device memory");
  }
  int dev = 0;
  TB_STATIC_CUDA(cudaGetDevice(&dev));
  char* scratch = nullptr;
  tb_status st = scratch_address(&scratch);
  if (st != TB_OK) return st;
  int sms = 0;
  TB_STATIC_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));

  // ---- coordinate range of the input (the key layout depends on it)
  ReadbackHeader* rb0 = (ReadbackHeader*)scratch;
  if (readback_bytes(B) + 4096 + sizeof(PassCtl) > kStaticScratchBytes)
    return static_fail(TB_ERR_TOO_LARGE, "tb_refine_static: too many grids for the static scratch");
  TB_STATIC_CUDA(cudaMemsetAsync(rb0, 0, sizeof(ReadbackHeader), stream));
  TB_STATIC_CUDA(launch_prepass_leaves(origins, masks, L, leaf_offsets, B, rb0,
                                       blocks_of(L, 256, (long long)sms * 4), stream));
  ReadbackHeader h;  // pageable host memory: nothing is allocated for the readback
  TB_STATIC_CUDA(cudaMemcpyAsync(&h, rb0, sizeof h, cudaMemcpyDeviceToHost, stream));
  TB_STATIC_CUDA(cudaStreamSynchronize(stream));
  if (h.err & kErrBadOffsets) return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: bad leaf offsets");
  if (h.err & kErrNotAligned) return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: origins must be multiples of 8");
  int32_t bb[6];
  for (int a = 0; a < 3; ++a) {
    bb[a] = dec_min(h.bbox_enc[a]);
    bb[3 + a] = dec_max(h.bbox_enc[3 + a]);
  }
  const bool empty = bb[0] > bb[3];
  int32_t ob[6] = {0, 0, 0, 0, 0, 0};
  if (!empty)
    for (int a = 0; a < 3; ++a) {
      const int64_t lo = 2 * (int64_t)bb[a], hi = 2 * (int64_t)bb[3 + a] + 1;
      if (lo < INT32_MIN || hi > INT32_MAX) return static_fail(TB_ERR_COORD_OVERFLOW, "tb_refine_static: coordinates leave int32");
      ob[a] = (int32_t)lo;
      ob[3 + a] = (int32_t)hi;
    }
  PassArgs a;
  std::memset(&a, 0, sizeof a);
  if (!make_layout(B, ob, empty, a.K)) return static_fail(TB_ERR_TOO_LARGE, "tb_refine_static: sort key wider than 64 bits");
  a.P = (a.K.W + 7) / 8;
  a.mid = a.P;  // the radix sort orders the leaves (no node tables here)

  // ---- carve the scratch array
  const long long S = 8 * L;
  const long long sort_tiles = std::max(1ll, (S + kSortTile - 1) / kSortTile);
  const long long dedup_tiles = std::max(1ll, (S + kDedupTile - 1) / kDedupTile);
  const size_t rbb = readback_bytes(B);
  size_t off = 256;  // the prepass header stays at offset 0
  auto take = [&](size_t n) {
    const size_t r = off;
    off = align256(off + n);
    return r;
  };
  const size_t o_err = take(4), o_bar = take(sizeof(GridBarrier)), o_rb = take(rbb), o_ctl = take(sizeof(PassCtl)),
               o_sort = take((size_t)a.P * sort_tiles * kBins * 4), o_dedup = take((size_t)dedup_tiles * 24),
               o_first = take((size_t)3 * B * 4);
  const size_t zero_begin = o_err, zero_end = off;
  const size_t o_k0 = take((size_t)S * 8), o_k1 = take((size_t)S * 8), o_v0 = take((size_t)S * 4),
               o_v1 = take((size_t)S * 4), o_run = take((size_t)(S + 1) * 4), o_ll = take((size_t)S * 4),
               o_lu = take((size_t)S * 4), o_voff = take((size_t)S * 8), o_pop = take((size_t)S * 4),
               o_lg = take((size_t)S * 4);
  const int G = sms * chain_occupancy();
  const size_t o_blk = take((size_t)G * 8), o_grp = take((size_t)G * 32 * 8), o_args = take(sizeof(PassArgs));
  if (off > kStaticScratchBytes)
    return static_fail(TB_ERR_TOO_LARGE,
                       "tb_refine_static: input needs more than the 32 MiB static scratch (about 75k leaves)");
  TB_STATIC_CUDA(cudaMemsetAsync(scratch + zero_begin, 0, zero_end - zero_begin, stream));

  a.op = kRefine;
  a.factor = 2;
  a.code_bits = pass_code_bits(kRefine, 2);
  a.B = B;
  a.last = 1;
  a.tchunk = (int32_t)std::max(1ll, std::min(8ll, (8 * L + (long long)G * 256 - 1) / ((long long)G * 256)));
  a.src_origins = origins;
  a.src_masks = masks;
  a.src_grid = nullptr;
  a.in_offsets = leaf_offsets;
  a.src_count = L;
  a.rb = (ReadbackHeader*)(scratch + o_rb);
  a.leaf_off = (int64_t*)(scratch + o_rb + sizeof(ReadbackHeader));
  a.lower_off = a.leaf_off + (B + 1);
  a.upper_off = a.lower_off + (B + 1);
  a.grid_vox = a.upper_off + (B + 1);
  a.gbox = (unsigned int*)(a.grid_vox + B);
  a.ctl = (PassCtl*)(scratch + o_ctl);
  a.sort_status = (uint32_t*)(scratch + o_sort);
  a.sort_tiles_cap = sort_tiles;
  a.dedup_status = (unsigned long long*)(scratch + o_dedup);
  a.first = (uint32_t*)(scratch + o_first);
  a.slot_cap = S;
  a.keys[0] = (uint64_t*)(scratch + o_k0);
  a.keys[1] = (uint64_t*)(scratch + o_k1);
  a.vals[0] = (uint32_t*)(scratch + o_v0);
  a.vals[1] = (uint32_t*)(scratch + o_v1);
  a.sorted = a.P & 1;
  a.run_start = (uint32_t*)(scratch + o_run);
  a.leaf_lower = (uint32_t*)(scratch + o_ll);
  a.leaf_upper = (uint32_t*)(scratch + o_lu);
  a.leaf_voff = (int64_t*)(scratch + o_voff);
  a.leaf_pop = (uint32_t*)(scratch + o_pop);
  a.leaf_g = (uint32_t*)(scratch + o_lg);
  a.blk_agg = (unsigned long long*)(scratch + o_blk);
  a.grp_agg = (unsigned long long*)(scratch + o_grp);
  a.err = (unsigned int*)(scratch + o_err);

  // ---- the same cooperative pass kernel as tb_refine
  // the pass arguments go to the scratch array from host stack memory
  TB_STATIC_CUDA(cudaMemcpyAsync(scratch + o_args, &a, sizeof a, cudaMemcpyHostToDevice, stream));
  ChainArgs ca{};
  ca.pass = (const PassArgs*)(scratch + o_args);
  ca.n_chain = 1;
  ca.n_stage = 1;
  ca.bar = (GridBarrier*)(scratch + o_bar);
  ca.err = (unsigned int*)(scratch + o_err);
  ca.front = 0;
  TB_STATIC_CUDA(launch_chain(ca, G, stream));
  ReadbackHeader r;
  unsigned int derr = 0;
  TB_STATIC_CUDA(cudaMemcpyAsync(&r, a.rb, sizeof r, cudaMemcpyDeviceToHost, stream));
  TB_STATIC_CUDA(cudaMemcpyAsync(&derr, a.err, sizeof derr, cudaMemcpyDeviceToHost, stream));
  TB_STATIC_CUDA(cudaStreamSynchronize(stream));
  r.err |= derr;
  if (r.err & kErrTimeout) return static_fail(TB_ERR_DEVICE_TIMEOUT, "tb_refine_static: a device wait timed out");
  if (r.err & kErrSlotOverflow) return static_fail(TB_ERR_INTERNAL, "tb_refine_static: internal slot bound exceeded");
  if (out_counts) {
    out_counts[0] = (int64_t)r.num_leaves;
    out_counts[1] = (int64_t)r.num_lowers;
    out_counts[2] = (int64_t)r.num_uppers;
  }
  if ((long long)r.num_leaves > out->leaf_capacity || (long long)r.num_lowers > out->lower_capacity ||
      (long long)r.num_uppers > out->upper_capacity)
    return static_fail(TB_ERR_TOO_LARGE, "tb_refine_static: output capacity too small (see out_counts)");
  if (B > 0 && (!out->leaf_offsets || !out->lower_offsets || !out->upper_offsets || !out->voxel_counts ||
                !out->grid_bbox || !out->node_counts))
    return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: per-grid output buffer missing");
  if (r.num_leaves > 0 && (!out->origins || !out->masks || !out->voxel_offset || !out->word_prefix ||
                           !out->leaf_bbox || !out->leaf_grid || !out->leaf_parent || !out->lower_origins ||
                           !out->lower_parent || !out->upper_origins))
    return static_fail(TB_ERR_INVALID_ARG, "tb_refine_static: per-leaf output buffer missing");

  // ---- writer into the caller's buffers
  WriteOut o;
  o.origins = out->origins;
  o.masks = out->masks;
  o.leaf_grid = out->leaf_grid;
  o.voxel_offset = out->voxel_offset;
  o.word_prefix = out->word_prefix;
  o.leaf_bbox = out->leaf_bbox;
  o.leaf_parent = out->leaf_parent;
  o.voxel_counts = out->voxel_counts;
  o.grid_bbox = out->grid_bbox;
  o.node_counts = out->node_counts;
  o.leaf_offsets = out->leaf_offsets;
  o.lower_offsets = out->lower_offsets;
  o.upper_offsets = out->upper_offsets;
  o.lower_origins = out->lower_origins;
  o.lower_parent = out->lower_parent;
  o.upper_origins = out->upper_origins;
  o.L_cap = (long long)r.num_leaves;  // the counts just read back
  o.NL_cap = (long long)r.num_lowers;
  o.NU_cap = (long long)r.num_uppers;
  const int wb = blocks_of(std::max<long long>((long long)r.num_leaves, B + 1), kWriteLeavesPerBlock,
                           (long long)sms * write_final_occupancy(kRefine));
  TB_STATIC_CUDA(launch_write_final(kRefine, a, o, wb, stream));
  return TB_OK;
}

}  // extern "C"
