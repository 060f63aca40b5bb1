// Host driver and C ABI of libtb.so (declared in include/tb.h).
//
// One call = one stream-ordered sequence (fVDB PR #757 "Batched leaf-mask
// topology construction for generated conv grids", Summary item 1): one
// cooperative launch of the pass kernel runs every pass of every chain of the
// call (intermediate passes hand their leaves to the next stage on the
// device), then the one count readback, the exact output allocation and one
// writer launch.  All buffers of a call are sized from host-known upper
// bounds (refine emits at most 8 leaves per source leaf, coarsen 1, a box
// dilation at most its box volume), so no readback is needed between passes.
//
// The sort key's width follows the batch's voxel bounding box, which the
// host tracks exactly: refine maps [lo, hi] to [2 lo, 2 hi + 1], coarsen to
// [floor(lo/2), floor(hi/2)], a box dilation to [lo + d_lo, hi + d_hi].  For
// the front ends the pass kernel reads the input's bbox and plans the key
// itself; the host repeats that plan after the readback.
#include <algorithm>
#include <array>
#include <atomic>
#include <chrono>
#include <cstddef>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/tb.h"
#include "tb_common.cuh"
#include "tb_launch.h"
#include "tb_layout.h"

using namespace tb;

struct tb_batch {
  int64_t build_slots = 0, build_sources = 0;
  int32_t build_key_bits = 0, build_digit_passes = 0, build_member_ctas = 0;
  int32_t B = 0;
  int device = 0;
  int64_t L = 0, NL = 0, NU = 0;
  bool has_alloc = false;
  tb_allocator alloc{};
  void* mem = nullptr;
  std::vector<int64_t> leaf_offsets_host;
  std::vector<int64_t> voxel_base_host;  // [B+1] exclusive prefix of the grids' voxel counts
  int32_t bbox[6] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MIN, INT32_MIN, INT32_MIN};
  int64_t* leaf_offsets = nullptr;
  int32_t* origins = nullptr;
  uint64_t* masks = nullptr;
  int64_t* voxel_offset = nullptr;
  uint64_t* word_prefix = nullptr;
  int32_t* leaf_bbox = nullptr;
  int32_t* leaf_grid = nullptr;
  int32_t* leaf_parent = nullptr;
  int64_t* voxel_counts = nullptr;
  int32_t* grid_bbox = nullptr;
  int32_t* node_counts = nullptr;
  int64_t* lower_offsets = nullptr;
  int64_t* upper_offsets = nullptr;
  int32_t* lower_origins = nullptr;
  int32_t* lower_parent = nullptr;
  int32_t* upper_origins = nullptr;
};

namespace {

thread_local std::string t_err;
thread_local long long t_launches = 0;

// ---------------------------------------------------------------- kernel timing

enum KernelKind {
  kKPrepassLeaves, kKChain, kKWrite0, kKValidate = kKWrite0 + kNumOps, kKWriteMulti, kKPrune, kKKmap, kKKmapPrep,
  kKExport, kKMember, kKNumKinds
};
const char* const kKernelNames[kKNumKinds] = {"prepass_leaves", "chain",         "write_ijk",
                                              "write_leaves",  "write_refine",   "write_coarsen", "write_dilate",
                                              "write_refine_dilate", "validate", "write_multi",   "prune",
                                              "kernel_map",    "kmap_prep",    "export",        "member"};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
thread_local int t_prof = 0;  // 1: kernel events, 2: also pass-phase stamps
constexpr int kNumGpuPhases = 5;
constexpr int kNumPhases = 11;
const char* const kPhaseNames[kNumPhases] = {"phase_emit",      "phase_sort",       "phase_dedup_merge",
                                             "phase_leaves",    "phase_offsets",    "phase_entry",
                                             "host_before_sync", "host_sync_wait",  "host_after_sync",
                                             "host_plan",       "host_alloc"};
double host_ms_since(const std::chrono::steady_clock::time_point& t0) {
  return std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
}
thread_local double t_phase_ms[kNumPhases] = {};
thread_local long long t_phase_n[kNumPhases] = {};
thread_local std::vector<ProfRec> t_recs;
thread_local std::vector<cudaEvent_t> t_events;

cudaEvent_t pooled_event() {
  if (!t_events.empty()) {
    cudaEvent_t e = t_events.back();
    t_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Launches through `f` (returning cudaError_t); counted, and timed when enabled.
template <class F>
cudaError_t launch(int kind, cudaStream_t s, F&& f) {
  ++t_launches;
  if (!t_prof) return f();
  cudaEvent_t a = pooled_event(), b = pooled_event();
  if (a) cudaEventRecord(a, s);
  const cudaError_t e = f();
  if (b) cudaEventRecord(b, s);
  if (a && b) t_recs.push_back({kind, a, b});
  return e;
}

tb_status fail(tb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

#define TB_CUDA(expr)                                                                          \
  do {                                                                                         \
    cudaError_t e_ = (expr);                                                                   \
    if (e_ != cudaSuccess) return fail(TB_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

// ---------------------------------------------------------------- device info

struct DeviceInfo {
  int sms = 0;
  int occ_chain = 1;
  int occ_member = 1;
  int member_fit[4] = {};  // clusters of 1, 2, 4, 8 CTAs of the member kernel the device runs at once
  int occ_write[kNumOps] = {};
  int occ_write_multi = 1;
  bool coop = false;
  bool ready = false;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

tb_status device_info(int dev, DeviceInfo** out) {
  if (dev < 0 || dev >= 64) return fail(TB_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    TB_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    int coop = 0;
    TB_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
    if (!coop) return fail(TB_ERR_CUDA, "device %d does not support cooperative launches", dev);
    d.coop = true;
    d.occ_chain = chain_occupancy();
    d.occ_member = member_occupancy();
    for (int i = 0; i < 4; ++i) d.member_fit[i] = i ? member_clusters(1 << i) : d.sms * d.occ_member;
    for (int op = 0; op < kNumOps; ++op) d.occ_write[op] = write_final_occupancy(op);
    d.occ_write_multi = write_multi_occupancy();
    // keep freed memory in the default pool between calls
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      uint64_t thr = UINT64_MAX;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
    cudaGetLastError();
    d.ready = true;
  }
  *out = &d;
  return TB_OK;
}

// ---------------------------------------------------------------- memory

struct Mem {
  const tb_allocator* a;
  cudaStream_t s;
  void* get(size_t n) const {
    if (n == 0) return nullptr;
    if (a) return a->alloc(a->ctx, n, (tb_stream)s);
    void* p = nullptr;
    if (cudaMallocAsync(&p, n, s) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return p;
  }
  void put(void* p) const {
    if (!p) return;
    if (a) a->free(a->ctx, p, (tb_stream)s);
    else cudaFreeAsync(p, s);
  }
};

// Frees a buffer at scope exit unless released.
struct Guard {
  const Mem* m;
  void* p;
  ~Guard() {
    if (p) m->put(p);
  }
};

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes, size_t align = 256) {
    off = (off + align - 1) & ~(align - 1);
    const size_t r = off;
    off += bytes;
    return r;
  }
};

struct Pinned {
  void* p = nullptr;
  size_t n = 0;
  ~Pinned() {
    if (p) cudaFreeHost(p);
  }
  void* get(size_t bytes) {
    if (bytes > n) {
      if (p) cudaFreeHost(p);
      p = nullptr;
      n = 0;
      if (cudaHostAlloc(&p, bytes, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
      n = bytes;
    }
    return p;
  }
};
thread_local Pinned t_pinned;
thread_local unsigned int t_seq = 0;  // readback flag values of this thread's calls

}  // namespace

bool tb::device_accessible(const void* p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

namespace {

// ---------------------------------------------------------------- pass plan

struct PassSpec {
  int op;
  int32_t factor;  // refine / coarsen
  int32_t lo[3], hi[3];
};

struct PassPlan {
  PassSpec spec;
  long long in_cap = 0, slot_cap = 0;
  bool empty = true;         // output has no voxels
  int32_t bbox[6];           // output voxel bbox (exact)
  KeyLayout K;
  int P = 0;
  // node path (see PassArgs): the bound on the output's lower nodes, and the
  // workspace of the node tables
  bool node = false;
  int node_zero = 0, mid = 0, node_cap = 0;
  long long node_bound = 0;
  uint32_t node_hslots = 0;
  size_t nh_key = 0, th_key = 0, node_mask = 0, gmin = 0, node_key = 0, node_lc = 0, node_tile = 0, node_rank = 0,
         node_wpre = 0, rank_cnt = 0, tile_rank = 0, node_list = 0, tile_list = 0, nref = 0;
  long long sort_tiles = 0, dedup_tiles = 0;
  size_t rb = 0, ctl = 0, sort_status = 0, dedup_status = 0, first = 0;
  size_t unit_ctl = 0;       // member launches: the members' control blocks
  long long ctl_stride = 0;  // and their size
};

// ---------------------------------------------------------------- launch shape

// 0: member launches where they pay, 1: always the whole-grid kernel, 2:
// member launches whenever possible (tb_set_launch_mode).
std::atomic<int> g_launch_mode{0};
// A member launch saves the whole-grid kernel's barriers and long look-backs
// but runs each grid's leaves phase on the member's own CTAs, so it pays
// where every grid's leaves are few for its CTAs (measured on GB300: single
// refine / coarsen / dilate calls on 16 or 48 grids of resolution 64, every
// front end tried) and loses where one chain's leaves dominate: several
// chains in one call, the fused refine-then-dilate merge, large grids.
constexpr long long kMemberSlotsPerCta = 2048;        // candidate leaves of one grid per member CTA
// Refinement alone: the whole-grid kernel's node path stores each target
// leaf's one slot directly (no clearing, no merge), so it wins from fewer
// candidates per member CTA (measured on GB300: 48 shells, about 400 per
// CTA, 76 us against 84 us; 16 shells, about 200, 72 us against 63 us).
constexpr long long kMemberRefineSlotsPerCta = 256;
constexpr long long kMemberVoxelsPerCta = 16384;      // front ends: input voxels of one grid per member CTA
constexpr int32_t kMemberMaxGrids = 4096;             // the last member scans its chain's grid counts alone

// CTAs per member of a member launch (1, 2, 4 or 8: the most whose clusters
// the device runs all at once, `fit[log2 cl]`), or 0 for the whole-grid
// kernel.  `nmax` is
// the most stage-0 sources of one grid (-1: not known on the host), `mmax`
// the largest slot capacity per stage-0 source of any pass, `heavy` whether a
// pass is the fused refine-then-dilate, `refine_only` whether every pass is
// a refinement.
int member_ctas(int n_chain, int32_t B, long long count, long long nmax, long long mmax, const int fit[4],
                bool front, bool heavy, bool refine_only) {
  const int mode = g_launch_mode.load();
  if (mode == 1 || B < 1 || count <= 0) return 0;
  int cl = 8, lg = 3;
  while (cl > 1 && (long long)n_chain * B > (long long)fit[lg]) {
    cl >>= 1;
    --lg;
  }
  if (mode == 2) return cl;
  if (B > kMemberMaxGrids || n_chain > 1 || heavy) return 0;
  const long long mean = (count + B - 1) / B;
  const long long per_cta = front ? kMemberVoxelsPerCta : refine_only ? kMemberRefineSlotsPerCta : kMemberSlotsPerCta;
  // a member launch lasts as long as its largest grid: with grids of very
  // unequal sizes (the largest above twice the mean) and a largest grid of
  // more than a quarter of the budget per CTA, the whole-grid kernel wins
  // (measured on GB300, 48 shells of 0.25x-4x the area: refinement 79 us
  // against 117 us, the {-1,0}^3 pad 78 against 96 us; coarsening, one
  // candidate per source, still 65 against 76 us as a member launch)
  if (nmax > 2 * mean && nmax * mmax > per_cta / 4 * cl) return 0;
  const long long n = nmax >= 0 ? nmax : 2 * mean;  // unknown: twice the mean
  return n * mmax <= per_cta * cl ? cl : 0;
}

long long slots_per_source(const PassSpec& s) { return pass_targets(s.op, s.factor, s.lo, s.hi); }

// 0: the node path wherever its bound allows (whole-grid launches), 1: never
// (tb_set_node_mode).
std::atomic<int> g_node_mode{0};
// Form of the kernel map (tb_set_kmap_mode): 0 picked by the host, 1 staged,
// 2 staged after the candidate look-up pass, 3 tabulated, 4 per entry.
std::atomic<int> g_kmap_mode{0};
// Staged masks of a node-path pass are cleared in its nodes phase (no phase
// of their own) when its slots' masks take at most this many bytes.
constexpr long long kNodeClearInline = 16ll << 20;

// Per axis, how many lower nodes the image of one source lower node spans
// after a pass, given `span` before it (a lower node spans 128 voxels per
// axis).  Refinement by f multiplies the span by f; coarsening by f maps a
// run of s nodes into at most (s - 1) / f + 2 nodes (one for s = 1); a box
// dilation by at most 7 voxels reaches one more node on each side it
// extends to; refinement by 2 then such a box does both.
long long node_span(const PassSpec& s, int axis, long long span) {
  const long long ext = (s.lo[axis] < 0 ? 1 : 0) + (s.hi[axis] > 0 ? 1 : 0);
  switch (s.op) {
    case kRefine: return span * s.factor;
    case kCoarsen: return span == 1 ? 1 : (span - 1) / s.factor + 2;
    case kDilate: return span + ext;
    case kRefineDilate: return 2 * span + ext;
    default: return span;  // the front ends: one node per source at most
  }
}

// Output bbox of one pass from its input bbox; false on int32 overflow.
bool propagate_bbox(const PassSpec& s, const int32_t in[6], int32_t out[6]) {
  const int32_t lo[3] = {s.lo[0], s.lo[1], s.lo[2]}, hi[3] = {s.hi[0], s.hi[1], s.hi[2]};
  return tb::propagate_bbox(s.op, s.factor, lo, hi, in, out);
}

tb_status plan_layouts(std::vector<PassPlan>& plans, int32_t B, const int32_t bbox_in[6], bool empty_in) {
  int32_t cur[6];
  std::memcpy(cur, bbox_in, sizeof cur);
  bool empty = empty_in;
  for (size_t p = 0; p < plans.size(); ++p) {
    PassPlan& pl = plans[p];
    if (!empty && !propagate_bbox(pl.spec, cur, pl.bbox))
      return fail(TB_ERR_COORD_OVERFLOW, "pass %zu would move voxel coordinates outside int32", p);
    if (empty) std::memcpy(pl.bbox, cur, sizeof cur);
    pl.empty = empty;
    if (!make_layout(B, pl.bbox, empty, pl.K))
      return fail(TB_ERR_TOO_LARGE, "pass %zu: the batch's grid count and coordinate range need a %d-bit sort key (max 64)",
                  p, pl.K.W);
    pl.P = (pl.K.W + 7) / 8;
    std::memcpy(cur, pl.bbox, sizeof cur);
  }
  return TB_OK;
}

// ---------------------------------------------------------------- sources

enum SrcKind { kSrcBatch, kSrcIjk, kSrcLeaves };

struct Source {
  SrcKind kind;
  const tb_batch* batch = nullptr;
  const int32_t* ijk = nullptr;
  const int32_t* origins = nullptr;
  const uint64_t* masks = nullptr;
  const int64_t* offsets = nullptr;
  int32_t B = 0;
  long long count = 0;
};

void batch_set_view(tb_batch* b, char* base, const size_t off[16]) {
  auto at = [&](int k) -> char* { return base ? base + off[k] : nullptr; };
  b->leaf_offsets = (int64_t*)at(0);
  b->origins = (int32_t*)at(1);
  b->masks = (uint64_t*)at(2);
  b->voxel_offset = (int64_t*)at(3);
  b->word_prefix = (uint64_t*)at(4);
  b->leaf_bbox = (int32_t*)at(5);
  b->leaf_grid = (int32_t*)at(6);
  b->leaf_parent = (int32_t*)at(7);
  b->voxel_counts = (int64_t*)at(8);
  b->grid_bbox = (int32_t*)at(9);
  b->node_counts = (int32_t*)at(10);
  b->lower_offsets = (int64_t*)at(11);
  b->upper_offsets = (int64_t*)at(12);
  b->lower_origins = (int32_t*)at(13);
  b->lower_parent = (int32_t*)at(14);
  b->upper_origins = (int32_t*)at(15);
}

int blocks_for(long long work, long long per_block, long long cap) {
  long long n = (work + per_block - 1) / per_block;
  if (n < 1) n = 1;
  if (n > cap) n = cap;
  return (int)n;
}

// ---------------------------------------------------------------- the driver

// Allocates the exact output arrays of a batch whose sizes (B, L, NL, NU)
// are set, in one allocation carved into 256-byte-aligned arrays.
tb_status alloc_outputs(tb_batch* b, const Mem& mem) {
  const int64_t B = b->B, L = b->L, NL = b->NL, NU = b->NU;
  Carve oc;
  size_t off[16];
  off[0] = oc.take((size_t)(B + 1) * 8);
  off[1] = oc.take((size_t)L * 12);
  off[2] = oc.take((size_t)L * 64);
  off[3] = oc.take((size_t)L * 8);
  off[4] = oc.take((size_t)L * 8);
  off[5] = oc.take((size_t)L * 24);
  off[6] = oc.take((size_t)L * 4);
  off[7] = oc.take((size_t)L * 4);
  off[8] = oc.take((size_t)B * 8);
  off[9] = oc.take((size_t)B * 24);
  off[10] = oc.take((size_t)B * 12);
  off[11] = oc.take((size_t)(B + 1) * 8);
  off[12] = oc.take((size_t)(B + 1) * 8);
  off[13] = oc.take((size_t)NL * 12);
  off[14] = oc.take((size_t)NL * 4);
  off[15] = oc.take((size_t)NU * 12);
  b->mem = mem.get(oc.off);
  if (!b->mem) return fail(TB_ERR_OOM, "output allocation of %zu bytes failed", oc.off);
  batch_set_view(b, (char*)b->mem, off);
  auto nz = [](void* p, int64_t n) { return n > 0 ? p : nullptr; };
  b->origins = (int32_t*)nz(b->origins, L);
  b->masks = (uint64_t*)nz(b->masks, L);
  b->voxel_offset = (int64_t*)nz(b->voxel_offset, L);
  b->word_prefix = (uint64_t*)nz(b->word_prefix, L);
  b->leaf_bbox = (int32_t*)nz(b->leaf_bbox, L);
  b->leaf_grid = (int32_t*)nz(b->leaf_grid, L);
  b->leaf_parent = (int32_t*)nz(b->leaf_parent, L);
  b->voxel_counts = (int64_t*)nz(b->voxel_counts, B);
  b->grid_bbox = (int32_t*)nz(b->grid_bbox, B);
  b->node_counts = (int32_t*)nz(b->node_counts, B);
  b->lower_origins = (int32_t*)nz(b->lower_origins, NL);
  b->lower_parent = (int32_t*)nz(b->lower_parent, NL);
  b->upper_origins = (int32_t*)nz(b->upper_origins, NU);
  return TB_OK;
}

void fill_write_out(const tb_batch* b, WriteOut& wo) {
  wo.origins = b->origins;
  wo.masks = b->masks;
  wo.leaf_grid = b->leaf_grid;
  wo.voxel_offset = b->voxel_offset;
  wo.word_prefix = b->word_prefix;
  wo.leaf_bbox = b->leaf_bbox;
  wo.leaf_parent = b->leaf_parent;
  wo.voxel_counts = b->voxel_counts;
  wo.grid_bbox = b->grid_bbox;
  wo.node_counts = b->node_counts;
  wo.leaf_offsets = b->leaf_offsets;
  wo.lower_offsets = b->lower_offsets;
  wo.upper_offsets = b->upper_offsets;
  wo.lower_origins = b->lower_origins;
  wo.lower_parent = b->lower_parent;
  wo.upper_origins = b->upper_origins;
  wo.L_cap = b->L;  // the counts the arrays were carved for
  wo.NL_cap = b->NL;
  wo.NU_cap = b->NU;
}

// Output counts of the last call of each shape on this thread (source kind,
// grids, source count, chains): the next call of that shape allocates its
// outputs with some room above them and queues its writers right behind the
// pass kernel, before the count readback.
thread_local std::unordered_map<uint64_t, std::vector<std::array<long long, 3>>> t_hints;

uint64_t mix(uint64_t h, long long v) {
  h ^= (uint64_t)v;
  return h * 0x100000001B3ull;
}

// Runs n chains of passes over one source in one cooperative launch and
// writes one output batch per chain (outs[c]).  A front-end source (ijk or
// leaves) takes exactly one chain.
tb_status run(const Source& src, const std::vector<std::vector<PassSpec>>& chains, const tb_allocator* alloc,
              cudaStream_t stream, tb_batch** outs) {
  const int n_chain = (int)chains.size();
  if (!outs) return fail(TB_ERR_INVALID_ARG, "out is NULL");
  for (int ch = 0; ch < n_chain; ++ch) outs[ch] = nullptr;
  if (alloc && (!alloc->alloc || !alloc->free)) return fail(TB_ERR_INVALID_ARG, "allocator without alloc/free");
  if (n_chain == 0) return fail(TB_ERR_INVALID_ARG, "no chains");
  for (const auto& c : chains)
    if (c.empty()) return fail(TB_ERR_INVALID_ARG, "a chain without passes");
  const auto t_entry = std::chrono::steady_clock::now();
  int dev = 0;
  TB_CUDA(cudaGetDevice(&dev));
  DeviceInfo* di = nullptr;
  tb_status st = device_info(dev, &di);
  if (st != TB_OK) return st;
  const Mem mem{alloc, stream};
  const int32_t B = src.B;
  const bool front = src.kind != kSrcBatch;
  if (front && n_chain != 1) return fail(TB_ERR_INVALID_ARG, "a front end runs one chain");
  const size_t rb_bytes = readback_bytes(B);
  const size_t rb_stride = (rb_bytes + 255) & ~(size_t)255;
  const int G = di->sms * di->occ_chain;  // every co-resident block

  // ---- bounds of every pass (host-known, no readback)
  std::vector<std::vector<PassPlan>> plans(n_chain);
  int n_stage = 0;
  for (int ch = 0; ch < n_chain; ++ch) {
    plans[ch].resize(chains[ch].size());
    n_stage = std::max(n_stage, (int)chains[ch].size());
    long long cap = src.count;
    for (size_t p = 0; p < chains[ch].size(); ++p) {
      PassPlan& pl = plans[ch][p];
      pl.spec = chains[ch][p];
      pl.in_cap = cap;
      const int cbits = pass_code_bits(pl.spec.op, pl.spec.factor);
      if (pl.spec.op != kIjk && cap >= (1ll << (32 - cbits)))
        return fail(TB_ERR_TOO_LARGE, "pass %zu: %lld source leaves exceed the limit of 2^%d", p, cap, 32 - cbits);
      pl.slot_cap = cap * slots_per_source(pl.spec);
      if (pl.slot_cap >= (1ll << 30))
        return fail(TB_ERR_TOO_LARGE, "pass %zu: up to %lld candidate leaves exceed the limit of 2^30", p,
                    pl.slot_cap);
      cap = pl.slot_cap;
    }
  }

  // ---- launch shape: a member launch (one cluster per grid of every chain)
  // where every grid is small, else the whole-grid kernel
  const bool off_on_host = front && src.offsets && !device_accessible(src.offsets);
  int cl = 0;
  {
    long long nmax = -1, mmax = 1;
    const int64_t* hoff = src.kind == kSrcBatch ? src.batch->leaf_offsets_host.data()
                                                : (off_on_host ? src.offsets : nullptr);
    if (hoff && B > 0) {
      nmax = 0;
      for (int32_t g = 0; g < B; ++g) nmax = std::max<long long>(nmax, hoff[g + 1] - hoff[g]);
    }
    bool heavy = false, refine_only = !front;
    for (const auto& pc : plans)
      for (const auto& pl : pc) {
        if (src.count > 0) mmax = std::max(mmax, pl.slot_cap / src.count);
        heavy |= pl.spec.op == kRefineDilate;
        refine_only &= pl.spec.op == kRefine;
      }
    cl = member_ctas(n_chain, B, src.count, nmax, mmax, di->member_fit, front, heavy, refine_only);
  }
  const int32_t B_key = cl ? 1 : B;  // a member's keys have no grid field

  // ---- key layouts (front ends: planned in the pass kernel from the input bbox)
  for (auto& pc : plans) {
    if (!front) {
      st = plan_layouts(pc, B_key, src.batch->bbox, src.batch->L == 0);
      if (st != TB_OK) return st;
    } else {
      for (auto& pl : pc) pl.P = kMaxDigitPasses;  // buffers sized for the widest key
    }
  }

  // ---- node path: passes of the whole-grid kernel whose output lower nodes
  // are bounded by kNodeCap (the bound follows the source's lower nodes
  // through the chain; a front end's is its source count)
  for (auto& pc : plans) {
    const long long base = src.kind == kSrcBatch ? std::max<long long>(src.batch->NL, 1) : std::max(src.count, 1ll);
    long long span[3] = {1, 1, 1};  // per axis, the nodes one source node reaches through the chain so far
    for (auto& pl : pc) {
      long long f = 1;
      for (int ax = 0; ax < 3; ++ax) {
        span[ax] = std::min(node_span(pl.spec, ax, span[ax]), 1ll << 20);
        f *= span[ax];
      }
      long long bound = base > pl.slot_cap / f ? pl.slot_cap : std::min(pl.slot_cap, base * f);
      bound = std::max(bound, 1ll);
      pl.node_bound = bound;
      pl.node = !cl && g_node_mode.load() == 0 && bound <= kNodeCap;
      if (pl.node) {
        pl.node_zero = pl.spec.op == kRefine ? 0 : (pl.slot_cap * 64 <= kNodeClearInline ? 1 : 2);
        pl.mid = pl.node_zero == 2 ? 3 : 2;
        pl.node_cap = (int)bound;
        uint32_t h = 64;  // ids are table slots: room for the bound with probes to spare
        while (h < (uint32_t)bound + (uint32_t)bound / 4u + 16u) h <<= 1;
        pl.node_hslots = h;
      } else {
        pl.mid = pl.P;
      }
    }
  }

  // ---- workspace: a zeroed control region (the call's error word and the
  // last passes' readback blocks first, so one copy reads them all), then the
  // slot buffers of every chain
  Carve c;
  const size_t o_err = c.take(256);
  std::vector<size_t> o_rb_last(n_chain);
  for (int ch = 0; ch < n_chain; ++ch) o_rb_last[ch] = c.take(rb_stride);
  const size_t readback_span = c.off;
  const size_t o_bar = c.take(sizeof(GridBarrier));
  const size_t o_done = c.take((size_t)n_chain * 4);  // finished members of each chain
  const size_t o_exit = c.take(16);                   // CTAs (or chains) out of the pass kernel
  const long long total = src.count;  // stage-0 sources of the call
  for (int ch = 0; ch < n_chain; ++ch)
    for (size_t p = 0; p < plans[ch].size(); ++p) {
      PassPlan& pl = plans[ch][p];
      if (cl) {  // members: the chain's readback block; their own control is carved below
        pl.rb = o_rb_last[ch];
        continue;
      }
      // status words for full tiles, or one short tile per block of a small pass
      pl.sort_tiles = std::max({1ll, (pl.slot_cap + kSortTile - 1) / kSortTile,
                                std::min<long long>(G, (pl.slot_cap + 255) / 256)});
      pl.dedup_tiles = std::max(1ll, (pl.slot_cap + kDedupTile - 1) / kDedupTile);
      pl.rb = p + 1 == plans[ch].size() ? o_rb_last[ch] : c.take(rb_bytes);
      pl.ctl = c.take(sizeof(PassCtl));
      pl.sort_status = c.take(pl.node ? 0 : (size_t)pl.P * pl.sort_tiles * kBins * 4);
      pl.dedup_status = c.take(pl.node ? 0 : (size_t)pl.dedup_tiles * 3 * 8);
      pl.first = c.take((size_t)3 * B * 4);
      if (pl.node) {  // the node tables that start empty
        pl.nh_key = c.take((size_t)pl.node_hslots * 8);
        pl.th_key = c.take((size_t)pl.node_hslots * 8);
        pl.node_mask = c.take((size_t)pl.node_hslots * 512);
        pl.gmin = c.take((size_t)2 * B * 4);
      }
    }
  size_t n_pass_total = 0;
  for (auto& pc : plans) n_pass_total += pc.size();
  const size_t o_ts = c.take(t_prof >= 2 ? n_pass_total * 8 * sizeof(unsigned long long) : 0);
  const size_t zero_bytes = c.off;
  // member launches: control blocks and status words per member and pass,
  // carved from the grids' source offsets and zeroed by the members
  const long long ctl_rb_bytes = (long long)((readback_bytes(1) + 15) & ~(size_t)15);
  if (cl)
    for (int ch = 0; ch < n_chain; ++ch)
      for (size_t p = 0; p < plans[ch].size(); ++p) {
        PassPlan& pl = plans[ch][p];
        const long long M = pl.slot_cap / total;
        pl.ctl_stride = (ctl_rb_bytes + (long long)offsetof(PassCtl, hist) + (long long)pl.P * kBins * 4 + 16 + 63) &
                        ~63ll;
        pl.unit_ctl = c.take((size_t)B * (size_t)pl.ctl_stride);
        pl.sort_status = c.take((size_t)member_first(total, M, kSortTile, cl, B) * pl.P * kBins * 4);
        pl.dedup_status = c.take((size_t)member_first(total, M, kDedupTile, 0, B) * 3 * 8);
      }
  struct ChainBufs {
    size_t keys0, keys1, vals0, vals1, run, llow, lup, voff, pop, lg, blk, grp, inter[2][3];
    long long m_slots, m_out[2];  // member launches: capacities per stage-0 source
  };
  std::vector<ChainBufs> cb(n_chain);
  for (int ch = 0; ch < n_chain; ++ch) {
    // merged leaves of pass p go to inter[p & 1]: the next pass's source, or
    // the last pass's staged records
    long long max_slots = 0, max_inter[2] = {0, 0};
    for (size_t p = 0; p < plans[ch].size(); ++p) {
      max_slots = std::max(max_slots, plans[ch][p].slot_cap);
      max_inter[p & 1] = std::max(max_inter[p & 1], plans[ch][p].slot_cap);
    }
    const long long last_slots = plans[ch].back().slot_cap;
    ChainBufs& b = cb[ch];
    b.keys0 = c.take((size_t)max_slots * 8);
    b.keys1 = c.take((size_t)max_slots * 8);
    b.vals0 = c.take((size_t)max_slots * 4);
    b.vals1 = c.take((size_t)max_slots * 4);
    // members index the per-leaf arrays like their slots; each adds one run sentinel
    const long long leaf_slots = cl ? max_slots : last_slots;
    const long long aggs = cl ? (long long)B * cl : G;
    b.run = c.take((size_t)(max_slots + 1 + (cl ? B : 0)) * 4);
    b.llow = c.take((size_t)leaf_slots * 4);
    b.lup = c.take((size_t)leaf_slots * 4);
    b.voff = c.take((size_t)leaf_slots * 8);
    b.pop = c.take((size_t)leaf_slots * 4);
    b.lg = c.take((size_t)leaf_slots * 4);
    b.blk = c.take((size_t)aggs * 8);
    b.grp = c.take((size_t)aggs * 32 * 8);
    b.m_slots = total > 0 ? max_slots / total : 0;
    b.m_out[0] = total > 0 ? max_inter[0] / total : 0;
    b.m_out[1] = total > 0 ? max_inter[1] / total : 0;
    for (int k = 0; k < 2; ++k) {
      b.inter[k][0] = c.take((size_t)max_inter[k] * 12);
      b.inter[k][1] = c.take((size_t)max_inter[k] * 64);
      b.inter[k][2] = c.take((size_t)max_inter[k] * 4);
    }
  }
  for (auto& pc : plans)
    for (auto& pl : pc)
      if (pl.node) {
        const size_t hs = (size_t)pl.node_hslots;
        pl.node_key = c.take(hs * 8);
        pl.node_lc = c.take(hs * 16);
        pl.node_tile = c.take(hs * 4);
        pl.node_rank = c.take(hs * 4);
        pl.node_wpre = c.take(hs * 256);
        pl.rank_cnt = c.take((size_t)pl.node_cap * 4);
        pl.tile_rank = c.take(hs * 4);
        pl.node_list = c.take((size_t)pl.node_cap * 4);
        pl.tile_list = c.take((size_t)pl.node_cap * 4);
        pl.nref = c.take((size_t)pl.slot_cap * 4);
      }
  const size_t o_args = c.take(sizeof(PassArgs) * (size_t)n_chain * n_stage);
  // staging of host-resident inputs
  const int32_t* in_ijk = src.ijk;
  const int32_t* in_orig = src.origins;
  const uint64_t* in_mask = src.masks;
  const int64_t* in_off = src.offsets;
  size_t o_st_a = 0, o_st_b = 0, o_st_off = 0;
  bool st_a = false, st_b = false, st_off = false;
  if (src.kind == kSrcIjk) {
    st_a = src.count > 0 && !device_accessible(src.ijk);
    if (st_a) o_st_a = c.take((size_t)src.count * 12);
  } else if (src.kind == kSrcLeaves) {
    st_a = src.count > 0 && !device_accessible(src.origins);
    st_b = src.count > 0 && !device_accessible(src.masks);
    if (st_a) o_st_a = c.take((size_t)src.count * 12);
    if (st_b) o_st_b = c.take((size_t)src.count * 64);
  }
  if (front) {
    st_off = off_on_host;
    if (st_off) o_st_off = c.take((size_t)(B + 1) * 8);
  }
  const size_t ws_bytes = c.off;
  const auto t_alloc = std::chrono::steady_clock::now();
  char* ws = (char*)mem.get(ws_bytes);
  const auto t_alloced = std::chrono::steady_clock::now();
  if (!ws && ws_bytes) return fail(TB_ERR_OOM, "workspace allocation of %zu bytes failed", ws_bytes);
  Guard ws_guard{&mem, ws};
  TB_CUDA(cudaMemsetAsync(ws, 0, zero_bytes, stream));
  if (st_a) {
    void* d = ws + o_st_a;
    TB_CUDA(cudaMemcpyAsync(d, src.kind == kSrcIjk ? (const void*)src.ijk : (const void*)src.origins,
                            (size_t)src.count * 12, cudaMemcpyDefault, stream));
    if (src.kind == kSrcIjk) in_ijk = (const int32_t*)d;
    else in_orig = (const int32_t*)d;
  }
  if (st_b) {
    TB_CUDA(cudaMemcpyAsync(ws + o_st_b, src.masks, (size_t)src.count * 64, cudaMemcpyDefault, stream));
    in_mask = (const uint64_t*)(ws + o_st_b);
  }
  if (st_off) {
    TB_CUDA(cudaMemcpyAsync(ws + o_st_off, src.offsets, (size_t)(B + 1) * 8, cudaMemcpyDefault, stream));
    in_off = (const int64_t*)(ws + o_st_off);
  }
  // pinned host memory: readback span | phase stamps | pass arguments
  const size_t args_bytes = sizeof(PassArgs) * (size_t)n_chain * n_stage;
  const size_t ts_bytes = t_prof >= 2 ? n_pass_total * 64 : 0;
  char* pinned = (char*)t_pinned.get(readback_span + ts_bytes + args_bytes + 64);
  if (!pinned) return fail(TB_ERR_OOM, "pinned host buffer failed");
  unsigned int* host_flag = (unsigned int*)(pinned + readback_span + ts_bytes + args_bytes);
  const bool flagged = t_prof < 2;  // profiling reads its stamps through the stream
  unsigned long long* host_ts = (unsigned long long*)(pinned + readback_span);
  PassArgs* host_args = (PassArgs*)(pinned + readback_span + ts_bytes);
  const ReadbackHeader* host_rb0 = (const ReadbackHeader*)(pinned + o_rb_last[0]);

  // ---- pass arguments, [chain][stage], copied to the device
  size_t pass_index = 0;
  std::vector<int> pass_stage;
  for (int ch = 0; ch < n_chain; ++ch) {
    const ChainBufs& bf = cb[ch];
    for (int k = 0; k < n_stage; ++k) {
      PassArgs& a = host_args[(size_t)ch * n_stage + k];
      std::memset(&a, 0, sizeof a);
      a.op = -1;
      if (k >= (int)plans[ch].size()) continue;
      const PassPlan& pl = plans[ch][k];
      a.K = pl.K;
      a.op = pl.spec.op;
      a.B = B;
      a.P = pl.node ? 0 : pl.P;
      a.mid = pl.mid;
      if (pl.node) {
        a.node = 1;
        a.node_zero = pl.node_zero;
        a.node_cap = pl.node_cap;
        a.node_hmask = pl.node_hslots - 1u;
        a.nh_key = (unsigned long long*)(ws + pl.nh_key);
        a.th_key = (unsigned long long*)(ws + pl.th_key);
        a.node_mask = (uint64_t*)(ws + pl.node_mask);
        a.gmin = (uint32_t*)(ws + pl.gmin);
        a.node_key = (uint64_t*)(ws + pl.node_key);
        a.node_lc = (int32_t*)(ws + pl.node_lc);
        a.node_tile = (uint32_t*)(ws + pl.node_tile);
        a.node_rank = (uint32_t*)(ws + pl.node_rank);
        a.node_wpre = (uint32_t*)(ws + pl.node_wpre);
        a.rank_cnt = (uint32_t*)(ws + pl.rank_cnt);
        a.tile_rank = (uint32_t*)(ws + pl.tile_rank);
        a.node_list = (uint32_t*)(ws + pl.node_list);
        a.tile_list = (uint32_t*)(ws + pl.tile_list);
        a.nref = (uint32_t*)(ws + pl.nref);
      }
      a.last = k + 1 == (int)plans[ch].size();
      {  // targets per emission thread: about one round of the grid's threads
        // (the node path: about four rounds, so the grid's blocks finish together)
        const long long T = slots_per_source(pl.spec);
        const long long want = (pl.in_cap * T + (long long)G * 256 - 1) / ((long long)G * 256);
        a.tchunk = (int32_t)std::max(1ll, std::min({T, want, 32ll}));
        if (pl.node) {
          const long long chunks = std::max(1ll, std::min(T, (4ll * G * 256 + pl.in_cap - 1) / std::max(1ll, pl.in_cap)));
          a.tchunk = (int32_t)std::max(1ll, std::min(32ll, (T + chunks - 1) / chunks));
        }
      }
      for (int ax = 0; ax < 3; ++ax) {
        a.lo[ax] = pl.spec.lo[ax];
        a.hi[ax] = pl.spec.hi[ax];
      }
      a.factor = pl.spec.factor;
      a.code_bits = pass_code_bits(pl.spec.op, pl.spec.factor);
      if (k == 0) {
        a.ijk = in_ijk;
        a.in_offsets = in_off;
        if (src.kind == kSrcBatch) {
          a.src_origins = src.batch->origins;
          a.src_masks = src.batch->masks;
          a.src_grid = src.batch->leaf_grid;
          a.src_count = src.batch->L;
        } else {
          a.src_origins = in_orig;
          a.src_masks = in_mask;
          a.src_count = src.count;
        }
      } else {
        const PassArgs& prev = host_args[(size_t)ch * n_stage + k - 1];
        a.src_origins = prev.out_origins;
        a.src_masks = prev.out_masks;
        a.src_grid = prev.out_grid;
        a.src_count_dev = &prev.rb->num_leaves;
      }
      a.err = (unsigned int*)(ws + o_err);
      a.rb = (ReadbackHeader*)(ws + pl.rb);
      a.leaf_off = (int64_t*)(ws + pl.rb + sizeof(ReadbackHeader));
      a.lower_off = a.leaf_off + (B + 1);
      a.upper_off = a.lower_off + (B + 1);
      a.grid_vox = a.upper_off + (B + 1);
      a.gbox = (unsigned int*)(a.grid_vox + B);
      a.ctl = (PassCtl*)(ws + pl.ctl);
      a.sort_status = (uint32_t*)(ws + pl.sort_status);
      a.sort_tiles_cap = pl.sort_tiles;
      a.dedup_status = (unsigned long long*)(ws + pl.dedup_status);
      a.first = (uint32_t*)(ws + pl.first);
      a.slot_cap = pl.slot_cap;
      a.keys[0] = (uint64_t*)(ws + bf.keys0);
      a.keys[1] = (uint64_t*)(ws + bf.keys1);
      a.vals[0] = (uint32_t*)(ws + bf.vals0);
      a.vals[1] = (uint32_t*)(ws + bf.vals1);
      a.sorted = pl.P & 1;
      a.run_start = (uint32_t*)(ws + bf.run);
      a.leaf_lower = (uint32_t*)(ws + bf.llow);
      a.leaf_upper = (uint32_t*)(ws + bf.lup);
      a.leaf_voff = (int64_t*)(ws + bf.voff);
      a.leaf_pop = (uint32_t*)(ws + bf.pop);
      a.leaf_g = (uint32_t*)(ws + bf.lg);
      a.blk_agg = (unsigned long long*)(ws + bf.blk);
      a.grp_agg = (unsigned long long*)(ws + bf.grp);
      a.phase_ts = t_prof >= 2 ? (unsigned long long*)(ws + o_ts) + 8 * pass_index : nullptr;
      ++pass_index;
      pass_stage.push_back(k);
      a.out_origins = (int32_t*)(ws + bf.inter[k & 1][0]);
      a.out_masks = (uint64_t*)(ws + bf.inter[k & 1][1]);
      a.out_grid = (int32_t*)(ws + bf.inter[k & 1][2]);
      if (cl) {  // a member template (see PassArgs)
        a.member = 1;
        a.cl = cl;
        a.unit_off = src.kind == kSrcBatch ? src.batch->leaf_offsets : in_off;
        a.m_stage = pl.slot_cap / total;
        a.m_slots = bf.m_slots;
        a.m_out = bf.m_out[k & 1];
        a.unit_ctl = ws + pl.unit_ctl;
        a.ctl_stride = pl.ctl_stride;
        a.ctl_rb_bytes = ctl_rb_bytes;
        a.ctl = nullptr;
        a.first = nullptr;
        const long long T = slots_per_source(pl.spec), mean = (total + B - 1) / B;
        const long long want = (mean * a.m_stage + (long long)cl * 256 - 1) / ((long long)cl * 256);
        a.tchunk = (int32_t)std::max(1ll, std::min({T, want, 32ll}));
      }
    }
  }
  TB_CUDA(cudaMemcpyAsync(ws + o_args, host_args, args_bytes, cudaMemcpyHostToDevice, stream));

  // ---- the cooperative pass kernel
  {
    ChainArgs ca{};
    ca.pass = (const PassArgs*)(ws + o_args);
    ca.n_chain = n_chain;
    ca.n_stage = n_stage;
    ca.bar = (GridBarrier*)(ws + o_bar);
    ca.err = (unsigned int*)(ws + o_err);
    ca.front = front ? 1 : 0;  // the kernel reads the input's bbox and plans the key itself
    if (flagged) {
      __atomic_store_n(host_flag, 0u, __ATOMIC_RELAXED);
      ca.host_span = pinned;
      ca.dev_span = ws;
      ca.span_bytes = (long long)readback_span;
      ca.exit_ctr = (unsigned int*)(ws + o_exit);
      ca.host_flag = host_flag;
      ca.seq = ++t_seq;
    }
    if (cl) {
      ca.B = B;
      ca.cl = cl;
      ca.done = (unsigned int*)(ws + o_done);
      TB_CUDA(launch(kKMember, stream, [&] { return launch_member(ca, n_chain * B, cl, stream); }));
    } else {
      TB_CUDA(launch(kKChain, stream, [&] { return launch_chain(ca, G, stream); }));
    }
  }

  // ---- outputs.  With the counts of the last call of the same shape, the
  // outputs are allocated now with room to spare and the writers queued
  // behind the pass kernel; a writer skips a chain that outgrew its room,
  // and that chain is written again after the readback.
  std::vector<tb_batch*> made(n_chain, nullptr);
  auto undo = [&] {
    for (tb_batch*& b : made)
      if (b) {
        mem.put(b->mem);
        delete b;
        b = nullptr;
      }
  };
  // a batch with arrays for L, NL, NU (counts or room)
  auto new_batch = [&](long long L, long long NL, long long NU) -> tb_batch* {
    tb_batch* b = new tb_batch();
    b->B = B;
    b->device = dev;
    b->L = L;
    b->NL = NL;
    b->NU = NU;
    b->has_alloc = alloc != nullptr;
    if (alloc) b->alloc = *alloc;
    if (alloc_outputs(b, mem) != TB_OK) {
      delete b;
      return nullptr;
    }
    return b;
  };
  // the writers of some chains: one launch for a one-chain call, else one per
  // kMaxWriteTasks chains with the tasks in its parameter
  auto launch_writers = [&](const std::vector<int>& chs) -> cudaError_t {
    if (n_chain == 1) {
      WriteOut wo;
      fill_write_out(made[0], wo);
      const int op_last = plans[0].back().spec.op;
      const int wb = blocks_for(std::max<long long>(wo.L_cap, B + 1), kWriteLeavesPerBlock,
                                (long long)di->sms * di->occ_write[op_last]);
      const PassArgs& a = host_args[plans[0].size() - 1];
      return launch(kKWrite0 + op_last, stream, [&] { return launch_write_final(op_last, a, wo, wb, stream); });
    }
    WriteTasks wt;
    for (size_t c0 = 0; c0 < chs.size(); c0 += kMaxWriteTasks) {
      const int nt = (int)std::min<size_t>(kMaxWriteTasks, chs.size() - c0);
      long long room = 0;
      std::memset(&wt, 0, sizeof wt);
      wt.n = nt;
      for (int j = 0; j < nt; ++j) {
        const int ch = chs[c0 + j];
        wt.t[j].a = host_args[(size_t)ch * n_stage + plans[ch].size() - 1];
        fill_write_out(made[ch], wt.t[j].o);
        room += (wt.t[j].o.L_cap + 3) / 4 * 4;
      }
      const int wb = blocks_for(std::max<long long>(room, B + 1), kWriteLeavesPerBlock,
                                (long long)di->sms * di->occ_write_multi);
      const cudaError_t e = launch(kKWriteMulti, stream, [&] { return launch_write_multi(wt, wb, stream); });
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  };
  uint64_t shape = mix(mix(mix(mix(0xCBF29CE484222325ull, src.kind), B), src.count), n_chain);
  for (const auto& pc : plans)
    for (const auto& pl : pc) {
      shape = mix(mix(mix(shape, pl.spec.op), pl.spec.factor), pc.size());
      for (int a = 0; a < 3; ++a) shape = mix(mix(shape, pl.spec.lo[a]), pl.spec.hi[a]);
    }
  std::vector<char> ahead(n_chain, 0);  // outputs allocated and written before the readback
  {
    const auto h = t_hints.find(shape);
    if (h != t_hints.end() && h->second.size() == (size_t)n_chain) {
      bool ok = true;
      for (int ch = 0; ch < n_chain && ok; ++ch) {
        const auto& c = h->second[ch];
        made[ch] = new_batch(c[0] + c[0] / 8 + 16, c[1] + c[1] / 8 + 4, c[2] + c[2] / 8 + 2);
        ok = made[ch] != nullptr;
      }
      std::vector<int> all(n_chain);
      for (int ch = 0; ch < n_chain; ++ch) all[ch] = ch;
      if (ok && launch_writers(all) == cudaSuccess) {
        for (int ch = 0; ch < n_chain; ++ch) ahead[ch] = 1;
      } else {
        cudaGetLastError();
        undo();
      }
    }
  }
  // every return from here on without outputs frees the batches made so far
  struct Release {
    decltype(undo)& f;
    bool armed = true;
    ~Release() {
      if (armed) f();
    }
  } release{undo};

  // ---- the one count readback of the call: the kernel's copy to pinned
  // memory, seen through the host flag; else (profiling, or a kernel that
  // stopped early) through the stream
  const auto t_sync = std::chrono::steady_clock::now();
  if (flagged) {
    const unsigned int seq = t_seq;
    bool seen = false;
    for (unsigned int it = 1;; ++it) {
      if (__atomic_load_n(host_flag, __ATOMIC_ACQUIRE) == seq) {
        seen = true;
        break;
      }
      if ((it & 63u) == 0 && cudaStreamQuery(stream) != cudaErrorNotReady) {
        seen = __atomic_load_n(host_flag, __ATOMIC_ACQUIRE) == seq;
        break;
      }
    }
    if (!seen) {
      TB_CUDA(cudaStreamSynchronize(stream));
      TB_CUDA(cudaMemcpy(pinned, ws, readback_span, cudaMemcpyDeviceToHost));
    }
  } else {
    if (t_prof >= 2) TB_CUDA(cudaMemcpyAsync(host_ts, ws + o_ts, ts_bytes, cudaMemcpyDeviceToHost, stream));
    TB_CUDA(cudaMemcpyAsync(pinned, ws, readback_span, cudaMemcpyDeviceToHost, stream));
    TB_CUDA(cudaStreamSynchronize(stream));
  }
  const auto t_synced = std::chrono::steady_clock::now();
  if (t_prof >= 2) {
    t_phase_ms[6] += std::chrono::duration<double, std::milli>(t_sync - t_entry).count();
    t_phase_ms[7] += std::chrono::duration<double, std::milli>(t_synced - t_sync).count();
    t_phase_n[6] += 1;
    t_phase_n[7] += 1;
    t_phase_ms[9] += std::chrono::duration<double, std::milli>(t_alloc - t_entry).count();
    t_phase_ms[10] += std::chrono::duration<double, std::milli>(t_alloced - t_alloc).count();
    t_phase_n[9] += 1;
    t_phase_n[10] += 1;
    // kernel entry (the first pass's slot 6, earliest block) to the first emission
    if (n_pass_total && host_ts[6] && ~host_ts[6] <= ~host_ts[0]) {
      t_phase_ms[5] += (double)(~host_ts[0] - ~host_ts[6]) * 1e-6;
      t_phase_n[5] += 1;
    }
    // phase j of stage k spans, over the chains' passes of the stage, from the
    // latest end of phase j-1 (the earliest start for j = 0) to the latest end
    for (int k = 0; k < n_stage; ++k)
      for (int j = 0; j < kNumGpuPhases; ++j) {
        unsigned long long t0 = j == 0 ? ~0ull : 0ull, t1 = 0;
        for (size_t p = 0; p < n_pass_total; ++p) {
          if (pass_stage[p] != k) continue;
          const unsigned long long s = j == 0 ? ~host_ts[8 * p] : host_ts[8 * p + j];
          t0 = j == 0 ? std::min(t0, s) : std::max(t0, s);
          t1 = std::max(t1, host_ts[8 * p + j + 1]);
        }
        if (t1 >= t0 && t0 && t0 != ~0ull) {
          t_phase_ms[j] += (double)(t1 - t0) * 1e-6;
          t_phase_n[j] += 1;
        }
      }
  }
  const unsigned int err = *(const unsigned int*)(pinned + o_err);
  if (err & kErrTimeout) return fail(TB_ERR_DEVICE_TIMEOUT, "a device-side wait timed out");
  if (err & kErrSlotOverflow) return fail(TB_ERR_INTERNAL, "internal: emitted slots exceeded the bound");
  if (front) {  // the layout the kernel planned, again on the host, for the batch and the writer
    if (err & kErrBadOffsets)
      return fail(TB_ERR_INVALID_ARG, "offsets must start at 0, be non-decreasing and end at %lld", src.count);
    if (err & kErrNotAligned) return fail(TB_ERR_INVALID_ARG, "leaf origins must be multiples of 8");
    int32_t bb[6];
    for (int a = 0; a < 3; ++a) {
      bb[a] = dec_min(host_rb0->bbox_enc[a]);
      bb[3 + a] = dec_max(host_rb0->bbox_enc[3 + a]);
    }
    st = plan_layouts(plans[0], B_key, bb, bb[0] > bb[3]);
    if (st != TB_OK) return st;
    if (err & kErrLayout) return fail(TB_ERR_CUDA, "internal: device and host key layouts disagree");
    PassArgs& a0 = host_args[0];
    a0.K = plans[0][0].K;
    a0.P = plans[0][0].P;
    a0.sorted = a0.P & 1;
  }

  // ---- each chain's batch: the one written ahead if its counts fit its
  // room, else a batch of the exact size written now
  std::vector<int> redo;
  std::vector<std::array<long long, 3>> counts(n_chain);
  for (int ch = 0; ch < n_chain; ++ch) {
    const PassPlan& last = plans[ch].back();
    const ReadbackHeader* hr = (const ReadbackHeader*)(pinned + o_rb_last[ch]);
    const int64_t L = (int64_t)hr->num_leaves, NL = (int64_t)hr->num_lowers, NU = (int64_t)hr->num_uppers;
    counts[ch] = {L, NL, NU};
    const int64_t* hoff = (const int64_t*)(hr + 1);
    tb_batch* b = made[ch];
    if (!(b && ahead[ch] && L <= b->L && NL <= b->NL && NU <= b->NU)) {
      if (b) {
        mem.put(b->mem);  // stream-ordered after the writer, which skipped it
        delete b;
        made[ch] = nullptr;
      }
      b = new_batch(L, NL, NU);
      if (!b) {
        undo();
        return fail(TB_ERR_OOM, "output allocation failed");
      }
      made[ch] = b;
      redo.push_back(ch);
    }
    b->L = L;
    b->NL = NL;
    b->NU = NU;
    // arrays of no elements read as NULL
    if (L == 0) {
      b->origins = nullptr;
      b->masks = nullptr;
      b->voxel_offset = nullptr;
      b->word_prefix = nullptr;
      b->leaf_bbox = nullptr;
      b->leaf_grid = nullptr;
      b->leaf_parent = nullptr;
    }
    if (NL == 0) {
      b->lower_origins = nullptr;
      b->lower_parent = nullptr;
    }
    if (NU == 0) b->upper_origins = nullptr;
    b->leaf_offsets_host.assign(hoff, hoff + B + 1);
    b->voxel_base_host.assign(B + 1, 0);
    for (int32_t g = 0; g < B; ++g) b->voxel_base_host[g + 1] = b->voxel_base_host[g] + hoff[3 * (B + 1) + g];
    std::memcpy(b->bbox, last.bbox, sizeof b->bbox);
    if (last.empty || L == 0) {
      const int32_t e[6] = {INT32_MAX, INT32_MAX, INT32_MAX, INT32_MIN, INT32_MIN, INT32_MIN};
      std::memcpy(b->bbox, e, sizeof e);
    }
    b->build_slots = (int64_t)hr->num_slots;
    b->build_sources = plans[ch].size() == 1 ? (int64_t)last.in_cap : -1;
    b->build_key_bits = last.K.W;
    b->build_digit_passes = last.node ? 0 : last.P;  // the node path sorts nothing
    b->build_member_ctas = cl;
  }
  if (!redo.empty()) {
    const cudaError_t e = launch_writers(redo);
    if (e != cudaSuccess) {
      undo();
      return fail(TB_ERR_CUDA, "writer launch: %s", cudaGetErrorString(e));
    }
  }
  if (t_hints.size() > 256) t_hints.clear();
  t_hints[shape] = counts;
  release.armed = false;
  for (int ch = 0; ch < n_chain; ++ch) outs[ch] = made[ch];
  if (t_prof >= 2) {
    t_phase_ms[8] += host_ms_since(t_synced);
    t_phase_n[8] += 1;
  }
  return TB_OK;
}

// The passes of a list of ops.  Consecutive ops are fused where one pass
// computes their composition exactly (the OR of the per-voxel images commutes
// with the union that dedups a pass): refinements (or coarsenings) whose
// factors multiply to at most 8, box dilations whose summed bounds stay
// within [-7, 7], and refinement by 2 followed by a box within [-1, 1]^3 --
// the last only for inputs of at most kFuseRefineDilateMax leaves: the fused
// merge does about four times the mask arithmetic per slot, which pays where
// a pass is latency-bound (saving a whole pass) and not on large inputs.
constexpr long long kFuseRefineDilateMax = 32768;

std::vector<PassSpec> expand_ops(const tb_op* ops, int32_t n, tb_status* st, long long in_leaves) {
  std::vector<PassSpec> v;
  *st = TB_OK;
  for (int32_t i = 0; i < n; ++i) {
    const tb_op& o = ops[i];
    PassSpec s;
    std::memset(&s, 0, sizeof s);
    if (o.kind == TB_OP_REFINE || o.kind == TB_OP_COARSEN) {
      if (o.factor != 2 && o.factor != 4 && o.factor != 8) {
        *st = fail(TB_ERR_INVALID_ARG, "op %d: factor %d is not 2, 4 or 8", i, o.factor);
        return {};
      }
      s.op = o.kind == TB_OP_REFINE ? kRefine : kCoarsen;
      s.factor = o.factor;
    } else if (o.kind == TB_OP_BOX_DILATE) {
      s.op = kDilate;
      for (int a = 0; a < 3; ++a) {
        if (o.lo[a] < -7 || o.lo[a] > 0 || o.hi[a] < 0 || o.hi[a] > 7) {
          *st = fail(TB_ERR_INVALID_ARG, "op %d: box bounds must be lo in [-7,0], hi in [0,7]", i);
          return {};
        }
        s.lo[a] = o.lo[a];
        s.hi[a] = o.hi[a];
      }
    } else {
      *st = fail(TB_ERR_INVALID_ARG, "op %d: unknown kind %d", i, o.kind);
      return {};
    }
    if (!v.empty()) {
      PassSpec& p = v.back();
      if ((p.op == kRefine || p.op == kCoarsen) && s.op == p.op && p.factor * s.factor <= 8) {
        p.factor *= s.factor;
        continue;
      }
      if (p.op == kDilate && s.op == kDilate) {
        bool fits = true;
        for (int a = 0; a < 3; ++a) fits &= p.lo[a] + s.lo[a] >= -7 && p.hi[a] + s.hi[a] <= 7;
        if (fits) {
          for (int a = 0; a < 3; ++a) {
            p.lo[a] += s.lo[a];
            p.hi[a] += s.hi[a];
          }
          continue;
        }
      }
      if (p.op == kRefine && p.factor == 2 && s.op == kDilate && in_leaves <= kFuseRefineDilateMax) {
        bool unit = true;
        for (int a = 0; a < 3; ++a) unit &= s.lo[a] >= -1 && s.hi[a] <= 1;
        if (unit) {
          p.op = kRefineDilate;
          for (int a = 0; a < 3; ++a) {
            p.lo[a] = s.lo[a];
            p.hi[a] = s.hi[a];
          }
          continue;
        }
      }
    }
    v.push_back(s);
  }
  return v;
}

tb_status check_batch(const tb_batch* b) {
  if (!b) return fail(TB_ERR_INVALID_ARG, "batch is NULL");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(TB_ERR_CUDA, "cudaGetDevice failed");
  if (dev != b->device) return fail(TB_ERR_INVALID_ARG, "batch lives on device %d, current device is %d", b->device, dev);
  return TB_OK;
}

tb_status run_ops(const tb_batch* in, const std::vector<std::vector<PassSpec>>& chains, const tb_allocator* alloc,
                  cudaStream_t s, tb_batch** outs) {
  tb_status st = check_batch(in);
  if (st != TB_OK) return st;
  Source src;
  src.kind = kSrcBatch;
  src.batch = in;
  src.B = in->B;
  src.count = in->L;
  return run(src, chains, alloc, s, outs);
}

// The passes of one chain of ops; an empty chain copies its input (one
// identity pass over the leaves).
tb_status chain_specs(const tb_op* ops, int32_t n_ops, std::vector<PassSpec>* specs, long long in_leaves) {
  tb_status st;
  *specs = expand_ops(ops, n_ops, &st, in_leaves);
  if (st != TB_OK) return st;
  if (specs->empty()) {
    PassSpec s;
    std::memset(&s, 0, sizeof s);
    s.op = kLeaves;
    specs->push_back(s);
  }
  return TB_OK;
}

}  // namespace

void tb::set_error_message(const char* msg) { t_err = msg; }

// ================================================================ C ABI

extern "C" {

tb_status tb_from_ijk(const int32_t* ijk, const int64_t* offsets, int32_t num_grids, int64_t num_voxels,
                      const tb_allocator* alloc, tb_stream stream, tb_batch** out) {
  if (out) *out = nullptr;
  if (!out || !offsets || num_grids < 0 || num_voxels < 0 || (num_voxels > 0 && !ijk))
    return fail(TB_ERR_INVALID_ARG, "tb_from_ijk: bad pointer or negative size");
  if (num_grids > (1 << 24)) return fail(TB_ERR_TOO_LARGE, "tb_from_ijk: more than 2^24 grids");
  if (num_voxels >= (1ll << 30)) return fail(TB_ERR_TOO_LARGE, "tb_from_ijk: 2^30 or more voxels");
  if (num_grids == 0 && num_voxels != 0) return fail(TB_ERR_INVALID_ARG, "tb_from_ijk: voxels without grids");
  Source src;
  src.kind = kSrcIjk;
  src.ijk = ijk;
  src.offsets = offsets;
  src.B = num_grids;
  src.count = num_voxels;
  std::vector<std::vector<PassSpec>> chains(1, std::vector<PassSpec>(1));
  std::memset(&chains[0][0], 0, sizeof(PassSpec));
  chains[0][0].op = kIjk;
  return run(src, chains, alloc, (cudaStream_t)stream, out);
}

tb_status tb_from_leaves(const int32_t* origins, const uint64_t* masks, const int64_t* leaf_offsets,
                         int32_t num_grids, int64_t num_leaves, const tb_allocator* alloc, tb_stream stream,
                         tb_batch** out) {
  if (out) *out = nullptr;
  if (!out || !leaf_offsets || num_grids < 0 || num_leaves < 0 || (num_leaves > 0 && (!origins || !masks)))
    return fail(TB_ERR_INVALID_ARG, "tb_from_leaves: bad pointer or negative size");
  if (num_grids > (1 << 24)) return fail(TB_ERR_TOO_LARGE, "tb_from_leaves: more than 2^24 grids");
  if (num_leaves >= (1ll << 27)) return fail(TB_ERR_TOO_LARGE, "tb_from_leaves: 2^27 or more leaves");
  if (num_grids == 0 && num_leaves != 0) return fail(TB_ERR_INVALID_ARG, "tb_from_leaves: leaves without grids");
  if (((uintptr_t)masks & 15) != 0) return fail(TB_ERR_INVALID_ARG, "tb_from_leaves: masks must be 16-byte aligned");
  Source src;
  src.kind = kSrcLeaves;
  src.origins = origins;
  src.masks = masks;
  src.offsets = leaf_offsets;
  src.B = num_grids;
  src.count = num_leaves;
  std::vector<std::vector<PassSpec>> chains(1, std::vector<PassSpec>(1));
  std::memset(&chains[0][0], 0, sizeof(PassSpec));
  chains[0][0].op = kLeaves;
  return run(src, chains, alloc, (cudaStream_t)stream, out);
}

tb_status tb_refine(const tb_batch* in, int32_t factor, const tb_allocator* alloc, tb_stream stream, tb_batch** out) {
  tb_op op{TB_OP_REFINE, factor, {0, 0, 0}, {0, 0, 0}};
  return tb_chain(in, &op, 1, alloc, stream, out);
}

tb_status tb_coarsen(const tb_batch* in, int32_t factor, const tb_allocator* alloc, tb_stream stream,
                     tb_batch** out) {
  tb_op op{TB_OP_COARSEN, factor, {0, 0, 0}, {0, 0, 0}};
  return tb_chain(in, &op, 1, alloc, stream, out);
}

tb_status tb_box_dilate(const tb_batch* in, const int32_t lo[3], const int32_t hi[3], const tb_allocator* alloc,
                        tb_stream stream, tb_batch** out) {
  if (out) *out = nullptr;
  if (!lo || !hi) return fail(TB_ERR_INVALID_ARG, "tb_box_dilate: lo/hi NULL");
  tb_op op{TB_OP_BOX_DILATE, 1, {lo[0], lo[1], lo[2]}, {hi[0], hi[1], hi[2]}};
  return tb_chain(in, &op, 1, alloc, stream, out);
}

tb_status tb_stride1_box(int32_t kernel_size, int32_t transpose, int32_t lo[3], int32_t hi[3]) {
  if (!lo || !hi) return fail(TB_ERR_INVALID_ARG, "tb_stride1_box: lo/hi NULL");
  if (kernel_size < 1 || kernel_size > 15)
    return fail(TB_ERR_INVALID_ARG, "tb_stride1_box: kernel size %d is outside 1..15", kernel_size);
  // [-floor((K-1)/2), ceil((K-1)/2)]: for even K the extra offset on the positive side
  int32_t l = -((kernel_size - 1) / 2), h = kernel_size / 2;
  if (transpose) {
    const int32_t t = l;
    l = -h;
    h = -t;
  }
  for (int a = 0; a < 3; ++a) {
    lo[a] = l;
    hi[a] = h;
  }
  return TB_OK;
}

tb_status tb_refine_masked(const tb_batch* in, const uint8_t* voxel_mask, int32_t factor, const tb_allocator* alloc,
                           tb_stream stream, tb_batch** out) {
  if (out) *out = nullptr;
  if (!out) return fail(TB_ERR_INVALID_ARG, "out is NULL");
  tb_status st = check_batch(in);
  if (st != TB_OK) return st;
  if (in->voxel_base_host.size() != (size_t)in->B + 1)
    return fail(TB_ERR_INVALID_ARG, "tb_refine_masked: batch without per-grid voxel counts");
  const int64_t V = in->voxel_base_host[in->B];
  if (V > 0 && !voxel_mask) return fail(TB_ERR_INVALID_ARG, "tb_refine_masked: voxel_mask is NULL");
  tb_op op{TB_OP_REFINE, factor, {0, 0, 0}, {0, 0, 0}};
  std::vector<std::vector<PassSpec>> chains(1);
  st = chain_specs(&op, 1, &chains[0], in->L);
  if (st != TB_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0;
  TB_CUDA(cudaGetDevice(&dev));
  DeviceInfo* di = nullptr;
  st = device_info(dev, &di);
  if (st != TB_OK) return st;
  // workspace: pruned masks | per-grid voxel bases | the flags, when they are host memory
  const Mem mem{alloc, s};
  const bool stage = V > 0 && !device_accessible(voxel_mask);
  Carve c;
  const size_t o_masks = c.take((size_t)in->L * 64), o_base = c.take((size_t)(in->B + 1) * 8),
               o_flags = c.take(stage ? (size_t)V : 0);
  char* ws = (char*)mem.get(c.off);
  if (!ws && c.off) return fail(TB_ERR_OOM, "tb_refine_masked: workspace of %zu bytes", c.off);
  Guard g{&mem, ws};
  const uint8_t* flags = voxel_mask;
  if (stage) {
    TB_CUDA(cudaMemcpyAsync(ws + o_flags, voxel_mask, (size_t)V, cudaMemcpyHostToDevice, s));
    flags = (const uint8_t*)(ws + o_flags);
  }
  // the voxel bases from the batch's device counts (no host copy, so the
  // host runs ahead of the stream)
  TB_CUDA(launch(kKPrune, s, [&] { return launch_voxel_bases(in->voxel_counts, in->B, (int64_t*)(ws + o_base), s); }));
  tb_batch pruned = *in;
  pruned.masks = in->L ? (uint64_t*)(ws + o_masks) : nullptr;
  if (in->L) {
    const int blocks = blocks_for(in->L, 32, (long long)di->sms * 8);
    TB_CUDA(launch(kKPrune, s, [&] {
      return launch_prune(in->masks, in->leaf_grid, in->voxel_offset, (const int64_t*)(ws + o_base), flags, in->L,
                          pruned.masks, blocks, s);
    }));
  }
  Source src;
  src.kind = kSrcBatch;
  src.batch = &pruned;
  src.B = in->B;
  src.count = in->L;
  return run(src, chains, alloc, s, out);
}

tb_status tb_kernel_map(const tb_batch* in, const tb_batch* out, const int32_t lo[3], const int32_t hi[3],
                        int32_t stride, int32_t transposed, int32_t* map, int64_t map_len, tb_stream stream) {
  tb_status st = check_batch(in);
  if (st != TB_OK) return st;
  st = check_batch(out);
  if (st != TB_OK) return st;
  if (!lo || !hi) return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: lo/hi NULL");
  if (in->B != out->B) return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: %d input grids, %d output grids", in->B, out->B);
  if (stride != 1 && stride != 2) return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: stride %d is not 1 or 2", stride);
  long long K = 1;
  for (int a = 0; a < 3; ++a) {
    if (lo[a] < -7 || hi[a] > 7 || lo[a] > hi[a])
      return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: box bounds must satisfy -7 <= lo <= hi <= 7");
    K *= hi[a] - lo[a] + 1;
  }
  if (in->voxel_base_host.size() != (size_t)in->B + 1 || out->voxel_base_host.size() != (size_t)out->B + 1)
    return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: batch without per-grid voxel counts");
  const int64_t Vin = in->voxel_base_host[in->B], Vout = out->voxel_base_host[out->B];
  if (Vin >= (1ll << 31)) return fail(TB_ERR_TOO_LARGE, "tb_kernel_map: 2^31 or more input voxels");
  if (map_len < Vout * K)
    return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: map holds %lld entries, %lld needed", (long long)map_len,
                (long long)(Vout * K));
  if (Vout > 0 && !map) return fail(TB_ERR_INVALID_ARG, "tb_kernel_map: map is NULL");
  if (out->L == 0) return TB_OK;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceInfo* di = nullptr;
  st = device_info(out->device, &di);
  if (st != TB_OK) return st;
  const Mem mem{out->has_alloc ? &out->alloc : nullptr, s};
  // workspace: the two voxel-base arrays, then a hash table of the input
  // leaves with at least twice as many slots as leaves
  const size_t nb = (size_t)(in->B + 1) * 8;
  unsigned long long cap = 64;
  while (cap < 2ull * (unsigned long long)in->L) cap <<= 1;
  // input leaves one output leaf's reach spans along an axis: origins are
  // multiples of 8, so eight residues of the origin cover every leaf
  int span = 0;
  for (int a = 0; a < 3; ++a)
    for (long long o = 0; o < 64; o += 8) {
      const int sh = stride == 2 ? 1 : 0;
      long long qlo, qhi;
      if (transposed) {
        qlo = floor_div(o - hi[a] + (1 << sh) - 1, 1ll << sh);
        qhi = floor_div(o + 7 - lo[a], 1ll << sh);
      } else {
        qlo = (o << sh) + lo[a];
        qhi = ((o + 7) << sh) + hi[a];
      }
      span = std::max(span, (int)(floor_div(qhi, 8) - floor_div(qlo, 8) + 1));
    }
  const bool staged = span <= 3 && K <= kKmapStagedColumns;
  // the tabulated reach (stride 1 or transposed): the same extents for every leaf
  long long halo = 1;
  for (int a = 0; a < 3; ++a)
    halo *= transposed ? floor_div(7 - lo[a], stride) + floor_div(hi[a], stride) + 1 : 8 + hi[a] - lo[a];
  const bool tabulable = span <= 3 && K <= kKmapTabColumns && (stride == 1 || transposed) && halo <= kKmapHaloMax;
  // measured on GB300 (L2 flushed, whole calls): the staged map wins once
  // the output has at least about 32 leaves per SM -- one leaf per warp
  // where the reach spans 3 leaves per axis (B = 48 shells k3s1, 8,164
  // leaves: 61 us against 67 us tabulated; stress batch, 83,722 leaves: 202
  // us against 381 us), chunks of 4 to 16 leaves per warp where it spans 1
  // (B = 16 k2s2 transpose, 10,547 leaves: 39 us against 45 us; B = 48: 55
  // against 100 us; stress: 145 against 747 us); below that the tabulated
  // map wins (B = 16 k3s1, 2,905 leaves: 35 us against 37 us).  The look-up
  // pass of its own measured slower than the staged map's own look-ups
  // everywhere; it stays as a form of its own.
  enum { kPerEntry, kStaged, kStagedPrepass, kTabulated } form = kPerEntry;
  switch (g_kmap_mode.load()) {
    case 0: {
      const bool many = out->L >= 32ll * di->sms;
      form = tabulable && (!many || !staged) ? kTabulated : staged ? kStaged : kPerEntry;
      break;
    }
    case 1: form = staged ? kStaged : kPerEntry; break;
    case 2: form = staged ? kStagedPrepass : kPerEntry; break;
    case 3: form = tabulable ? kTabulated : kPerEntry; break;
    default: form = kPerEntry; break;
  }
  const long long cand_max = (long long)span * span * span;
  const bool prepass = form == kStagedPrepass;
  const size_t cand_bytes = prepass ? (size_t)(out->L * cand_max) * 4 : 0;
  // workspace: the two voxel-base arrays, the leaf table, the staged map's
  // chunk counter (16 bytes), the candidates of the look-up pass
  char* ws = (char*)mem.get(2 * nb + cap * 4 + 16 + cand_bytes);
  if (!ws) return fail(TB_ERR_OOM, "tb_kernel_map: workspace");
  Guard g{&mem, ws};
  int32_t* table = (int32_t*)(ws + 2 * nb);
  unsigned int* next_chunk = (unsigned int*)(ws + 2 * nb + cap * 4);
  TB_CUDA(cudaMemsetAsync(table, 0xFF, cap * 4, s));
  KmapPrep kp;
  kp.in_counts = in->voxel_counts;
  kp.out_counts = out->voxel_counts;
  kp.B = in->B;
  kp.in_vbase = (int64_t*)ws;
  kp.out_vbase = (int64_t*)(ws + nb);
  kp.origins = in->origins;
  kp.leaf_grid = in->leaf_grid;
  kp.L = in->L;
  kp.table = table;
  kp.mask = cap - 1;
  kp.next_chunk = next_chunk;
  const int prep_blocks = in->L ? blocks_for(in->L, 256, (long long)di->sms * 8) : 1;
  TB_CUDA(launch(kKKmapPrep, s, [&] { return launch_kmap_prep(kp, prep_blocks, s); }));
  KmapArgs k;
  k.in_origins = in->origins;
  k.in_masks = in->masks;
  k.in_wp = in->word_prefix;
  k.in_voff = in->voxel_offset;
  k.in_grid = in->leaf_grid;
  k.table = table;
  k.table_mask = cap - 1;
  k.in_vbase = (const int64_t*)ws;
  k.out_origins = out->origins;
  k.out_masks = out->masks;
  k.out_voff = out->voxel_offset;
  k.out_wp = out->word_prefix;
  k.out_grid = out->leaf_grid;
  k.out_vbase = (const int64_t*)(ws + nb);
  k.L_out = out->L;
  for (int a = 0; a < 3; ++a) {
    k.lo[a] = lo[a];
    k.hi[a] = hi[a];
  }
  k.stride = stride;
  k.transposed = transposed ? 1 : 0;
  k.map = map;
  k.cands = prepass ? (int32_t*)(ws + 2 * nb + cap * 4 + 16) : nullptr;
  k.next_chunk = next_chunk;
  k.cand_max = (int32_t)cand_max;
  k.span = span;
  if (prepass) {
    const int cb = blocks_for(out->L * cand_max, 256, (long long)di->sms * 8);
    TB_CUDA(launch(kKKmap, s, [&] { return launch_kmap_cands(k, cb, s); }));
  }
  if (form == kTabulated) {
    const int hb = blocks_for(out->L, 4, (long long)di->sms * 7);
    TB_CUDA(launch(kKKmap, s, [&] { return launch_kmap_halo(k, hb, s); }));
  } else if (form == kStaged || form == kStagedPrepass) {
    TB_CUDA(launch(kKKmap, s, [&] { return launch_kmap_staged(k, di->sms, s); }));
  } else {
    const int blocks = blocks_for(out->L, 8, (long long)di->sms * 8);
    TB_CUDA(launch(kKKmap, s, [&] { return launch_kmap(k, blocks, s); }));
  }
  return TB_OK;
}

tb_status tb_chain(const tb_batch* in, const tb_op* ops, int32_t n_ops, const tb_allocator* alloc, tb_stream stream,
                   tb_batch** out) {
  if (out) *out = nullptr;
  if (!out) return fail(TB_ERR_INVALID_ARG, "out is NULL");
  if (n_ops < 0 || (n_ops > 0 && !ops)) return fail(TB_ERR_INVALID_ARG, "tb_chain: bad op list");
  std::vector<std::vector<PassSpec>> chains(1);
  tb_status st = chain_specs(ops, n_ops, &chains[0], in ? in->L : 0);
  if (st != TB_OK) return st;
  return run_ops(in, chains, alloc, (cudaStream_t)stream, out);
}

tb_status tb_multi(const tb_batch* in, const tb_op* ops, const int32_t* chain_lengths, int32_t n_chains,
                   const tb_allocator* alloc, tb_stream stream, tb_batch** outs) {
  if (!outs || n_chains <= 0 || !chain_lengths) return fail(TB_ERR_INVALID_ARG, "tb_multi: bad chain list");
  for (int32_t c = 0; c < n_chains; ++c) outs[c] = nullptr;
  if (n_chains > 1024) return fail(TB_ERR_TOO_LARGE, "tb_multi: more than 1024 chains");
  std::vector<std::vector<PassSpec>> chains(n_chains);
  long long first = 0;
  for (int32_t c = 0; c < n_chains; ++c) {
    if (chain_lengths[c] < 0 || (chain_lengths[c] > 0 && !ops))
      return fail(TB_ERR_INVALID_ARG, "tb_multi: bad length of chain %d", c);
    tb_status st = chain_specs(ops + first, chain_lengths[c], &chains[c], in ? in->L : 0);
    if (st != TB_OK) return st;
    first += chain_lengths[c];
  }
  return run_ops(in, chains, alloc, (cudaStream_t)stream, outs);
}

tb_status tb_selftest_wait(int32_t set_flag, int32_t spin_limit, tb_stream stream) {
  if (spin_limit < 1) return fail(TB_ERR_INVALID_ARG, "tb_selftest_wait: spin_limit must be positive");
  cudaStream_t s = (cudaStream_t)stream;
  const Mem mem{nullptr, s};
  uint32_t* d = (uint32_t*)mem.get(8);  // [0] the flag, [1] the error word
  if (!d) return fail(TB_ERR_OOM, "tb_selftest_wait: allocation failed");
  Guard g{&mem, d};
  TB_CUDA(cudaMemsetAsync(d, 0, 8, s));
  if (set_flag) TB_CUDA(cudaMemsetAsync(d, 1, 1, s));
  TB_CUDA(launch(kKValidate, s, [&] { return launch_wait_selftest(d, (uint32_t)spin_limit, d + 1, s); }));
  unsigned int* h = (unsigned int*)t_pinned.get(64);
  if (!h) return fail(TB_ERR_OOM, "pinned buffer");
  TB_CUDA(cudaMemcpyAsync(h, d + 1, 4, cudaMemcpyDeviceToHost, s));
  TB_CUDA(cudaStreamSynchronize(s));
  if (*h & kErrTimeout) return fail(TB_ERR_DEVICE_TIMEOUT, "a device-side wait timed out (self-test)");
  return TB_OK;
}

tb_status tb_validate(const tb_batch* b, tb_stream stream) {
  tb_status st = check_batch(b);
  if (st != TB_OK) return st;
  const Mem mem{b->has_alloc ? &b->alloc : nullptr, (cudaStream_t)stream};
  unsigned int* err = (unsigned int*)mem.get(4);
  if (!err) return fail(TB_ERR_OOM, "tb_validate: allocation failed");
  Guard g{&mem, err};
  TB_CUDA(cudaMemsetAsync(err, 0, 4, (cudaStream_t)stream));
  DeviceInfo* di = nullptr;
  st = device_info(b->device, &di);
  if (st != TB_OK) return st;
  const int blocks = blocks_for(std::max<long long>(b->L, b->B + 1), 256, (long long)di->sms * 4);
  TB_CUDA(launch(kKValidate, (cudaStream_t)stream, [&] {
    return launch_validate(b->origins, b->masks, b->leaf_grid, b->leaf_offsets, b->L, b->B, err, blocks,
                           (cudaStream_t)stream);
  }));
  unsigned int* h = (unsigned int*)t_pinned.get(64);
  if (!h) return fail(TB_ERR_OOM, "pinned buffer");
  TB_CUDA(cudaMemcpyAsync(h, err, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
  TB_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  if (*h) return fail(TB_ERR_NOT_CANONICAL, "batch violates the canonical-order invariants");
  return TB_OK;
}

tb_status tb_batch_get_view(const tb_batch* b, tb_batch_view* v) {
  if (!b || !v) return fail(TB_ERR_INVALID_ARG, "tb_batch_get_view: NULL argument");
  v->num_grids = b->B;
  v->device = b->device;
  v->num_leaves = b->L;
  v->num_lowers = b->NL;
  v->num_uppers = b->NU;
  v->leaf_offsets_host = b->leaf_offsets_host.data();
  std::memcpy(v->bbox, b->bbox, sizeof v->bbox);
  v->leaf_offsets = b->leaf_offsets;
  v->origins = b->origins;
  v->masks = b->masks;
  v->voxel_offset = b->voxel_offset;
  v->word_prefix = b->word_prefix;
  v->leaf_bbox = b->leaf_bbox;
  v->leaf_grid = b->leaf_grid;
  v->leaf_parent = b->leaf_parent;
  v->voxel_counts = b->voxel_counts;
  v->grid_bbox = b->grid_bbox;
  v->node_counts = b->node_counts;
  v->lower_offsets = b->lower_offsets;
  v->upper_offsets = b->upper_offsets;
  v->lower_origins = b->lower_origins;
  v->lower_parent = b->lower_parent;
  v->upper_origins = b->upper_origins;
  v->build_slots = b->build_slots;
  v->build_source_leaves = b->build_sources;
  v->build_key_bits = b->build_key_bits;
  v->build_digit_passes = b->build_digit_passes;
  v->build_member_ctas = b->build_member_ctas;
  v->num_voxels = b->voxel_base_host.empty() ? 0 : b->voxel_base_host.back();
  return TB_OK;
}

// Arrays at least this large are exported by the copy engines.
constexpr unsigned long long kExportEngineBytes = 1ull << 20;

tb_status tb_batch_export_many(const tb_batch* const* batches, int32_t n, int32_t* const* origins,
                               uint64_t* const* masks, int64_t* const* voxel_offset, int64_t* const* leaf_offsets,
                               tb_stream stream) {
  if (n < 0 || (n > 0 && !batches)) return fail(TB_ERR_INVALID_ARG, "tb_batch_export_many: bad batch list");
  for (int32_t i = 0; i < n; ++i)
    if (!batches[i]) return fail(TB_ERR_INVALID_ARG, "tb_batch_export_many: batch %d is NULL", i);
  cudaStream_t s = (cudaStream_t)stream;
  CopyTasks tasks;
  tasks.n = 0;
  // arrays of kExportEngineBytes or more go to the copy engines (measured on
  // GB300: the same device-to-host rate as the copy kernel, and no SM time,
  // so they overlap kernels on other streams); the smaller ones whose
  // destination the device can write (device memory, or pinned host memory
  // through its mapped address) to one copy kernel; plain copies for the rest
  auto add = [&](const void* src, void* dst, unsigned long long bytes) -> tb_status {
    if (!dst || !bytes) return TB_OK;
    if (bytes >= kExportEngineBytes) {
      TB_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s));
      return TB_OK;
    }
    void* dev = nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, dst) == cudaSuccess &&
        (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged || at.type == cudaMemoryTypeHost))
      dev = at.devicePointer;
    cudaGetLastError();
    if (!dev) {
      TB_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s));
      return TB_OK;
    }
    if (tasks.n == kMaxCopyTasks) {
      TB_CUDA(launch(kKExport, s, [&] { return launch_copies(tasks, s); }));
      tasks.n = 0;
    }
    tasks.t[tasks.n++] = CopyTask{src, dev, bytes};
    return TB_OK;
  };
  for (int32_t i = 0; i < n; ++i) {
    const tb_batch* b = batches[i];
    tb_status st = TB_OK;
    if (origins && st == TB_OK) st = add(b->origins, origins[i], (unsigned long long)b->L * 12);
    if (masks && st == TB_OK) st = add(b->masks, masks[i], (unsigned long long)b->L * 64);
    if (voxel_offset && st == TB_OK) st = add(b->voxel_offset, voxel_offset[i], (unsigned long long)b->L * 8);
    if (leaf_offsets && st == TB_OK) st = add(b->leaf_offsets, leaf_offsets[i], (unsigned long long)(b->B + 1) * 8);
    if (st != TB_OK) return st;
  }
  if (tasks.n) TB_CUDA(launch(kKExport, s, [&] { return launch_copies(tasks, s); }));
  return TB_OK;
}

tb_status tb_batch_export(const tb_batch* b, int32_t* origins, uint64_t* masks, int64_t* voxel_offset,
                          int64_t* leaf_offsets, tb_stream stream) {
  if (!b) return fail(TB_ERR_INVALID_ARG, "tb_batch_export: batch is NULL");
  return tb_batch_export_many(&b, 1, origins ? &origins : nullptr, masks ? &masks : nullptr,
                              voxel_offset ? &voxel_offset : nullptr, leaf_offsets ? &leaf_offsets : nullptr, stream);
}

tb_status tb_batch_free(tb_batch* b, tb_stream stream) {
  if (!b) return TB_OK;
  const Mem mem{b->has_alloc ? &b->alloc : nullptr, (cudaStream_t)stream};
  mem.put(b->mem);
  delete b;
  return TB_OK;
}

const char* tb_last_error(void) { return t_err.c_str(); }

const char* tb_status_string(tb_status s) {
  switch (s) {
    case TB_OK: return "TB_OK";
    case TB_ERR_INVALID_ARG: return "TB_ERR_INVALID_ARG";
    case TB_ERR_OOM: return "TB_ERR_OOM";
    case TB_ERR_CUDA: return "TB_ERR_CUDA";
    case TB_ERR_COORD_OVERFLOW: return "TB_ERR_COORD_OVERFLOW";
    case TB_ERR_NOT_CANONICAL: return "TB_ERR_NOT_CANONICAL";
    case TB_ERR_DEVICE_TIMEOUT: return "TB_ERR_DEVICE_TIMEOUT";
    case TB_ERR_TOO_LARGE: return "TB_ERR_TOO_LARGE";
    case TB_ERR_INTERNAL: return "TB_ERR_INTERNAL";
  }
  return "TB_ERR_UNKNOWN";
}

int32_t tb_version(void) { return 100; }

int64_t tb_kernel_launch_count(void) { return t_launches; }

int32_t tb_set_launch_mode(int32_t mode) {
  if (mode < 0 || mode > 2) return -1;
  return g_launch_mode.exchange(mode);
}

int32_t tb_set_node_mode(int32_t mode) {
  if (mode < 0 || mode > 1) return -1;
  return g_node_mode.exchange(mode);
}

int32_t tb_set_kmap_mode(int32_t mode) {
  if (mode < 0 || mode > 4) return -1;
  return g_kmap_mode.exchange(mode);
}

tb_status tb_profile_enable(int32_t on) {
  t_prof = on < 0 ? 0 : on;
  return TB_OK;
}

int32_t tb_profile_read(tb_kernel_stat* stats, int32_t max) {
  double ms[kKNumKinds] = {};
  int64_t n[kKNumKinds] = {};
  for (const ProfRec& r : t_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      ms[r.kind] += t;
      n[r.kind] += 1;
    }
    cudaGetLastError();
    t_events.push_back(r.a);
    t_events.push_back(r.b);
  }
  t_recs.clear();
  int32_t k = 0;
  for (int i = 0; i < kKNumKinds; ++i) {
    if (!n[i]) continue;
    if (stats && k < max) stats[k] = tb_kernel_stat{kKernelNames[i], n[i], ms[i]};
    ++k;
  }
  for (int i = 0; i < kNumPhases; ++i) {
    if (!t_phase_n[i]) continue;
    if (stats && k < max) stats[k] = tb_kernel_stat{kPhaseNames[i], t_phase_n[i], t_phase_ms[i]};
    ++k;
    t_phase_n[i] = 0;
    t_phase_ms[i] = 0.0;
  }
  return k;
}

}  // extern "C"
