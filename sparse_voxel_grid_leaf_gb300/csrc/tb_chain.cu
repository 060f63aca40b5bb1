// The batched pass as one cooperative, persistent kernel per call, and the
// final writers (fVDB PR #757 "Batched leaf-mask topology construction for
// generated conv grids", Summary item 1; item 2 for the box dilation).
//
// k_chain runs every pass of a call -- one or several chains of passes over
// the same input, stage by stage, the chains of a stage side by side on
// shares of the grid -- with all blocks co-resident; phases are separated by
// a bounded software grid barrier:
//   [front ends: input bbox -> key plan]
//   emission -> digit pass 0 .. P-1 -> index -> leaves (merge, popcounts,
//   bboxes, staged records; or the hand-off of an intermediate pass) ->
//   voxel offsets.
// Everything the host needs to size the outputs then comes back in one
// readback, and the writers copy the staged records into the exact outputs.
//
// Emission: one thread per (source leaf or input voxel, chunk of targets)
// writes one slot per non-empty target leaf -- the f^3 children of a
// refinement by f, the coarse leaf of a coarsening, up to 27 neighbours of a
// box dilation, up to 64 fine leaves of a fused refinement then dilation --
// with warp-aggregated slot claims, and counts the first digit's histogram.
// Sort: the grid index is the key's most significant field, so one global LSD
// sort over the varying key bits replaces the PR's segmented sorts.  A digit
// pass is a onesweep tile loop: warp multisplit ranking (match.any), per-digit
// decoupled look-back, shared-memory staging, coalesced scatter, and the next
// digit's histogram.
// Index: head flags on the sorted keys (new leaf / lower node / upper node /
// grid), a tile scan with warp-window look-back.
#include "tb_common.cuh"
#include "tb_launch.h"
#include "tb_layout.h"

namespace tb {

namespace {

constexpr int kThreads = 256;

struct SmemSort {
  uint32_t whist[kThreads / 32][kBins];
  uint32_t binstart[kBins];
  uint32_t glob[kBins];
  uint32_t binbase[kBins];
  unsigned int next_hist[kBins];  // histogram of the next digit over this block's tiles
  uint64_t keys[kSortTile];
  uint32_t vals[kSortTile];
  uint32_t scan[8];
  uint32_t tile;
};
struct SmemEmit {
  unsigned int hist[kMaxDigitPasses][kBins];
};
// Node path emission: the child-mask bits of a few lower nodes gathered per
// block and flushed to the node tables once at the end of the phase.
constexpr int kNodeSlots = 8;
struct SmemNodes {
  uint32_t id[kNodeSlots];              // node id + 1, 0: free
  uint32_t mask[kNodeSlots][128];       // child mask as 32-bit words
};
struct SmemDedup {
  unsigned long long scan[8];
  unsigned long long base[3];
  uint32_t tile;
};
struct SmemLeaves {
  uint32_t grp_f[kThreads / 8];            // per 8-lane group: segmented aggregate of its leaves
  unsigned long long grp_v[kThreads / 8];
  uint32_t grp_g[kThreads / 8];            // grid of its pending bbox
  unsigned int grp_box[kThreads / 8][6];   // its pending encoded bbox
  unsigned long long blk_prefix;           // voxels before the block's first leaf in the same grid
  unsigned long long grp_prefix[kThreads / 8];
};
struct SmemFinish {
  uint32_t s[kThreads];
};
struct SmemPlace {
  uint32_t base[kNodeCap];  // leaves before the node of each rank
  uint32_t scan[8];
};
union Smem {
  SmemPlace place;
  SmemNodes nodes;
  SmemSort sort;
  SmemEmit emit;
  SmemDedup dedup;
  SmemFinish fin;
  SmemLeaves lv;
};

// Profiling stamps of the GPU global timer over all blocks: slot 0 holds the
// earliest block start (as the max of its complement), slot k in 1..5 the
// latest block end of phase k, slot 6 the earliest kernel entry (complemented).
__device__ __forceinline__ void stamp(const PassArgs& a, int k) {
  if (a.phase_ts && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    atomicMax(&a.phase_ts[k], k == 0 ? ~t : t);
  }
}

// ---------------------------------------------------------------- node path: lower-node child masks

// Hash of a node or tile key (the splitmix64 finaliser).
__device__ __forceinline__ uint32_t mix_key(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return (uint32_t)(z ^ (z >> 31));
}

// Id of `key` in an open-addressing table of key + 1 per slot (0: free;
// zeroed): the key's slot, claimed by compare-and-swap when the key is new,
// in which case `made(id)` runs in the claiming thread.  The id is the slot
// itself, so a thread that finds the key needs nothing more (no counter, no
// wait); what made() writes is read after a grid barrier.  Relaxed loads at
// GPU scope.
template <class Made>
__device__ __forceinline__ uint32_t table_id(const PassArgs& a, unsigned long long* keys, uint64_t key, Made made) {
  const unsigned long long want = key + 1ull;
  uint32_t h = mix_key(key) & a.node_hmask;
  for (uint32_t probe = 0; probe <= a.node_hmask; ++probe, h = (h + 1u) & a.node_hmask) {
    unsigned long long cur = ld_relaxed(keys + h);
    if (cur == 0ull) {
      cur = atomicCAS(keys + h, 0ull, want);
      if (cur == 0ull) {
        made(h);
        return h;
      }
    }
    if (cur == want) return h;
  }
  atomicOr(a.err, kErrSlotOverflow);  // table full: the host's bound was wrong
  return 0;
}

// Lower node `nk` (key >> lower_bits of target leaf tl in grid g): its id,
// made if new, and its slot in the block's cache of child masks (-1: none).
// The cache is direct-mapped: a node may only take slot id mod kNodeSlots,
// claimed by its id; a node whose slot another holds ORs its bits into the
// node table directly.  (One shared-memory compare per look-up; scanning
// every slot measured 4 % slower on the seven-chain call at stress size.)
__device__ __forceinline__ uint32_t node_lookup(const PassArgs& a, SmemNodes* sn, uint64_t nk, uint64_t key,
                                                const int32_t tl[3], uint32_t g, int& slot) {
  const KeyLayout& K = a.K;
  const uint32_t id = table_id(a, a.nh_key, nk, [&](uint32_t nid) {
    a.node_key[nid] = nk;
    int32_t* nl = a.node_lc + 4ull * nid;
    nl[0] = tl[0] >> 4;
    nl[1] = tl[1] >> 4;
    nl[2] = tl[2] >> 4;
    nl[3] = (int32_t)g;
    const uint64_t tk = shr64(key, K.node_bits);
    a.node_tile[nid] = table_id(a, a.th_key, tk, [&](uint32_t tid) {
      const uint32_t li = atomicAdd(&a.ctl->n_tiles, 1u);  // the compact list of tiles
      if (li < (uint32_t)a.node_cap) a.tile_list[li] = tid;
    });
    const uint32_t li = atomicAdd(&a.ctl->n_nodes, 1u);  // the compact list of nodes
    if (li < (uint32_t)a.node_cap) a.node_list[li] = nid;
    else atomicOr(a.err, kErrSlotOverflow);
  });
  slot = -1;
  if (!sn) return id;
  {
    const int j = (int)(id & (uint32_t)(kNodeSlots - 1));
    const uint32_t v = *reinterpret_cast<volatile uint32_t*>(&sn->id[j]);
    if (v == id + 1u) {
      slot = j;
    } else if (v == 0u) {
      const uint32_t old = atomicCAS(&sn->id[j], 0u, id + 1u);
      if (old == 0u || old == id + 1u) slot = j;
    }
  }
  return id;
}

// A run of child-mask bits of one 32-bit word of one node, merged in
// registers before its one atomic OR (into the block cache, or the node
// table for a node without a cache slot).
struct NodeRun {
  uint32_t id, w32, bits;
  int slot;
};
__device__ __forceinline__ void run_flush(const PassArgs& a, SmemNodes& sn, NodeRun& run) {
  if (!run.bits) return;
  if (run.slot >= 0) {
    atomicOr(&sn.mask[run.slot][run.w32], run.bits);
  } else {
    atomicOr(reinterpret_cast<unsigned int*>(a.node_mask + 64ull * run.id) + run.w32, run.bits);
  }
  run.bits = 0;
}

// The end of a node-path emission: the block's gathered child-mask bits go
// to the node tables, one atomic OR per non-zero 64-bit word.
__device__ __forceinline__ void emit_flush(const PassArgs& a, SmemNodes& sn) {
  __syncthreads();
  for (int i = threadIdx.x; i < kNodeSlots * 64; i += kThreads) {
    const int j = i >> 6, w = i & 63;
    const uint32_t id1 = sn.id[j];
    if (!id1) continue;  // a slot is used only once its id is set
    const unsigned long long v = (unsigned long long)sn.mask[j][2 * w] | ((unsigned long long)sn.mask[j][2 * w + 1] << 32);
    if (v) atomicOr(reinterpret_cast<unsigned long long*>(a.node_mask) + 64ull * (id1 - 1u) + w, v);
  }
}

__device__ __forceinline__ void put_node_slot(const PassArgs& a, unsigned long long pos, uint32_t nref, uint32_t val) {
  if (pos < (unsigned long long)a.slot_cap) {
    a.nref[pos] = nref;
    a.vals[0][pos] = val;
  } else {
    atomicOr(a.err, kErrSlotOverflow);
  }
}

// ---------------------------------------------------------------- emission

__device__ __forceinline__ int grid_of(const int64_t* offsets, int32_t B, long long i) {
  int lo = 0, hi = B;  // last g with offsets[g] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(offsets + mid) <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// Claims `n` consecutive slots for this lane within one warp-wide range;
// returns the lane's first slot and the warp's range [wbase, wbase + wtotal).
__device__ __forceinline__ unsigned long long claim_slots(const PassArgs& a, uint32_t n, unsigned long long& wbase,
                                                          uint32_t& wtotal) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  wtotal = __shfl_sync(0xffffffffu, incl, 31);
  unsigned long long base = 0;
  if (lane == 31 && wtotal) base = atomicAdd(&a.rb->num_slots, (unsigned long long)wtotal);
  wbase = __shfl_sync(0xffffffffu, base, 31);
  return wbase + incl - n;
}

__device__ __forceinline__ void put_slot(const PassArgs& a, unsigned long long pos, uint64_t key, uint32_t val) {
  if (pos < (unsigned long long)a.slot_cap) {
    a.keys[0][pos] = key;
    a.vals[0][pos] = val;
  } else {
    atomicOr(a.err, kErrSlotOverflow);
  }
}

// Adds digit `pass` of one key per lane (valid lanes only) to a shared
// histogram, one shared-memory atomic per distinct digit value in the warp.
__device__ __forceinline__ void hist_digit(unsigned int* hist, uint64_t key, int pass, bool valid) {
  const int lane = threadIdx.x & 31;
  const uint32_t d = valid ? ((uint32_t)(key >> (8 * pass)) & 255u) : kBins;
  const uint32_t peers = __match_any_sync(0xffffffffu, d);
  if (valid && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(&hist[d], (unsigned int)__popc(peers));
}

// Is target `t` (an index into the op's target set) of a source leaf with
// mask m non-empty?  Sets the target's slot code and leaf coordinate.
template <int OP>
__device__ __forceinline__ bool target_nonempty(const PassArgs& a, const uint64_t m[8], const int32_t lc[3],
                                                uint32_t t, uint32_t& code, int32_t out[3]) {
  if (OP == kRefine) {
    const int f = a.factor;
    if (f == 2) {  // child t = 4*cx + 2*cy + cz: the parent's octant t holds a voxel
      const int cx = (t >> 2) & 1, cy = (t >> 1) & 1, cz = t & 1;
      const uint64_t h = m[4 * cx] | m[4 * cx + 1] | m[4 * cx + 2] | m[4 * cx + 3];
      code = t;
      out[0] = 2 * lc[0] + cx;
      out[1] = 2 * lc[1] + cy;
      out[2] = 2 * lc[2] + cz;
      return (h & (0x0F0F0F0Full << (32 * cy + 4 * cz))) != 0;
    }
    // child t = (cx f + cy) f + cz of a refinement by f = 4 or 8: the parent's
    // block [c 8/f, (c + 1) 8/f) per axis holds a voxel
    const int bs = 8 / f, cx = (int)t / (f * f), cy = ((int)t / f) % f, cz = (int)t % f;
    uint64_t h = 0, ym = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k / bs == cx) h |= m[k];
      if (k / bs == cy) ym |= 0xFFull << (8 * k);
    }
    const uint64_t zm = 0x0101010101010101ull * ((((1u << bs) - 1u) << (cz * bs)) & 0xFFu);
    code = t;
    out[0] = f * lc[0] + cx;
    out[1] = f * lc[1] + cy;
    out[2] = f * lc[2] + cz;
    return (h & ym & zm) != 0;
  }
  uint64_t all = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) all |= m[k];
  if (OP == kLeaves || OP == kCoarsen) {
    // coarsen by f: the code is the source leaf's position q = lc mod f inside
    // its coarse leaf, (qx f + qy) f + qz
    const int sh = OP == kCoarsen ? log2_factor(a.factor) : 0, fm = (1 << sh) - 1;
    code = OP == kCoarsen ? (uint32_t)((((lc[0] & fm) << sh) | (lc[1] & fm)) << sh | (lc[2] & fm)) : 0u;
    out[0] = lc[0] >> sh;
    out[1] = lc[1] >> sh;
    out[2] = lc[2] >> sh;
    return all != 0;
  }
  if (OP == kRefineDilate) {
    // refinement by 2, then a box within [-1, 1]^3: targets are fine leaves at
    // offsets t (relative to the first child) per axis; the source voxels s
    // that reach target t along an axis are [(8t - hi) / 2, (8t + 7 - lo) / 2]
    // (floors), clamped to 0..7
    const int tlx = refine_dilate_lo(a.lo[0]), tly = refine_dilate_lo(a.lo[1]), tlz = refine_dilate_lo(a.lo[2]);
    const int ny = refine_dilate_hi(a.hi[1]) - tly + 1, nz = refine_dilate_hi(a.hi[2]) - tlz + 1;
    const int tz = tlz + (int)(t % nz), ty = tly + (int)((t / nz) % ny), tx = tlx + (int)(t / (nz * ny));
    const int tt[3] = {tx, ty, tz};
    uint32_t zone[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      int s0 = (8 * tt[ax] - a.hi[ax]) >> 1, s1 = (8 * tt[ax] + 7 - a.lo[ax]) >> 1;
      s0 = s0 < 0 ? 0 : s0;
      s1 = s1 > 7 ? 7 : s1;
      zone[ax] = s0 > s1 ? 0u : (((0xFFu >> (7 - s1)) & (0xFFu << s0)) & 0xFFu);
    }
    uint64_t xs = 0, ym = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((zone[0] >> k) & 1u) xs |= m[k];
      if ((zone[1] >> k) & 1u) ym |= 0xFFull << (8 * k);
    }
    const uint64_t zm = 0x0101010101010101ull * zone[2];
    code = (uint32_t)(((tx + 1) * 4 + (ty + 1)) * 4 + (tz + 1));
    out[0] = 2 * lc[0] + tx;
    out[1] = 2 * lc[1] + ty;
    out[2] = 2 * lc[2] + tz;
    return (xs & ym & zm) != 0;
  }
  // box dilation: targets enumerate the offsets t in {-1 if lo < 0, 0, +1 if
  // hi > 0} per axis; target t is reached iff a voxel lies in its zone
  // (dilate_zone) on all three axes
  const int tlx = a.lo[0] < 0 ? -1 : 0, tly = a.lo[1] < 0 ? -1 : 0, tlz = a.lo[2] < 0 ? -1 : 0;
  const int ny = (a.hi[1] > 0 ? 1 : 0) - tly + 1, nz = (a.hi[2] > 0 ? 1 : 0) - tlz + 1;
  const int tz = tlz + (int)(t % nz), ty = tly + (int)((t / nz) % ny), tx = tlx + (int)(t / (nz * ny));
  uint64_t xs = 0, ym = 0, zm;
  if (a.lo[0] >= -1 && a.lo[1] >= -1 && a.lo[2] >= -1 && a.hi[0] <= 1 && a.hi[1] <= 1 && a.hi[2] <= 1) {
    // a box within [-1, 1]^3: the zones are the whole leaf (offset 0) or the
    // facing plane (offset +-1)
    xs = tx < 0 ? m[0] : (tx > 0 ? m[7] : all);
    ym = ty < 0 ? 0x00000000000000FFull : (ty > 0 ? 0xFF00000000000000ull : ~0ull);
    zm = tz < 0 ? 0x0101010101010101ull : (tz > 0 ? 0x8080808080808080ull : ~0ull);
  } else {
    const uint32_t zx = dilate_zone(tx, a.lo[0], a.hi[0]), zy = dilate_zone(ty, a.lo[1], a.hi[1]),
                   zz = dilate_zone(tz, a.lo[2], a.hi[2]);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((zx >> k) & 1u) xs |= m[k];
      if ((zy >> k) & 1u) ym |= 0xFFull << (8 * k);
    }
    zm = 0x0101010101010101ull * zz;
  }
  code = (uint32_t)(9 * (tx + 1) + 3 * (ty + 1) + (tz + 1));
  out[0] = lc[0] + tx;
  out[1] = lc[1] + ty;
  out[2] = lc[2] + tz;
  return (xs & ym & zm) != 0;
}

// The slot code and leaf coordinate of target `t` of a source leaf at leaf
// coordinate lc (the geometry of target_nonempty, without its test).
template <int OP>
__device__ __forceinline__ void target_geometry(const PassArgs& a, const int32_t lc[3], uint32_t t, uint32_t& code,
                                                int32_t out[3]) {
  if constexpr (OP == kRefine) {
    const int f = a.factor;
    const int cx = (int)t / (f * f), cy = ((int)t / f) % f, cz = (int)t % f;
    code = t;
    out[0] = f * lc[0] + cx;
    out[1] = f * lc[1] + cy;
    out[2] = f * lc[2] + cz;
  } else if constexpr (OP == kLeaves || OP == kCoarsen) {
    const int sh = OP == kCoarsen ? log2_factor(a.factor) : 0, fm = (1 << sh) - 1;
    code = OP == kCoarsen ? (uint32_t)((((lc[0] & fm) << sh) | (lc[1] & fm)) << sh | (lc[2] & fm)) : 0u;
    out[0] = lc[0] >> sh;
    out[1] = lc[1] >> sh;
    out[2] = lc[2] >> sh;
  } else if constexpr (OP == kRefineDilate) {
    const int tlx = refine_dilate_lo(a.lo[0]), tly = refine_dilate_lo(a.lo[1]), tlz = refine_dilate_lo(a.lo[2]);
    const int ny = refine_dilate_hi(a.hi[1]) - tly + 1, nz = refine_dilate_hi(a.hi[2]) - tlz + 1;
    const int tz = tlz + (int)(t % nz), ty = tly + (int)((t / nz) % ny), tx = tlx + (int)(t / (nz * ny));
    code = (uint32_t)(((tx + 1) * 4 + (ty + 1)) * 4 + (tz + 1));
    out[0] = 2 * lc[0] + tx;
    out[1] = 2 * lc[1] + ty;
    out[2] = 2 * lc[2] + tz;
  } else {  // kDilate
    const int tlx = a.lo[0] < 0 ? -1 : 0, tly = a.lo[1] < 0 ? -1 : 0, tlz = a.lo[2] < 0 ? -1 : 0;
    const int ny = (a.hi[1] > 0 ? 1 : 0) - tly + 1, nz = (a.hi[2] > 0 ? 1 : 0) - tlz + 1;
    const int tz = tlz + (int)(t % nz), ty = tly + (int)((t / nz) % ny), tx = tlx + (int)(t / (nz * ny));
    code = (uint32_t)(9 * (tx + 1) + 3 * (ty + 1) + (tz + 1));
    out[0] = lc[0] + tx;
    out[1] = lc[1] + ty;
    out[2] = lc[2] + tz;
  }
}

// Targets per source leaf of an op.
template <int OP>
__device__ __forceinline__ uint32_t targets_per_source(const PassArgs& a) {
  return (uint32_t)pass_targets(OP, a.factor, a.lo, a.hi);
}

// One thread per (source, chunk of a.tchunk targets): it tests its targets,
// claims one warp-aggregated range of slots for the non-empty ones, and
// writes them in warp-synchronous rounds that also feed the block's digit
// histograms.  The host sizes the chunk so that all candidates of a pass are
// covered by about one round of the grid's threads.
template <int OP>
__device__ void phase_emit(const PassArgs& a, Smem& sm, int vb, int vg) {
  for (int i = threadIdx.x; i < kBins; i += kThreads) sm.emit.hist[0][i] = 0;
  __syncthreads();
  const long long n = a.src_count_dev ? (long long)__ldcg(a.src_count_dev) : a.src_count;
  const uint32_t T = targets_per_source<OP>(a);
  uint32_t k = (a.tchunk > 0 && (uint32_t)a.tchunk < T) ? (uint32_t)a.tchunk : T;
  if (k > 32) k = 32;  // a thread's targets are one 32-bit set
  const uint32_t nchunks = (T + k - 1) / k;
  const long long items = n * (long long)nchunks;
  const long long stride = (long long)vg * kThreads;
  for (long long base = (long long)vb * kThreads; base < items; base += stride) {
    const long long idx = base + threadIdx.x;
    uint32_t bits = 0, t0 = 0, g = 0;
    long long i = 0;
    uint64_t m[8];
    int32_t lc[3] = {0, 0, 0};
    if (idx < items) {
      i = idx / nchunks;
      t0 = (uint32_t)(idx - i * nchunks) * k;
      const uint32_t t1 = t0 + k < T ? t0 + k : T;
      if (OP == kIjk) {
        lc[0] = __ldg(a.ijk + 3 * i);
        lc[1] = __ldg(a.ijk + 3 * i + 1);
        lc[2] = __ldg(a.ijk + 3 * i + 2);
        g = (uint32_t)grid_of(a.in_offsets, a.B, i);
        bits = 1u;
      } else {
        load_mask(a.src_masks, i, m);
        lc[0] = __ldcg(a.src_origins + 3 * i) >> 3;
        lc[1] = __ldcg(a.src_origins + 3 * i + 1) >> 3;
        lc[2] = __ldcg(a.src_origins + 3 * i + 2) >> 3;
        for (uint32_t t = t0; t < t1; ++t) {
          uint32_t code;
          int32_t tl[3];
          if (target_nonempty<OP>(a, m, lc, t, code, tl)) bits |= 1u << (t - t0);
        }
        if (bits) g = a.src_grid ? (uint32_t)__ldcg(a.src_grid + i) : (uint32_t)grid_of(a.in_offsets, a.B, i);
      }
    }
    const uint32_t nt = __popc(bits);
    unsigned long long wbase;
    uint32_t wtotal;
    unsigned long long pos = claim_slots(a, nt, wbase, wtotal);
    const uint32_t rounds = __reduce_max_sync(0xffffffffu, nt);
    for (uint32_t r = 0; r < rounds; ++r) {
      const bool valid = bits != 0;
      uint64_t key = 0;
      if (valid) {
        const uint32_t t = t0 + (uint32_t)(__ffs(bits) - 1);
        bits &= bits - 1;
        uint32_t val;
        if (OP == kIjk) {
          // the voxel's bit in its leaf, n = 64 x + 8 y + z: all the merge needs
          key = encode_key(a.K, g, lc[0] >> 3, lc[1] >> 3, lc[2] >> 3);
          val = (uint32_t)(((lc[0] & 7) << 6) | ((lc[1] & 7) << 3) | (lc[2] & 7));
        } else {
          uint32_t code;
          int32_t tl[3];
          target_nonempty<OP>(a, m, lc, t, code, tl);
          key = encode_key(a.K, g, tl[0], tl[1], tl[2]);
          val = ((uint32_t)i << a.code_bits) | code;
        }
        put_slot(a, pos++, key, val);
      }
      if (a.P > 0) hist_digit(sm.emit.hist[0], key, 0, valid);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += kThreads) {
    const unsigned int c = sm.emit.hist[0][i];
    if (c && a.P > 0) atomicAdd(&a.ctl->hist[0][i], c);
  }
}

// ---------------------------------------------------------------- radix digit pass

// Tiles vb, vb + ... : a block's first tile is its virtual block index; only
// when a pass has more tiles than the chain has blocks do the rest come from
// an atomic counter, in increasing order (so every tile's predecessors are
// held by running blocks, as the look-back needs).
__device__ __forceinline__ long long next_tile(unsigned int* ctr, long long ntiles, int vg, uint32_t& shared_tile) {
  if (ntiles <= vg) return ntiles;
  __syncthreads();
  if (threadIdx.x == 0) shared_tile = (uint32_t)vg + atomicAdd(ctr, 1u);
  __syncthreads();
  return (long long)shared_tile;
}

// A digit pass.  Tiles hold `ipt` slots per thread (1..kSortItems), chosen so
// that the chain's blocks get one tile each where the status words allow: a
// small pass then runs as many short tiles side by side instead of a few long
// ones.
__device__ void phase_sort(const PassArgs& a, int pass, Smem& sm, int vb, int vg) {
  constexpr int NW = kThreads / 32;
  SmemSort& s = sm.sort;
  const int shift = 8 * pass;
  const uint64_t* kin = a.keys[pass & 1];
  const uint32_t* vin = a.vals[pass & 1];
  uint64_t* kout = a.keys[(pass + 1) & 1];
  uint32_t* vout = a.vals[(pass + 1) & 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the slot count, this pass's digit counts and (speculatively, within the
  // buffers' capacity) the first tile's keys are loaded together
  long long S = (long long)__ldcg(&a.rb->num_slots);
  const uint32_t hist = __ldcg(&a.ctl->hist[pass][tid]);
  const long long cap = a.slot_cap;
  if (S > cap) S = cap;
  const long long per_blk = (S + (long long)vg * kThreads - 1) / ((long long)vg * kThreads);
  const long long per_cap = (S + a.sort_tiles_cap * kThreads - 1) / (a.sort_tiles_cap * kThreads);
  long long ipt_l = per_blk > per_cap ? per_blk : per_cap;
  const int ipt = ipt_l < 1 ? 1 : (ipt_l > kSortItems ? kSortItems : (int)ipt_l);
  const long long TS = (long long)kThreads * ipt;
  const long long ntiles = (S + TS - 1) / TS;
  uint32_t* status = a.sort_status + (long long)pass * a.sort_tiles_cap * kBins;
  unsigned int* ctr = &a.ctl->sort_tile_ctr[pass];
  const bool count_next = pass + 1 < a.P;
  s.next_hist[tid] = 0;
  bool based = false;
  for (long long tile = vb; tile < ntiles; tile = next_tile(ctr, ntiles, vg, s.tile)) {
    const long long base = tile * TS + (long long)warp * 32 * ipt;
    uint64_t k[kSortItems];
    uint32_t v[kSortItems], d[kSortItems], r[kSortItems];
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const long long idx = base + j * 32 + lane;
      k[j] = 0;
      v[j] = 0;
      if (j < ipt && idx < cap) {
        k[j] = __ldcg(kin + idx);
        v[j] = __ldcg(vin + idx);
      }
    }
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const long long idx = base + j * 32 + lane;
      d[j] = (j < ipt && idx < S) ? ((uint32_t)(k[j] >> shift) & 255u) : kBins;  // kBins: ranked nowhere
    }
    if (!based) {
      uint32_t total;
      s.binbase[tid] = block_excl_scan_256(hist, s.scan, &total);
      based = true;
    }
    for (int i = tid; i < NW * kBins; i += kThreads) (&s.whist[0][0])[i] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      if (j >= ipt) break;  // block-uniform
      const uint32_t peers = __match_any_sync(0xffffffffu, d[j]);
      const uint32_t lt = peers & ((1u << lane) - 1u);
      uint32_t cnt = 0;
      if (d[j] < kBins) cnt = s.whist[warp][d[j]];
      __syncwarp();
      if (d[j] < kBins && lt == 0) s.whist[warp][d[j]] = cnt + __popc(peers);
      __syncwarp();
      r[j] = cnt + __popc(lt);
    }
    __syncthreads();
    uint32_t tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t c = s.whist[w][tid];
      s.whist[w][tid] = tot;
      tot += c;
    }
    uint32_t all;
    const uint32_t ex = block_excl_scan_256(tot, s.scan, &all);
    s.binstart[tid] = ex;
    const uint32_t prefix = lookback32(status + tid, kBins, tile, tot, a.err);
    s.glob[tid] = s.binbase[tid] + prefix - ex;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      if (j < ipt && d[j] < kBins) {
        const uint32_t lp = s.binstart[d[j]] + s.whist[warp][d[j]] + r[j];
        s.keys[lp] = k[j];
        s.vals[lp] = v[j];
      }
    }
    __syncthreads();
    const long long rem = S - tile * TS;
    const int nvalid = rem < TS ? (int)rem : (int)TS;
    for (int i = tid; i < nvalid; i += kThreads) {
      const uint64_t key = s.keys[i];
      const uint32_t gp = s.glob[(uint32_t)(key >> shift) & 255u] + (uint32_t)i;
      if (gp < (uint64_t)S) {  // always true when the histograms match the slots
        kout[gp] = key;
        vout[gp] = s.vals[i];
      }
      if (count_next) atomicAdd(&s.next_hist[(uint32_t)(key >> (shift + 8)) & 255u], 1u);
    }
  }
  __syncthreads();
  if (count_next && s.next_hist[tid]) atomicAdd(&a.ctl->hist[pass + 1][tid], s.next_hist[tid]);
}

// ---------------------------------------------------------------- merged masks

// Word w (this lane's, within an aligned group of 8 lanes) of the OR of the
// run of slots [s0, s1).  Refinement runs have one slot per leaf, so each lane
// recomputes its own word; the other ops spread the run's slots over the 8
// lanes, build full 8-word contributions and reduce-scatter them.
template <int OP>
__device__ __forceinline__ uint64_t merge_run(const PassArgs& a, const uint32_t* vals, uint32_t s0, uint32_t s1,
                                              int w) {
  if constexpr (OP == kRefine) {
    const int f = a.factor, cb = a.code_bits;
    uint64_t word = 0;
    for (uint32_t s = s0; s < s1; ++s) {
      const uint32_t val = __ldcg(vals + s);
      const long long src = (long long)(val >> cb);
      const int code = (int)(val & ((1u << cb) - 1u));
      if (f == 2) {
        const int cx = (code >> 2) & 1, cy = (code >> 1) & 1, cz = code & 1;
        word |= refine_word(__ldcg(a.src_masks + 8 * src + 4 * cx + (w >> 1)), cy, cz);
      } else {
        const int cx = code / (f * f), cy = (code / f) % f, cz = code % f;
        word |= refine_word_f(__ldcg(a.src_masks + 8 * src + (8 * cx + w) / f), cy, cz, f);
      }
    }
    return word;
  } else if constexpr (OP == kRefineDilate) {
    // lane w builds target word w: along x, the fine positions 8 tx + w - d
    // (d in [lo, hi]) inside the refined 16^3 block, i.e. source words
    // (8 tx + w - d) / 2; along y and z, the child quadrants (cy, cz) whose
    // dilation reaches the target, each refined and dilated as a plane.
    // The run's slot values come 8 at a time (lane w holds slot 8 j + w) and
    // the next slot's source words are loaded while this slot's are combined.
    const int cb = a.code_bits;
    const uint32_t gmask = 0xFFu << (threadIdx.x & 24u);  // this lane's group of 8
    auto xword = [&](uint32_t val) {  // lane w's x-dilated source word of a slot
      const long long src = (long long)(val >> cb);
      const int tx = (int)((val & 63u) >> 4) - 1;
      uint64_t mx = 0;
      for (int d = a.lo[0]; d <= a.hi[0]; ++d) {
        const int fx = 8 * tx + w - d;
        if (fx >= 0 && fx < 16) mx |= __ldcg(a.src_masks + 8 * src + (fx >> 1));
      }
      return mx;
    };
    uint64_t word = 0;
    const uint32_t n = s1 - s0;
    uint32_t vcache = 0, val_next = 0;
    uint64_t mx_next = 0;
    if (n) {
      vcache = __ldcg(vals + s0 + min((uint32_t)w, n - 1u));
      val_next = __shfl_sync(gmask, vcache, 0, 8);
      mx_next = xword(val_next);
    }
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t val = val_next;
      const uint64_t mx = mx_next;
      if (i + 1 < n) {
        if (((i + 1) & 7u) == 0) vcache = __ldcg(vals + s0 + i + 1 + min((uint32_t)w, n - i - 2u));
        val_next = __shfl_sync(gmask, vcache, (int)((i + 1) & 7u), 8);
        mx_next = xword(val_next);
      }
      if (!mx) continue;
      const int code = (int)(val & 63u);
      const int ty = ((code >> 2) & 3) - 1, tz = (code & 3) - 1;
#pragma unroll
      for (int cy = 0; cy < 2; ++cy) {
        const int dy = ty - cy;
        if (dy < -1 || dy > 1 || (dy < 0 && a.lo[1] >= 0) || (dy > 0 && a.hi[1] <= 0)) continue;
#pragma unroll
        for (int cz = 0; cz < 2; ++cz) {
          const int dz = tz - cz;
          if (dz < -1 || dz > 1 || (dz < 0 && a.lo[2] >= 0) || (dz > 0 && a.hi[2] <= 0)) continue;
          if (!(mx & (0x0F0F0F0Full << (32 * cy + 4 * cz)))) continue;  // an empty quadrant adds nothing
          word |= dilate_y1(dilate_z1(refine_word(mx, cy, cz), dz, a.lo[2], a.hi[2]), dy, a.lo[1], a.hi[1]);
        }
      }
    }
    return word;
  } else {
  uint64_t c[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) c[k] = 0;
  // a box within [-1, 1] per axis takes the constant-mask path
  const bool unit = OP == kDilate && a.lo[0] >= -1 && a.lo[1] >= -1 && a.lo[2] >= -1 && a.hi[0] <= 1 &&
                    a.hi[1] <= 1 && a.hi[2] <= 1;
  (void)unit;
  for (uint32_t s = s0 + w; s < s1; s += 8) {
    const uint32_t val = __ldcg(vals + s);
    if constexpr (OP == kIjk) {  // the slot holds the voxel's bit n = 64 x + 8 y + z
      const uint64_t bit = 1ull << (val & 63u);
#pragma unroll
      for (int k = 0; k < 8; ++k) c[k] |= ((int)(val >> 6) == k) ? bit : 0ull;
    } else {
    uint64_t m[8];
    load_mask(a.src_masks, (long long)(val >> a.code_bits), m);
    const uint32_t code = val & ((1u << a.code_bits) - 1u);
    if (OP == kLeaves) {
#pragma unroll
      for (int k = 0; k < 8; ++k) c[k] |= m[k];
    } else if (OP == kCoarsen) {
      const int f = a.factor;
      if (f == 2) {
        const int qx = (code >> 2) & 1, qy = (code >> 1) & 1, qz = code & 1;
        uint64_t cw[4];
#pragma unroll
        for (int X = 0; X < 4; ++X) cw[X] = coarsen_word(m[2 * X] | m[2 * X + 1], qy, qz);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] |= ((k >> 2) == qx) ? cw[k & 3] : 0ull;
      } else {
        // coarse word k takes source words f (k - qx 8/f) .. + f - 1 when k
        // lies in the source's share qx 8/f .. (qx + 1) 8/f - 1
        const int sh = log2_factor(f), fm = f - 1, cs = 8 / f;
        const int qx = (int)(code >> (2 * sh)), qy = (int)(code >> sh) & fm, qz = (int)code & fm;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int X = k - qx * cs;
          if (X < 0 || X >= cs) continue;
          uint64_t t = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j / f == X) t |= m[j];
          c[k] |= coarsen_word_f(t, qy, qz, f);
        }
      }
    } else {  // kDilate
      const int tx = (int)(code / 9) - 1, ty = (int)((code / 3) % 3) - 1, tz = (int)(code % 3) - 1;
      if (unit) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          c[k] |= dilate_y1(dilate_z1(dilate_x1(m, k, tx, a.lo[0], a.hi[0]), tz, a.lo[2], a.hi[2]), ty, a.lo[1],
                            a.hi[1]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          c[k] |= dilate_y(dilate_z(dilate_x(m, k, tx, a.lo[0], a.hi[0]), tz, a.lo[2], a.hi[2]), ty, a.lo[1],
                           a.hi[1]);
      }
    }
    }
  }
  return reduce_scatter8(c, w);
  }
}

__device__ __forceinline__ uint32_t bits_of_bytes(uint64_t m) {
  uint32_t b = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if ((m >> (8 * r)) & 0xFFull) b |= 1u << r;
  return b;
}

// Inclusive min/max of the set voxels of a leaf from its 8-lane group's word
// (lane w holds word w); valid in every lane of the group.
__device__ __forceinline__ void leaf_bounds(uint64_t word, int w, int lane, int32_t mn[3], int32_t mx[3]) {
  uint64_t orm = word;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) orm |= __shfl_xor_sync(0xffffffffu, orm, off);
  const uint32_t xb = (__ballot_sync(0xffffffffu, word != 0) >> (lane & ~7)) & 0xFFu;
  const uint32_t yb = bits_of_bytes(orm);
  uint64_t z = orm | (orm >> 32);
  z |= z >> 16;
  z |= z >> 8;
  const uint32_t zb = (uint32_t)(z & 0xFFull);
  (void)w;
  mn[0] = __ffs(xb) - 1;
  mx[0] = 31 - __clz(xb);
  mn[1] = __ffs(yb) - 1;
  mx[1] = 31 - __clz(yb);
  mn[2] = __ffs(zb) - 1;
  mx[2] = 31 - __clz(zb);
}

// ---------------------------------------------------------------- dedup and index

constexpr uint32_t kGridFirst = 0x80000000u;  // leaf_upper flag: first leaf of its grid

// Head flags on the sorted keys -- a new leaf where the key changes, a new
// lower node where (grid, tile, upper child) changes, a new upper node where
// (grid, tile) changes, a new grid where the grid field changes -- and a
// 1024-slot tile scan of the three head counts with a warp-window look-back.
// Every unique leaf u gets its run start and (last pass) its lower / upper
// node indices, the upper index flagged when u is its grid's first leaf;
// each grid gets its first leaf / lower / upper indices.
__device__ void phase_index(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemDedup& s = sm.dedup;
  const uint64_t* keys = a.keys[a.sorted];
  long long S = (long long)__ldcg(&a.rb->num_slots);
  if (S > a.slot_cap) S = a.slot_cap;
  const long long ntiles = (S + kDedupTile - 1) / kDedupTile;
  const int lb = a.K.lower_bits, nb = a.K.node_bits, gsh = a.K.gw ? a.K.gshift : 64;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t B = a.B;
  constexpr unsigned long long M21 = (1ull << 21) - 1;
  for (long long tile = vb; tile < ntiles; tile = next_tile(&a.ctl->dedup_tile_ctr, ntiles, vg, s.tile)) {
    const long long i0 = tile * kDedupTile + (long long)tid * kDedupItems;
    uint64_t prev = (i0 > 0 && i0 - 1 < S) ? __ldcg(keys + i0 - 1) : 0ull;
    uint64_t kk[kDedupItems];
    uint32_t fl[kDedupItems];
    unsigned long long c = 0;
#pragma unroll
    for (int j = 0; j < kDedupItems; ++j) {
      const long long i = i0 + j;
      fl[j] = 0;
      kk[j] = 0;
      if (i < S) {
        const uint64_t key = __ldcg(keys + i);
        kk[j] = key;
        const bool first = (i == 0);
        const bool hl = first || key != prev;
        const bool hlo = first || shr64(key, lb) != shr64(prev, lb);
        const bool hup = first || shr64(key, nb) != shr64(prev, nb);
        const bool hg = first || shr64(key, gsh) != shr64(prev, gsh);
        fl[j] = (hl ? 1u : 0u) | (hlo ? 2u : 0u) | (hup ? 4u : 0u) | (hg ? 8u : 0u);
        c += (hl ? 1ull : 0ull) | (hlo ? (1ull << 21) : 0ull) | (hup ? (1ull << 42) : 0ull);
        prev = key;
      }
    }
    unsigned long long tot;
    const unsigned long long ex = block_excl_scan_256(c, s.scan, &tot);
    if (warp < 3) {
      const unsigned long long field = (tot >> (21 * warp)) & M21;
      lb64_publish(a.dedup_status + warp, 3, tile, field, false);
      const unsigned long long b = lb64_resolve(a.dedup_status + warp, 3, tile, field, false, a.err);
      if (lane == 0) {
        s.base[warp] = b;
        if (field) atomicAdd(&a.ctl->head_totals[warp], field);
      }
    }
    __syncthreads();
    unsigned long long cl = s.base[0] + (ex & M21);
    unsigned long long clo = s.base[1] + ((ex >> 21) & M21);
    unsigned long long cup = s.base[2] + ((ex >> 42) & M21);
#pragma unroll
    for (int j = 0; j < kDedupItems; ++j) {
      if (!(fl[j] & 1u)) continue;
      if (fl[j] & 2u) ++clo;
      if (fl[j] & 4u) ++cup;
      const unsigned long long u = cl++;
      a.run_start[u] = (uint32_t)(i0 + j);
      if (!a.last) continue;
      a.leaf_lower[u] = (uint32_t)(clo - 1);
      a.leaf_upper[u] = (uint32_t)(cup - 1) | ((fl[j] & 8u) ? kGridFirst : 0u);
      if (fl[j] & 8u) {
        const uint32_t g = (uint32_t)shr64(kk[j], gsh);
        if (g < (uint32_t)B) {
          a.first[g] = (uint32_t)(u + 1);
          a.first[B + g] = (uint32_t)clo;
          a.first[2 * B + g] = (uint32_t)cup;
        }
      }
    }
    __syncthreads();
  }
}

// out[g] = first index of the first non-empty grid >= g, or `total`; out[B] = total.
__device__ void suffix_fill(const uint32_t* first, int32_t B, unsigned long long total, int64_t* out, Smem& sm) {
  uint32_t* s = sm.fin.s;
  const int tid = threadIdx.x;
  uint32_t carry = 0xFFFFFFFFu;
  if (B > 0) {
    for (long long base = ((long long)(B - 1) / kThreads) * kThreads; base >= 0; base -= kThreads) {
      const long long g = base + tid;
      uint32_t v = 0xFFFFFFFFu;
      if (g < B) {
        const uint32_t f = __ldcg(first + g);
        if (f) v = f - 1;
      }
      s[tid] = v;
      __syncthreads();
      for (int off = 1; off < kThreads; off <<= 1) {
        const uint32_t t = (tid + off < kThreads) ? s[tid + off] : 0xFFFFFFFFu;
        __syncthreads();
        s[tid] = min(s[tid], t);
        __syncthreads();
      }
      const uint32_t res = min(s[tid], carry);
      if (g < B) out[g] = (res == 0xFFFFFFFFu) ? (int64_t)total : (int64_t)res;
      carry = min(carry, s[0]);
      __syncthreads();
    }
  }
  if (tid == 0) out[B] = (int64_t)total;
}

// Block 0 after the index phase: totals, run sentinel, per-grid offsets.
__device__ void phase_finish(const PassArgs& a, Smem& sm) {
  long long S = (long long)__ldcg(&a.rb->num_slots);
  if (S > a.slot_cap) S = a.slot_cap;
  const unsigned long long U = __ldcg(&a.ctl->head_totals[0]);
  const unsigned long long NL = __ldcg(&a.ctl->head_totals[1]);
  const unsigned long long NU = __ldcg(&a.ctl->head_totals[2]);
  if (threadIdx.x == 0) {
    a.rb->num_leaves = U;
    a.rb->num_lowers = NL;
    a.rb->num_uppers = NU;
    a.run_start[U] = (uint32_t)S;
  }
  if (a.last) {
    suffix_fill(a.first, a.B, U, a.leaf_off, sm);
    suffix_fill(a.first + a.B, a.B, NL, a.lower_off, sm);
    suffix_fill(a.first + 2 * a.B, a.B, NU, a.upper_off, sm);
  }
}

// Leaves of the pass, spread over the whole grid: block b takes a contiguous
// range of leaves and each of its 8-lane groups a contiguous sub-range, so a
// group sees its leaves in grid order.  Per leaf the run of slots is merged;
//  - last pass: popcount and bbox (grid bboxes accumulate per group and reach
//    memory once per grid change), per-leaf voxels, and the segmented voxel
//    aggregate of each group and block (segments start at grid-first leaves);
//  - intermediate pass: the merged leaves for the next pass.
template <int OP>
__device__ void phase_leaves(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemLeaves& s = sm.lv;
  const uint64_t* keys = a.keys[a.sorted];
  const uint32_t* vals = a.vals[a.sorted];
  long long S = (long long)__ldcg(&a.rb->num_slots);
  if (S > a.slot_cap) S = a.slot_cap;
  const long long U = (long long)__ldcg(&a.ctl->head_totals[0]);
  const int tid = threadIdx.x, lane = tid & 31, w = tid & 7, grp = tid >> 3;
  const long long C = (U + vg - 1) / vg;
  const long long c = (C + kThreads / 8 - 1) / (kThreads / 8);
  const long long bbeg = (long long)vb * C, bend = bbeg + C < U ? bbeg + C : U;
  const long long gbeg = bbeg + grp * c, gend = gbeg + c < bend ? gbeg + c : bend;
  constexpr int kU = OP == kRefine ? 4 : 1;
  uint32_t acc_g = 0xFFFFFFFFu, F = 0;
  unsigned int acc_e = 0;
  unsigned long long V = 0;
  for (long long q = 0; q < c; q += kU) {
    uint64_t word[kU];
    uint32_t gg[kU];
    int32_t lcs[kU][3];
    bool valid[kU];
#pragma unroll
    for (int r = 0; r < kU; ++r) {
      const long long u = gbeg + q + r;
      valid[r] = u < gend;
      uint32_t s0 = 0, s1 = 0;
      gg[r] = 0;
      lcs[r][0] = lcs[r][1] = lcs[r][2] = 0;
      if (valid[r]) {
        if (S == U) {  // every run is one slot (refinement): leaf u is slot u
          s0 = (uint32_t)u;
          s1 = (uint32_t)u + 1;
        } else {
          s0 = __ldcg(a.run_start + u);
          s1 = u + 1 < U ? __ldcg(a.run_start + u + 1) : (uint32_t)S;
        }
        decode_key(a.K, __ldcg(keys + s0), gg[r], lcs[r]);
      }
      word[r] = merge_run<OP>(a, vals, s0, s1, w);
    }
#pragma unroll
    for (int r = 0; r < kU; ++r) {
      const long long u = gbeg + q + r;
      const uint32_t g = gg[r];
      if (a.last) {
        uint32_t pop = __popcll(word[r]);
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) pop += __shfl_xor_sync(0xffffffffu, pop, off);
        int32_t mn[3], mx[3];
        leaf_bounds(word[r], w, lane, mn, mx);
        if (valid[r]) {
          if (w < 6) {
            const int ax = w < 3 ? w : w - 3;
            const int32_t o = (int32_t)((uint32_t)lcs[r][ax] << 3);
            const unsigned int e = w < 3 ? enc_min(o + mn[ax]) : enc_max(o + mx[ax]);
            if (g != acc_g) {
              if (acc_g != 0xFFFFFFFFu) atomicMax(&a.gbox[6 * acc_g + w], acc_e);
              acc_g = g;
              acc_e = e;
            } else {
              acc_e = max(acc_e, e);
            }
          }
          if (w == 0) {
            a.leaf_pop[u] = pop;
            a.leaf_g[u] = g;
          }
          if (a.out_masks) {
            a.out_masks[8 * u + w] = word[r];
            if (w < 3) a.out_origins[3 * u + w] = (int32_t)((uint32_t)lcs[r][w] << 3);
          }
          if (__ldcg(a.leaf_upper + u) & kGridFirst) {
            F = 1;
            V = pop;
          } else {
            V += pop;
          }
        }
      } else if (valid[r]) {
        a.out_masks[8 * u + w] = word[r];
        if (w < 3) a.out_origins[3 * u + w] = (int32_t)((uint32_t)lcs[r][w] << 3);
        if (w == 3) a.out_grid[u] = (int32_t)g;
      }
    }
  }
  if (!a.last) return;
  if (w == 0) {
    s.grp_f[grp] = F;
    s.grp_v[grp] = V;
    s.grp_g[grp] = acc_g;
    a.grp_agg[(long long)vb * (kThreads / 8) + grp] = ((unsigned long long)F << 63) | V;
  }
  if (w < 6) s.grp_box[grp][w] = acc_e;
  __syncthreads();
  if (tid < 6) {  // grid bboxes: one atomic per grid run of the groups
    uint32_t cg = 0xFFFFFFFFu;
    unsigned int ce = 0;
    for (int j = 0; j < kThreads / 8; ++j) {
      const uint32_t gj = s.grp_g[j];
      if (gj == 0xFFFFFFFFu) continue;
      const unsigned int ej = s.grp_box[j][tid];
      if (gj == cg) {
        ce = max(ce, ej);
      } else {
        if (cg != 0xFFFFFFFFu) atomicMax(&a.gbox[6 * cg + tid], ce);
        cg = gj;
        ce = ej;
      }
    }
    if (cg != 0xFFFFFFFFu) atomicMax(&a.gbox[6 * cg + tid], ce);
  }
  if (tid == 32) {  // the block's segmented voxel aggregate
    uint32_t bf = 0;
    unsigned long long bv = 0;
    for (int j = 0; j < kThreads / 8; ++j) {
      bv = s.grp_f[j] ? s.grp_v[j] : bv + s.grp_v[j];
      bf |= s.grp_f[j];
    }
    a.blk_agg[vb] = ((unsigned long long)bf << 63) | bv;
  }
}

// After a grid barrier: each block reads the aggregates of the blocks before
// it (complete, so no waiting) for its carried-in voxel count; each group then
// scans its leaves eight at a time and writes their per-grid voxel offsets,
// and every grid's last leaf writes the grid's voxel total.
__device__ void phase_voxel_offsets(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemLeaves& s = sm.lv;
  const long long U = (long long)__ldcg(&a.ctl->head_totals[0]);
  const int tid = threadIdx.x, lane = tid & 31, w = tid & 7, grp = tid >> 3;
  if (tid < 32) {
    unsigned long long carry = 0;
    for (long long base = (long long)vb - 1; base >= 0; base -= 32) {
      const long long b = base - lane;
      const unsigned long long e = b >= 0 ? __ldcg(a.blk_agg + b) : (1ull << 63);
      const uint32_t stop = __ballot_sync(0xffffffffu, (e >> 63) != 0);
      const int first = stop ? __ffs(stop) - 1 : 32;
      unsigned long long v = (lane <= first && b >= 0) ? (e & ~(1ull << 63)) : 0ull;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      carry += v;
      if (first < 32) break;
    }
    // carried-in value of each group: the block's prefix, then the groups before it
    const unsigned long long ga = __ldcg(a.grp_agg + (long long)vb * (kThreads / 8) + lane);
    const uint32_t gf = (uint32_t)(ga >> 63);
    unsigned long long gv = ga & ~(1ull << 63);
    uint32_t F = gf;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t F2 = __shfl_up_sync(0xffffffffu, F, off);
      const unsigned long long V2 = __shfl_up_sync(0xffffffffu, gv, off);
      if (lane >= off) {
        if (!F) gv += V2;
        F |= F2;
      }
    }
    uint32_t Fe = __shfl_up_sync(0xffffffffu, F, 1);
    unsigned long long Ve = __shfl_up_sync(0xffffffffu, gv, 1);
    if (lane == 0) {
      Fe = 0;
      Ve = 0;
    }
    s.grp_prefix[lane] = Fe ? Ve : carry + Ve;
  }
  __syncthreads();
  const long long C = (U + vg - 1) / vg;
  const long long c = (C + kThreads / 8 - 1) / (kThreads / 8);
  const long long bbeg = (long long)vb * C, bend = bbeg + C < U ? bbeg + C : U;
  const long long gbeg = bbeg + grp * c, gend = gbeg + c < bend ? gbeg + c : bend;
  unsigned long long cv = s.grp_prefix[grp];
  const uint32_t gmask = 0xFFu << (lane & ~7);
  for (long long base = gbeg; base < gend; base += 8) {  // uniform within the group
    const long long u = base + w;
    const bool valid = u < gend;
    const uint32_t pop = valid ? __ldcg(a.leaf_pop + u) : 0u;
    const uint32_t f = valid ? ((__ldcg(a.leaf_upper + u) & kGridFirst) ? 1u : 0u) : 0u;
    uint32_t Fi = f;
    unsigned long long Vi = pop;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const uint32_t F2 = __shfl_up_sync(gmask, Fi, off, 8);
      const unsigned long long V2 = __shfl_up_sync(gmask, Vi, off, 8);
      if (w >= off) {
        if (!Fi) Vi += V2;
        Fi |= F2;
      }
    }
    uint32_t Fe = __shfl_up_sync(gmask, Fi, 1, 8);
    unsigned long long Ve = __shfl_up_sync(gmask, Vi, 1, 8);
    if (w == 0) {
      Fe = 0;
      Ve = 0;
    }
    const unsigned long long off = f ? 0ull : (Fe ? Ve : cv + Ve);
    if (valid) {
      a.leaf_voff[u] = (long long)off;
      const bool last = (u + 1 == U) || (__ldcg(a.leaf_upper + u + 1) & kGridFirst);
      if (last) a.grid_vox[__ldcg(a.leaf_g + u)] = (long long)(off + pop);
    }
    const uint32_t Ft = __shfl_sync(gmask, Fi, 7, 8);
    const unsigned long long Vt = __shfl_sync(gmask, Vi, 7, 8);
    cv = Ft ? Vt : cv + Vt;
  }
}

// ---------------------------------------------------------------- node path phases

// After the emission: a warp per lower node (in the list the emission kept)
// takes its child mask's popcount prefix per word and its leaf count,
// and ranks the node among all nodes by canonical key (node keys are
// unique); a warp per tile ranks the tile.  The per-grid first node and tile
// ranks and the totals follow.  With node_zero == 1 the staged masks of the
// pass's slots are cleared here too.
__device__ __noinline__ void phase_nodes(const PassArgs& a, int vb, int vg) {
  const uint32_t n = min(__ldcg(&a.ctl->n_nodes), (uint32_t)a.node_cap);
  const uint32_t nt = min(__ldcg(&a.ctl->n_tiles), (uint32_t)a.node_cap);
  const int lane = threadIdx.x & 31;
  const KeyLayout& K = a.K;
  const long long nw = (long long)vg * (kThreads / 32);
  for (long long it = (long long)vb * (kThreads / 32) + (threadIdx.x >> 5); it < (long long)n + nt; it += nw) {
    if (it < (long long)n) {  // a lower node
      const uint32_t id = __ldcg(a.node_list + it);
      const unsigned long long k1 = __ldcg(a.nh_key + id);
      const uint64_t* m = a.node_mask + 64ull * id;
      const uint64_t x0 = __ldcg(m + 2 * lane), x1 = __ldcg(m + 2 * lane + 1);
      const uint32_t c0 = __popcll(x0), c = c0 + __popcll(x1);
      uint32_t incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      a.node_wpre[64ull * id + 2 * lane] = incl - c;
      a.node_wpre[64ull * id + 2 * lane + 1] = incl - c + c0;
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t r = 0;  // the nodes that sort before this one
      for (uint32_t j = lane; j < n; j += 32) r += __ldcg(a.nh_key + __ldcg(a.node_list + j)) < k1 ? 1u : 0u;
      r = __reduce_add_sync(0xffffffffu, r);
      if (lane == 0) {
        a.node_rank[id] = r;
        a.rank_cnt[r] = total;
        atomicAdd(&a.ctl->head_totals[0], (unsigned long long)total);
        atomicMax(a.gmin + __ldcg(a.node_lc + 4ull * id + 3), ~r);
      }
    } else {  // a tile
      const uint32_t t = __ldcg(a.tile_list + (it - n));
      const unsigned long long k1 = __ldcg(a.th_key + t);
      uint32_t r = 0;
      for (uint32_t j = lane; j < nt; j += 32) r += __ldcg(a.th_key + __ldcg(a.tile_list + j)) < k1 ? 1u : 0u;
      r = __reduce_add_sync(0xffffffffu, r);
      if (lane == 0) {
        a.tile_rank[t] = r;
        const uint32_t g = K.gw ? (uint32_t)shr64(k1 - 1ull, K.gshift - K.node_bits) : 0u;
        atomicMax(a.gmin + a.B + g, ~r);
      }
    }
  }
  if (a.node_zero == 1) {  // clear the staged masks of up to one leaf per slot
    long long S = (long long)__ldcg(&a.rb->num_slots);
    if (S > a.slot_cap) S = a.slot_cap;
    uint4* z = reinterpret_cast<uint4*>(a.out_masks);
    for (long long i = (long long)vb * kThreads + threadIdx.x; i < 4 * S; i += (long long)vg * kThreads)
      z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The clear phase of node_zero == 2: the staged masks of the pass's leaves.
__device__ void phase_clear(const PassArgs& a, int vb, int vg) {
  const long long U = (long long)__ldcg(&a.ctl->head_totals[0]);
  uint4* z = reinterpret_cast<uint4*>(a.out_masks);
  for (long long i = (long long)vb * kThreads + threadIdx.x; i < 4 * U; i += (long long)vg * kThreads)
    z[i] = make_uint4(0u, 0u, 0u, 0u);
}

// The eight words of one target's contribution to its target leaf, from the
// source leaf's mask m (target code `code`; for the ijk front end `code` is
// the voxel's bit n = 64 x + 8 y + z in its leaf).
template <int OP>
__device__ __forceinline__ void contrib_words(const PassArgs& a, const uint64_t m[8], uint32_t code, uint64_t c[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) c[k] = 0;
  if constexpr (OP == kIjk) {
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = ((int)(code >> 6) == k) ? 1ull << (code & 63u) : 0ull;
  } else if constexpr (OP == kLeaves) {
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = m[k];
  } else if constexpr (OP == kRefine) {
    const int f = a.factor;
    if (f == 2) {  // child (cx, cy, cz): word k from parent word 4 cx + k / 2
      const int cx = (code >> 2) & 1, cy = (code >> 1) & 1, cz = code & 1;
#pragma unroll
      for (int k = 0; k < 8; ++k) c[k] = refine_word(cx ? m[4 + (k >> 1)] : m[k >> 1], cy, cz);
      return;
    }
    const int cx = (int)code / (f * f), cy = ((int)code / f) % f, cz = (int)code % f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int j = (8 * cx + k) / f;
      uint64_t pw = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) pw = q == j ? m[q] : pw;
      c[k] = refine_word_f(pw, cy, cz, f);
    }
  } else if constexpr (OP == kCoarsen) {
    const int f = a.factor;
    if (f == 2) {
      const int qx = (code >> 2) & 1, qy = (code >> 1) & 1, qz = code & 1;
#pragma unroll
      for (int X = 0; X < 4; ++X) {
        const uint64_t cw = coarsen_word(m[2 * X] | m[2 * X + 1], qy, qz);
        c[X] = qx == 0 ? cw : 0ull;
        c[4 + X] = qx == 1 ? cw : 0ull;
      }
    } else {
      const int sh = log2_factor(f), fm = f - 1, cs = 8 / f;
      const int qx = (int)(code >> (2 * sh)), qy = (int)(code >> sh) & fm, qz = (int)code & fm;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int X = k - qx * cs;
        if (X < 0 || X >= cs) continue;
        uint64_t t = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j / f == X) t |= m[j];
        c[k] = coarsen_word_f(t, qy, qz, f);
      }
    }
  } else if constexpr (OP == kRefineDilate) {
    // word w: along x the fine positions 8 tx + w - d inside the refined
    // 16^3 block (source words (8 tx + w - d) / 2), along y and z the child
    // quadrants whose dilation reaches the target
    const int tx = (int)(code >> 4) - 1, ty = ((int)(code >> 2) & 3) - 1, tz = ((int)code & 3) - 1;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint64_t mx = 0;
      for (int d = a.lo[0]; d <= a.hi[0]; ++d) {
        const int fx = 8 * tx + w - d;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (fx >= 0 && fx < 16 && (fx >> 1) == q) mx |= m[q];
      }
      if (!mx) continue;
      uint64_t word = 0;
#pragma unroll
      for (int cy = 0; cy < 2; ++cy) {
        const int dy = ty - cy;
        if (dy < -1 || dy > 1 || (dy < 0 && a.lo[1] >= 0) || (dy > 0 && a.hi[1] <= 0)) continue;
#pragma unroll
        for (int cz = 0; cz < 2; ++cz) {
          const int dz = tz - cz;
          if (dz < -1 || dz > 1 || (dz < 0 && a.lo[2] >= 0) || (dz > 0 && a.hi[2] <= 0)) continue;
          if (!(mx & (0x0F0F0F0Full << (32 * cy + 4 * cz)))) continue;
          word |= dilate_y1(dilate_z1(refine_word(mx, cy, cz), dz, a.lo[2], a.hi[2]), dy, a.lo[1], a.hi[1]);
        }
      }
      c[w] = word;
    }
  } else {  // kDilate
    const int tx = (int)(code / 9) - 1, ty = (int)((code / 3) % 3) - 1, tz = (int)(code % 3) - 1;
    if (a.lo[0] >= -1 && a.lo[1] >= -1 && a.lo[2] >= -1 && a.hi[0] <= 1 && a.hi[1] <= 1 && a.hi[2] <= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        c[k] = dilate_y1(dilate_z1(dilate_x1(m, k, tx, a.lo[0], a.hi[0]), tz, a.lo[2], a.hi[2]), ty, a.lo[1],
                         a.hi[1]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        c[k] = dilate_y(dilate_z(dilate_x(m, k, tx, a.lo[0], a.hi[0]), tz, a.lo[2], a.hi[2]), ty, a.lo[1], a.hi[1]);
    }
  }
}

// One item of a node-path sweep: source idx / nchunks (a leaf, or a voxel
// for the ijk front end) and its chunk of targets.  Loads the source (mask
// m, leaf coordinate lc -- voxel coordinate for the ijk front end -- and
// grid g) and tests the chunk's targets: bit t - t0 of `bits` is set for
// each non-empty target t.
template <int OP>
__device__ __forceinline__ void node_item(const PassArgs& a, long long idx, uint32_t k, uint32_t T, uint32_t nchunks,
                                          uint64_t m[8], int32_t lc[3], uint32_t& g, long long& i, uint32_t& t0,
                                          uint32_t& bits) {
  i = idx / nchunks;
  t0 = (uint32_t)(idx - i * nchunks) * k;
  const uint32_t t1 = t0 + k < T ? t0 + k : T;
  bits = 0;
  if (OP == kIjk) {
    lc[0] = __ldg(a.ijk + 3 * i);
    lc[1] = __ldg(a.ijk + 3 * i + 1);
    lc[2] = __ldg(a.ijk + 3 * i + 2);
    g = (uint32_t)grid_of(a.in_offsets, a.B, i);
    bits = 1u;
    return;
  }
  load_mask(a.src_masks, i, m);
  lc[0] = __ldcg(a.src_origins + 3 * i) >> 3;
  lc[1] = __ldcg(a.src_origins + 3 * i + 1) >> 3;
  lc[2] = __ldcg(a.src_origins + 3 * i + 2) >> 3;
  for (uint32_t t = t0; t < t1; ++t) {
    uint32_t code;
    int32_t tl[3];
    if (target_nonempty<OP>(a, m, lc, t, code, tl)) bits |= 1u << (t - t0);
  }
  g = bits ? (a.src_grid ? (uint32_t)__ldcg(a.src_grid + i) : (uint32_t)grid_of(a.in_offsets, a.B, i)) : 0u;
}

// Target t of an item: its code (the ijk front end: the voxel's bit in its
// leaf), leaf coordinate tl and canonical key.
template <int OP>
__device__ __forceinline__ uint64_t node_target(const PassArgs& a, const int32_t lc[3], uint32_t g, uint32_t t,
                                                uint32_t& code, int32_t tl[3]) {
  if (OP == kIjk) {
    tl[0] = lc[0] >> 3;
    tl[1] = lc[1] >> 3;
    tl[2] = lc[2] >> 3;
    code = (uint32_t)(((lc[0] & 7) << 6) | ((lc[1] & 7) << 3) | (lc[2] & 7));
  } else {
    target_geometry<OP>(a, lc, t, code, tl);
  }
  return encode_key(a.K, g, tl[0], tl[1], tl[2]);
}

// The warp's first look-ups of an item step: each lane's first non-empty
// target's lower node, one table look-up per distinct node of the warp (the
// lanes of a warp work on neighbouring sources), into the lanes' caches.
template <int OP>
__device__ __forceinline__ void node_prime(const PassArgs& a, SmemNodes* sn, const int32_t lc[3], uint32_t g,
                                           uint32_t bits, uint32_t t0, uint64_t& cache_nk, uint32_t& cache_id,
                                           int& cache_slot) {
  const int lane = threadIdx.x & 31;
  uint64_t nk = 0, key = 0;
  int32_t tl[3] = {0, 0, 0};
  if (bits) {
    uint32_t code;
    key = node_target<OP>(a, lc, g, t0 + (uint32_t)(__ffs(bits) - 1), code, tl);
    nk = shr64(key, a.K.lower_bits);
  }
  const bool need = bits && nk + 1ull != cache_nk;
  const uint32_t nmask = __ballot_sync(0xffffffffu, need);
  if (!nmask) return;
  const uint32_t peers = __match_any_sync(0xffffffffu, nk) & nmask;
  const int leader = need ? __ffs(peers) - 1 : lane;
  uint32_t id = 0;
  int slot = -1;
  if (need && lane == leader) id = node_lookup(a, sn, nk, key, tl, g, slot);
  id = __shfl_sync(0xffffffffu, id, leader);
  slot = __shfl_sync(0xffffffffu, slot, leader);
  if (need) {
    cache_nk = nk + 1ull;
    cache_id = id;
    cache_slot = slot;
  }
}

// Leaves before the node of each rank (exclusive scan of the nodes' leaf
// counts in rank order) into shared memory, by every block for itself.
__device__ __forceinline__ uint32_t scan_node_bases(const PassArgs& a, SmemPlace& s) {
  const uint32_t n = min(__ldcg(&a.ctl->n_nodes), (uint32_t)a.node_cap);
  uint32_t carry = 0;
  for (uint32_t c0 = 0; c0 < n; c0 += kThreads) {
    const uint32_t i = c0 + threadIdx.x;
    const uint32_t v = i < n ? __ldcg(a.rank_cnt + i) : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan_256(v, s.scan, &tot);
    if (i < n) s.base[i] = carry + ex;
    carry += tot;
  }
  __syncthreads();
  return n;
}

// The place phase.  Every block scans the node leaf counts in rank order
// into shared memory (the leaves before each node).  Then, a thread per slot
// over the whole grid: the slot's target leaf is one set bit of its lower
// node's child mask, and its index is the node's base plus the set bits
// before it; the leaf's record (origin, grid, links) is written -- by every
// slot of the leaf alike -- and the slot's contribution, computed from its
// source mask, is merged into the leaf's staged mask (stored where each leaf
// has one slot, else OR-ed into the cleared masks).
template <int OP>
__device__ __noinline__ void phase_place(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemPlace& s = sm.place;
  const int tid = threadIdx.x;
  scan_node_bases(a, s);
  const int32_t B = a.B;
  if (vb == 0 && tid == 0) {  // the pass's lower and upper node totals
    a.ctl->head_totals[1] = __ldcg(&a.ctl->n_nodes);
    a.ctl->head_totals[2] = __ldcg(&a.ctl->n_tiles);
  }
  if (vb == 0 && a.last) {  // 1 + first leaf / lower / upper index of every grid (0: empty grid)
    for (int g = tid; g < B; g += kThreads) {
      const uint32_t el = __ldcg(a.gmin + g), eu = __ldcg(a.gmin + B + g);
      a.first[g] = el ? s.base[~el] + 1u : 0u;
      a.first[B + g] = el ? ~el + 1u : 0u;
      a.first[2 * B + g] = eu ? ~eu + 1u : 0u;
    }
  }
  // Node tables are read-only from here on and no SM has loaded them into its
  // L1 before (they were written by stores and atomics and read at L2), so
  // they are read through L1.
  const long long nthreads = (long long)vg * kThreads, gt = (long long)vb * kThreads + tid;
  long long S = (long long)__ldcg(&a.rb->num_slots);
  if (S > a.slot_cap) S = a.slot_cap;
  for (long long sl = gt; sl < S; sl += nthreads) {
    const uint32_t nref = __ldcg(a.nref + sl), val = __ldcg(a.vals[0] + sl);
    const uint32_t id = nref >> 12, bit = nref & 4095u;
    const uint64_t mw = __ldca(a.node_mask + 64ull * id + (bit >> 6));
    const uint32_t rank = __ldca(a.node_rank + id), wpre = __ldca(a.node_wpre + 64ull * id + (bit >> 6));
    const int32_t* lc = a.node_lc + 4ull * id;
    const int32_t g = __ldca(lc + 3);
    const long long u = (long long)s.base[rank] + wpre + __popcll(mw & ((1ull << (bit & 63u)) - 1ull));
    // the leaf's record (every slot of a leaf writes the same one)
    int32_t* o = a.out_origins + 3 * u;
    o[0] = (int32_t)(((uint32_t)__ldca(lc) << 7) | ((bit >> 8) << 3));
    o[1] = (int32_t)(((uint32_t)__ldca(lc + 1) << 7) | (((bit >> 4) & 15u) << 3));
    o[2] = (int32_t)(((uint32_t)__ldca(lc + 2) << 7) | ((bit & 15u) << 3));
    if (a.last) {
      const bool f = ~__ldca(a.gmin + g) == rank && u == (long long)s.base[rank];
      a.leaf_g[u] = (uint32_t)g;
      a.leaf_lower[u] = rank;
      a.leaf_upper[u] = __ldca(a.tile_rank + __ldca(a.node_tile + id)) | (f ? kGridFirst : 0u);
    } else {
      a.out_grid[u] = g;
    }
    uint64_t m[8];
    uint32_t code = val;
    if (OP != kIjk) {
      load_mask(a.src_masks, (long long)(val >> a.code_bits), m);
      code = val & ((1u << a.code_bits) - 1u);
    }
    uint64_t c[8];
    contrib_words<OP>(a, m, code, c);
    if (a.node_zero == 0) {  // the leaf's only contribution
      uint4* d = reinterpret_cast<uint4*>(a.out_masks + 8 * u);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        d[w] = make_uint4((uint32_t)c[2 * w], (uint32_t)(c[2 * w] >> 32), (uint32_t)c[2 * w + 1],
                          (uint32_t)(c[2 * w + 1] >> 32));
    } else {
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (c[w]) atomicOr(reinterpret_cast<unsigned long long*>(a.out_masks + 8 * u + w), (unsigned long long)c[w]);
    }
  }
}

__device__ void dispatch_place(const PassArgs& a, Smem& sm, int vb, int vg) {
  switch (a.op) {
    case kIjk: phase_place<kIjk>(a, sm, vb, vg); break;
    case kLeaves: phase_place<kLeaves>(a, sm, vb, vg); break;
    case kRefine: phase_place<kRefine>(a, sm, vb, vg); break;
    case kCoarsen: phase_place<kCoarsen>(a, sm, vb, vg); break;
    case kRefineDilate: phase_place<kRefineDilate>(a, sm, vb, vg); break;
    default: phase_place<kDilate>(a, sm, vb, vg); break;
  }
}

// Middle phase d of a node-path pass: nodes, [clear,] place.
__device__ void node_middle(const PassArgs& a, int d, Smem& sm, int vb, int vg) {
  if (d == 0) {
    phase_nodes(a, vb, vg);
  } else if (d + 1 < a.mid) {
    phase_clear(a, vb, vg);
  } else {
    stamp(a, 2);
    dispatch_place(a, sm, vb, vg);
    stamp(a, 3);
  }
}

// The node path's emission: calls of their own, so that their node tables'
// state does not weigh on the rest of the kernel's registers.
// Items of one thread tested before one slot claim in a node-path emission.
constexpr int kNodeItems = 8;

template <int OP>
__device__ __noinline__ void emit_node(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemNodes& sn = sm.nodes;
  for (int i = threadIdx.x; i < kNodeSlots * 129; i += kThreads) {
    if (i < kNodeSlots) sn.id[i] = 0u;
    else (&sn.mask[0][0])[i - kNodeSlots] = 0u;
  }
  __syncthreads();
  const long long ns = a.src_count_dev ? (long long)__ldcg(a.src_count_dev) : a.src_count;
  const uint32_t T = targets_per_source<OP>(a);
  uint32_t k = (a.tchunk > 0 && (uint32_t)a.tchunk < T) ? (uint32_t)a.tchunk : T;
  if (k > 32) k = 32;  // a thread's targets are one 32-bit set
  const uint32_t nchunks = (T + k - 1) / k;
  const long long items = ns * (long long)nchunks;
  const long long stride = (long long)vg * kThreads;
  // each thread a run of consecutive items (neighbouring sources share nodes)
  const long long gt = (long long)vb * kThreads + threadIdx.x;
  const long long per = (items + stride - 1) / stride;
  uint64_t cache_nk = 0;  // the thread's last lower node (key + 1; 0: none), its id and block slot
  uint32_t cache_id = 0;
  int cache_slot = -1;
  NodeRun run{0u, 0u, 0u, -1};
  for (long long qb = 0; qb < per; qb += kNodeItems) {  // uniform
  // first the tests of up to kNodeItems items, so the warp claims their slots at once
  uint32_t bits[kNodeItems];
  uint32_t cnt = 0;
#pragma unroll
  for (int q = 0; q < kNodeItems; ++q) {
    bits[q] = 0;
    const long long idx = gt * per + qb + q;
    if (qb + q < per && idx < items) {
      uint64_t m[8];
      int32_t lc[3];
      uint32_t g, t0;
      long long i;
      node_item<OP>(a, idx, k, T, nchunks, m, lc, g, i, t0, bits[q]);
      cnt += __popc(bits[q]);
    }
  }
  unsigned long long wbase;
  uint32_t wtotal;
  unsigned long long pos = claim_slots(a, cnt, wbase, wtotal);
#pragma unroll 1
  for (int q = 0; q < kNodeItems; ++q) {  // uniform
    if (qb + q >= per) break;
    const long long idx = gt * per + qb + q;
    uint32_t b = bits[0];
#pragma unroll
    for (int j = 1; j < kNodeItems; ++j) b = j == q ? bits[j] : b;
    int32_t lc[3] = {0, 0, 0};
    uint32_t g = 0, t0 = 0;
    long long i = 0;
    if (b) {  // the item's source again (its mask is not needed)
      i = idx / nchunks;
      t0 = (uint32_t)(idx - i * nchunks) * k;
      if (OP == kIjk) {
        lc[0] = __ldg(a.ijk + 3 * i);
        lc[1] = __ldg(a.ijk + 3 * i + 1);
        lc[2] = __ldg(a.ijk + 3 * i + 2);
        g = (uint32_t)grid_of(a.in_offsets, a.B, i);
      } else {
        lc[0] = __ldcg(a.src_origins + 3 * i) >> 3;
        lc[1] = __ldcg(a.src_origins + 3 * i + 1) >> 3;
        lc[2] = __ldcg(a.src_origins + 3 * i + 2) >> 3;
        g = a.src_grid ? (uint32_t)__ldcg(a.src_grid + i) : (uint32_t)grid_of(a.in_offsets, a.B, i);
      }
    }
    node_prime<OP>(a, &sn, lc, g, b, t0, cache_nk, cache_id, cache_slot);
    while (b) {
      const uint32_t t = t0 + (uint32_t)(__ffs(b) - 1);
      b &= b - 1;
      uint32_t code;
      int32_t tl[3];
      const uint64_t key = node_target<OP>(a, lc, g, t, code, tl);
      const uint64_t nk = shr64(key, a.K.lower_bits);
      if (nk + 1ull != cache_nk) {
        cache_id = node_lookup(a, &sn, nk, key, tl, g, cache_slot);
        cache_nk = nk + 1ull;
      }
      const uint32_t bit = ((uint32_t)(tl[0] & 15) << 8) | ((uint32_t)(tl[1] & 15) << 4) | (uint32_t)(tl[2] & 15);
      if (run.bits && (run.id != cache_id || run.w32 != (bit >> 5))) run_flush(a, sn, run);
      run.id = cache_id;
      run.slot = cache_slot;
      run.w32 = bit >> 5;
      run.bits |= 1u << (bit & 31u);
      put_node_slot(a, pos++, (cache_id << 12) | bit,
                    OP == kIjk ? code : (((uint32_t)i << a.code_bits) | code));
    }
  }
  }
  run_flush(a, sn, run);
  emit_flush(a, sn);
}

__device__ void dispatch_emit(const PassArgs& a, Smem& sm, int vb, int vg) {
  if (a.node) {
    switch (a.op) {
      case kIjk: emit_node<kIjk>(a, sm, vb, vg); break;
      case kLeaves: emit_node<kLeaves>(a, sm, vb, vg); break;
      case kRefine: emit_node<kRefine>(a, sm, vb, vg); break;
      case kCoarsen: emit_node<kCoarsen>(a, sm, vb, vg); break;
      case kRefineDilate: emit_node<kRefineDilate>(a, sm, vb, vg); break;
      default: emit_node<kDilate>(a, sm, vb, vg); break;
    }
    return;
  }
  switch (a.op) {
    case kIjk: phase_emit<kIjk>(a, sm, vb, vg); break;
    case kLeaves: phase_emit<kLeaves>(a, sm, vb, vg); break;
    case kRefine: phase_emit<kRefine>(a, sm, vb, vg); break;
    case kCoarsen: phase_emit<kCoarsen>(a, sm, vb, vg); break;
    case kRefineDilate: phase_emit<kRefineDilate>(a, sm, vb, vg); break;
    default: phase_emit<kDilate>(a, sm, vb, vg); break;
  }
}

// The fused refine-then-dilate leaves phase as a call of its own: inlined,
// its register peak would push the whole kernel past 128 registers a thread.
__device__ __noinline__ void leaves_refine_dilate(const PassArgs& a, Smem& sm, int vb, int vg) {
  phase_leaves<kRefineDilate>(a, sm, vb, vg);
}

// The node path's leaves phase (last pass), a call of its own: the records
// are placed already, so a thread takes a leaf -- each 8-lane group eight
// consecutive leaves of its range at a time -- for its popcount and bbox, and
// the group carries the segmented voxel aggregate and the grid bbox as the
// leaves phase above does.
__device__ __noinline__ void leaves_staged(const PassArgs& a, Smem& sm, int vb, int vg) {
  SmemLeaves& s = sm.lv;
  const long long U = (long long)__ldcg(&a.ctl->head_totals[0]);
  const int tid = threadIdx.x, lane = tid & 31, w = tid & 7, grp = tid >> 3;
  const long long C = (U + vg - 1) / vg;
  const long long c = (C + kThreads / 8 - 1) / (kThreads / 8);
  const long long bbeg = (long long)vb * C, bend = bbeg + C < U ? bbeg + C : U;
  const long long gbeg = bbeg + grp * c, gend = gbeg + c < bend ? gbeg + c : bend;
  const uint32_t gmask = 0xFFu << (lane & ~7);
  uint32_t acc_g = 0xFFFFFFFFu, F = 0;
  unsigned int acc_e[6] = {0, 0, 0, 0, 0, 0};
  unsigned long long V = 0;
  for (long long base = gbeg; base < gend; base += 8) {  // uniform within the group
    const long long u = base + w;
    const bool valid = u < gend;
    uint32_t pop = 0, f = 0;
    if (valid) {
      uint64_t m[8];
      load_mask(a.out_masks, u, m);
      const uint32_t g = __ldcg(a.leaf_g + u);
      int32_t o[3];
#pragma unroll
      for (int k = 0; k < 3; ++k) o[k] = __ldcg(a.out_origins + 3 * u + k);
      f = (__ldcg(a.leaf_upper + u) & kGridFirst) ? 1u : 0u;
      uint64_t orw = 0;
      uint32_t xb = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pop += __popcll(m[k]);
        orw |= m[k];
        xb |= m[k] ? 1u << k : 0u;
      }
      const uint32_t yb = bits_of_bytes(orw);
      uint64_t z = orw | (orw >> 32);
      z |= z >> 16;
      z |= z >> 8;
      const uint32_t zb = (uint32_t)(z & 0xFFull);
      const unsigned int e[6] = {enc_min(o[0] + __ffs(xb) - 1), enc_min(o[1] + __ffs(yb) - 1),
                                 enc_min(o[2] + __ffs(zb) - 1), enc_max(o[0] + 31 - __clz(xb)),
                                 enc_max(o[1] + 31 - __clz(yb)), enc_max(o[2] + 31 - __clz(zb))};
      if (g != acc_g) {
        if (acc_g != 0xFFFFFFFFu)
#pragma unroll
          for (int k = 0; k < 6; ++k) atomicMax(&a.gbox[6 * acc_g + k], acc_e[k]);
        acc_g = g;
#pragma unroll
        for (int k = 0; k < 6; ++k) acc_e[k] = e[k];
      } else {
#pragma unroll
        for (int k = 0; k < 6; ++k) acc_e[k] = max(acc_e[k], e[k]);
      }
      a.leaf_pop[u] = pop;
    }
    // segmented scan of (grid-first flag, voxels) over the group's 8 leaves
    uint32_t Fi = f;
    unsigned long long Vi = pop;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const uint32_t F2 = __shfl_up_sync(gmask, Fi, off, 8);
      const unsigned long long V2 = __shfl_up_sync(gmask, Vi, off, 8);
      if (w >= off) {
        if (!Fi) Vi += V2;
        Fi |= F2;
      }
    }
    const uint32_t Ft = __shfl_sync(gmask, Fi, 7, 8);
    const unsigned long long Vt = __shfl_sync(gmask, Vi, 7, 8);
    V = Ft ? Vt : V + Vt;
    F |= Ft;
  }
  // the group's pending grid bbox: its last leaf's grid, merged over the
  // lanes that hold it; a lane left on an earlier grid reaches memory itself
  const int wl = gend > gbeg ? (int)((gend - 1 - gbeg) & 7) : 0;
  const uint32_t lg = __shfl_sync(gmask, acc_g, wl, 8);
  if (acc_g != lg && acc_g != 0xFFFFFFFFu)
#pragma unroll
    for (int k = 0; k < 6; ++k) atomicMax(&a.gbox[6 * acc_g + k], acc_e[k]);
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    unsigned int v = acc_g == lg ? acc_e[k] : 0u;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) v = max(v, __shfl_xor_sync(gmask, v, off, 8));
    if (w == 0) s.grp_box[grp][k] = v;
  }
  if (w == 0) {
    s.grp_f[grp] = F;
    s.grp_v[grp] = V;
    s.grp_g[grp] = lg;
    a.grp_agg[(long long)vb * (kThreads / 8) + grp] = ((unsigned long long)F << 63) | V;
  }
  __syncthreads();
  if (tid < 6) {  // grid bboxes: one atomic per grid run of the groups
    uint32_t cg = 0xFFFFFFFFu;
    unsigned int ce = 0;
    for (int j = 0; j < kThreads / 8; ++j) {
      const uint32_t gj = s.grp_g[j];
      if (gj == 0xFFFFFFFFu) continue;
      const unsigned int ej = s.grp_box[j][tid];
      if (gj == cg) {
        ce = max(ce, ej);
      } else {
        if (cg != 0xFFFFFFFFu) atomicMax(&a.gbox[6 * cg + tid], ce);
        cg = gj;
        ce = ej;
      }
    }
    if (cg != 0xFFFFFFFFu) atomicMax(&a.gbox[6 * cg + tid], ce);
  }
  if (tid == 32) {  // the block's segmented voxel aggregate
    uint32_t bf = 0;
    unsigned long long bv = 0;
    for (int j = 0; j < kThreads / 8; ++j) {
      bv = s.grp_f[j] ? s.grp_v[j] : bv + s.grp_v[j];
      bf |= s.grp_f[j];
    }
    a.blk_agg[vb] = ((unsigned long long)bf << 63) | bv;
  }
}

__device__ void dispatch_leaves(const PassArgs& a, Smem& sm, int vb, int vg) {
  if (a.node) {  // the place phase merged the leaves; a last pass counts them
    if (a.last) leaves_staged(a, sm, vb, vg);
    return;
  }
  switch (a.op) {
    case kIjk: phase_leaves<kIjk>(a, sm, vb, vg); break;
    case kLeaves: phase_leaves<kLeaves>(a, sm, vb, vg); break;
    case kRefine: phase_leaves<kRefine>(a, sm, vb, vg); break;
    case kCoarsen: phase_leaves<kCoarsen>(a, sm, vb, vg); break;
    case kRefineDilate: leaves_refine_dilate(a, sm, vb, vg); break;
    default: phase_leaves<kDilate>(a, sm, vb, vg); break;
  }
}

// The pass held in a block's shared copy.
struct Loaded {
  int ch, k;
};

// A front end's key layout, planned by every block for itself.
struct FrontPlan {
  KeyLayout K;
  int32_t P;
  int32_t valid;
};

// Copies pass (ch, k) into the block's shared copy unless it is already
// there (with a front end's planned layout in place of its placeholder);
// returns its op (< 0: none).  The pass array is read-only in the launch.
__device__ __forceinline__ int load_pass(const ChainArgs& c, int ch, int k, PassArgs& dst, Loaded& held,
                                         const FrontPlan& fp) {
  static_assert(sizeof(PassArgs) % 8 == 0 && sizeof(PassArgs) / 8 <= kThreads, "pass argument copy");
  __syncthreads();  // the previous phase is done with dst (and held is settled)
  if (ch != held.ch || k != held.k) {
    const unsigned long long* from = reinterpret_cast<const unsigned long long*>(c.pass + ch * c.n_stage + k);
    if (threadIdx.x < sizeof(PassArgs) / 8) reinterpret_cast<unsigned long long*>(&dst)[threadIdx.x] = __ldg(from + threadIdx.x);
    __syncthreads();
    if (threadIdx.x == 0) {
      if (fp.valid && ch == 0 && k == 0) {
        dst.K = fp.K;
        if (!dst.node) {
          dst.P = fp.P;
          dst.mid = fp.P;
          dst.sorted = fp.P & 1;
        }
      }
      held.ch = ch;
      held.k = k;
    }
    __syncthreads();
  }
  return dst.op;
}

// ---------------------------------------------------------------- chains side by side

// The phases of the chains of one stage are independent, so each phase splits
// the grid's blocks over the chains that take part in it, in proportion to
// their work (candidates, slots, or unique leaves plus weighted slots), at
// least one block each.
// Every block computes the same split from the same counters, so no
// coordination is needed; a chain's blocks then run its phase as a virtual
// grid of `vg` blocks.  With more chains than blocks, every block runs every
// chain in turn instead.
enum SplitKind { kSplitEmit, kSplitSort, kSplitIndex, kSplitLeaves };

struct Split {
  int ch, vb, vg;  // this block's chain (< 0: none), its virtual block index and grid size
  int serial;      // 1: more chains take part than there are blocks
  int maxP, more;  // emission split: most middle phases of the stage; some pass is intermediate
  int any_index;   // emission split: some pass of the stage sorts (and so runs the index phase)
};

// Relative cost of merging one slot in the leaves phase: a leaf costs its
// record (1) plus this per slot; the fused refine-then-dilate merge runs a
// leaf's slots one after another in every lane, the others spread them over
// the 8 lanes of a group or have one slot per leaf.
__device__ __forceinline__ unsigned long long leaves_slot_cost(int op) { return op == kRefineDilate ? 3ull : 1ull; }

constexpr unsigned long long kSplitOne = 1ull << 52;  // chain count unit in a packed (count, weight)
constexpr unsigned long long kSplitWCap = 1ull << 40;  // weights above this are clamped

// Work of chain ch in a phase of stage k, or -1 when it takes no part.
__device__ __forceinline__ long long split_weight(const ChainArgs& c, int ch, int k, int kind, int d, Split& sp) {
  const PassArgs* p = c.pass + ch * c.n_stage + k;
  const int op = p->op;
  if (op < 0) return -1;
  unsigned long long w;
  if (kind == kSplitEmit) {
    const unsigned long long* cd = p->src_count_dev;
    const unsigned long long n = cd ? __ldcg(cd) : (unsigned long long)p->src_count;
    const int32_t lo[3] = {p->lo[0], p->lo[1], p->lo[2]};
    const int32_t hi[3] = {p->hi[0], p->hi[1], p->hi[2]};
    const unsigned long long T = (unsigned long long)pass_targets(op, p->factor, lo, hi);
    w = n < kSplitWCap ? n * T : kSplitWCap;
    atomicMax(&sp.maxP, p->mid);
    if (!p->last) sp.more = 1;
    if (!p->node) sp.any_index = 1;
  } else if (kind == kSplitLeaves) {
    const PassCtl* ctl = p->ctl;
    const ReadbackHeader* rb = p->rb;
    w = __ldcg(&ctl->head_totals[0]) + leaves_slot_cost(op) * __ldcg(&rb->num_slots);
  } else {
    if (kind == kSplitSort && d >= p->mid) return -1;
    if (kind == kSplitIndex && p->node) return -1;
    const ReadbackHeader* rb = p->rb;
    w = __ldcg(&rb->num_slots);
  }
  return (long long)(w < kSplitWCap ? w : kSplitWCap);
}

// What the split needs of each chain's pass at the current stage, for calls
// of up to 32 chains: loaded once per stage, so a split costs one load of
// the chains' counters, a warp scan and one block barrier.
constexpr int kWarpChains = 32;
struct StageInfo {
  const ReadbackHeader* rb;
  const PassCtl* ctl;
  const unsigned long long* src_count_dev;
  long long src_count;
  int op, mid, node, last, T;
};

__device__ void load_stage(const ChainArgs& c, int k, StageInfo* si, const FrontPlan& fp) {
  __syncthreads();  // the previous stage's splits are done with si
  const int ch = threadIdx.x;
  if (ch < c.n_chain && ch < kWarpChains) {
    const PassArgs* p = c.pass + ch * c.n_stage + k;
    StageInfo& e = si[ch];
    e.op = p->op;
    e.node = p->node;
    // a sorting front end's planned digit passes
    e.mid = (fp.valid && ch == 0 && k == 0 && !p->node) ? fp.P : p->mid;
    e.last = p->last;
    e.rb = p->rb;
    e.ctl = p->ctl;
    e.src_count_dev = p->src_count_dev;
    e.src_count = p->src_count;
    const int32_t lo[3] = {p->lo[0], p->lo[1], p->lo[2]};
    const int32_t hi[3] = {p->hi[0], p->hi[1], p->hi[2]};
    e.T = pass_targets(e.op, p->factor, lo, hi);
  }
  __syncthreads();
}

// The split of split_grid for up to 32 chains, by warp 0.
__device__ void split_warp(const ChainArgs& c, const StageInfo* si, int kind, int d, Split& sp) {
  const unsigned long long G = gridDim.x, b = blockIdx.x;
  const int n = c.n_chain;
  __syncthreads();  // the previous phase is done with sp
  if (threadIdx.x < 32) {
    const int ch = threadIdx.x;
    long long w = -1;
    int P = 0, more = 0, sorts = 0;
    if (ch < n && si[ch].op >= 0) {
      const StageInfo& e = si[ch];
      unsigned long long v = 0;
      bool on = true;
      if (n == 1) {
        v = 1;  // one chain takes the whole grid whatever its work
      } else if (kind == kSplitEmit) {
        const unsigned long long ns = e.src_count_dev ? __ldcg(e.src_count_dev) : (unsigned long long)e.src_count;
        v = ns < kSplitWCap ? ns * (unsigned long long)e.T : kSplitWCap;
      } else if (kind == kSplitLeaves) {
        v = __ldcg(&e.ctl->head_totals[0]) + leaves_slot_cost(e.op) * __ldcg(&e.rb->num_slots);
      } else {
        on = !(kind == kSplitSort && d >= e.mid) && !(kind == kSplitIndex && e.node);
        if (on) v = __ldcg(&e.rb->num_slots);
      }
      if (on) w = (long long)(v < kSplitWCap ? v : kSplitWCap);
      P = e.mid;
      more = !e.last;
      sorts = !e.node;
    }
    const unsigned long long own = w >= 0 ? kSplitOne + (unsigned long long)w : 0ull;
    unsigned long long incl = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (ch >= off) incl += y;
    }
    const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31), ex = incl - own;
    const int maxP = __reduce_max_sync(0xffffffffu, (unsigned)P);
    const bool any_more = __any_sync(0xffffffffu, more);
    const bool any_sort = __any_sync(0xffffffffu, sorts);
    const unsigned long long nact = total / kSplitOne, wt = total % kSplitOne;
    if (ch == 0) {
      sp.ch = -1;
      sp.vb = 0;
      sp.vg = 0;
      sp.serial = nact > G ? 1 : 0;
      sp.maxP = maxP;
      sp.more = any_more ? 1 : 0;
      sp.any_index = any_sort ? 1 : 0;
    }
    __syncwarp();
    if (w >= 0 && nact <= G) {
      const unsigned long long ai = ex / kSplitOne, wex = ex % kSplitOne, extra = G - nact;
      const unsigned long long s0 = ai + (wt ? extra * wex / wt : extra * ai / nact);
      const unsigned long long s1 = ai + 1 + (wt ? extra * (wex + (unsigned long long)w) / wt : extra * (ai + 1) / nact);
      if (b >= s0 && b < s1) {
        sp.ch = ch;
        sp.vb = (int)(b - s0);
        sp.vg = (int)(s1 - s0);
      }
    }
  }
  __syncthreads();
}

__device__ void split_grid(const ChainArgs& c, int k, int kind, int d, Split& sp, Smem& sm) {
  const int tid = threadIdx.x;
  const unsigned long long G = gridDim.x, b = blockIdx.x;
  __syncthreads();  // the previous phase is done with sp
  if (tid == 0) {
    sp.ch = -1;
    sp.vb = 0;
    sp.vg = 0;
    sp.maxP = 0;
    sp.more = 0;
    sp.any_index = 0;
  }
  __syncthreads();
  const int n = c.n_chain;
  unsigned long long total = 0, carry = 0, t;
  if (n > kThreads) {  // totals first when the chains do not fit one scan
    for (int base = 0; base < n; base += kThreads) {
      const int ch = base + tid;
      const long long w = ch < n ? split_weight(c, ch, k, kind, d, sp) : -1;
      block_excl_scan_256(w >= 0 ? kSplitOne + (unsigned long long)w : 0ull, sm.dedup.scan, &t);
      total += t;
    }
    __syncthreads();
    if (tid == 0) {
      sp.maxP = 0;
      sp.more = 0;
      sp.any_index = 0;
    }
    __syncthreads();
  }
  for (int base = 0; base < n; base += kThreads) {
    const int ch = base + tid;
    const long long w = ch < n ? split_weight(c, ch, k, kind, d, sp) : -1;
    const unsigned long long v = w >= 0 ? kSplitOne + (unsigned long long)w : 0ull;
    const unsigned long long ex = carry + block_excl_scan_256(v, sm.dedup.scan, &t);
    if (n <= kThreads) total = t;
    carry += t;
    const unsigned long long nact = total / kSplitOne, wt = total % kSplitOne;
    if (w >= 0 && nact <= G) {
      const unsigned long long ai = ex / kSplitOne, wex = ex % kSplitOne, extra = G - nact;
      const unsigned long long s0 = ai + (wt ? extra * wex / wt : extra * ai / nact);
      const unsigned long long s1 = ai + 1 + (wt ? extra * (wex + (unsigned long long)w) / wt : extra * (ai + 1) / nact);
      if (b >= s0 && b < s1) {
        sp.ch = ch;
        sp.vb = (int)(b - s0);
        sp.vg = (int)(s1 - s0);
      }
    }
  }
  if (tid == 0) sp.serial = total / kSplitOne > G ? 1 : 0;
  __syncthreads();
}

// Runs `body(a, vb, vg)` for this block's share of a phase: its own chain, or
// in serial mode every chain that takes part, as block blockIdx.x of the grid.
template <class Body>
__device__ __forceinline__ void for_share(const ChainArgs& c, int k, int kind, int d, const Split& sp, PassArgs& a,
                                          Loaded& held, const FrontPlan& fp, Body body) {
  const int serial = sp.serial;
  const int nit = serial ? c.n_chain : (sp.ch >= 0 ? 1 : 0);
  for (int it = 0; it < nit; ++it) {
    const int ch = serial ? it : sp.ch;
    if (load_pass(c, ch, k, a, held, fp) < 0) continue;
    if (kind == kSplitSort && d >= a.mid) continue;
    if (kind == kSplitIndex && a.node) continue;
    body(a, ch, serial ? (int)blockIdx.x : sp.vb, serial ? (int)gridDim.x : sp.vg);
  }
}

// ---------------------------------------------------------------- front ends

// The input's voxel bbox (into the pass's readback block) and the checks of
// the jagged offsets and leaf origins (into the call's error word), over the
// whole grid.
__device__ void phase_front(const PassArgs& a) {
  int32_t mn[3], mx[3];
  if (a.op == kIjk) {
    ijk_bounds(a.ijk, a.src_count, mn, mx, (int)blockIdx.x, (int)gridDim.x);
  } else {
    leaves_bounds(a.src_origins, a.src_masks, a.src_count, mn, mx, a.err, (int)blockIdx.x, (int)gridDim.x);
  }
  reduce_bbox(mn, mx, a.rb->bbox_enc);
  check_offsets(a.in_offsets, a.B, a.src_count, a.err);
}

// After a grid barrier: every block reads the bbox and the checks, and plans
// the pass's key layout for itself (into fp).  Returns false (in every block
// alike) when the call must stop: bad offsets or origins, or a key wider than
// 64 bits.
__device__ bool front_plan(const ChainArgs& c, const PassArgs& a, FrontPlan& fp) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    const unsigned int err = __ldcg(c.err);
    bool good = (err & (kErrBadOffsets | kErrNotAligned | kErrTimeout)) == 0;
    if (good) {
      int32_t bb[6];
      for (int ax = 0; ax < 3; ++ax) {
        bb[ax] = dec_min(__ldcg(&a.rb->bbox_enc[ax]));
        bb[3 + ax] = dec_max(__ldcg(&a.rb->bbox_enc[3 + ax]));
      }
      KeyLayout K;
      good = make_layout(a.B, bb, bb[0] > bb[3], K);
      if (!good) {
        if (blockIdx.x == 0) atomicOr(c.err, kErrLayout);
      } else {
        fp.K = K;
        fp.P = (K.W + 7) / 8;
        fp.valid = 1;
      }
    }
    ok = good ? 1 : 0;
  }
  __syncthreads();
  return ok != 0;
}

// The last CTA out of a pass kernel (`expected` arrivals) copies the call's
// readback span to pinned host memory, then sets the host flag to the call's
// sequence number (system-scope fences order the copy before the flag), so
// the host can take the counts without a stream synchronisation.  A kernel
// that stops early never sets the flag; the host then falls back to the
// stream.
__device__ void publish_readback(const ChainArgs& c, unsigned int expected) {
  if (!c.host_span) return;
  __shared__ unsigned int out_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    out_last = atomicAdd(c.exit_ctr, 1u) + 1u == expected ? 1u : 0u;
    if (out_last) __threadfence();
  }
  __syncthreads();
  if (!out_last) return;
  const uint4* src = reinterpret_cast<const uint4*>(c.dev_span);
  uint4* dst = reinterpret_cast<uint4*>(c.host_span);
  for (long long i = threadIdx.x; i < c.span_bytes / 16; i += blockDim.x) dst[i] = __ldcg(src + i);
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    *reinterpret_cast<volatile unsigned int*>(c.host_flag) = c.seq;
  }
}

// One stage of the launch runs stage k of every chain, phase by phase, the
// chains of a phase side by side on their shares of the grid.  Stamps:
// 1 emission, 2 digit passes, 3 index, 4 leaves and voxel offsets.
// Two blocks per SM at least: the register cap this sets keeps every phase
// inlined into the kernel within 128 registers a thread.
__global__ void __launch_bounds__(kThreads, 2) k_chain(const ChainArgs c) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  __shared__ __align__(16) PassArgs a;
  __shared__ Split sp;
  __shared__ Loaded held;
  __shared__ StageInfo si[kWarpChains];
  __shared__ FrontPlan fp;
  if (threadIdx.x == 0) {
    held.ch = -1;
    held.k = -1;
    fp.valid = 0;
    unsigned long long* ts = c.pass[0].phase_ts;
    if (ts) {  // kernel entry, earliest block
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      atomicMax(ts + 6, ~t);
    }
  }
  if (c.front) {  // one one-pass chain: plan its key from the input's bbox
    load_pass(c, 0, 0, a, held, fp);
    phase_front(a);
    grid_sync(c.bar, c.err);
    if (!front_plan(c, a, fp)) return;
    if (threadIdx.x == 0) held.ch = -1;  // reload with the planned layout
  }
  const bool small = c.n_chain <= kWarpChains;
  // one chain takes the whole grid in every phase: its split is set once a
  // stage (after the stage's emission split, which also reads maxP and more)
  const bool one = c.n_chain == 1;
  auto split = [&](int k, int kind, int d) {
    if (one && kind != kSplitEmit) return;
    if (small) {
      split_warp(c, si, kind, d, sp);
    } else {
      split_grid(c, k, kind, d, sp, sm);
    }
  };
  for (int k = 0; k < c.n_stage; ++k) {
    if (small) load_stage(c, k, si, fp);
    split(k, kSplitEmit, 0);
    const int maxP = sp.maxP;
    const bool more = sp.more != 0;
    for_share(c, k, kSplitEmit, 0, sp, a, held, fp, [&](const PassArgs& pa, int, int vb, int vg) {
      stamp(pa, 0);
      dispatch_emit(pa, sm, vb, vg);
      stamp(pa, 1);
    });
    grid_sync(c.bar, c.err);
    const bool any_index = sp.any_index != 0;
    for (int d = 0; d < maxP; ++d) {
      split(k, kSplitSort, d);
      for_share(c, k, kSplitSort, d, sp, a, held, fp, [&](const PassArgs& pa, int, int vb, int vg) {
        if (pa.node) {
          node_middle(pa, d, sm, vb, vg);
        } else {
          phase_sort(pa, d, sm, vb, vg);
        }
      });
      grid_sync(c.bar, c.err);
    }
    if (any_index) {
      split(k, kSplitIndex, 0);
      for_share(c, k, kSplitIndex, 0, sp, a, held, fp, [&](const PassArgs& pa, int, int vb, int vg) {
        stamp(pa, 2);
        phase_index(pa, sm, vb, vg);
        stamp(pa, 3);
      });
      grid_sync(c.bar, c.err);
    }
    // the leaves and voxel offsets share one split: the block aggregates of
    // the leaves phase are indexed by virtual block
    split(k, kSplitLeaves, 0);
    for_share(c, k, kSplitLeaves, 0, sp, a, held, fp, [&](const PassArgs& pa, int ch, int vb, int vg) {
      // the totals and per-grid offsets: a block near the end of the chain's
      // share, which holds few leaves
      if (sp.serial ? (int)blockIdx.x == (int)gridDim.x - 1 - (ch % (int)gridDim.x) : vb == vg - 1) {
        phase_finish(pa, sm);
        __syncthreads();
      }
      dispatch_leaves(pa, sm, vb, vg);
      stamp(pa, 4);
    });
    grid_sync(c.bar, c.err);
    for_share(c, k, -1, 0, sp, a, held, fp, [&](const PassArgs& pa, int, int vb, int vg) {
      if (pa.last) phase_voxel_offsets(pa, sm, vb, vg);
      stamp(pa, 5);
    });
    if (more) grid_sync(c.bar, c.err);
  }
  publish_readback(c, gridDim.x);
}

// ---------------------------------------------------------------- member launches

// k_member runs every grid of every chain of a call on its own: member
// u = ch * B + g, one cluster of `cl` CTAs, takes grid g of chain ch through
// all of the chain's passes as a batch of one grid (its keys have no grid
// field) on its share of the chain's buffers.  Phases are separated by
// cluster barriers and look-backs span the member's own CTAs, so no member
// waits on another; the last member to finish turns the members' counts into
// each chain's per-grid offsets and totals, and the writer reads every leaf
// from its member's share.  This is the launch for batches of small grids,
// where the whole-grid phases of k_chain are bound by the latency of their
// barriers and look-backs rather than by their work.

// A barrier over the member's CTAs that also orders their global-memory
// accesses (release / acquire at cluster scope).
__device__ __forceinline__ void member_sync(int cl) {
  __syncthreads();
  if (cl > 1)
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct MemberInfo {
  long long o0, n;  // the grid's first stage-0 source and its count
  int ok;
};

// Stage k of chain ch for grid g: the stage template made the member's own
// (sources, slot arrays, control block, status words), and the member's
// control block zeroed by its CTAs.  False in every thread when the grid's
// source offsets are out of order (flagged in the error word).
__device__ bool member_args(const ChainArgs& c, int ch, int k, int g, int vb, PassArgs& a, MemberInfo& mi) {
  __syncthreads();  // the previous stage is done with a
  const unsigned long long* from = reinterpret_cast<const unsigned long long*>(c.pass + ch * c.n_stage + k);
  if (threadIdx.x < sizeof(PassArgs) / 8) reinterpret_cast<unsigned long long*>(&a)[threadIdx.x] = __ldg(from + threadIdx.x);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int32_t B = a.B;
    const long long o0 = __ldg(a.unit_off + g), o1 = __ldg(a.unit_off + g + 1);
    bool ok = true;
    if (k == 0) {  // every member checks its own offsets (later stages reuse them)
      const long long total = a.src_count;
      ok = o0 >= 0 && o1 >= o0 && o1 <= total && (g > 0 || o0 == 0) && (g + 1 < B || o1 == total);
      if (!ok && vb == 0) atomicOr(a.err, kErrBadOffsets);
    }
    mi.ok = ok ? 1 : 0;
    const long long n = ok ? o1 - o0 : 0;
    mi.o0 = o0;
    mi.n = n;
    const long long cap = n * a.m_stage;
    char* blk = a.unit_ctl + (long long)g * a.ctl_stride;
    a.rb = reinterpret_cast<ReadbackHeader*>(blk);
    a.leaf_off = reinterpret_cast<int64_t*>(blk + sizeof(ReadbackHeader));
    a.lower_off = a.leaf_off + 2;
    a.upper_off = a.lower_off + 2;
    a.grid_vox = a.upper_off + 2;
    a.gbox = reinterpret_cast<unsigned int*>(a.grid_vox + 1);
    a.ctl = reinterpret_cast<PassCtl*>(blk + a.ctl_rb_bytes);
    a.first = reinterpret_cast<uint32_t*>(blk + a.ctl_stride - 16);
    a.sort_status += member_first(o0, a.m_stage, kSortTile, a.cl, g) * a.P * kBins;
    a.sort_tiles_cap = (cap + kSortTile - 1) / kSortTile + a.cl;
    a.dedup_status += member_first(o0, a.m_stage, kDedupTile, 0, g) * 3;
    const long long xs = o0 * a.m_slots, xo = o0 * a.m_out;
    a.keys[0] += xs;
    a.keys[1] += xs;
    a.vals[0] += xs;
    a.vals[1] += xs;
    a.run_start += xs + g;
    a.leaf_lower += xs;
    a.leaf_upper += xs;
    a.leaf_voff += xs;
    a.leaf_pop += xs;
    a.leaf_g += xs;
    a.blk_agg += (long long)g * a.cl;  // the chain's [B][cl] block and [B][cl][32] group aggregates
    a.grp_agg += (long long)g * a.cl * (kThreads / 8);
    a.out_origins += 3 * xo;
    a.out_masks += 8 * xo;
    a.out_grid += xo;
    if (k == 0) {
      if (a.op == kIjk) {
        a.ijk += 3 * o0;
      } else {
        a.src_origins += 3 * o0;
        a.src_masks += 8 * o0;
      }
      a.src_count = n;
    } else {  // the member's leaves of the previous stage
      const PassArgs* p = c.pass + ch * c.n_stage + k - 1;
      const long long po = o0 * p->m_out;
      a.src_origins = p->out_origins + 3 * po;
      a.src_masks = p->out_masks + 8 * po;
      a.src_count_dev =
          &reinterpret_cast<const ReadbackHeader*>(p->unit_ctl + (long long)g * p->ctl_stride)->num_leaves;
    }
    a.src_grid = nullptr;
    a.slot_cap = cap;
    a.B = 1;
    a.sorted = a.P & 1;
  }
  __syncthreads();
  if (!mi.ok) return false;
  uint32_t* blk = reinterpret_cast<uint32_t*>(a.rb);
  const long long words = a.ctl_stride / 4, stride = (long long)a.cl * kThreads;
  for (long long i = (long long)vb * kThreads + threadIdx.x; i < words; i += stride) blk[i] = 0u;
  return true;
}

// The member's status words of the stage's digit passes and index phase,
// zeroed by its CTAs (after a front end has planned its digit passes).
__device__ void member_zero_status(const PassArgs& a, int vb) {
  const long long stride = (long long)a.cl * kThreads, first = (long long)vb * kThreads + threadIdx.x;
  const long long sw = a.sort_tiles_cap * a.P * kBins;
  for (long long i = first; i < sw; i += stride) a.sort_status[i] = 0u;
  const long long dw = 3 * ((a.slot_cap + kDedupTile - 1) / kDedupTile);
  for (long long i = first; i < dw; i += stride) a.dedup_status[i] = 0ull;
}

// A front end's member: its grid's voxel bbox, then every CTA plans the
// member's key from it (a batch of one grid); the chain's bbox (for the
// host) accumulates the members'.  False in every thread if the key needs
// more than 64 bits.
__device__ bool member_front(const ChainArgs& c, PassArgs& a, int vb) {
  int32_t mn[3], mx[3];
  if (a.op == kIjk) {
    ijk_bounds(a.ijk, a.src_count, mn, mx, vb, a.cl);
  } else {
    leaves_bounds(a.src_origins, a.src_masks, a.src_count, mn, mx, a.err, vb, a.cl);
  }
  reduce_bbox(mn, mx, a.rb->bbox_enc);
  member_sync(a.cl);
  __shared__ int ok;
  if (threadIdx.x == 0) {
    int32_t bb[6];
    for (int ax = 0; ax < 3; ++ax) {
      bb[ax] = dec_min(__ldcg(&a.rb->bbox_enc[ax]));
      bb[3 + ax] = dec_max(__ldcg(&a.rb->bbox_enc[3 + ax]));
    }
    KeyLayout K;
    const bool good = make_layout(1, bb, bb[0] > bb[3], K);
    if (good) {
      a.K = K;
      a.P = (K.W + 7) / 8;
      a.sorted = a.P & 1;
    } else if (vb == 0) {
      atomicOr(a.err, kErrLayout);
    }
    ok = good ? 1 : 0;
  }
  if (vb == 0 && threadIdx.x < 6) {
    const unsigned int e = __ldcg(&a.rb->bbox_enc[threadIdx.x]);
    if (e) atomicMax(&c.pass[0].rb->bbox_enc[threadIdx.x], e);
  }
  __syncthreads();
  return ok != 0;
}

// The last member of chain ch: the chain's per-grid leaf / lower / upper
// offsets (exclusive scans of its members' counts), voxel counts, bboxes and
// totals.  Counts stay below 2^30, so two of them share a 64-bit scan.
__device__ void member_epilogue(const ChainArgs& c, int ch, Smem& sm) {
  unsigned long long* scratch = sm.dedup.scan;
  const int B = c.B, tid = threadIdx.x;
  int kl = c.n_stage - 1;
  while (kl > 0 && c.pass[ch * c.n_stage + kl].op < 0) --kl;
  const PassArgs* t = c.pass + ch * c.n_stage + kl;
  const char* ub = t->unit_ctl;
  const long long st = t->ctl_stride;
  constexpr unsigned long long lo32 = 0xFFFFFFFFull;
  unsigned long long carry_a = 0, carry_b = 0;  // (leaves | lowers << 32), (uppers | slots << 32)
  for (int base = 0; base < B; base += kThreads) {
    const int g = base + tid;
    const ReadbackHeader* r = g < B ? reinterpret_cast<const ReadbackHeader*>(ub + (long long)g * st) : nullptr;
    unsigned long long va = 0, vc = 0;
    if (r) {
      va = __ldcg(&r->num_leaves) | (__ldcg(&r->num_lowers) << 32);
      vc = __ldcg(&r->num_uppers) | (__ldcg(&r->num_slots) << 32);
    }
    unsigned long long ta, tc;
    const unsigned long long ea = carry_a + block_excl_scan_256(va, scratch, &ta);
    const unsigned long long eb = carry_b + block_excl_scan_256(vc, scratch, &tc);
    if (r) {
      t->leaf_off[g] = (int64_t)(ea & lo32);
      t->lower_off[g] = (int64_t)(ea >> 32);
      t->upper_off[g] = (int64_t)(eb & lo32);
      const int64_t* uo = reinterpret_cast<const int64_t*>(r + 1);  // leaf | lower | upper offsets, voxels, bbox
      t->grid_vox[g] = __ldcg(uo + 6);
      const unsigned int* ugb = reinterpret_cast<const unsigned int*>(uo + 7);
#pragma unroll
      for (int e = 0; e < 6; ++e) t->gbox[6 * g + e] = __ldcg(ugb + e);
    }
    carry_a += ta;
    carry_b += tc;
  }
  if (tid == 0) {
    t->leaf_off[B] = (int64_t)(carry_a & lo32);
    t->lower_off[B] = (int64_t)(carry_a >> 32);
    t->upper_off[B] = (int64_t)(carry_b & lo32);
    t->rb->num_leaves = carry_a & lo32;
    t->rb->num_lowers = carry_a >> 32;
    t->rb->num_uppers = carry_b & lo32;
    t->rb->num_slots = carry_b >> 32;
  }
}

__global__ void __launch_bounds__(kThreads, 2) k_member(const ChainArgs c) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  __shared__ __align__(16) PassArgs a;
  __shared__ MemberInfo mi;
  const int cl = c.cl;
  const int vb = (int)(blockIdx.x % (unsigned)cl), u = (int)(blockIdx.x / (unsigned)cl);
  const int ch = u / c.B, g = u % c.B;
  if (threadIdx.x == 0) {
    unsigned long long* ts = c.pass[0].phase_ts;
    if (ts) {  // kernel entry, earliest block
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      atomicMax(ts + 6, ~t);
    }
  }
  for (int k = 0; k < c.n_stage; ++k) {
    if (c.pass[ch * c.n_stage + k].op < 0) break;
    if (!member_args(c, ch, k, g, vb, a, mi)) return;
    member_sync(cl);
    if (c.front && k == 0 && !member_front(c, a, vb)) return;
    member_zero_status(a, vb);
    member_sync(cl);
    stamp(a, 0);
    dispatch_emit(a, sm, vb, cl);
    stamp(a, 1);
    member_sync(cl);
    for (int d = 0; d < a.P; ++d) {
      phase_sort(a, d, sm, vb, cl);
      member_sync(cl);
    }
    stamp(a, 2);
    phase_index(a, sm, vb, cl);
    stamp(a, 3);
    member_sync(cl);
    if (vb == cl - 1) {
      phase_finish(a, sm);
      __syncthreads();
    }
    dispatch_leaves(a, sm, vb, cl);
    stamp(a, 4);
    member_sync(cl);
    if (a.last) {
      phase_voxel_offsets(a, sm, vb, cl);
      stamp(a, 5);
      member_sync(cl);
    }
  }
  // the member is done: count it; the chain's last one writes its offsets
  if (vb != 0) return;
  __shared__ unsigned int last;
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(c.done + ch, 1u) + 1u == (unsigned int)c.B ? 1u : 0u;
    if (last) __threadfence();
  }
  __syncthreads();
  if (!last) return;
  member_epilogue(c, ch, sm);
  publish_readback(c, (unsigned int)c.n_chain);  // the chains' last members
}

// ---------------------------------------------------------------- final writer

// After the readback: per-grid arrays, and one 8-lane group per output leaf
// writing its record (origin, merged mask, voxel offset, word prefix, bbox,
// grid, parent) and the node records at node heads.
__device__ __forceinline__ void write_grid_arrays(const PassArgs& a, const WriteOut& o, long long g) {
  o.leaf_offsets[g] = a.leaf_off[g];
  o.lower_offsets[g] = a.lower_off[g];
  o.upper_offsets[g] = a.upper_off[g];
  if (g == a.B) return;
  o.node_counts[3 * g + 0] = (int32_t)(a.upper_off[g + 1] - a.upper_off[g]);
  o.node_counts[3 * g + 1] = (int32_t)(a.lower_off[g + 1] - a.lower_off[g]);
  o.node_counts[3 * g + 2] = (int32_t)(a.leaf_off[g + 1] - a.leaf_off[g]);
  o.voxel_counts[g] = a.grid_vox[g];
#pragma unroll
  for (int c = 0; c < 6; ++c) {
    const unsigned int e = a.gbox[6 * g + c];
    o.grid_bbox[6 * g + c] = c < 3 ? dec_min(e) : dec_max(e);
  }
}

// A leaf's links to its grid and nodes, each in the lanes that write it.
struct LeafLinks {
  long long voff = 0;         // lane 0: voxels before the leaf in its grid
  uint32_t parent = 0;        // lane 3: its lower node, index within the grid
  long long lower = 0;        // lane 4: its lower node, index within the batch
  bool new_lower = false;     // lane 4: the leaf is its lower node's first
  uint32_t lower_parent = 0;  // lane 4: its upper node, index within the grid
  long long upper = 0;        // lane 5: its upper node, index within the batch
  bool new_upper = false;     // lane 5: the leaf is its upper node's first
};

// Links of leaf u of a whole-batch pass (node indices are the batch's).
__device__ __forceinline__ LeafLinks links_batch(const PassArgs& a, long long u, uint32_t g, int w) {
  LeafLinks lk;
  if (w == 0) lk.voff = a.leaf_voff[u];
  if (w == 3 || w == 4) {
    const uint32_t lw = a.leaf_lower[u];
    lk.parent = (uint32_t)((long long)lw - a.lower_off[g]);
    lk.lower = lw;
    lk.new_lower = u == 0 || a.leaf_lower[u - 1] != lw;
  }
  if (w == 4 || w == 5) {
    const uint32_t up = a.leaf_upper[u] & ~kGridFirst;
    lk.lower_parent = (uint32_t)((long long)up - a.upper_off[g]);
    lk.upper = up;
    lk.new_upper = u == 0 || (a.leaf_upper[u - 1] & ~kGridFirst) != up;
  }
  return lk;
}

// The record of leaf u of the calling lane's 8-lane group from its merged
// mask (lane w holds word w), grid, origin and links; all 32 lanes of the
// warp call it.
__device__ __forceinline__ void write_record(const WriteOut& o, long long u, bool valid, uint64_t word, uint32_t g,
                                             const int32_t org[3], const LeafLinks& lk) {
  const int lane = threadIdx.x & 31, w = lane & 7;
  const uint32_t pop = __popcll(word);
  uint32_t incl = pop;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off, 8);
    if (w >= off) incl += y;
  }
  uint64_t wp = w ? ((uint64_t)(incl - pop) << (9 * (w - 1))) : 0ull;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) wp |= __shfl_xor_sync(0xffffffffu, wp, off);
  int32_t mn[3], mx[3];
  leaf_bounds(word, w, lane, mn, mx);
  if (!valid) return;
  // this lane's axis (lanes 0-5: min x y z, max x y z), by selects rather than
  // a dynamic index into local arrays
  const int ax = w < 3 ? w : w - 3;
  const int32_t oa = ax == 0 ? org[0] : (ax == 1 ? org[1] : org[2]);
  const int32_t ma = w < 3 ? (ax == 0 ? mn[0] : (ax == 1 ? mn[1] : mn[2]))
                           : (ax == 0 ? mx[0] : (ax == 1 ? mx[1] : mx[2]));
  o.masks[8 * u + w] = word;
  if (w < 3) o.origins[3 * u + w] = oa;
  if (w < 6) o.leaf_bbox[6 * u + w] = oa + ma;
  if (w == 6) o.word_prefix[u] = wp;
  if (w == 7) o.leaf_grid[u] = (int32_t)g;
  if (w == 0) o.voxel_offset[u] = lk.voff;
  if (w == 3) o.leaf_parent[u] = (int32_t)lk.parent;
  if (w == 4 && lk.new_lower) {
#pragma unroll
    for (int c = 0; c < 3; ++c) o.lower_origins[3 * lk.lower + c] = (int32_t)((uint32_t)org[c] & ~127u);
    o.lower_parent[lk.lower] = (int32_t)lk.lower_parent;
  }
  if (w == 5 && lk.new_upper) {
#pragma unroll
    for (int c = 0; c < 3; ++c) o.upper_origins[3 * lk.upper + c] = (int32_t)((uint32_t)org[c] & ~4095u);
  }
}

// Leaf u (< U or not) of a member launch's chain: its grid g is the last whose
// first leaf is at most u, and its record sits in member g's share at the
// leaf's index within the grid; node indices there are the grid's own.
__device__ __forceinline__ void write_leaf_member(const PassArgs& a, const WriteOut& o, long long u, long long U) {
  const int w = threadIdx.x & 7;
  const bool valid = u < U;
  uint32_t g = 0;
  int32_t org[3] = {0, 0, 0};
  uint64_t word = 0;
  LeafLinks lk;
  if (valid) {
    int lo = 0, hi = a.B;  // leaf_off comes from an earlier kernel: read-only cached loads see it
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(a.leaf_off + mid) <= u) lo = mid; else hi = mid;
    }
    g = (uint32_t)lo;
    const long long ul = u - __ldg(a.leaf_off + g);
    const long long o0 = __ldg(a.unit_off + g);
    const long long xs = o0 * a.m_slots + ul, xo = o0 * a.m_out + ul;
    word = __ldcg(a.out_masks + 8 * xo + w);
#pragma unroll
    for (int c = 0; c < 3; ++c) org[c] = __ldcg(a.out_origins + 3 * xo + c);
    if (w == 0) lk.voff = __ldcg(a.leaf_voff + xs);
    if (w == 3 || w == 4) {
      const uint32_t lw = __ldcg(a.leaf_lower + xs);
      lk.parent = lw;
      lk.lower = __ldg(a.lower_off + g) + lw;
      lk.new_lower = ul == 0 || __ldcg(a.leaf_lower + xs - 1) != lw;
    }
    if (w == 4 || w == 5) {
      const uint32_t up = __ldcg(a.leaf_upper + xs) & ~kGridFirst;
      lk.lower_parent = up;
      lk.upper = __ldg(a.upper_off + g) + up;
      lk.new_upper = ul == 0 || (__ldcg(a.leaf_upper + xs - 1) & ~kGridFirst) != up;
    }
  }
  write_record(o, u, valid, word, g, org, lk);
}

// Leaf u (< U or not) from the records staged by the leaves phase.
__device__ __forceinline__ void write_leaf_staged(const PassArgs& a, const WriteOut& o, long long u, long long U) {
  if (a.member) {
    write_leaf_member(a, o, u, U);
    return;
  }
  const int w = threadIdx.x & 7;
  const bool valid = u < U;
  uint32_t g = 0;
  int32_t org[3] = {0, 0, 0};
  uint64_t word = 0;
  LeafLinks lk;
  if (valid) {
    word = __ldcg(a.out_masks + 8 * u + w);
    g = __ldcg(a.leaf_g + u);
#pragma unroll
    for (int c = 0; c < 3; ++c) org[c] = __ldcg(a.out_origins + 3 * u + c);
    lk = links_batch(a, u, g, w);
  }
  write_record(o, u, valid, word, g, org, lk);
}

// Leaf u from the records staged by a whole-batch pass, one thread per leaf:
// a warp's 32 consecutive leaves make every load and store coalesced (masks
// as 16-byte vectors).
__device__ __forceinline__ void write_leaf_thread(const PassArgs& a, const WriteOut& o, long long u) {
  uint64_t m[8];
  load_mask(a.out_masks, u, m);
  const uint32_t g = __ldcg(a.leaf_g + u);
  int32_t org[3];
#pragma unroll
  for (int c = 0; c < 3; ++c) org[c] = __ldcg(a.out_origins + 3 * u + c);
  const long long voff = __ldcg(a.leaf_voff + u);
  const uint32_t lw = __ldcg(a.leaf_lower + u), up = __ldcg(a.leaf_upper + u) & ~kGridFirst;
  const bool new_lower = u == 0 || __ldcg(a.leaf_lower + u - 1) != lw;
  const bool new_upper = u == 0 || (__ldcg(a.leaf_upper + u - 1) & ~kGridFirst) != up;
  // word prefix: field k = voxels in words 0..k (k = 0..6); bbox of the set bits
  uint64_t wp = 0, orw = 0;
  uint32_t run = 0, xb = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    run += __popcll(m[k]);
    if (k < 7) wp |= (uint64_t)run << (9 * k);
    orw |= m[k];
    xb |= m[k] ? 1u << k : 0u;
  }
  const uint32_t yb = bits_of_bytes(orw);
  uint64_t z = orw | (orw >> 32);
  z |= z >> 16;
  z |= z >> 8;
  const uint32_t zb = (uint32_t)(z & 0xFFull);
  uint4* dm = reinterpret_cast<uint4*>(o.masks + 8 * u);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    dm[q] = make_uint4((uint32_t)m[2 * q], (uint32_t)(m[2 * q] >> 32), (uint32_t)m[2 * q + 1],
                       (uint32_t)(m[2 * q + 1] >> 32));
#pragma unroll
  for (int c = 0; c < 3; ++c) o.origins[3 * u + c] = org[c];
  int32_t* bb = o.leaf_bbox + 6 * u;
  bb[0] = org[0] + __ffs(xb) - 1;
  bb[1] = org[1] + __ffs(yb) - 1;
  bb[2] = org[2] + __ffs(zb) - 1;
  bb[3] = org[0] + 31 - __clz(xb);
  bb[4] = org[1] + 31 - __clz(yb);
  bb[5] = org[2] + 31 - __clz(zb);
  o.word_prefix[u] = wp;
  o.leaf_grid[u] = (int32_t)g;
  o.voxel_offset[u] = voff;
  o.leaf_parent[u] = (int32_t)((long long)lw - a.lower_off[g]);
  if (new_lower) {
#pragma unroll
    for (int c = 0; c < 3; ++c) o.lower_origins[3 * (long long)lw + c] = (int32_t)((uint32_t)org[c] & ~127u);
    o.lower_parent[lw] = (int32_t)((long long)up - a.upper_off[g]);
  }
  if (new_upper) {
#pragma unroll
    for (int c = 0; c < 3; ++c) o.upper_origins[3 * (long long)up + c] = (int32_t)((uint32_t)org[c] & ~4095u);
  }
}

// Leaf u of a pass: from the staged records when there are any, else by
// merging its run of slots here.
template <int OP>
__device__ __forceinline__ void write_leaf(const PassArgs& a, const WriteOut& o, long long u, long long U) {
  if (a.out_masks) {
    write_leaf_staged(a, o, u, U);
    return;
  }
  const int w = threadIdx.x & 7;
  const bool valid = u < U;
  const uint64_t* keys = a.keys[a.sorted];
  const uint32_t* vals = a.vals[a.sorted];
  uint32_t s0 = 0, s1 = 0, g = 0;
  int32_t lc[3] = {0, 0, 0}, org[3] = {0, 0, 0};
  if (valid) {
    s0 = a.run_start[u];
    s1 = a.run_start[u + 1];
    decode_key(a.K, keys[s0], g, lc);
#pragma unroll
    for (int c = 0; c < 3; ++c) org[c] = (int32_t)((uint32_t)lc[c] << 3);
  }
  const uint64_t word = merge_run<OP>(a, vals, s0, s1, w);
  LeafLinks lk;
  if (valid) lk = links_batch(a, u, g, w);
  write_record(o, u, valid, word, g, org, lk);
}

// Whether a chain's counts fit the room of its outputs.
__device__ __forceinline__ bool write_fits(const PassArgs& a, const WriteOut& o) {
  return (long long)__ldcg(&a.rb->num_leaves) <= o.L_cap && (long long)__ldcg(&a.rb->num_lowers) <= o.NL_cap &&
         (long long)__ldcg(&a.rb->num_uppers) <= o.NU_cap;
}

template <int OP>
__global__ void __launch_bounds__(kThreads) k_write_final(const PassArgs a, const WriteOut o) {
  if (!write_fits(a, o)) return;
  const long long U = (long long)a.rb->num_leaves;
  const int tid = threadIdx.x, lane = tid & 31;
  const long long gtid = (long long)blockIdx.x * kThreads + tid, nthreads = (long long)gridDim.x * kThreads;
  for (long long g = gtid; g <= a.B; g += nthreads) write_grid_arrays(a, o, g);
  if (a.out_masks && !a.member) {  // staged records of a whole-batch pass
    for (long long u = gtid; u < U; u += nthreads) write_leaf_thread(a, o, u);
    return;
  }
  const long long groups = (long long)gridDim.x * (kThreads / 8);
  for (long long ub = (long long)blockIdx.x * (kThreads / 8) + (tid >> 5) * 4; ub < U; ub += groups)
    write_leaf<OP>(a, o, ub + (lane >> 3), U);
}

// The writers of several chains in one launch, from the records their leaves
// phases staged.  Tasks (one per chain, up to kMaxWriteTasks) come as one
// kernel parameter; every block reads the chains' counts and lays the leaves
// of the chains that fit their room out as one index space in units of 32
// leaves, a warp's unit within one chain: one thread per leaf for a
// whole-batch pass, 8 lanes per leaf for a member launch's shares.
__global__ void __launch_bounds__(kThreads) k_write_multi(const __grid_constant__ WriteTasks wt) {
  const WriteTask* t = wt.t;  // read in place: the lanes of a warp read the same task
  const int n_task = wt.n;
  __shared__ long long qbase[kMaxWriteTasks + 1], leaves[kMaxWriteTasks];
  if (threadIdx.x == 0) {
    long long q = 0;
    for (int i = 0; i < n_task; ++i) {
      const long long U = write_fits(t[i].a, t[i].o) ? (long long)__ldcg(&t[i].a.rb->num_leaves) : -1;
      leaves[i] = U;
      qbase[i] = q;
      if (U > 0) q += (U + 31) / 32;
    }
    qbase[n_task] = q;
  }
  __syncthreads();
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = t[0].a.B;
  const long long gtid = (long long)blockIdx.x * kThreads + tid, nthreads = (long long)gridDim.x * kThreads;
  for (long long i = gtid; i < (long long)n_task * (B + 1); i += nthreads)
    if (leaves[i / (B + 1)] >= 0) write_grid_arrays(t[i / (B + 1)].a, t[i / (B + 1)].o, i % (B + 1));
  const long long total = qbase[n_task];
  const long long nwarps = nthreads / 32;
  for (long long q = gtid / 32; q < total; q += nwarps) {
    int ch = 0;
    while (ch + 1 < n_task && qbase[ch + 1] <= q) ++ch;
    const long long u0 = (q - qbase[ch]) * 32;
    if (t[ch].a.member) {  // a member launch's shares: 8 lanes per leaf, 4 leaves at a time
      for (int j = 0; j < 8; ++j) write_leaf_member(t[ch].a, t[ch].o, u0 + 4 * j + (lane >> 3), leaves[ch]);
    } else if (u0 + lane < leaves[ch]) {
      write_leaf_thread(t[ch].a, t[ch].o, u0 + lane);
    }
  }
}

template <int OP>
int write_occupancy() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_write_final<OP>, kThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

}  // namespace

size_t chain_smem_bytes() { return sizeof(Smem); }

int chain_occupancy() {
  int n = 0;
  if (cudaFuncSetAttribute(k_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem)) != cudaSuccess)
    return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_chain, kThreads, sizeof(Smem)) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_chain(const ChainArgs& c, int blocks, cudaStream_t s) {
  void* args[] = {(void*)&c};
  return cudaLaunchCooperativeKernel((const void*)k_chain, dim3(blocks), dim3(kThreads), args, sizeof(Smem), s);
}

int member_occupancy() {
  int n = 0;
  if (cudaFuncSetAttribute(k_member, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem)) != cudaSuccess)
    return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_member, kThreads, sizeof(Smem)) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

// How many clusters of `cl` CTAs of k_member the device runs at once (the
// GPCs' SM counts decide; for cl = 1 the resident blocks).
int member_clusters(int cl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_member, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_member(const ChainArgs& c, int members, int cl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(members * cl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = cl > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_member, c);
}

int write_final_occupancy(int op) {
  switch (op) {
    case kIjk: return write_occupancy<kIjk>();
    case kLeaves: return write_occupancy<kLeaves>();
    case kRefine: return write_occupancy<kRefine>();
    case kCoarsen: return write_occupancy<kCoarsen>();
    case kRefineDilate: return write_occupancy<kRefineDilate>();
    default: return write_occupancy<kDilate>();
  }
}

int write_multi_occupancy() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_write_multi, kThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_write_multi(const WriteTasks& tasks, int blocks, cudaStream_t s) {
  k_write_multi<<<blocks, kThreads, 0, s>>>(tasks);
  return cudaGetLastError();
}

cudaError_t launch_write_final(int op, const PassArgs& a, const WriteOut& o, int blocks, cudaStream_t s) {
  switch (op) {
    case kIjk: k_write_final<kIjk><<<blocks, kThreads, 0, s>>>(a, o); break;
    case kLeaves: k_write_final<kLeaves><<<blocks, kThreads, 0, s>>>(a, o); break;
    case kRefine: k_write_final<kRefine><<<blocks, kThreads, 0, s>>>(a, o); break;
    case kCoarsen: k_write_final<kCoarsen><<<blocks, kThreads, 0, s>>>(a, o); break;
    case kDilate: k_write_final<kDilate><<<blocks, kThreads, 0, s>>>(a, o); break;
    case kRefineDilate: k_write_final<kRefineDilate><<<blocks, kThreads, 0, s>>>(a, o); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tb
