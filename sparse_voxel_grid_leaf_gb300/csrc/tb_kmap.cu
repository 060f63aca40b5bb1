// Kernel maps between two batches: for every active voxel p of the output
// batch and every offset d of a box, the index of the input voxel that a
// sparse convolution reads through d, or -1 (the step after topology
// generation in fVDB's ConvolutionPlan: issue #755 "Generated-topology grid
// construction dominates per-iteration ConvolutionPlan cost", which times the
// k3s1 same-topology map and the k2s2 transpose map).
//
//   stride 1:            input voxel p + d
//   stride s, forward:   input voxel s p + d
//   stride s, transposed: input voxel (p - d) / s where p - d divides by s
//
// Voxel indices follow the batch's voxel order (grid by grid, leaf by leaf,
// ascending bit index), the order of every other per-voxel array.  A hash
// table of the input leaves is built first; then warps take output leaves:
// their candidate input leaves (the few leaves any of their voxels can reach)
// are looked up and kept in shared memory; the leaves' active voxels are
// listed in shared memory; then the warp writes the voxels x K entries, which
// are contiguous in the map.  Three forms of that work, picked by the host
// from the box and the output's size:
//   k_kmap_halo    one leaf per warp; the input index of every voxel in the
//                  leaf's reach is tabulated once; an entry is one
//                  shared-memory word
//   k_kmap_staged  (reaches of up to 2 leaves per axis) batches of up to 16
//                  leaves per warp, k_kmap_leafwarp (3 per axis) one leaf
//                  per warp; the candidates' mask words and word bases are
//                  staged; an entry is a packed-coordinate add, a bit test
//                  and a popcount (optionally after k_kmap_cands has done
//                  the look-ups)
//   k_kmap         any box, one leaf per warp: an entry computes its input
//                  leaf and reads it
#include <algorithm>

#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

constexpr int kKmapThreads = 256;
constexpr int kKmapWarps = kKmapThreads / 32;

// Hash table of the input leaves: open addressing with linear probing over a
// power-of-two array of leaf indices (-1: empty), keyed by (grid, leaf
// coordinates); a probe checks the stored leaf's grid and origin.
__device__ __forceinline__ unsigned long long leaf_hash(int32_t g, long long lx, long long ly, long long lz) {
  unsigned long long h = (unsigned long long)(uint32_t)g * 0x9E3779B97F4A7C15ull;
  h ^= (unsigned long long)(uint32_t)lx * 0xC2B2AE3D27D4EB4Full;
  h ^= (unsigned long long)(uint32_t)ly * 0x165667B19E3779F9ull;
  h ^= (unsigned long long)(uint32_t)lz * 0xD6E8FEB86659FD93ull;
  h ^= h >> 29;
  h *= 0xBF58476D1CE4E5B9ull;
  return h ^ (h >> 32);
}

// The set-up of a kernel map, one launch: block 0 writes both batches'
// per-grid voxel bases (the exclusive prefix of their voxel counts) and
// zeroes the staged map's chunk counter; every thread inserts input leaves
// into the hash table.  The host sizes the table to at least twice the
// leaves, so every insert finds an empty slot within the bounded probe loop.
__global__ void __launch_bounds__(256) k_kmap_prep(KmapPrep p) {
  if (blockIdx.x == 0) {
    __shared__ long long part[8];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    for (int side = 0; side < 2; ++side) {
      const int64_t* c = side ? p.out_counts : p.in_counts;
      int64_t* vb = side ? p.out_vbase : p.in_vbase;
      if (threadIdx.x == 0) vb[0] = 0;
      long long carry = 0;
      for (int base = 0; base < p.B; base += 256) {
        const int i = base + threadIdx.x;
        long long v = i < p.B ? c[i] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += y;
        }
        if (lane == 31) part[wib] = v;
        __syncthreads();
        long long before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          before += w < wib ? part[w] : 0;
          total += part[w];
        }
        if (i < p.B) vb[i + 1] = carry + before + v;
        carry += total;
        __syncthreads();
      }
    }
    if (threadIdx.x == 0 && p.next_chunk) *p.next_chunk = 0u;
  }
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.L; i += stride) {
    unsigned long long h = leaf_hash(p.leaf_grid[i], p.origins[3 * i] >> 3, p.origins[3 * i + 1] >> 3,
                                     p.origins[3 * i + 2] >> 3);
    for (unsigned long long probe = 0; probe <= p.mask; ++probe, ++h)  // at most the table's size
      if (atomicCAS(p.table + (h & p.mask), -1, (int32_t)i) == -1) break;
  }
}

// Index of the input leaf of grid g at leaf coordinates (lx, ly, lz), or -1.
__device__ __forceinline__ int32_t find_leaf(const KmapArgs& k, int32_t g, long long lx, long long ly, long long lz) {
  unsigned long long h = leaf_hash(g, lx, ly, lz);
  for (unsigned long long probe = 0; probe <= k.table_mask; ++probe, ++h) {
    const int32_t e = __ldg(k.table + (h & k.table_mask));
    if (e < 0) return -1;
    if (__ldg(k.in_grid + e) == g && __ldg(k.in_origins + 3 * (long long)e) == (int32_t)(lx * 8) &&
        __ldg(k.in_origins + 3 * (long long)e + 1) == (int32_t)(ly * 8) &&
        __ldg(k.in_origins + 3 * (long long)e + 2) == (int32_t)(lz * 8))
      return e;
  }
  return -1;
}

// Box offsets d of column k, x-major, packed as three bytes (d + 8); kept in
// shared memory for boxes of up to kKmapTab offsets.
constexpr int kKmapTab = 1024;

__global__ void __launch_bounds__(kKmapThreads, 4) k_kmap(const KmapArgs k) {
  __shared__ int32_t cand[kKmapWarps][kKmapMaxCand];
  __shared__ uint16_t vox[kKmapWarps][512];
  __shared__ uint32_t dtab[kKmapTab];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const long long nwarps = (long long)gridDim.x * kKmapWarps;
  const int nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = (k.hi[0] - k.lo[0] + 1) * nb1 * nb2;
  const int sh = k.stride == 2 ? 1 : 0;  // strides 1 and 2
  const bool tab = K <= kKmapTab;
  for (int i = threadIdx.x; i < K && tab; i += kKmapThreads)
    dtab[i] = (uint32_t)(k.lo[0] + i / (nb1 * nb2) + 8) | ((uint32_t)(k.lo[1] + (i / nb2) % nb1 + 8) << 8) |
              ((uint32_t)(k.lo[2] + i % nb2 + 8) << 16);
  __syncthreads();
  for (long long u = (long long)blockIdx.x * kKmapWarps + wib; u < k.L_out; u += nwarps) {
    const int32_t g = __ldg(k.out_grid + u);
    const long long o[3] = {__ldg(k.out_origins + 3 * u), __ldg(k.out_origins + 3 * u + 1),
                            __ldg(k.out_origins + 3 * u + 2)};
    // input leaf coordinate range per axis (coordinates >> 3 is a floor)
    long long a[3];
    int n[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      long long qlo, qhi;
      if (k.transposed) {
        qlo = (o[ax] - k.hi[ax] + (1 << sh) - 1) >> sh;  // ceil((p_min - hi) / s)
        qhi = (o[ax] + 7 - k.lo[ax]) >> sh;
      } else {
        qlo = (o[ax] << sh) + k.lo[ax];
        qhi = ((o[ax] + 7) << sh) + k.hi[ax];
      }
      a[ax] = qlo >> 3;
      n[ax] = (int)((qhi >> 3) - a[ax] + 1);
    }
    const int C = n[0] * n[1] * n[2];  // <= kKmapMaxCand, checked by the host's bounds
    for (int c = lane; c < C; c += 32) {
      const long long lx = a[0] + c / (n[1] * n[2]), ly = a[1] + (c / n[2]) % n[1], lz = a[2] + c % n[2];
      cand[wib][c] = find_leaf(k, g, lx, ly, lz);
    }
    // the output leaf's active voxels in order: lane l lists bits 16 l .. 16 l + 15
    // (mask word l / 4, quarter l % 4)
    const uint32_t chunk = (uint32_t)(__ldg(k.out_masks + 8 * u + (lane >> 2)) >> (16 * (lane & 3))) & 0xFFFFu;
    const uint32_t cnt = __popc(chunk);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const uint32_t nvox = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = incl - cnt, rest = chunk;
    while (rest) {
      const int b = __ffs(rest) - 1;
      rest &= rest - 1;
      vox[wib][pos++] = (uint16_t)(16 * lane + b);
    }
    __syncwarp();
    // the leaf's entries: map rows j0 .. j0 + nvox - 1, K entries each,
    // contiguous in the map; lane entry e = lane + 32 i walks (row r, column
    // kk) without dividing, and the column's offset comes from a shared table
    const long long j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
    const long long E = (long long)nvox * K;
    const long long vin = __ldg(k.in_vbase + g);
    int32_t* row = k.map + j0 * K;
    int r = lane / K, kk = lane % K;
    const int step_r = 32 / K, step_k = 32 % K;
    for (long long e = lane; e < E; e += 32) {
      const int nbit = vox[wib][r];
      int d0, d1, d2;
      if (tab) {
        const uint32_t dp = dtab[kk];
        d0 = (int)(dp & 0xFFu) - 8;
        d1 = (int)((dp >> 8) & 0xFFu) - 8;
        d2 = (int)((dp >> 16) & 0xFFu) - 8;
      } else {
        d0 = k.lo[0] + kk / (nb1 * nb2);
        d1 = k.lo[1] + (kk / nb2) % nb1;
        d2 = k.lo[2] + kk % nb2;
      }
      const long long p0 = o[0] + (nbit >> 6), p1 = o[1] + ((nbit >> 3) & 7), p2 = o[2] + (nbit & 7);
      long long q0, q1, q2;
      bool ok = true;
      if (k.transposed) {
        const long long t0 = p0 - d0, t1 = p1 - d1, t2 = p2 - d2;
        ok = ((t0 | t1 | t2) & ((1 << sh) - 1)) == 0;
        q0 = t0 >> sh;
        q1 = t1 >> sh;
        q2 = t2 >> sh;
      } else {
        q0 = (p0 << sh) + d0;
        q1 = (p1 << sh) + d1;
        q2 = (p2 << sh) + d2;
      }
      int32_t idx = -1;
      if (ok) {
        const int c = ((int)((q0 >> 3) - a[0]) * n[1] + (int)((q1 >> 3) - a[1])) * n[2] + (int)((q2 >> 3) - a[2]);
        const int32_t ci = cand[wib][c];
        if (ci >= 0) {
          const int wx = (int)(q0 & 7), by = (int)(8 * (q1 & 7) + (q2 & 7));
          const uint64_t w = __ldg(k.in_masks + 8 * (long long)ci + wx);
          if ((w >> by) & 1ull) {
            const uint64_t wp = __ldg(k.in_wp + ci);
            const long long before = wx ? (long long)((wp >> (9 * (wx - 1))) & 511ull) : 0ll;
            idx = (int32_t)(vin + __ldg(k.in_voff + ci) + before + __popcll(w & ((1ull << by) - 1ull)));
          }
        }
      }
      row[e] = idx;
      r += step_r;
      kk += step_k;
      if (kk >= K) {
        kk -= K;
        ++r;
      }
    }
    __syncwarp();
  }
}

// The same map for boxes whose reach from an output leaf spans at most 3
// input leaves per axis (span^3 <= 27 candidates per output leaf; the host
// checks).  Every output leaf gets the same candidate layout: a span^3 block
// of input leaves, x-major, starting at the first leaf its reach touches
// (candidates past the leaf's own reach are absent).  Coordinates relative to
// that first candidate leaf's origin Q_b: stride 1 q = o + p + d, so
// o - Q_b + p + d; forward stride 2, 2o - Q_b + 2p + d; transposed stride 1,
// o - Q_b + p - d; transposed stride 2 (p - d even),
// o/2 - Q_b + floor(p/2) - floor(d/2).
constexpr int kStagedCand = 27;

// The first and count of the input leaves along one axis that an output leaf
// at voxel coordinate o reaches (leaf coordinates).
__device__ __forceinline__ void reach(const KmapArgs& k, int ax, long long o, long long& a, int& n) {
  const int sh = k.stride == 2 ? 1 : 0;
  long long qlo, qhi;
  if (k.transposed) {
    qlo = (o - k.hi[ax] + (1 << sh) - 1) >> sh;  // ceil((o - hi) / s)
    qhi = (o + 7 - k.lo[ax]) >> sh;
  } else {
    qlo = (o << sh) + k.lo[ax];
    qhi = ((o + 7) << sh) + k.hi[ax];
  }
  a = qlo >> 3;
  n = (int)((qhi >> 3) - a + 1);
}

// Candidate input leaves of every output leaf, one thread per (leaf,
// candidate) in the span^3 layout: the hash look-ups of all leaves run side
// by side here, and the map kernel then reads each leaf's candidates with
// coalesced loads.  An optional pass (the "staged after a look-up pass"
// form): on GB300 the staged kernels' own look-ups measured faster.
__global__ void __launch_bounds__(256) k_kmap_cands(const KmapArgs k) {
  const long long total = k.L_out * k.cand_max;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int S = k.span, S2 = S * S;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long u = i / k.cand_max;
    const int c = (int)(i - u * k.cand_max);
    const int cx = c / S2, cy = (c / S) % S, cz = c % S;
    long long a[3];
    int n[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) reach(k, ax, __ldg(k.out_origins + 3 * u + ax), a[ax], n[ax]);
    int32_t ci = -1;
    if (cx < n[0] && cy < n[1] && cz < n[2]) ci = find_leaf(k, __ldg(k.out_grid + u), a[0] + cx, a[1] + cy, a[2] + cz);
    k.cands[i] = ci;
  }
}

// The staged map one output leaf per warp, for reaches of up to 3 input
// leaves per axis (27 candidates, which fill a warp's look-ups and staged
// words on their own) and boxes of up to kKmapStagedColumns columns: the
// candidates are looked up (or read from the look-up pass), their words
// staged, the leaf's active voxels listed in shared memory (a lane per 16
// bits of the mask) and the leaf's voxels x K entries taken flat over the
// lanes with coalesced stores.
constexpr int kLeafWarps = 8;
struct LeafWarp {
  uint64_t mask[kStagedCand * 8];  // word w of candidate c at 8 c + w (0: no candidate)
  int32_t base[kStagedCand * 8];   // first voxel index of that word
  int32_t cand[kStagedCand];
  uint32_t vpk[512];               // per active voxel: coordinate bytes (biased by 8) | parity << 24
};

__global__ void __launch_bounds__(kLeafWarps * 32, 4) k_kmap_leafwarp(const KmapArgs k) {
  __shared__ LeafWarp sw[kLeafWarps];
  __shared__ uint32_t dpk[kKmapStagedColumns];  // per column: 3 offset bytes (biased by 8) | parity << 24
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  LeafWarp& W = sw[wib];
  const long long nwarps = (long long)gridDim.x * kLeafWarps;
  const int nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = (k.hi[0] - k.lo[0] + 1) * nb1 * nb2;
  const int sh = k.stride == 2 ? 1 : 0, tr = k.transposed, par2 = tr && sh;
  for (int i = threadIdx.x; i < K; i += kLeafWarps * 32) {
    const int d[3] = {k.lo[0] + i / (nb1 * nb2), k.lo[1] + (i / nb2) % nb1, k.lo[2] + i % nb2};
    uint32_t v = 0, par = 0;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const int gv = tr ? -(d[ax] >> sh) : d[ax];
      v |= (uint32_t)(gv + 8) << (8 * ax);
      if (par2) par |= (uint32_t)(d[ax] & 1) << (2 - ax);
    }
    dpk[i] = v | (par << 24);
  }
  __syncthreads();
  const int S = k.span, S2 = S * S, Cn = S2 * S;
  const uint32_t nm = (uint32_t)(8 * Cn - 1);
  const int step_r = 32 / K, step_k = 32 % K, r_0 = lane / K, k_0 = lane - r_0 * K;
  for (long long u = (long long)blockIdx.x * kLeafWarps + wib; u < k.L_out; u += nwarps) {
    const int32_t g = __ldg(k.out_grid + u);
    long long a[3];
    int n[3];
    uint32_t Apk = 0;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const long long o = __ldg(k.out_origins + 3 * u + ax);
      reach(k, ax, o, a[ax], n[ax]);
      Apk |= (uint32_t)((tr ? (o >> sh) : (o << sh)) - (a[ax] << 3) + 8) << (8 * ax);
    }
    if (k.cands) {
      if (lane < Cn) W.cand[lane] = __ldcg(k.cands + u * Cn + lane);
    } else if (lane < Cn) {
      const int cx = lane / S2, cy = (lane / S) % S, cz = lane % S;
      W.cand[lane] = cx < n[0] && cy < n[1] && cz < n[2] ? find_leaf(k, g, a[0] + cx, a[1] + cy, a[2] + cz) : -1;
    }
    __syncwarp();
    const long long vin = __ldg(k.in_vbase + g);
    for (int j = lane; j < 8 * Cn; j += 32) {
      const int ci = W.cand[j >> 3], w = j & 7;
      uint64_t m = 0;
      int32_t b = 0;
      if (ci >= 0) {
        m = __ldg(k.in_masks + 8 * (long long)ci + w);
        const uint64_t wp = __ldg(k.in_wp + ci);
        b = (int32_t)(vin + __ldg(k.in_voff + ci) + (w ? (long long)((wp >> (9 * (w - 1))) & 511ull) : 0ll));
      }
      W.mask[j] = m;
      W.base[j] = b;
    }
    // the output leaf's active voxels in order (lane l lists bits 16 l .. 16 l + 15)
    const uint32_t chunk = (uint32_t)(__ldg(k.out_masks + 8 * u + (lane >> 2)) >> (16 * (lane & 3))) & 0xFFFFu;
    const uint32_t cnt = __popc(chunk);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const uint32_t nvox = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = incl - cnt, rest = chunk;
    while (rest) {
      const int bn = 16 * lane + __ffs(rest) - 1;
      rest &= rest - 1;
      const int p[3] = {bn >> 6, (bn >> 3) & 7, bn & 7};
      uint32_t v = Apk, par = 0;
#pragma unroll
      for (int ax = 0; ax < 3; ++ax) {
        v += (uint32_t)(tr ? (p[ax] >> sh) : (p[ax] << sh)) << (8 * ax);
        if (par2) par |= (uint32_t)(p[ax] & 1) << (2 - ax);
      }
      W.vpk[pos++] = v | (par << 24);
    }
    __syncwarp();
    const long long j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
    const int Etot = (int)nvox * K;
    int32_t* row = k.map + j0 * K;
    int r = r_0, kk = k_0;
    for (int e = lane; e < Etot; e += 32) {
      const uint32_t vp = W.vpk[r], dp = dpk[kk];
      // both packs carry a bias of 8 per byte; a column of the wrong parity
      // (transposed stride 2) reads a clamped slot and is then masked out
      const uint32_t rel = (vp & 0xFFFFFFu) + (dp & 0xFFFFFFu) - 0x101010u;
      const uint32_t rx = rel & 0xFFu, ry = (rel >> 8) & 0xFFu, rz = (rel >> 16) & 0xFFu;
      const uint32_t slot =
          min((((rx >> 3) * (uint32_t)S2 + (ry >> 3) * (uint32_t)S + (rz >> 3)) << 3) | (rx & 7u), nm);
      const uint64_t word = W.mask[slot];
      const uint32_t bit = ((ry & 7u) << 3) | (rz & 7u);
      const uint64_t upto = word << (63u - bit);  // bit 63: the voxel; the rest: the voxels before it
      const bool on = (vp >> 24) == (dp >> 24) && (upto >> 63);
      __stcs(row + e, on ? W.base[slot] + __popcll(upto) - 1 : -1);
      r += step_r;
      kk += step_k;
      if (kk >= K) {
        kk -= K;
        ++r;
      }
    }
    __syncwarp();
  }
}

// The staged map for reaches of up to 2 input leaves per axis (8 candidates)
// and boxes of up to kKmapBatchColumns columns.  A warp takes a chunk of
// consecutive output leaves (16 with one candidate each, else 8, halved
// down to 4 where the output has too few leaves for two chunks per warp;
// small enough that the chunks, handed out one at a time, end together)
// and cuts it into batches of as many leaves as fit kStagedSlots candidate
// mask words (8 per candidate).  For a batch it
//   1. looks up the candidates, a lane per leaf and candidate,
//   2. stages the candidates' mask words and the first input voxel index of
//      each word in shared memory, a lane per word,
//   3. writes the batch's rows, which are contiguous in the map (the output's
//      voxel order runs leaf after leaf, grid after grid), a lane per row:
//      the lane finds its voxel from the row number alone (the leaf by a
//      binary search over the chunk's running voxel counts, the mask word by
//      one over the leaf's word prefix, the bit by popcounts), packs its
//      coordinate relative to the leaf's candidate block, and computes the
//      row's entries.  Only the columns of the voxel's parity class are
//      computed (one of the 8 for the k2s2 transpose), and rows of 4 or 8
//      entries leave from registers as 16-byte stores; for other widths the
//      warp packs 32 voxels, then takes their entries flat over the lanes
//      (every lane busy however few the rows) with coalesced stores.
// An entry is a byte-wise add, a shared-memory word, a bit test and a
// popcount.  With sparse leaves (a few dozen voxels each) one leaf's setup
// would cost more than its entries; a batch of up to 16 leaves shares it.
constexpr int kStagedWarps = 8;
constexpr int kStagedSlots = 256;

struct StagedSmem {
  uint32_t dpk[kKmapBatchColumns];  // per column: 3 offset bytes (biased by 8) | parity << 24
  uint8_t pcol[8][kKmapBatchColumns];  // columns of each parity class
  int32_t pcnt[8];
};
struct StagedWarp {
  uint64_t mask[kStagedSlots];  // word w of candidate c of batch leaf t at 8 (t C + c) + w
  int32_t base[kStagedSlots];   // input voxel index of that word's first voxel
};

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(unsigned long long)v, src);
  const int hi = __shfl_sync(0xffffffffu, (int)((unsigned long long)v >> 32), src);
  return (long long)(((unsigned long long)(uint32_t)hi << 32) | (uint32_t)lo);
}

// Position of set bit number r (from 0, counting from bit 0) of m; r < popcount(m).
__device__ __forceinline__ int select_bit(uint64_t m, int r) {
  uint32_t x = (uint32_t)m;
  int pos = 0;
  const int c = __popc(x);
  if (r >= c) {
    r -= c;
    x = (uint32_t)(m >> 32);
    pos = 32;
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const int cl = __popc(x & ((1u << s) - 1u));
    if (r >= cl) {
      r -= cl;
      x >>= s;
      pos += s;
    }
  }
  return pos;
}

// One entry of the staged map: a voxel's pack vp and a column's pack dp
// (kMatched: the column is of the voxel's parity class).
template <bool kMatched = false>
__device__ __forceinline__ int32_t staged_value(const StagedWarp& W, uint32_t vp, uint32_t dp, int S, int S2,
                                                int words) {
  // both packs carry a bias of 8 per byte, so no byte borrows where the
  // entry exists; a column of the wrong parity (transposed stride 2) may
  // read a clamped slot and is masked out
  const uint32_t rel = (vp & 0xFFFFFFu) + (dp & 0xFFFFFFu) - 0x101010u;
  const uint32_t rx = rel & 0xFFu, ry = (rel >> 8) & 0xFFu, rz = (rel >> 16) & 0xFFu;
  const uint32_t local = min((((rx >> 3) * (uint32_t)S2 + (ry >> 3) * (uint32_t)S + (rz >> 3)) << 3) | (rx & 7u),
                             (uint32_t)(words - 1));
  const uint32_t slot = (vp >> 27) * (uint32_t)words + local;
  const uint64_t word = W.mask[slot];
  const uint32_t bit = ((ry & 7u) << 3) | (rz & 7u);
  const uint64_t upto = word << (63u - bit);  // bit 63: the voxel; the rest: the voxels before it
  const bool on = (kMatched || ((vp >> 24) & 7u) == (dp >> 24)) && (upto >> 63);
  return on ? W.base[slot] + __popcll(upto) - 1 : -1;
}

__global__ void __launch_bounds__(kStagedWarps * 32, 4) k_kmap_staged(const KmapArgs k) {
  extern __shared__ __align__(16) unsigned char kmap_smem[];
  StagedSmem& C = *reinterpret_cast<StagedSmem*>(kmap_smem);
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = (k.hi[0] - k.lo[0] + 1) * nb1 * nb2;  // <= kKmapBatchColumns (checked at launch)
  const bool vec = (K == 4 || K == 8) && (((uintptr_t)k.map & 15u) == 0);
  StagedWarp& W = *reinterpret_cast<StagedWarp*>(kmap_smem + sizeof(StagedSmem) + (size_t)wib * (sizeof(StagedWarp) + 128));
  uint32_t* vps = reinterpret_cast<uint32_t*>(&W + 1);  // a round's 32 voxel packs
  const int sh = k.stride == 2 ? 1 : 0, tr = k.transposed, par2 = tr && sh;
  for (int i = threadIdx.x; i < K; i += kStagedWarps * 32) {
    const int d[3] = {k.lo[0] + i / (nb1 * nb2), k.lo[1] + (i / nb2) % nb1, k.lo[2] + i % nb2};
    uint32_t v = 0, par = 0;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const int gv = tr ? -(d[ax] >> sh) : d[ax];
      v |= (uint32_t)(gv + 8) << (8 * ax);
      if (par2) par |= (uint32_t)(d[ax] & 1) << (2 - ax);
    }
    C.dpk[i] = v | (par << 24);
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    int c = 0;
    for (int kk = 0; kk < K; ++kk)
      if ((int)(C.dpk[kk] >> 24) == (int)threadIdx.x) C.pcol[threadIdx.x][c++] = (uint8_t)kk;
    C.pcnt[threadIdx.x] = c;
  }
  __syncthreads();
  // a class of at most one column (the k2s2 transpose): a row is that entry and -1s
  int single = 1;
#pragma unroll
  for (int pc = 0; pc < 8; ++pc) single &= C.pcnt[pc] <= 1;
  const int S = k.span, S2 = S * S, Cn = S2 * S, words = 8 * Cn;
  const int gmax = kStagedSlots / words;  // leaves per batch (>= 4: Cn <= 8)
  // leaves per chunk: 16 (8 for a span of 2), halved down to 4 while there
  // are fewer than two chunks per warp of the grid
  int cs = gmax >= 16 ? 16 : 8;
  while (cs > 4 && (k.L_out + cs - 1) / cs < 2ll * gridDim.x * kStagedWarps) cs >>= 1;
  const long long nchunks = (k.L_out + cs - 1) / cs;
  // this lane's place in step 1 (batch leaf, candidate and its offsets) and
  // in the flat entry rounds, divided out once
  const int l_lt = lane / Cn, l_c = lane - l_lt * Cn;
  const int l_cx = l_c / S2, l_cy = (l_c / S) % S, l_cz = l_c % S;
  const int f_r = lane / K, f_k = lane - f_r * K, f_sr = 32 / K, f_sk = 32 % K;
  for (;;) {
    // chunks are handed out one at a time: their costs vary with their voxels
    unsigned int chu = 0;
    if (lane == 0) chu = atomicAdd(k.next_chunk, 1u);
    const long long ch = (long long)__shfl_sync(full, chu, 0);
    if (ch >= nchunks) break;
    const long long u0 = ch * cs, u = u0 + lane;
    const int nleaf = (int)min((long long)cs, k.L_out - u0);
    // lane t holds chunk leaf t: grid, reach, packed offset, first voxel,
    // word prefix, voxels before it in the chunk
    int32_t g = 0;
    int a[3] = {0, 0, 0}, n[3] = {0, 0, 0};
    uint32_t Apk = 0;
    long long j0 = 0;
    uint64_t owp = 0;
    int cnt = 0, vin = 0;
    if (lane < nleaf) {
      g = __ldg(k.out_grid + u);
#pragma unroll
      for (int ax = 0; ax < 3; ++ax) {
        const long long o = __ldg(k.out_origins + 3 * u + ax);
        long long al;
        reach(k, ax, o, al, n[ax]);
        a[ax] = (int)al;
        Apk |= (uint32_t)((tr ? (o >> sh) : (o << sh)) - (al << 3) + 8) << (8 * ax);
      }
      j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
      vin = (int)__ldg(k.in_vbase + g);
      owp = __ldg(k.out_wp + u);
      cnt = (int)((owp >> 54) & 511ull) + __popcll(__ldg(k.out_masks + 8 * u + 7));
    }
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(full, incl, off);
      if (lane >= off) incl += y;
    }
    const int excl = incl - cnt;
    for (int t0 = 0; t0 < nleaf;) {
      const int t1 = min(t0 + gmax, nleaf), nb = t1 - t0;
      const int vb = __shfl_sync(full, excl, t0);
      const int nv = __shfl_sync(full, incl, t1 - 1) - vb;
      const long long jb = shfl_ll(j0, t0);
      // 1. the candidates, a lane per (leaf, candidate): nb Cn <= kStagedSlots / 8 = 32
      int32_t ci = -1, cvin = 0;
      {
        const int src = t0 + min(l_lt, nb - 1);
        const int gs = __shfl_sync(full, g, src);
        const int a0 = __shfl_sync(full, a[0], src), a1 = __shfl_sync(full, a[1], src),
                  a2 = __shfl_sync(full, a[2], src);
        const int n0 = __shfl_sync(full, n[0], src), n1 = __shfl_sync(full, n[1], src),
                  n2 = __shfl_sync(full, n[2], src);
        cvin = __shfl_sync(full, vin, src);
        if (lane < nb * Cn) {
          if (k.cands)
            ci = __ldcg(k.cands + (u0 + src) * Cn + l_c);
          else if (l_cx < n0 && l_cy < n1 && l_cz < n2)
            ci = find_leaf(k, gs, a0 + l_cx, a1 + l_cy, a2 + l_cz);
        }
      }
      // 2. the candidates' mask words and word bases, a lane per word
#pragma unroll
      for (int i = 0; i < kStagedSlots / 32; ++i) {
        if (32 * i >= nb * words) break;
        const int j = 32 * i + lane, src = min(j >> 3, 31);
        const int cj = __shfl_sync(full, ci, src), vj = __shfl_sync(full, cvin, src);
        if (j < nb * words) {
          const int w = j & 7;
          uint64_t m = 0;
          int32_t b = 0;
          if (cj >= 0) {
            m = __ldg(k.in_masks + 8 * (long long)cj + w);
            const uint64_t wp = __ldg(k.in_wp + cj);
            b = vj + (int32_t)__ldg(k.in_voff + cj) + (w ? (int32_t)((wp >> (9 * (w - 1))) & 511ull) : 0);
          }
          W.mask[j] = m;
          W.base[j] = b;
        }
      }
      __syncwarp();
      // 3. the rows, a lane each: rows jb .. jb + nv - 1 of the map
      for (int r0 = 0; r0 < nv; r0 += 32) {
        const int r = r0 + lane, R = vb + r;  // R: voxels of the chunk before this one
        // the leaf: the round's first row lies in the last batch leaf starting
        // at or before it; each leaf starting inside the round moves the
        // rows from its start on to the next leaf (leaves are never empty)
        const bool inb = lane >= t0 && lane < t1;
        const unsigned lead = __ballot_sync(full, inb && excl - vb <= r0);
        const int st = excl - vb - r0;
        const unsigned starts = __reduce_or_sync(full, inb && st > 0 && st < 32 ? 1u << st : 0u);
        const int lt = (31 - __clz(lead)) + __popc(starts & (0xFFFFFFFFu >> (31 - lane)));
        const int ex = __shfl_sync(full, excl, lt);
        const unsigned long long wpl = (unsigned long long)shfl_ll((long long)owp, lt);
        const uint32_t A = __shfl_sync(full, Apk, lt);
        int32_t* rowp = k.map + (jb + r) * K;
        uint32_t vp = 0;
        int pc = 0;
        if (r < nv) {
          // the word: the last x whose first voxel is at or before the rank
          const int rank = R - ex;
          int x = 0;
          if ((int)((wpl >> 27) & 511ull) <= rank) x = 4;
          if ((int)((wpl >> (9 * (x + 1))) & 511ull) <= rank) x += 2;
          if ((int)((wpl >> (9 * x)) & 511ull) <= rank) x += 1;
          const int before = x ? (int)((wpl >> (9 * (x - 1))) & 511ull) : 0;
          const int b = select_bit(__ldg(k.out_masks + 8 * (u0 + lt) + x), rank - before);
          const int py = b >> 3, pz = b & 7;
          vp = A + (uint32_t)(tr ? (x >> sh) : (x << sh)) + ((uint32_t)(tr ? (py >> sh) : (py << sh)) << 8) +
               ((uint32_t)(tr ? (pz >> sh) : (pz << sh)) << 16) + ((uint32_t)(lt - t0) << 27);
          if (par2) {
            pc = ((x & 1) << 2) | ((py & 1) << 1) | (pz & 1);
            vp += (uint32_t)pc << 24;
          }
        }
        if (vec) {
          if (r < nv) {
            int32_t v[8];
            if (single) {
              const int kk0 = C.pcnt[pc] ? C.pcol[pc][0] : -1;
              const int32_t val = kk0 >= 0 ? staged_value<true>(W, vp, C.dpk[kk0], S, S2, words) : -1;
#pragma unroll
              for (int c = 0; c < 8; ++c) v[c] = c == kk0 ? val : -1;
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c) v[c] = c < K ? staged_value(W, vp, C.dpk[c], S, S2, words) : -1;
            }
            int4* dst = reinterpret_cast<int4*>(rowp);
            __stcs(dst, make_int4(v[0], v[1], v[2], v[3]));
            if (K == 8) __stcs(dst + 1, make_int4(v[4], v[5], v[6], v[7]));
          }
        } else {
          // the round's 32 voxels, then its nr x K entries flat over the lanes
          // (every lane busy however few the rows; coalesced stores)
          const int nr = min(32, nv - r0);
          vps[lane] = vp;
          __syncwarp();
          int32_t* dst = k.map + (jb + r0) * K;
          int rr = f_r, kc = f_k;
          for (int i = lane; i < nr * K; i += 32) {
            __stcs(dst + i, staged_value(W, vps[rr], C.dpk[kc], S, S2, words));
            rr += f_sr;
            kc += f_sk;
            if (kc >= K) {
              kc -= K;
              ++rr;
            }
          }
          __syncwarp();
        }
      }
      __syncwarp();
      t0 = t1;
    }
  }
}

// The map for reaches small enough to tabulate: the input voxel index of
// every voxel of the output leaf's reach (the halo: E0 x E1 x E2 <= kHaloMax
// voxels, the same extents for every leaf) is computed once per leaf, and an
// entry is then one shared-memory word at halo offset base(p) + delta(d):
//   stride 1          q = o + p + d          base p,        delta d - lo
//   transposed 1      q = o + p - d          base p,        delta hi - d
//   transposed 2      q = (o + p - d) / 2    base p / 2,    delta hi / 2 - d / 2 (floors;
//                     p - d even on every axis, else no entry)
// Each output leaf pays for its halo once; an entry costs two shared loads,
// an add and the store, so the map is written at close to store rate.
constexpr int kHaloMax = kKmapHaloMax;
constexpr int kHaloWarps = 4;
struct HaloWarp {
  uint64_t mask[kStagedCand * 8];
  int32_t base[kStagedCand * 8];
  int32_t cand[kStagedCand];
  int32_t H[kHaloMax];   // input voxel index of each halo voxel, or -1
  uint16_t vh[512];      // per active output voxel: halo offset of base(p) | parity << 10
};

__global__ void __launch_bounds__(kHaloWarps * 32, 7) k_kmap_halo(const KmapArgs k) {
  __shared__ HaloWarp sw[kHaloWarps];
  __shared__ uint16_t dh[kKmapTabColumns];  // per column: delta(d) | parity << 10
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  HaloWarp& W = sw[wib];
  const long long nwarps = (long long)gridDim.x * kHaloWarps;
  const int nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = (k.hi[0] - k.lo[0] + 1) * nb1 * nb2;
  const int sh = k.stride == 2 ? 1 : 0, tr = k.transposed;
  int E[3];
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
    E[ax] = tr ? ((7 - k.lo[ax]) >> sh) + (k.hi[ax] >> sh) + 1 : 8 + k.hi[ax] - k.lo[ax];
  const int E12 = E[1] * E[2];
  for (int i = threadIdx.x; i < K; i += kHaloWarps * 32) {
    const int d[3] = {k.lo[0] + i / (nb1 * nb2), k.lo[1] + (i / nb2) % nb1, k.lo[2] + i % nb2};
    int delta[3];
    uint32_t par = 0;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      delta[ax] = tr ? (k.hi[ax] >> sh) - (d[ax] >> sh) : d[ax] - k.lo[ax];
      if (tr && sh) par |= (uint32_t)(d[ax] & 1) << (2 - ax);
    }
    dh[i] = (uint16_t)((delta[0] * E12 + delta[1] * E[2] + delta[2]) | (par << 10));
  }
  __syncthreads();
  for (long long u = (long long)blockIdx.x * kHaloWarps + wib; u < k.L_out; u += nwarps) {
    const int32_t g = __ldg(k.out_grid + u);
    long long a[3];
    int n[3], off[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const long long o = __ldg(k.out_origins + 3 * u + ax);
      reach(k, ax, o, a[ax], n[ax]);
      const long long qlo = tr ? (o - k.hi[ax] + (1 << sh) - 1) >> sh : o + k.lo[ax];
      off[ax] = (int)(qlo - (a[ax] << 3));  // the halo's first voxel within the first candidate leaf
    }
    const int n12 = n[1] * n[2], C = n[0] * n12;
    for (int c = lane; c < C; c += 32)
      W.cand[c] = find_leaf(k, g, a[0] + c / n12, a[1] + (c / n[2]) % n[1], a[2] + c % n[2]);
    __syncwarp();
    const long long vin = __ldg(k.in_vbase + g);
    for (int j = lane; j < 8 * C; j += 32) {
      const int ci = W.cand[j >> 3], w = j & 7;
      uint64_t m = 0;
      int32_t b = 0;
      if (ci >= 0) {
        m = __ldg(k.in_masks + 8 * (long long)ci + w);
        const uint64_t wp = __ldg(k.in_wp + ci);
        const long long before = w ? (long long)((wp >> (9 * (w - 1))) & 511ull) : 0ll;
        b = (int32_t)(vin + __ldg(k.in_voff + ci) + before);
      }
      W.mask[j] = m;
      W.base[j] = b;
    }
    __syncwarp();
    // the halo: lanes take (x, y) rows of E2 voxels
    for (int t = lane; t < E[0] * E[1]; t += 32) {
      const int hx = t / E[1], hy = t - hx * E[1];
      const int rx = off[0] + hx, ry = off[1] + hy;
      const int rowc = (rx >> 3) * n12 + (ry >> 3) * n[2];
      const int bity = (ry & 7) << 3;
      int32_t* hrow = W.H + t * E[2];
      for (int hz = 0; hz < E[2]; ++hz) {
        const int rz = off[2] + hz;
        const int slot = (rowc + (rz >> 3)) * 8 + (rx & 7);
        const uint64_t word = W.mask[slot];
        const int bit = bity | (rz & 7);
        hrow[hz] = ((word >> bit) & 1ull) ? W.base[slot] + __popcll(word & ((1ull << bit) - 1ull)) : -1;
      }
    }
    // the output leaf's active voxels in order (lane l lists bits 16 l .. 16 l + 15)
    const uint32_t chunk = (uint32_t)(__ldg(k.out_masks + 8 * u + (lane >> 2)) >> (16 * (lane & 3))) & 0xFFFFu;
    const uint32_t cnt = __popc(chunk);
    uint32_t incl = cnt;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o2);
      if (lane >= o2) incl += y;
    }
    const int nvox = (int)__shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = incl - cnt, rest = chunk;
    while (rest) {
      const int bn = 16 * lane + __ffs(rest) - 1;
      rest &= rest - 1;
      const int p[3] = {bn >> 6, (bn >> 3) & 7, bn & 7};
      int hb = 0;
      uint32_t par = 0;
#pragma unroll
      for (int ax = 0; ax < 3; ++ax) {
        hb = hb * E[ax] + (tr ? (p[ax] >> sh) : p[ax]);
        if (tr && sh) par |= (uint32_t)(p[ax] & 1) << (2 - ax);
      }
      W.vh[pos++] = (uint16_t)(hb | (par << 10));
    }
    __syncwarp();
    const long long j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
    const int Etot = nvox * K;
    int32_t* row = k.map + j0 * K;
    int r = lane / K, kk = lane % K;
    const int step_r = 32 / K, step_k = 32 % K;
    for (int e = lane; e < Etot; e += 32) {
      const uint32_t vp = W.vh[r], dp = dh[kk];
      row[e] = ((vp ^ dp) >> 10) ? -1 : W.H[(vp & 1023u) + (dp & 1023u)];
      r += step_r;
      kk += step_k;
      if (kk >= K) {
        kk -= K;
        ++r;
      }
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_kmap_prep(const KmapPrep& p, int blocks, cudaStream_t s) {
  k_kmap_prep<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kmap(const KmapArgs& k, int blocks, cudaStream_t s) {
  k_kmap<<<blocks, kKmapThreads, 0, s>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_kmap_cands(const KmapArgs& k, int blocks, cudaStream_t s) {
  k_kmap_cands<<<blocks, 256, 0, s>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_kmap_halo(const KmapArgs& k, int blocks, cudaStream_t s) {
  k_kmap_halo<<<blocks, kHaloWarps * 32, 0, s>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_kmap_staged(const KmapArgs& k, int sms, cudaStream_t s) {
  const int K = (k.hi[0] - k.lo[0] + 1) * (k.hi[1] - k.lo[1] + 1) * (k.hi[2] - k.lo[2] + 1);
  const int S = k.span;
  if (S == 3 || K > kKmapBatchColumns) {
    const int blocks = (int)std::max(1ll, std::min((k.L_out + kLeafWarps - 1) / kLeafWarps, 4ll * sms));
    k_kmap_leafwarp<<<blocks, kLeafWarps * 32, 0, s>>>(k);
    return cudaGetLastError();
  }
  // chunks of 4 to 16 output leaves per warp (the kernel picks the size
  // from the grid), handed out by the counter; the grid is sized for chunks
  // of 4.  Shared memory: the column tables, then per warp the staged words
  // and a round's 32 voxel packs
  const long long chunks = (k.L_out + 3) / 4;
  const size_t smem = sizeof(StagedSmem) + (size_t)kStagedWarps * (sizeof(StagedWarp) + 128);
  const int blocks = (int)std::max(1ll, std::min((chunks + kStagedWarps - 1) / kStagedWarps, 4ll * sms));
  k_kmap_staged<<<blocks, kStagedWarps * 32, smem, s>>>(k);
  return cudaGetLastError();
}

}  // namespace tb
