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
// table of the input leaves is built first; then one warp per output leaf:
// its candidate input leaves (the few leaves any of its voxels can reach) are
// looked up and kept in shared memory; the leaf's active voxels are listed in
// shared memory; then the warp writes the leaf's voxels x K entries, which
// are contiguous in the map.  Three forms of that warp's work, picked by the
// host from the box and the output's size:
//   k_kmap_halo    the input index of every voxel in the leaf's reach is
//                  tabulated once; an entry is one shared-memory word
//   k_kmap_staged  the candidates' mask words and word bases are staged; an
//                  entry is a packed-coordinate add, a bit test and a
//                  popcount (with k_kmap_cands doing the look-ups first for
//                  large outputs)
//   k_kmap         any box: an entry computes its input leaf and reads it
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

// The host sizes the table to at least twice the leaves, so every insert
// finds an empty slot within the bounded probe loop.
__global__ void __launch_bounds__(256) k_leaf_table(const int32_t* origins, const int32_t* leaf_grid, long long L,
                                                    int32_t* table, unsigned long long mask) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < L; i += stride) {
    unsigned long long h = leaf_hash(leaf_grid[i], origins[3 * i] >> 3, origins[3 * i + 1] >> 3, origins[3 * i + 2] >> 3);
    for (unsigned long long probe = 0; probe <= mask; ++probe, ++h)  // at most the table's size
      if (atomicCAS(table + (h & mask), -1, (int32_t)i) == -1) break;
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
// input leaves per axis (27 candidates; the host checks): the candidates'
// mask words and the first voxel index of each word are staged in shared
// memory, each active output voxel's position is packed once as three bytes
// (its coordinate relative to the first candidate leaf, minus the column's
// part), and each column's offset likewise, so an entry costs a byte-wise
// add, one shared-memory word, a bit test and a popcount.  Coordinates
// relative to the first candidate leaf's origin Q_b: stride 1 q = o + p + d,
// so o - Q_b + p + d; forward stride 2, 2o - Q_b + 2p + d; transposed
// stride 1, o - Q_b + p - d; transposed stride 2 (p - d even),
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
// candidate): the hash look-ups of all leaves run side by side here, so the
// map kernel starts each leaf from one coalesced load.
__global__ void __launch_bounds__(256) k_kmap_cands(const KmapArgs k) {
  const long long total = k.L_out * k.cand_max;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long u = i / k.cand_max;
    const int c = (int)(i - u * k.cand_max);
    long long a[3];
    int n[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) reach(k, ax, __ldg(k.out_origins + 3 * u + ax), a[ax], n[ax]);
    int32_t ci = -1;
    if (c < n[0] * n[1] * n[2]) {
      const int n12 = n[1] * n[2];
      ci = find_leaf(k, __ldg(k.out_grid + u), a[0] + c / n12, a[1] + (c / n[2]) % n[1], a[2] + c % n[2]);
    }
    k.cands[i] = ci;
  }
}
constexpr int kStagedWarps = 8;
struct KmapWarp {
  uint64_t mask[kStagedCand * 8];  // word w of candidate c at 8 c + w (0: no candidate)
  int32_t base[kStagedCand * 8];   // first voxel index of that word
  int32_t cand[kStagedCand];
  uint32_t vpk[512];               // per active voxel: 3 relative-coordinate bytes | parity << 24
};

__global__ void __launch_bounds__(kStagedWarps * 32, 4) k_kmap_staged(const KmapArgs k) {
  __shared__ KmapWarp sw[kStagedWarps];
  __shared__ uint32_t dpk[kKmapTab];  // per column: 3 offset bytes (biased by 8) | parity << 24
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  KmapWarp& W = sw[wib];
  const long long nwarps = (long long)gridDim.x * kStagedWarps;
  const int nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = (k.hi[0] - k.lo[0] + 1) * nb1 * nb2;
  const int sh = k.stride == 2 ? 1 : 0, tr = k.transposed;
  for (int i = threadIdx.x; i < K; i += kStagedWarps * 32) {
    const int d[3] = {k.lo[0] + i / (nb1 * nb2), k.lo[1] + (i / nb2) % nb1, k.lo[2] + i % nb2};
    uint32_t v = 0, par = 0;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const int gv = tr ? -(d[ax] >> sh) : d[ax];
      v |= (uint32_t)(gv + 8) << (8 * ax);
      if (tr && sh) par |= (uint32_t)(d[ax] & 1) << (2 - ax);
    }
    dpk[i] = v | (par << 24);
  }
  __syncthreads();
  for (long long u = (long long)blockIdx.x * kStagedWarps + wib; u < k.L_out; u += nwarps) {
    const int32_t g = __ldg(k.out_grid + u);
    long long a[3];
    int n[3], A[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const long long o = __ldg(k.out_origins + 3 * u + ax);
      reach(k, ax, o, a[ax], n[ax]);
      A[ax] = (int)((tr ? (o >> sh) : (o << sh)) - (a[ax] << 3));
    }
    const int n12 = n[1] * n[2], C = n[0] * n12;
    if (k.cands) {
      if (lane < C) W.cand[lane] = __ldcg(k.cands + u * k.cand_max + lane);
    } else {
      for (int c = lane; c < C; c += 32)
        W.cand[c] = find_leaf(k, g, a[0] + c / n12, a[1] + (c / n[2]) % n[1], a[2] + c % n[2]);
    }
    __syncwarp();
    const long long vin = __ldg(k.in_vbase + g);
    for (int j = lane; j < 8 * C; j += 32) {
      const int ci = W.cand[j >> 3], w = j & 7;
      uint64_t m = 0;
      int32_t b = -1;
      if (ci >= 0) {
        m = __ldg(k.in_masks + 8 * (long long)ci + w);
        const uint64_t wp = __ldg(k.in_wp + ci);
        const long long before = w ? (long long)((wp >> (9 * (w - 1))) & 511ull) : 0ll;
        b = (int32_t)(vin + __ldg(k.in_voff + ci) + before);
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
      uint32_t v = 0, par = 0;
#pragma unroll
      for (int ax = 0; ax < 3; ++ax) {
        const int f = tr ? (p[ax] >> sh) : (p[ax] << sh);
        v |= (uint32_t)(A[ax] + f) << (8 * ax);
        if (tr && sh) par |= (uint32_t)(p[ax] & 1) << (2 - ax);
      }
      W.vpk[pos++] = v | (par << 24);
    }
    __syncwarp();
    const long long j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
    const int Etot = (int)nvox * K;
    int32_t* row = k.map + j0 * K;
    int r = lane / K, kk = lane % K;
    const int step_r = 32 / K, step_k = 32 % K;
    const uint32_t n2 = (uint32_t)n[2], nm = (uint32_t)(8 * C - 1);
    for (int e = lane; e < Etot; e += 32) {
      const uint32_t vp = W.vpk[r], dp = dpk[kk];
      // branch-free: a column of the wrong parity (transposed stride 2) reads
      // a clamped slot and is then masked out
      const uint32_t rel = (vp & 0xFFFFFFu) + (dp & 0xFFFFFFu) - 0x080808u;
      const uint32_t rx = rel & 0xFFu, ry = (rel >> 8) & 0xFFu, rz = (rel >> 16) & 0xFFu;
      const uint32_t slot = min((((rx >> 3) * (uint32_t)n12 + (ry >> 3) * n2 + (rz >> 3)) << 3) | (rx & 7u), nm);
      const uint64_t word = W.mask[slot];
      const uint32_t bit = ((ry & 7u) << 3) | (rz & 7u);
      const uint64_t upto = word << (63u - bit);  // bit 63: the voxel; the rest: the voxels before it
      const bool on = (vp >> 24) == (dp >> 24) && (upto >> 63);
      row[e] = on ? W.base[slot] + __popcll(upto) - 1 : -1;
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
  __shared__ uint16_t dh[kKmapStagedColumns];  // per column: delta(d) | parity << 10
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
    if (k.cands) {
      if (lane < C) W.cand[lane] = __ldcg(k.cands + u * k.cand_max + lane);
    } else {
      for (int c = lane; c < C; c += 32)
        W.cand[c] = find_leaf(k, g, a[0] + c / n12, a[1] + (c / n[2]) % n[1], a[2] + c % n[2]);
    }
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

cudaError_t launch_leaf_table(const int32_t* origins, const int32_t* leaf_grid, long long L, int32_t* table,
                              unsigned long long mask, int blocks, cudaStream_t s) {
  k_leaf_table<<<blocks, 256, 0, s>>>(origins, leaf_grid, L, table, mask);
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

cudaError_t launch_kmap_staged(const KmapArgs& k, int blocks, cudaStream_t s) {
  k_kmap_staged<<<blocks, kStagedWarps * 32, 0, s>>>(k);
  return cudaGetLastError();
}

}  // namespace tb
