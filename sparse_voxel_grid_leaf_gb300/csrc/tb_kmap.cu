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
// ascending bit index), the order of every other per-voxel array.  One warp
// per output leaf: its candidate input leaves (the few leaves any of its
// voxels can reach) are found by binary search in the input grid's canonical
// leaf list and kept in shared memory; the leaf's active voxels are listed in
// shared memory; then the warp writes the leaf's voxels x K entries, which
// are contiguous in the map.
#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

constexpr int kKmapThreads = 256;
constexpr int kKmapWarps = kKmapThreads / 32;

// Canonical order of leaf coordinates (origin >> 3): signed root tile
// (coordinate >> 9) x, y, z, then the upper child (>> 4 & 31) and the lower
// child (& 15), x-major; as a 128-bit (hi, lo) pair.
__device__ __forceinline__ void leaf_order_key(long long lx, long long ly, long long lz, unsigned long long& hi,
                                               unsigned long long& lo) {
  const unsigned long long bias = 1ull << 20;
  hi = ((unsigned long long)((lx >> 9) + bias) << 42) | ((unsigned long long)((ly >> 9) + bias) << 21) |
       (unsigned long long)((lz >> 9) + bias);
  lo = ((unsigned long long)((lx >> 4) & 31) << 22) | ((unsigned long long)((ly >> 4) & 31) << 17) |
       ((unsigned long long)((lz >> 4) & 31) << 12) | ((unsigned long long)(lx & 15) << 8) |
       ((unsigned long long)(ly & 15) << 4) | (unsigned long long)(lz & 15);
}

// Index of the leaf with coordinates (lx, ly, lz) among leaves [b, e) of a
// canonically ordered list, or -1.
__device__ long long find_leaf(const int32_t* origins, long long b, long long e, long long lx, long long ly,
                               long long lz) {
  unsigned long long kh, kl;
  leaf_order_key(lx, ly, lz, kh, kl);
  while (b < e) {
    const long long m = b + (e - b) / 2;
    unsigned long long mh, ml;
    leaf_order_key(__ldg(origins + 3 * m) >> 3, __ldg(origins + 3 * m + 1) >> 3, __ldg(origins + 3 * m + 2) >> 3, mh,
                   ml);
    if (mh == kh && ml == kl) return m;
    if (mh < kh || (mh == kh && ml < kl)) {
      b = m + 1;
    } else {
      e = m;
    }
  }
  return -1;
}

__device__ __forceinline__ long long floor_div_d(long long a, long long b) {
  const long long q = a / b;
  return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

__global__ void __launch_bounds__(kKmapThreads) k_kmap(const KmapArgs k) {
  __shared__ int32_t cand[kKmapWarps][kKmapMaxCand];
  __shared__ uint16_t vox[kKmapWarps][512];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const long long nwarps = (long long)gridDim.x * kKmapWarps;
  const int nb0 = k.hi[0] - k.lo[0] + 1, nb1 = k.hi[1] - k.lo[1] + 1, nb2 = k.hi[2] - k.lo[2] + 1;
  const int K = nb0 * nb1 * nb2, s = k.stride;
  for (long long u = (long long)blockIdx.x * kKmapWarps + wib; u < k.L_out; u += nwarps) {
    const int32_t g = __ldg(k.out_grid + u);
    const long long o[3] = {__ldg(k.out_origins + 3 * u), __ldg(k.out_origins + 3 * u + 1),
                            __ldg(k.out_origins + 3 * u + 2)};
    // input leaf coordinate range per axis
    long long a[3], n[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      long long qlo, qhi;
      if (k.transposed) {
        qlo = -floor_div_d(-(o[ax] - k.hi[ax]), s);  // ceil((p_min - hi) / s)
        qhi = floor_div_d(o[ax] + 7 - k.lo[ax], s);
      } else {
        qlo = (long long)s * o[ax] + k.lo[ax];
        qhi = (long long)s * (o[ax] + 7) + k.hi[ax];
      }
      a[ax] = floor_div_d(qlo, 8);
      n[ax] = floor_div_d(qhi, 8) - a[ax] + 1;
    }
    const int C = (int)(n[0] * n[1] * n[2]);  // <= kKmapMaxCand, checked by the host's bounds
    const long long ib = __ldg(k.in_leaf_off + g), ie = __ldg(k.in_leaf_off + g + 1);
    for (int c = lane; c < C; c += 32) {
      const long long lx = a[0] + c / (n[1] * n[2]), ly = a[1] + (c / n[2]) % n[1], lz = a[2] + c % n[2];
      cand[wib][c] = (int32_t)find_leaf(k.in_origins, ib, ie, lx, ly, lz);
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
    // the leaf's entries: map rows j0 .. j0 + nvox - 1, K entries each
    const long long j0 = __ldg(k.out_vbase + g) + __ldg(k.out_voff + u);
    const long long E = (long long)nvox * K;
    const long long vin = __ldg(k.in_vbase + g);
    int32_t* row = k.map + j0 * K;
    for (long long e = lane; e < E; e += 32) {
      const int r = (int)(e / K), kk = (int)(e % K);
      const int nbit = vox[wib][r];
      const long long p[3] = {o[0] + (nbit >> 6), o[1] + ((nbit >> 3) & 7), o[2] + (nbit & 7)};
      const int d[3] = {k.lo[0] + kk / (nb1 * nb2), k.lo[1] + (kk / nb2) % nb1, k.lo[2] + kk % nb2};
      long long q[3];
      bool ok = true;
#pragma unroll
      for (int ax = 0; ax < 3; ++ax) {
        if (k.transposed) {
          const long long t = p[ax] - d[ax];
          ok = ok && (t % s == 0);
          q[ax] = floor_div_d(t, s);
        } else {
          q[ax] = (long long)s * p[ax] + d[ax];
        }
      }
      int32_t idx = -1;
      if (ok) {
        const long long c = ((floor_div_d(q[0], 8) - a[0]) * n[1] + (floor_div_d(q[1], 8) - a[1])) * n[2] +
                            (floor_div_d(q[2], 8) - a[2]);
        const int32_t ci = cand[wib][c];
        if (ci >= 0) {
          const int wx = (int)(q[0] & 7), by = (int)(8 * (q[1] & 7) + (q[2] & 7));
          const uint64_t w = __ldg(k.in_masks + 8 * (long long)ci + wx);
          if ((w >> by) & 1ull) {
            const uint64_t wp = __ldg(k.in_wp + ci);
            const long long before = wx ? (long long)((wp >> (9 * (wx - 1))) & 511ull) : 0ll;
            idx = (int32_t)(vin + __ldg(k.in_voff + ci) + before + __popcll(w & ((1ull << by) - 1ull)));
          }
        }
      }
      row[e] = idx;
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_kmap(const KmapArgs& k, int blocks, cudaStream_t s) {
  k_kmap<<<blocks, kKmapThreads, 0, s>>>(k);
  return cudaGetLastError();
}

}  // namespace tb
