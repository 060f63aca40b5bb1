// Emission: one kernel over all source leaves (or voxels) of all grids writes
// candidate output-leaf slots (canonical key, source reference), fVDB PR #757
// "Batched leaf-mask topology construction for generated conv grids", Summary
// item 1 (first bullet) and item 2 (box-dilate scatter with up to 27 target
// leaves per source leaf).  Empty candidates are never emitted.  The same
// kernel builds the radix histograms of every digit pass of the sort, and its
// last block turns them into global digit offsets.
//
// Also: the range prepasses of the two front ends (coordinate bbox and input
// checks), whose readback sizes the sort key.
#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

constexpr int kEmitThreads = 256;

__device__ __forceinline__ int grid_of(const int64_t* offsets, int32_t B, long long i) {
  // last g with offsets[g] <= i (offsets non-decreasing, offsets[0] == 0)
  int lo = 0, hi = B;  // answer in [0, B)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(offsets + mid) <= i) lo = mid; else hi = mid;
  }
  return lo;
}

struct Target {
  int32_t lc[3];
  uint32_t code;
};

// Per-source targets of each op.  Returns a bit set of non-empty target codes.
template <int OP>
__device__ __forceinline__ uint32_t targets_of(const PassArgs& a, const uint64_t m[8]);

template <>
__device__ __forceinline__ uint32_t targets_of<kLeaves>(const PassArgs&, const uint64_t m[8]) {
  uint64_t any = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) any |= m[w];
  return any ? 1u : 0u;
}

template <>
__device__ __forceinline__ uint32_t targets_of<kCoarsen>(const PassArgs& a, const uint64_t m[8]) {
  return targets_of<kLeaves>(a, m);
}

// Child c = 4*cx + 2*cy + cz is non-empty iff the parent's octant c holds a voxel.
template <>
__device__ __forceinline__ uint32_t targets_of<kRefine>(const PassArgs&, const uint64_t m[8]) {
  uint32_t bits = 0;
#pragma unroll
  for (int cx = 0; cx < 2; ++cx) {
    const uint64_t t = m[4 * cx] | m[4 * cx + 1] | m[4 * cx + 2] | m[4 * cx + 3];
#pragma unroll
    for (int cy = 0; cy < 2; ++cy)
#pragma unroll
      for (int cz = 0; cz < 2; ++cz) {
        const uint64_t oct = 0x0F0F0F0Full << (32 * cy + 4 * cz);
        if (t & oct) bits |= 1u << (4 * cx + 2 * cy + cz);
      }
  }
  return bits;
}

// Target offset t (per axis in {-1,0,1}, code 9*(tx+1) + 3*(ty+1) + (tz+1)) is
// non-empty iff a voxel lies in the zone that reaches it: any position for
// t = 0, the last plane for t = +1 (needs hi = 1), the first for t = -1
// (needs lo = -1).
template <>
__device__ __forceinline__ uint32_t targets_of<kDilate>(const PassArgs& a, const uint64_t m[8]) {
  uint64_t all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) all |= m[w];
  const uint64_t xs[3] = {m[0], all, m[7]};  // zones for tx = -1, 0, +1
  const uint64_t ym[3] = {0x00000000000000FFull, ~0ull, 0xFF00000000000000ull};
  const uint64_t zm[3] = {0x0101010101010101ull, ~0ull, 0x8080808080808080ull};
  uint32_t bits = 0;
#pragma unroll
  for (int tx = -1; tx <= 1; ++tx)
#pragma unroll
    for (int ty = -1; ty <= 1; ++ty)
#pragma unroll
      for (int tz = -1; tz <= 1; ++tz) {
        if (tx < a.lo[0] || tx > a.hi[0] || ty < a.lo[1] || ty > a.hi[1] || tz < a.lo[2] || tz > a.hi[2])
          continue;
        if (xs[tx + 1] & ym[ty + 1] & zm[tz + 1]) bits |= 1u << (9 * (tx + 1) + 3 * (ty + 1) + (tz + 1));
      }
  return bits;
}

template <int OP>
__device__ __forceinline__ void target_lc(const int32_t lc[3], uint32_t code, int32_t out[3]) {
  if (OP == kRefine) {
    out[0] = 2 * lc[0] + (int32_t)((code >> 2) & 1);
    out[1] = 2 * lc[1] + (int32_t)((code >> 1) & 1);
    out[2] = 2 * lc[2] + (int32_t)(code & 1);
  } else if (OP == kCoarsen) {
    out[0] = lc[0] >> 1;
    out[1] = lc[1] >> 1;
    out[2] = lc[2] >> 1;
  } else if (OP == kDilate) {
    out[0] = lc[0] + (int32_t)(code / 9) - 1;
    out[1] = lc[1] + (int32_t)((code / 3) % 3) - 1;
    out[2] = lc[2] + (int32_t)(code % 3) - 1;
  } else {
    out[0] = lc[0];
    out[1] = lc[1];
    out[2] = lc[2];
  }
}

__device__ __forceinline__ void hist_add(unsigned int (*s_hist)[kBins], int P, uint64_t key) {
  for (int p = 0; p < P; ++p) atomicAdd(&s_hist[p][(uint32_t)(key >> (8 * p)) & 255u], 1u);
}

// Writes `n` slots of this thread at warp-aggregated positions; returns the
// first position.
__device__ __forceinline__ unsigned long long claim_slots(const PassArgs& a, uint32_t n) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  unsigned long long base = 0;
  if (lane == 31 && total) base = atomicAdd(&a.rb->num_slots, (unsigned long long)total);
  base = __shfl_sync(0xffffffffu, base, 31);
  return base + incl - n;
}

__device__ void finish_histograms(const PassArgs& a, unsigned int (*s_hist)[kBins]) {
  __syncthreads();
  for (int i = threadIdx.x; i < a.P * kBins; i += blockDim.x) {
    const unsigned int c = (&s_hist[0][0])[i];
    if (c) atomicAdd(&(&a.ctl->hist[0][0])[i], c);
  }
  if (!last_block_done(&a.ctl->emit_ticket)) return;
  __shared__ unsigned int s_scan[8];
  for (int p = 0; p < a.P; ++p) {
    const unsigned int v = __ldcg(&a.ctl->hist[p][threadIdx.x]);
    unsigned int total;
    const unsigned int ex = block_excl_scan_256(v, s_scan, &total);
    a.ctl->bin_base[p][threadIdx.x] = ex;
  }
  if (threadIdx.x == 0 && __ldcg(&a.rb->num_slots) > (unsigned long long)a.slot_cap)
    atomicOr(&a.rb->err, kErrSlotOverflow);
}

// One thread per source leaf.
template <int OP>
__global__ void __launch_bounds__(kEmitThreads) k_emit_leaves(const PassArgs a) {
  __shared__ unsigned int s_hist[kMaxDigitPasses][kBins];
  for (int i = threadIdx.x; i < a.P * kBins; i += blockDim.x) (&s_hist[0][0])[i] = 0;
  __syncthreads();
  const long long L = a.src_count_dev ? (long long)*a.src_count_dev : a.src_count;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x; base < L; base += stride) {
    const long long i = base + threadIdx.x;
    uint32_t bits = 0;
    int32_t lc[3] = {0, 0, 0};
    uint32_t g = 0;
    if (i < L) {
      uint64_t m[8];
      load_mask(a.src_masks, i, m);
      bits = targets_of<OP>(a, m);
      lc[0] = __ldg(a.src_origins + 3 * i) >> 3;
      lc[1] = __ldg(a.src_origins + 3 * i + 1) >> 3;
      lc[2] = __ldg(a.src_origins + 3 * i + 2) >> 3;
      g = a.src_grid ? (uint32_t)__ldg(a.src_grid + i) : (uint32_t)grid_of(a.in_offsets, a.B, i);
    }
    unsigned long long pos = claim_slots(a, __popc(bits));
    while (bits) {
      const uint32_t code = __ffs(bits) - 1;
      bits &= bits - 1;
      int32_t t[3];
      target_lc<OP>(lc, code, t);
      uint32_t ref_code = code;
      if (OP == kCoarsen)  // octant of the source leaf inside its coarse leaf
        ref_code = (uint32_t)(((lc[0] & 1) << 2) | ((lc[1] & 1) << 1) | (lc[2] & 1));
      const uint64_t key = encode_key(a.K, g, t[0], t[1], t[2]);
      if (pos < (unsigned long long)a.slot_cap) {
        a.keys[0][pos] = key;
        a.vals[0][pos] = ((uint32_t)i << kSrcShift) | ref_code;
      }
      ++pos;
      hist_add(s_hist, a.P, key);
    }
  }
  finish_histograms(a, s_hist);
}

// One thread per input voxel (ijk front end); slot value = voxel index.
__global__ void __launch_bounds__(kEmitThreads) k_emit_ijk(const PassArgs a) {
  __shared__ unsigned int s_hist[kMaxDigitPasses][kBins];
  for (int i = threadIdx.x; i < a.P * kBins; i += blockDim.x) (&s_hist[0][0])[i] = 0;
  __syncthreads();
  const long long N = a.src_count;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x; base < N; base += stride) {
    const long long i = base + threadIdx.x;
    const bool valid = i < N;
    const unsigned long long pos = claim_slots(a, valid ? 1u : 0u);
    if (valid) {
      const int32_t x = __ldg(a.ijk + 3 * i), y = __ldg(a.ijk + 3 * i + 1), z = __ldg(a.ijk + 3 * i + 2);
      const uint32_t g = (uint32_t)grid_of(a.in_offsets, a.B, i);
      const uint64_t key = encode_key(a.K, g, x >> 3, y >> 3, z >> 3);
      if (pos < (unsigned long long)a.slot_cap) {
        a.keys[0][pos] = key;
        a.vals[0][pos] = (uint32_t)i;
      }
      hist_add(s_hist, a.P, key);
    }
  }
  finish_histograms(a, s_hist);
}

// ---------------------------------------------------------------- front-end prepasses

__device__ void reduce_bbox(const int32_t mn[3], const int32_t mx[3], unsigned int* enc) {
  // block-level reduction of the encoded bounds, then one atomic per block
  __shared__ unsigned int s_enc[6];
  if (threadIdx.x < 6) s_enc[threadIdx.x] = 0;
  __syncthreads();
  unsigned int e[6] = {enc_min(mn[0]), enc_min(mn[1]), enc_min(mn[2]), enc_max(mx[0]), enc_max(mx[1]),
                       enc_max(mx[2])};
#pragma unroll
  for (int k = 0; k < 6; ++k) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) e[k] = max(e[k], __shfl_xor_sync(0xffffffffu, e[k], off));
  }
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 6; ++k) atomicMax(&s_enc[k], e[k]);
  __syncthreads();
  if (threadIdx.x < 6 && s_enc[threadIdx.x]) atomicMax(&enc[threadIdx.x], s_enc[threadIdx.x]);
}

__device__ void check_offsets(const int64_t* off, int32_t B, long long n, unsigned int* err) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g <= B; g += stride) {
    const int64_t v = off[g];
    bool bad = (g == 0 && v != 0) || (g == B && v != n) || v < 0 || v > n;
    if (g > 0 && off[g - 1] > v) bad = true;
    if (bad) atomicOr(err, kErrBadOffsets);
  }
}

__global__ void __launch_bounds__(256) k_prepass_ijk(const int32_t* ijk, long long N, const int64_t* off,
                                                     int32_t B, ReadbackHeader* rb) {
  int32_t mn[3] = {INT32_MAX, INT32_MAX, INT32_MAX}, mx[3] = {INT32_MIN, INT32_MIN, INT32_MIN};
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride)
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const int32_t v = __ldg(ijk + 3 * i + a);
      mn[a] = min(mn[a], v);
      mx[a] = max(mx[a], v);
    }
  reduce_bbox(mn, mx, rb->bbox_enc);
  check_offsets(off, B, N, &rb->err);
}

// Exact voxel bbox of a leaf list (from the set bits), plus origin alignment.
__global__ void __launch_bounds__(256) k_prepass_leaves(const int32_t* origins, const uint64_t* masks,
                                                        long long L, const int64_t* off, int32_t B,
                                                        ReadbackHeader* rb) {
  int32_t mn[3] = {INT32_MAX, INT32_MAX, INT32_MAX}, mx[3] = {INT32_MIN, INT32_MIN, INT32_MIN};
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < L; i += stride) {
    uint64_t m[8];
    load_mask(masks, i, m);
    uint64_t all = 0;
    uint32_t xbits = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      all |= m[w];
      if (m[w]) xbits |= 1u << w;
    }
    const int32_t o[3] = {__ldg(origins + 3 * i), __ldg(origins + 3 * i + 1), __ldg(origins + 3 * i + 2)};
    if ((o[0] | o[1] | o[2]) & 7) atomicOr(&rb->err, kErrNotAligned);
    if (!all) continue;
    uint32_t ybits = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if ((all >> (8 * r)) & 0xFFull) ybits |= 1u << r;
    uint64_t z = all | (all >> 32);
    z |= z >> 16;
    z |= z >> 8;
    const uint32_t zbits = (uint32_t)(z & 0xFFull);
    const uint32_t b[3] = {xbits, ybits, zbits};
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      mn[a] = min(mn[a], o[a] + (__ffs(b[a]) - 1));
      mx[a] = max(mx[a], o[a] + (31 - __clz(b[a])));
    }
  }
  reduce_bbox(mn, mx, rb->bbox_enc);
  check_offsets(off, B, L, &rb->err);
}

}  // namespace

// ---------------------------------------------------------------- launchers

cudaError_t launch_emit(int op, const PassArgs& a, int blocks, cudaStream_t s) {
  switch (op) {
    case kIjk: k_emit_ijk<<<blocks, kEmitThreads, 0, s>>>(a); break;
    case kLeaves: k_emit_leaves<kLeaves><<<blocks, kEmitThreads, 0, s>>>(a); break;
    case kRefine: k_emit_leaves<kRefine><<<blocks, kEmitThreads, 0, s>>>(a); break;
    case kCoarsen: k_emit_leaves<kCoarsen><<<blocks, kEmitThreads, 0, s>>>(a); break;
    case kDilate: k_emit_leaves<kDilate><<<blocks, kEmitThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_prepass_ijk(const int32_t* ijk, long long N, const int64_t* off, int32_t B,
                               ReadbackHeader* rb, int blocks, cudaStream_t s) {
  k_prepass_ijk<<<blocks, 256, 0, s>>>(ijk, N, off, B, rb);
  return cudaGetLastError();
}

cudaError_t launch_prepass_leaves(const int32_t* origins, const uint64_t* masks, long long L, const int64_t* off,
                                  int32_t B, ReadbackHeader* rb, int blocks, cudaStream_t s) {
  k_prepass_leaves<<<blocks, 256, 0, s>>>(origins, masks, L, off, B, rb);
  return cudaGetLastError();
}

}  // namespace tb
