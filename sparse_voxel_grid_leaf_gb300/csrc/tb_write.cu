// Batched writers (fVDB PR #757 "Batched leaf-mask topology construction for
// generated conv grids", Summary item 1, fourth bullet): after the single
// count readback, one kernel writes every grid's leaf records -- origin,
// mask, voxel offset (a per-grid segmented scan), word popcount prefix and
// bbox -- plus node linkage and per-grid counts/bboxes; empty grids become
// valid empty grids.  An intermediate pass of a chain uses the same kernel
// without the readback and writes only (origin, mask, grid) for the next pass.
//
// Eight lanes handle one output leaf, lane w owning mask word w.  A leaf's
// mask is the OR over its run of sorted slots of each slot's contribution,
// recomputed from the 64-byte source mask (refine / coarsen / box-dilate bit
// arithmetic of Summary items 1-2).
#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

template <int OP>
__device__ __forceinline__ uint64_t contrib(const PassArgs& a, uint32_t val, int w) {
  const long long src = (long long)(val >> kSrcShift);
  const uint32_t code = val & 31u;
  const uint64_t* __restrict__ sm = a.src_masks + 8 * src;
  if (OP == kLeaves) {
    return __ldg(sm + w);
  } else if (OP == kRefine) {
    const int cx = (code >> 2) & 1, cy = (code >> 1) & 1, cz = code & 1;
    return refine_word(__ldg(sm + 4 * cx + (w >> 1)), cy, cz);
  } else if (OP == kCoarsen) {
    const int qx = (code >> 2) & 1, qy = (code >> 1) & 1, qz = code & 1;
    if ((w >> 2) != qx) return 0ull;
    const int X = w & 3;
    return coarsen_word(__ldg(sm + 2 * X) | __ldg(sm + 2 * X + 1), qy, qz);
  } else {  // kDilate
    const int tx = (int)(code / 9) - 1, ty = (int)((code / 3) % 3) - 1, tz = (int)(code % 3) - 1;
    uint64_t r = 0;
    if (tx == 0) {
      for (int d = a.lo[0]; d <= a.hi[0]; ++d) {
        const int xs = w - d;
        if (xs >= 0 && xs < 8) r |= __ldg(sm + xs);
      }
    } else if (tx > 0) {
      if (w == 0) r = __ldg(sm + 7);
    } else {
      if (w == 7) r = __ldg(sm + 0);
    }
    return dilate_y(dilate_z(r, tz, a.lo[2], a.hi[2]), ty, a.lo[1], a.hi[1]);
  }
}

template <int OP>
__device__ __forceinline__ uint64_t merge_run(const PassArgs& a, const uint32_t* __restrict__ vals, uint32_t s0,
                                              uint32_t s1, int w) {
  uint64_t word = 0;
  if (OP == kIjk) {
    for (uint32_t s = s0; s < s1; ++s) {
      const long long n = vals[s];
      const int32_t x = __ldg(a.ijk + 3 * n), y = __ldg(a.ijk + 3 * n + 1), z = __ldg(a.ijk + 3 * n + 2);
      if ((x & 7) == w) word |= 1ull << (8 * (y & 7) + (z & 7));
    }
  } else {
    for (uint32_t s = s0; s < s1; ++s) word |= contrib<OP>(a, vals[s], w);
  }
  return word;
}

__device__ __forceinline__ uint32_t bits_of_bytes(uint64_t m) {
  uint32_t b = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if ((m >> (8 * r)) & 0xFFull) b |= 1u << r;
  return b;
}

template <int OP, bool FINAL>
__global__ void __launch_bounds__(kWriteThreads) k_write(const PassArgs a, const WriteOut o) {
  __shared__ uint32_t s_pop[kWriteTile];
  __shared__ uint32_t s_head[kWriteTile];
  __shared__ long long s_off[kWriteTile];
  __shared__ uint32_t s_tile;

  const uint64_t* __restrict__ keys = a.keys[a.sorted];
  const uint32_t* __restrict__ vals = a.vals[a.sorted];
  const long long U = (long long)a.rb->num_leaves;
  const long long ntiles = (U + kWriteTile - 1) / kWriteTile;
  const int tid = threadIdx.x, lane = tid & 31, w = tid & 7, slot = tid >> 3;
  long long iter = 0;

  for (;;) {
    long long tile;
    if (FINAL) {
      if (tid == 0) s_tile = atomicAdd(&a.ctl->write_tile_ctr, 1u);
      __syncthreads();
      tile = s_tile;
    } else {
      tile = (long long)blockIdx.x + iter * gridDim.x;
      ++iter;
    }
    if (tile >= ntiles) break;

    uint32_t g_row[kWriteRows];
#pragma unroll
    for (int r = 0; r < kWriteRows; ++r) {
      const int e = r * 32 + slot;
      const long long u = tile * kWriteTile + e;
      const bool valid = u < U;
      uint64_t word = 0;
      int32_t lc[3] = {0, 0, 0};
      uint32_t g = 0;
      if (valid) {
        const uint32_t s0 = a.run_start[u], s1 = a.run_start[u + 1];
        decode_key(a.K, keys[s0], g, lc);
        word = merge_run<OP>(a, vals, s0, s1, w);
      }
      g_row[r] = g;
      const int32_t org[3] = {(int32_t)((uint32_t)lc[0] << 3), (int32_t)((uint32_t)lc[1] << 3),
                              (int32_t)((uint32_t)lc[2] << 3)};
      if (!FINAL) {
        if (valid) {
          o.masks[8 * u + w] = word;
          if (w < 3) o.origins[3 * u + w] = org[w];
          if (w == 3) o.leaf_grid[u] = (int32_t)g;
        }
        continue;
      }
      // popcounts and the 7 x 9-bit word prefix
      const uint32_t pop = __popcll(word);
      uint32_t incl = pop;
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off, 8);
        if (w >= off) incl += y;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 7, 8);
      uint64_t wp = w ? ((uint64_t)(incl - pop) << (9 * (w - 1))) : 0ull;
      uint64_t orm = word;
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) {
        wp |= __shfl_xor_sync(0xffffffffu, wp, off);
        orm |= __shfl_xor_sync(0xffffffffu, orm, off);
      }
      const uint32_t ballot = __ballot_sync(0xffffffffu, word != 0);
      const uint32_t xbits = (ballot >> (lane & ~7)) & 0xFFu;
      const uint32_t ybits = bits_of_bytes(orm);
      uint64_t zz = orm | (orm >> 32);
      zz |= zz >> 16;
      zz |= zz >> 8;
      const uint32_t zbits = (uint32_t)(zz & 0xFFull);
      if (valid) {
        const uint32_t bits[3] = {xbits, ybits, zbits};
        o.masks[8 * u + w] = word;
        if (w < 3) o.origins[3 * u + w] = org[w];
        if (w < 6) {
          const int ax = w < 3 ? w : w - 3;
          const int32_t v = w < 3 ? org[ax] + (__ffs(bits[ax]) - 1) : org[ax] + (31 - __clz(bits[ax]));
          o.leaf_bbox[6 * u + w] = v;
          atomicMax(&a.gbox[6 * g + w], w < 3 ? enc_min(v) : enc_max(v));
        }
        if (w == 6) o.word_prefix[u] = wp;
        if (w == 7) o.leaf_grid[u] = (int32_t)g;
        if (w == 3) o.leaf_parent[u] = (int32_t)((long long)a.leaf_lower[u] - a.lower_off[g]);
        if (w == 4) {
          const uint32_t lw = a.leaf_lower[u];
          if (u == 0 || a.leaf_lower[u - 1] != lw) {
#pragma unroll
            for (int c = 0; c < 3; ++c) o.lower_origins[3 * (long long)lw + c] = (int32_t)((uint32_t)org[c] & ~127u);
            o.lower_parent[lw] = (int32_t)((long long)a.leaf_upper[u] - a.upper_off[g]);
          }
        }
        if (w == 5) {
          const uint32_t up = a.leaf_upper[u];
          if (u == 0 || a.leaf_upper[u - 1] != up) {
#pragma unroll
            for (int c = 0; c < 3; ++c) o.upper_origins[3 * (long long)up + c] = (int32_t)((uint32_t)org[c] & ~4095u);
          }
        }
      }
      if (w == 0) {
        s_pop[e] = valid ? total : 0u;
        s_head[e] = (valid && u == a.leaf_off[g]) ? 1u : 0u;
      }
    }
    if (!FINAL) continue;
    __syncthreads();

    // per-grid segmented exclusive scan of voxel counts over the tile's leaves
    if (tid < 32) {
      uint32_t p[4], h[4];
      uint32_t f = 0;
      unsigned long long v = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p[q] = s_pop[4 * lane + q];
        h[q] = s_head[4 * lane + q];
        if (h[q]) {
          f = 1;
          v = p[q];
        } else {
          v += p[q];
        }
      }
      uint32_t F = f;
      unsigned long long V = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t F2 = __shfl_up_sync(0xffffffffu, F, off);
        const unsigned long long V2 = __shfl_up_sync(0xffffffffu, V, off);
        if (lane >= off) {
          if (!F) V += V2;
          F |= F2;
        }
      }
      uint32_t Fe = __shfl_up_sync(0xffffffffu, F, 1);
      unsigned long long Ve = __shfl_up_sync(0xffffffffu, V, 1);
      if (lane == 0) {
        Fe = 0;
        Ve = 0;
      }
      const uint32_t Ft = __shfl_sync(0xffffffffu, F, 31);
      const unsigned long long Vt = __shfl_sync(0xffffffffu, V, 31);
      unsigned long long excl_tile = 0;
      if (lane == 0) excl_tile = lookback64(a.write_status, 1, tile, Vt, Ft != 0, &a.rb->err);
      excl_tile = __shfl_sync(0xffffffffu, excl_tile, 0);
      uint32_t fr = Fe;
      unsigned long long vr = Ve;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const long long off_v = h[q] ? 0ll : (long long)(vr + (fr ? 0ull : excl_tile));
        s_off[4 * lane + q] = off_v;
        if (h[q]) {
          fr = 1;
          vr = p[q];
        } else {
          vr += p[q];
        }
      }
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
      for (int r = 0; r < kWriteRows; ++r) {
        const int e = r * 32 + slot;
        const long long u = tile * kWriteTile + e;
        if (u < U) {
          o.voxel_offset[u] = s_off[e];
          const uint32_t g = g_row[r];
          if (u == a.leaf_off[g + 1] - 1) o.voxel_counts[g] = s_off[e] + (long long)s_pop[e];
        }
      }
    }
    __syncthreads();
  }

  if (!FINAL) return;
  if (!last_block_done(&a.ctl->write_ticket)) return;
  for (long long g = tid; g <= a.B; g += blockDim.x) {
    o.leaf_offsets[g] = a.leaf_off[g];
    o.lower_offsets[g] = a.lower_off[g];
    o.upper_offsets[g] = a.upper_off[g];
    if (g == a.B) break;
    const int64_t nleaf = a.leaf_off[g + 1] - a.leaf_off[g];
    o.node_counts[3 * g + 0] = (int32_t)(a.upper_off[g + 1] - a.upper_off[g]);
    o.node_counts[3 * g + 1] = (int32_t)(a.lower_off[g + 1] - a.lower_off[g]);
    o.node_counts[3 * g + 2] = (int32_t)nleaf;
    if (nleaf == 0) o.voxel_counts[g] = 0;
#pragma unroll
    for (int c = 0; c < 6; ++c) {
      const unsigned int e = __ldcg(&a.gbox[6 * g + c]);
      o.grid_bbox[6 * g + c] = c < 3 ? dec_min(e) : dec_max(e);
    }
  }
}

// Canonical-order comparison of two leaf origins: signed tile, then x-major
// upper child offset, then x-major lower child offset.
__device__ __forceinline__ bool canon_less(const int32_t a[3], const int32_t b[3]) {
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
    if ((a[ax] >> 12) != (b[ax] >> 12)) return (a[ax] >> 12) < (b[ax] >> 12);
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
    if (((a[ax] >> 7) & 31) != ((b[ax] >> 7) & 31)) return ((a[ax] >> 7) & 31) < ((b[ax] >> 7) & 31);
#pragma unroll
  for (int ax = 0; ax < 3; ++ax)
    if (((a[ax] >> 3) & 15) != ((b[ax] >> 3) & 15)) return ((a[ax] >> 3) & 15) < ((b[ax] >> 3) & 15);
  return false;
}

__global__ void __launch_bounds__(256) k_validate(const int32_t* origins, const uint64_t* masks,
                                                  const int32_t* leaf_grid, const int64_t* off, long long L,
                                                  int32_t B, unsigned int* err) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g <= B; g += stride) {
    const int64_t v = off[g];
    if ((g == 0 && v != 0) || (g == B && v != L) || (g > 0 && off[g - 1] > v)) atomicOr(err, kErrNotCanonical);
  }
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < L; i += stride) {
    const int32_t o[3] = {origins[3 * i], origins[3 * i + 1], origins[3 * i + 2]};
    bool bad = ((o[0] | o[1] | o[2]) & 7) != 0;
    uint64_t m[8];
    load_mask(masks, i, m);
    uint64_t any = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) any |= m[w];
    bad |= (any == 0);
    const int32_t g = leaf_grid[i];
    if (g < 0 || g >= B || i < off[g] || i >= off[g + 1]) {
      bad = true;
    } else if (i > off[g]) {
      const int32_t p[3] = {origins[3 * i - 3], origins[3 * i - 2], origins[3 * i - 1]};
      if (!canon_less(p, o)) bad = true;
    }
    if (bad) atomicOr(err, kErrNotCanonical);
  }
}

template <int OP, bool FINAL>
cudaError_t launch_one(const PassArgs& a, const WriteOut& o, int blocks, cudaStream_t s) {
  k_write<OP, FINAL><<<blocks, kWriteThreads, 0, s>>>(a, o);
  return cudaGetLastError();
}

template <int OP, bool FINAL>
int occ_one() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_write<OP, FINAL>, kWriteThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_write(int op, bool final_pass, const PassArgs& a, const WriteOut& o, int blocks, cudaStream_t s) {
  switch (op * 2 + (final_pass ? 1 : 0)) {
    case kIjk * 2 + 0: return launch_one<kIjk, false>(a, o, blocks, s);
    case kIjk * 2 + 1: return launch_one<kIjk, true>(a, o, blocks, s);
    case kLeaves * 2 + 0: return launch_one<kLeaves, false>(a, o, blocks, s);
    case kLeaves * 2 + 1: return launch_one<kLeaves, true>(a, o, blocks, s);
    case kRefine * 2 + 0: return launch_one<kRefine, false>(a, o, blocks, s);
    case kRefine * 2 + 1: return launch_one<kRefine, true>(a, o, blocks, s);
    case kCoarsen * 2 + 0: return launch_one<kCoarsen, false>(a, o, blocks, s);
    case kCoarsen * 2 + 1: return launch_one<kCoarsen, true>(a, o, blocks, s);
    case kDilate * 2 + 0: return launch_one<kDilate, false>(a, o, blocks, s);
    case kDilate * 2 + 1: return launch_one<kDilate, true>(a, o, blocks, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_write(int op, bool final_pass) {
  switch (op * 2 + (final_pass ? 1 : 0)) {
    case kIjk * 2 + 0: return occ_one<kIjk, false>();
    case kIjk * 2 + 1: return occ_one<kIjk, true>();
    case kLeaves * 2 + 0: return occ_one<kLeaves, false>();
    case kLeaves * 2 + 1: return occ_one<kLeaves, true>();
    case kRefine * 2 + 0: return occ_one<kRefine, false>();
    case kRefine * 2 + 1: return occ_one<kRefine, true>();
    case kCoarsen * 2 + 0: return occ_one<kCoarsen, false>();
    case kCoarsen * 2 + 1: return occ_one<kCoarsen, true>();
    case kDilate * 2 + 0: return occ_one<kDilate, false>();
    default: return occ_one<kDilate, true>();
  }
}

cudaError_t launch_validate(const int32_t* origins, const uint64_t* masks, const int32_t* leaf_grid,
                            const int64_t* leaf_offsets, long long L, int32_t B, unsigned int* err, int blocks,
                            cudaStream_t s) {
  k_validate<<<blocks, 256, 0, s>>>(origins, masks, leaf_grid, leaf_offsets, L, B, err);
  return cudaGetLastError();
}

}  // namespace tb
