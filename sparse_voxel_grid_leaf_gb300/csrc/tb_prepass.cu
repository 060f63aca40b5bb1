// Auxiliary kernels: the leaf-range prepass of the allocation-free refinement
// (its input's voxel bounding box sizes the sort key; fVDB PR #757 "Batched
// leaf-mask topology construction for generated conv grids"), masked
// refinement's pruning, batched exports, the bounded-wait self-test, and the
// canonical-batch validator (tb_validate: canonical order per grid, non-zero
// masks, aligned origins).
#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

// ---------------------------------------------------------------- front-end prepasses

// Exact voxel bbox of a leaf list (from the set bits), plus origin alignment.
__global__ void __launch_bounds__(256) k_prepass_leaves(const int32_t* origins, const uint64_t* masks,
                                                        long long L, const int64_t* off, int32_t B,
                                                        ReadbackHeader* rb) {
  int32_t mn[3], mx[3];
  leaves_bounds(origins, masks, L, mn, mx, &rb->err, (int)blockIdx.x, (int)gridDim.x);
  reduce_bbox(mn, mx, rb->bbox_enc);
  check_offsets(off, B, L, &rb->err);
}

// Masked refinement's pruning step (fVDB PR #757, Summary item 1: masked
// subdivision prunes upstream, then refines): each leaf keeps the voxels whose
// flag is set.  Voxel v of grid g sits at flag index vbase[g] + voxel_offset
// of its leaf + its rank among the leaf's set bits (ascending bit index).
// One 8-lane group per leaf, lane w on mask word w.
__global__ void __launch_bounds__(256) k_prune(const uint64_t* masks, const int32_t* leaf_grid,
                                               const int64_t* voxel_offset, const int64_t* vbase,
                                               const uint8_t* flags, long long L, uint64_t* out) {
  const int lane = threadIdx.x & 31, w = lane & 7;
  const long long groups = (long long)gridDim.x * (blockDim.x / 8);
  // ub is uniform within the warp, so the group shuffles see all 32 lanes
  for (long long ub = (long long)blockIdx.x * (blockDim.x / 8) + (threadIdx.x >> 5) * 4; ub < L; ub += groups) {
    const long long u = ub + (lane >> 3);
    const bool valid = u < L;
    const uint64_t word = valid ? __ldg(masks + 8 * u + w) : 0ull;
    const uint32_t pop = __popcll(word);
    uint32_t incl = pop;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off, 8);
      if (w >= off) incl += y;
    }
    if (!valid) continue;
    const long long first = vbase[leaf_grid[u]] + voxel_offset[u] + (incl - pop);
    uint64_t kept = 0, rest = word;
    for (uint32_t j = 0; rest; ++j) {
      const uint64_t bit = rest & (~rest + 1);
      if (__ldg(flags + first + j)) kept |= bit;
      rest ^= bit;
    }
    out[8 * u + w] = kept;
  }
}

// Several copies in one launch: blockIdx.y picks the task; 16-byte vectors
// where both ends are 16-byte aligned, bytes otherwise.
__global__ void __launch_bounds__(256) k_copies(const CopyTasks c) {
  const CopyTask& t = c.t[blockIdx.y];
  const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  const bool vec = (((uintptr_t)t.src | (uintptr_t)t.dst) & 15u) == 0;
  unsigned long long done = 0;
  if (vec) {
    const unsigned long long nv = t.bytes / 16;
    const int4* s4 = (const int4*)t.src;
    int4* d4 = (int4*)t.dst;
    for (unsigned long long i = tid; i < nv; i += stride) d4[i] = __ldg(s4 + i);
    done = nv * 16;
  }
  const unsigned char* s1 = (const unsigned char*)t.src;
  unsigned char* d1 = (unsigned char*)t.dst;
  for (unsigned long long i = done + tid; i < t.bytes; i += stride) d1[i] = s1[i];
}

// Per-grid voxel bases: vbase[0] = 0, vbase[g + 1] = vbase[g] + counts[g],
// one block scanning 256 grids at a time.
__global__ void __launch_bounds__(256) k_voxel_bases(const int64_t* counts, int32_t B, int64_t* vbase) {
  __shared__ long long part[8];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  if (threadIdx.x == 0) vbase[0] = 0;
  long long carry = 0;
  for (int base = 0; base < B; base += 256) {
    const int i = base + threadIdx.x;
    long long v = i < B ? counts[i] : 0;
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
    if (i < B) vbase[i + 1] = carry + before + v;
    carry += total;
    __syncthreads();
  }
}

// Self-test of the bounded waits: one thread waits for *flag to reach 1 with
// the same bounded spin as the grid barrier, `limit` polls at most.
__global__ void k_wait_selftest(const uint32_t* flag, uint32_t limit, unsigned int* err) {
  if (threadIdx.x == 0 && blockIdx.x == 0) wait_reach(flag, 1u, limit, err);
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

}  // namespace

cudaError_t launch_prepass_leaves(const int32_t* origins, const uint64_t* masks, long long L, const int64_t* off,
                                  int32_t B, ReadbackHeader* rb, int blocks, cudaStream_t s) {
  k_prepass_leaves<<<blocks, 256, 0, s>>>(origins, masks, L, off, B, rb);
  return cudaGetLastError();
}

cudaError_t launch_prune(const uint64_t* masks, const int32_t* leaf_grid, const int64_t* voxel_offset,
                         const int64_t* vbase, const uint8_t* flags, long long L, uint64_t* out, int blocks,
                         cudaStream_t s) {
  k_prune<<<blocks, 256, 0, s>>>(masks, leaf_grid, voxel_offset, vbase, flags, L, out);
  return cudaGetLastError();
}

cudaError_t launch_copies(const CopyTasks& c, cudaStream_t s) {
  if (c.n <= 0) return cudaSuccess;
  unsigned long long most = 0;
  for (int i = 0; i < c.n; ++i) most = c.t[i].bytes > most ? c.t[i].bytes : most;
  unsigned long long bx = (most / 16 + 255) / 256;
  bx = bx < 1 ? 1 : (bx > 64 ? 64 : bx);
  k_copies<<<dim3((unsigned)bx, (unsigned)c.n), 256, 0, s>>>(c);
  return cudaGetLastError();
}

cudaError_t launch_voxel_bases(const int64_t* counts, int32_t B, int64_t* vbase, cudaStream_t s) {
  k_voxel_bases<<<1, 256, 0, s>>>(counts, B, vbase);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const uint32_t* flag, uint32_t limit, unsigned int* err, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(flag, limit, err);
  return cudaGetLastError();
}

cudaError_t launch_validate(const int32_t* origins, const uint64_t* masks, const int32_t* leaf_grid,
                            const int64_t* leaf_offsets, long long L, int32_t B, unsigned int* err, int blocks,
                            cudaStream_t s) {
  k_validate<<<blocks, 256, 0, s>>>(origins, masks, leaf_grid, leaf_offsets, L, B, err);
  return cudaGetLastError();
}

}  // namespace tb
