// Segmented radix sort of the slots into canonical order, and the head-flag
// dedup scan (fVDB PR #757 "Batched leaf-mask topology construction for
// generated conv grids", Summary item 1, second and third bullets).
//
// The PR sorts with two stable segmented radix sorts; here the grid index is
// the most significant key field, so one global LSD sort over only the key
// bits that vary in the batch does the segmentation.  Each digit pass is a
// single "onesweep" kernel: a tile ranks its keys with warp-level multisplit
// (match.any), publishes its per-digit counts, and finds its global offsets
// by a bounded decoupled look-back over the preceding tiles.  Digit offsets
// come from the histograms the emission kernel already built.
#include "tb_common.cuh"
#include "tb_launch.h"

namespace tb {

namespace {

__global__ void __launch_bounds__(kSortThreads) k_sort_pass(const PassArgs a, int pass) {
  constexpr int NW = kSortThreads / 32;
  constexpr int WITEMS = 32 * kSortItems;
  __shared__ uint32_t s_whist[NW][kBins];
  __shared__ uint32_t s_binstart[kBins];
  __shared__ uint32_t s_glob[kBins];
  __shared__ uint64_t s_keys[kSortTile];
  __shared__ uint32_t s_vals[kSortTile];
  __shared__ uint32_t s_scan[8];
  __shared__ uint32_t s_tile;

  const int shift = 8 * pass;
  const uint64_t* __restrict__ kin = a.keys[pass & 1];
  const uint32_t* __restrict__ vin = a.vals[pass & 1];
  uint64_t* __restrict__ kout = a.keys[(pass + 1) & 1];
  uint32_t* __restrict__ vout = a.vals[(pass + 1) & 1];
  long long S = (long long)a.rb->num_slots;
  if (S > a.slot_cap) S = a.slot_cap;
  const long long ntiles = (S + kSortTile - 1) / kSortTile;
  uint32_t* status = a.sort_status + (long long)pass * a.sort_tiles_cap * kBins;
  unsigned int* ctr = &a.ctl->sort_tile_ctr[pass];
  const uint32_t* bin_base = a.ctl->bin_base[pass];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (;;) {
    if (tid == 0) s_tile = atomicAdd(ctr, 1u);
    for (int k = tid; k < NW * kBins; k += kSortThreads) (&s_whist[0][0])[k] = 0;
    __syncthreads();
    const long long tile = s_tile;
    if (tile >= ntiles) break;

    // warp-contiguous, lane-striped load; stable rank within the warp
    const long long base = tile * kSortTile + (long long)warp * WITEMS;
    uint64_t k[kSortItems];
    uint32_t v[kSortItems], d[kSortItems], r[kSortItems];
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const long long idx = base + j * 32 + lane;
      if (idx < S) {
        k[j] = kin[idx];
        v[j] = vin[idx];
        d[j] = (uint32_t)(k[j] >> shift) & 255u;
      } else {
        k[j] = 0;
        v[j] = 0;
        d[j] = kBins;  // padding: ranked nowhere
      }
    }
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const uint32_t peers = __match_any_sync(0xffffffffu, d[j]);
      const uint32_t lt = peers & ((1u << lane) - 1u);
      uint32_t cnt = 0;
      if (d[j] < kBins) cnt = s_whist[warp][d[j]];
      __syncwarp();
      if (d[j] < kBins && lt == 0) s_whist[warp][d[j]] = cnt + __popc(peers);
      __syncwarp();
      r[j] = cnt + __popc(lt);
    }
    __syncthreads();

    // thread b owns digit b: per-warp offsets, tile-local start, global base
    uint32_t tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t c = s_whist[w][tid];
      s_whist[w][tid] = tot;
      tot += c;
    }
    uint32_t all;
    const uint32_t ex = block_excl_scan_256(tot, s_scan, &all);
    s_binstart[tid] = ex;
    const uint32_t prefix = lookback32(status + tid, kBins, tile, tot, &a.rb->err);
    s_glob[tid] = bin_base[tid] + prefix - ex;
    __syncthreads();

    // local scatter into digit order, then coalesced global write
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      if (d[j] < kBins) {
        const uint32_t lp = s_binstart[d[j]] + s_whist[warp][d[j]] + r[j];
        s_keys[lp] = k[j];
        s_vals[lp] = v[j];
      }
    }
    __syncthreads();
    const long long rem = S - tile * kSortTile;
    const int nvalid = rem < kSortTile ? (int)rem : kSortTile;
    for (int i = tid; i < nvalid; i += kSortThreads) {
      const uint64_t key = s_keys[i];
      const uint32_t gp = s_glob[(uint32_t)(key >> shift) & 255u] + (uint32_t)i;
      if (gp < (uint64_t)S) {  // always true when the histograms match the slots
        kout[gp] = key;
        vout[gp] = s_vals[i];
      }
    }
    __syncthreads();
  }
}

// Suffix fill: out[g] = first leaf (node) index of the first non-empty grid
// >= g, or `total` if none; out[B] = total.  One block.
__device__ void suffix_fill(const uint32_t* first, int32_t B, unsigned long long total, int64_t* out) {
  __shared__ uint32_t s[kDedupThreads];
  const int tid = threadIdx.x;
  uint32_t carry = 0xFFFFFFFFu;
  if (B > 0) {
    for (long long base = ((long long)(B - 1) / kDedupThreads) * kDedupThreads; base >= 0;
         base -= kDedupThreads) {
      const long long g = base + tid;
      uint32_t v = 0xFFFFFFFFu;
      if (g < B) {
        const uint32_t f = __ldcg(first + g);
        if (f) v = f - 1;
      }
      s[tid] = v;
      __syncthreads();
      for (int off = 1; off < kDedupThreads; off <<= 1) {
        const uint32_t t = (tid + off < kDedupThreads) ? s[tid + off] : 0xFFFFFFFFu;
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

// Head flags on the sorted keys: a new leaf where the key changes, a new
// lower node where (grid, tile, upper offset) changes, a new upper node where
// (grid, tile) changes, a new grid where the grid field changes.  A blocked
// 1024-slot tile scans the three head counts and gets its global base by a
// bounded look-back.  Outputs: run_start[u] (first slot of unique leaf u),
// the global lower/upper index of each leaf, and each grid's first indices;
// the last block derives per-grid offsets and totals.
__global__ void __launch_bounds__(kDedupThreads) k_dedup(const PassArgs a) {
  __shared__ unsigned long long s_scan[8];
  __shared__ unsigned long long s_base[3];
  __shared__ uint32_t s_tile;
  const uint64_t* __restrict__ keys = a.keys[a.sorted];
  long long S = (long long)a.rb->num_slots;
  if (S > a.slot_cap) S = a.slot_cap;
  const long long ntiles = (S + kDedupTile - 1) / kDedupTile;
  const int lb = a.K.lower_bits, nb = a.K.node_bits, gsh = a.K.gw ? a.K.gshift : 64;
  const int tid = threadIdx.x;
  const int32_t B = a.B;
  constexpr unsigned long long M21 = (1ull << 21) - 1;

  for (;;) {
    if (tid == 0) s_tile = atomicAdd(&a.ctl->dedup_tile_ctr, 1u);
    __syncthreads();
    const long long tile = s_tile;
    if (tile >= ntiles) break;
    const long long i0 = tile * kDedupTile + (long long)tid * kDedupItems;
    uint64_t prev = (i0 > 0 && i0 - 1 < S) ? keys[i0 - 1] : 0ull;
    uint64_t kk[kDedupItems];
    uint32_t fl[kDedupItems];
    unsigned long long c = 0;
#pragma unroll
    for (int j = 0; j < kDedupItems; ++j) {
      const long long i = i0 + j;
      fl[j] = 0;
      kk[j] = 0;
      if (i < S) {
        const uint64_t key = keys[i];
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
    const unsigned long long ex = block_excl_scan_256(c, s_scan, &tot);
    if (tid < 3) {
      const unsigned long long field = (tot >> (21 * tid)) & M21;
      s_base[tid] = lookback64(a.dedup_status + tid, 3, tile, field, false, &a.rb->err);
      if (field) atomicAdd(&a.ctl->head_totals[tid], field);
    }
    __syncthreads();
    unsigned long long cl = s_base[0] + (ex & M21);
    unsigned long long clo = s_base[1] + ((ex >> 21) & M21);
    unsigned long long cup = s_base[2] + ((ex >> 42) & M21);
#pragma unroll
    for (int j = 0; j < kDedupItems; ++j) {
      if (!(fl[j] & 1u)) continue;
      const long long i = i0 + j;
      if (fl[j] & 2u) ++clo;
      if (fl[j] & 4u) ++cup;
      const unsigned long long u = cl++;
      a.run_start[u] = (uint32_t)i;
      a.leaf_lower[u] = (uint32_t)(clo - 1);
      a.leaf_upper[u] = (uint32_t)(cup - 1);
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

  if (!last_block_done(&a.ctl->dedup_ticket)) return;
  const unsigned long long U = __ldcg(&a.ctl->head_totals[0]);
  const unsigned long long NL = __ldcg(&a.ctl->head_totals[1]);
  const unsigned long long NU = __ldcg(&a.ctl->head_totals[2]);
  if (tid == 0) {
    a.rb->num_leaves = U;
    a.rb->num_lowers = NL;
    a.rb->num_uppers = NU;
    a.run_start[U] = (uint32_t)S;
  }
  suffix_fill(a.first, B, U, a.leaf_off);
  suffix_fill(a.first + B, B, NL, a.lower_off);
  suffix_fill(a.first + 2 * B, B, NU, a.upper_off);
}

}  // namespace

cudaError_t launch_sort_pass(const PassArgs& a, int pass, int blocks, cudaStream_t s) {
  k_sort_pass<<<blocks, kSortThreads, 0, s>>>(a, pass);
  return cudaGetLastError();
}

cudaError_t launch_dedup(const PassArgs& a, int blocks, cudaStream_t s) {
  k_dedup<<<blocks, kDedupThreads, 0, s>>>(a);
  return cudaGetLastError();
}

int occupancy_sort() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_sort_pass, kSortThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

int occupancy_dedup() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_dedup, kDedupThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

}  // namespace tb
