// Host-side launchers of the pass kernels (internal to libtb.so).
#pragma once

#include <cuda_runtime.h>

#include "tb_common.cuh"

namespace tb {

constexpr int kSortItems = 8;
constexpr int kSortTile = 256 * kSortItems;   // slots per digit-pass tile
constexpr int kDedupItems = 4;
constexpr int kDedupTile = 256 * kDedupItems;  // slots per dedup tile
constexpr int kWriteLeavesPerBlock = 32;       // 8 lanes per leaf, 256 threads

// Bytes of a pass's readback block for B grids:
// header | leaf_off[B+1] | lower_off[B+1] | upper_off[B+1] | voxels[B] | gbox[6B]
inline size_t readback_bytes(int32_t B) {
  return sizeof(ReadbackHeader) + 3 * sizeof(int64_t) * (size_t)(B + 1) + sizeof(int64_t) * (size_t)B +
         6 * sizeof(unsigned int) * (size_t)B;
}

// Voxel bbox and checks of a raw leaf list (the allocation-free refinement).
cudaError_t launch_prepass_leaves(const int32_t* origins, const uint64_t* masks, long long L,
                                  const int64_t* off, int32_t B, ReadbackHeader* rb, int blocks,
                                  cudaStream_t s);

// Kernel map between two batches (tb_kmap.cu).  Box offsets d enumerate
// [lo, hi] x-major; stride 1 or 2, forward or transposed.
constexpr int kKmapMaxCand = 128;  // candidate input leaves of one output leaf
struct KmapArgs {
  const int32_t* in_origins;
  const uint64_t* in_masks;
  const uint64_t* in_wp;
  const int64_t* in_voff;
  const int32_t* in_grid;    // [L_in] grid of each input leaf
  const int32_t* table;      // hash table of the input leaves (leaf index or -1)
  unsigned long long table_mask;  // table size - 1 (a power of two minus one)
  const int64_t* in_vbase;   // [B+1] first voxel index of each input grid
  const int32_t* out_origins;
  const uint64_t* out_masks;
  const int64_t* out_voff;
  const uint64_t* out_wp;    // [L_out] output word prefixes
  const int32_t* out_grid;
  const int64_t* out_vbase;  // [B+1] first voxel index of each output grid
  long long L_out;
  int32_t lo[3], hi[3];
  int32_t stride, transposed;
  int32_t* map;              // [V_out, K]
  int32_t* cands;            // staged map: [L_out, cand_max] candidate input leaves (-1: none), or NULL
  int32_t cand_max;          // span^3 of the staged map
  int32_t span;              // input leaves a leaf's reach spans per axis, at most (1..3 in the staged map)
  unsigned int* next_chunk;  // staged map: the next chunk of output leaves (zeroed by the set-up)
};
// Set-up of a kernel map: both batches' per-grid voxel bases from their
// device voxel counts, the staged map's chunk counter, the input leaf table.
struct KmapPrep {
  const int64_t* in_counts;
  const int64_t* out_counts;  // [B] voxels per grid
  int32_t B;
  int64_t* in_vbase;
  int64_t* out_vbase;         // [B+1] written
  const int32_t* origins;
  const int32_t* leaf_grid;   // the input's leaves
  long long L;
  int32_t* table;             // all -1 on entry
  unsigned long long mask;
  unsigned int* next_chunk;   // zeroed (or NULL)
};
cudaError_t launch_kmap_prep(const KmapPrep& p, int blocks, cudaStream_t s);
cudaError_t launch_kmap(const KmapArgs& k, int blocks, cudaStream_t s);
// The staged map: boxes whose reach from an output leaf spans at most 3 input
// leaves per axis, with at most kKmapStagedColumns columns (a batch of output
// leaves per warp for spans of up to 2 and at most kKmapBatchColumns
// columns, else one leaf per warp).
constexpr int kKmapStagedColumns = 1024;
constexpr int kKmapBatchColumns = 32;
cudaError_t launch_kmap_cands(const KmapArgs& k, int blocks, cudaStream_t s);
// The tabulated map: stride 1 or transposed, the reach of an output leaf at
// most kKmapHaloMax voxels (E0 x E1 x E2) and at most 3 input leaves per
// axis, at most kKmapTabColumns columns.
constexpr int kKmapTabColumns = 1024;
constexpr int kKmapHaloMax = 1024;
cudaError_t launch_kmap_halo(const KmapArgs& k, int blocks, cudaStream_t s);
cudaError_t launch_kmap_staged(const KmapArgs& k, int sms, cudaStream_t s);

// Masked refinement: keeps the voxels of each leaf whose flag (one byte per
// voxel, in the batch's voxel order) is non-zero.
cudaError_t launch_prune(const uint64_t* masks, const int32_t* leaf_grid, const int64_t* voxel_offset,
                         const int64_t* vbase, const uint8_t* flags, long long L, uint64_t* out, int blocks,
                         cudaStream_t s);
// Copies of several arrays in one launch (tb_batch_export_many): task t
// copies `bytes` from src to dst; both device-accessible (device memory, or
// pinned host memory seen through unified addressing).
constexpr int kMaxCopyTasks = 64;
struct CopyTask {
  const void* src;
  void* dst;
  unsigned long long bytes;
};
struct CopyTasks {
  CopyTask t[kMaxCopyTasks];
  int32_t n;
};
cudaError_t launch_copies(const CopyTasks& c, cudaStream_t s);

// Per-grid voxel bases [B+1] (exclusive prefix, then the total) of a
// batch's device voxel counts [B], one block.
cudaError_t launch_voxel_bases(const int64_t* counts, int32_t B, int64_t* vbase, cudaStream_t s);

// Self-test of the bounded device waits (tb_selftest_wait).
cudaError_t launch_wait_selftest(const uint32_t* flag, uint32_t limit, unsigned int* err, cudaStream_t s);
cudaError_t launch_validate(const int32_t* origins, const uint64_t* masks, const int32_t* leaf_grid,
                            const int64_t* leaf_offsets, long long L, int32_t B, unsigned int* err,
                            int blocks, cudaStream_t s);

// The cooperative pass kernel (all blocks co-resident) and the final writer.
size_t chain_smem_bytes();
int chain_occupancy();
cudaError_t launch_chain(const ChainArgs& c, int blocks, cudaStream_t s);
// The member launch: one cluster of `cl` CTAs (1, 2, 4 or 8) per grid of
// every chain (`members` = chains x grids), nothing co-resident required.
int member_occupancy();
int member_clusters(int cl);
cudaError_t launch_member(const ChainArgs& c, int members, int cl, cudaStream_t s);
int write_final_occupancy(int op);
cudaError_t launch_write_final(int op, const PassArgs& a, const WriteOut& o, int blocks, cudaStream_t s);
int write_multi_occupancy();
cudaError_t launch_write_multi(const WriteTasks& tasks, int blocks, cudaStream_t s);

// Sets the calling thread's tb_last_error() message.
void set_error_message(const char* msg);

// True for device or managed memory (cudaPointerGetAttributes); false for
// NULL, pageable or pinned host memory.
bool device_accessible(const void* p);

}  // namespace tb
