// Host-side launchers of the pass kernels (internal to libtb.so).
#pragma once

#include <cuda_runtime.h>

#include "tb_common.cuh"

namespace tb {

constexpr int kSortThreads = 256;
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortThreads * kSortItems;   // slots per digit-pass tile
constexpr int kDedupThreads = 256;
constexpr int kDedupItems = 4;
constexpr int kDedupTile = kDedupThreads * kDedupItems;
constexpr int kWriteThreads = 256;                      // 8 lanes per leaf
constexpr int kWriteRows = 4;
constexpr int kWriteTile = (kWriteThreads / 8) * kWriteRows;  // leaves per writer tile

cudaError_t launch_emit(int op, const PassArgs& a, int blocks, cudaStream_t s);
cudaError_t launch_prepass_ijk(const int32_t* ijk, long long N, const int64_t* off, int32_t B,
                               ReadbackHeader* rb, int blocks, cudaStream_t s);
cudaError_t launch_prepass_leaves(const int32_t* origins, const uint64_t* masks, long long L,
                                  const int64_t* off, int32_t B, ReadbackHeader* rb, int blocks,
                                  cudaStream_t s);
cudaError_t launch_sort_pass(const PassArgs& a, int pass, int blocks, cudaStream_t s);
cudaError_t launch_dedup(const PassArgs& a, int blocks, cudaStream_t s);
cudaError_t launch_write(int op, bool final_pass, const PassArgs& a, const WriteOut& o, int blocks,
                         cudaStream_t s);
cudaError_t launch_validate(const int32_t* origins, const uint64_t* masks, const int32_t* leaf_grid,
                            const int64_t* leaf_offsets, long long L, int32_t B, unsigned int* err,
                            int blocks, cudaStream_t s);

// Sets the calling thread's tb_last_error() message.
void set_error_message(const char* msg);

// Occupancy-derived resident block counts (per SM) of the persistent kernels.
int occupancy_sort();
int occupancy_dedup();
int occupancy_write(int op, bool final_pass);

}  // namespace tb
