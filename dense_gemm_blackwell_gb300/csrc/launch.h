// launch.h -- host entry points of the kernel translation units (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace dgb {

// Single-CTA kernel: grid = batch, block = 128 threads.
cudaError_t launch_single_cta(const SingleParams& p, int dtype_d, int batch, size_t smem_bytes,
                              cudaStream_t stream);

// Persistent kernel: grid = CTAs (a multiple of cta_group), block = 352 threads (kThreads: two producer
// warps, the MMA warp and eight epilogue warps).
cudaError_t launch_persistent(const PersistentParams& p, int cta_group, int dtype_d, int grid,
                              size_t smem_bytes, cudaStream_t stream);

// How many clusters of `cta_group` CTAs with `smem_bytes` of dynamic shared
// memory can be resident at once (0 if the query fails).
int persistent_max_active_clusters(int cta_group, int dtype_d, size_t smem_bytes);

// Block-scaled e4m3 kernel: grid = CTAs (a multiple of cta_group), block = 384 threads (kFp8Threads:
// producers, MMA warp and an idle warp, then eight promotion/epilogue warps).
cudaError_t launch_fp8_block(const PersistentParams& p, int cta_group, int dtype_d, int grid, size_t smem_bytes,
                             cudaStream_t stream);
int fp8_max_active_clusters(int cta_group, int tile_n, int dtype_d, size_t smem_bytes);

// Zero fill of D (K == 0).
cudaError_t launch_zero_fill(void* D, int dtype_d, int64_t M, int64_t N, int64_t batch, int64_t ldd,
                             int64_t stride_d, int sm_count, cudaStream_t stream);

}  // namespace dgb
