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

// Hardware block-scaled kernel (MXFP8, MXFP4, NVFP4): the persistent
// schedule and operand maps of `base` (tile_k counts bytes of K per stage, the
// operand maps are byte matrices), plus the scale tiles' maps.
struct MxParams {
    PersistentParams base;
    CUtensorMap tmap_sfa;         // A's scale tiles: (128 words, ceil(KB/4), ceil(M/128), batch), box (128, chunks, 1, 1)
    CUtensorMap tmap_sfb;         // B's scale tiles, same shape over N
    const float* tensor_scales;   // NVFP4: {tA, tB} (device); nullptr for MX
    int32_t chunks;               // 512-byte scale slabs per 128 rows per ring stage: 1 (MXFP8), 2 (MXFP4), 4 (NVFP4)
    uint32_t sf_stage_bytes;      // shared memory per stage for scales: A's slabs and B's two row blocks
    uint32_t sf_ring_offset;      // bytes from the operand ring to the scale ring
};

// kind: 1 = mxf8f6f4, 2 = mxf4, 3 = mxf4nvf4.  grid = CTAs (a multiple of
// cta_group), block = 384 threads (producers of A, B and scales, MMA warp,
// eight epilogue warps).
cudaError_t launch_mx(const MxParams& q, int kind, int cta_group, int dtype_d, int grid, size_t smem_bytes,
                      cudaStream_t stream);
int mx_max_active_clusters(int kind, int cta_group, int dtype_d, size_t smem_bytes);

// Zero fill of D (K == 0).
cudaError_t launch_zero_fill(void* D, int dtype_d, int64_t M, int64_t N, int64_t batch, int64_t ldd,
                             int64_t stride_d, int sm_count, cudaStream_t stream);

}  // namespace dgb
