// mx_ptx.cuh -- inline-PTX wrappers for hardware block-scaled MMA (MXFP8,
// MXFP4, NVFP4) on sm_103a: 4-D tensor copies of the scale tiles, the
// shared-to-tensor-memory copy of scale factors and the block-scaled
// tcgen05.mma forms.  One instruction per wrapper.
//
// Protocol ("TMEM -- the accumulator's new home", section "Block-scaled MMA";
// "Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling"): the
// scale factors of a block-scaled MMA are read from tensor memory while A and
// B stay in shared memory, so every ring stage's scales take one more hop:
// TMA brings them into shared memory as 32-row x 16-byte slabs (row r of a
// 128-row block at lane r mod 32, 4-byte word r / 32), and tcgen05.cp copies
// each slab into 4 tensor-memory columns of lanes 0..31, replicated into the
// other three 32-lane windows (.warpx4), where each warp of the reading
// warpgroup finds its rows.  Field layouts of the descriptors follow the
// public PTX ISA (the pages do not print them).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace dgb {

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z, int32_t w) {
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5, %6}], [%2];"
                 :: "r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// CTA-pair form: the completing barrier may be the pair leader's.
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y, int32_t z, int32_t w) {
    asm volatile("cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5, %6}], [%2];"
                 :: "r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// Shared-memory descriptor of one 32-row x 16-byte scale slab (no swizzle,
// K-major): rows 16 bytes apart inside 8-row core matrices of 128 bytes, core
// matrices 128 bytes apart along the rows (stride-dim offset); one core
// matrix wide, so the leading-dim offset is unused.
__host__ __device__ constexpr uint64_t smem_desc_scale_slab(uint32_t smem_addr) {
    return uint64_t((smem_addr >> 4) & 0x3FFFu) |
           (uint64_t(128 >> 4) << 16) |     // leading-dim offset (one core matrix; unused)
           (uint64_t(128 >> 4) << 32) |     // stride-dim offset: next 8 rows
           (uint64_t(1) << 46);             // descriptor version for tcgen05; swizzle none
}

// Copy one 32-row x 128-bit slab from shared memory into tensor-memory
// columns [col, col + 4) of lanes 0..31 and of the three other 32-lane windows.
template <int CG>
__device__ __forceinline__ void tmem_cp_scales(uint32_t taddr, uint64_t sdesc) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

// Block-scaled MMA kinds.
enum MxKind : int {
    kMxF8 = 1,    // kind::mxf8f6f4, 8-bit elements, one E8M0 scale per 32 (scale_vec::1X), K = 32
    kMxF4 = 2,    // kind::mxf4, packed E2M1, one E8M0 scale per 32 (scale_vec::2X), K = 64
    kNvF4 = 3     // kind::mxf4nvf4, packed E2M1, one E4M3 scale per 16 (scale_vec::4X), K = 64
};

// D[tmem] (+)= (A . SA)[smem] * ((B . SB)[smem])^T with the scale factors of
// A and B read from tensor memory at sa_tmem / sb_tmem.
template <int CG, int KIND>
__device__ __forceinline__ void mma_block_scaled(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sa_tmem, uint32_t sb_tmem, uint32_t accumulate) {
#define DGB_MMA_BS(CGS, KINDS, VEC)                                                                          \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"                                          \
                 "tcgen05.mma.cta_group::" CGS ".kind::" KINDS ".block_scale.scale_vec::" VEC               \
                 " [%0], %1, %2, %3, [%4], [%5], p;\n\t}"                                                    \
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sa_tmem), "r"(sb_tmem),          \
                    "r"(accumulate) : "memory")
    if constexpr (CG == 1) {
        if constexpr (KIND == kMxF8) DGB_MMA_BS("1", "mxf8f6f4", "1X");
        else if constexpr (KIND == kMxF4) DGB_MMA_BS("1", "mxf4", "2X");
        else DGB_MMA_BS("1", "mxf4nvf4", "4X");
    } else {
        if constexpr (KIND == kMxF8) DGB_MMA_BS("2", "mxf8f6f4", "1X");
        else if constexpr (KIND == kMxF4) DGB_MMA_BS("2", "mxf4", "2X");
        else DGB_MMA_BS("2", "mxf4nvf4", "4X");
    }
#undef DGB_MMA_BS
}

// Instruction descriptor of the block-scaled kinds (public PTX ISA):
//   [4,6) B scale-factor id   [7,10) A format   [10,13) B format
//   [15] A major (0 = K)      [16] B major      [17,23) N >> 3
//   [23] scale format (0 = UE4M3, 1 = UE8M0)    [24,29) M >> 4
//   [29,31) A scale-factor id [31] K size (0: K = 32 for mxf8f6f4, 64 for mxf4 / mxf4nvf4)
// Formats: mxf8f6f4 0 = E4M3, 1 = E5M2; mxf4 and mxf4nvf4 1 = E2M1.  The
// scale-factor ids pick which byte (1X), byte pair (2X) or the whole word
// (4X, id 0) of each 32-bit tensor-memory cell holds the MMA's scales.
// The major bits may be 1 (MN-major) for 8-bit elements only.
__host__ __device__ constexpr uint32_t make_idesc_block_scaled(uint32_t a_format, uint32_t b_format, uint32_t m,
                                                               uint32_t n, uint32_t scale_ue8m0, uint32_t a_mn_major = 0,
                                                               uint32_t b_mn_major = 0) {
    return (a_format << 7) | (b_format << 10) | (a_mn_major << 15) | (b_mn_major << 16) | ((n >> 3) << 17) |
           (scale_ue8m0 << 23) | ((m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_with_scale_ids(uint32_t idesc, uint32_t sf_id) {
    return idesc | (sf_id << 29) | (sf_id << 4);
}

}  // namespace dgb
