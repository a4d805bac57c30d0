// gemm_api.cu -- the C ABI declared in include/gemm.h: planner, TMA tensor-map
// builder, launches and status reporting.  Host code only.
//
// Planner gates (cuBLASDx "API Card: Blackwell Pipeline (tcgen05)", section
// "Descriptor" and "Depth and shared memory"):
//   * 16-bit inputs (f16 x f16 or bf16 x bf16) with f32 accumulation; 8-bit
//     e4m3 x e4m3 only with block scales;
//   * one MMA tile is 128 rows per SM (256 for an SM pair) by tile_n columns,
//     tile_n a multiple of 16 up to 256, and its fp32 accumulator (tile_n
//     32-bit columns, two buffers) must fit the 512 tensor-memory columns;
//   * 16-byte alignment of A, B and D;
//   * ring depth = the largest that fits the opt-in shared-memory limit, where
//     one stage holds one A and one B tile, (M*K + N*K) * sizeof(input), and
//     each barrier costs 8 bytes (two per stage, two per TMEM stage) plus a
//     4-byte tensor-memory handle.
// Unsupported requests fail with GEMM_ERR_UNSUPPORTED instead of running
// another path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm.h"
#include "common.cuh"
#include "launch.h"
#include "mx_ptx.cuh"
#include "units.cuh"

namespace {

using dgb::PersistentParams;
using dgb::SingleParams;

constexpr int kVersion = 10000;  // 1.0.0
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kPersistentThreads = 352;   // two producer warps, MMA warp and 8 epilogue warps
constexpr int kSkFlagsPerCta = 8;         // stream-K: one published flag per epilogue warp
// stream-K launch counter: two words in the plan's 256-byte status area, past
// the error record (which gemm_sync_status clears) and zeroed with it at creation
constexpr size_t kSkEpochOffset = 128;
static_assert(sizeof(gemm_device_error_t) <= kSkEpochOffset, "error record overlaps the launch counter");
constexpr int64_t kStagingBytes = 8 * 32 * 128;   // 8 epilogue warps x one 4 KB buffer
constexpr int64_t kAlignSlack = 1024;                  // dynamic smem is re-aligned to 1024 B
constexpr int kDefaultRasterGroup = 8;                 // m blocks per raster group (least DRAM traffic on GB300)
// 512-wide tiles with at least 32 m blocks: groups of 16 read less from DRAM
// (8192^3: 0.70 vs 0.78 GB per launch) and, under the power cap, run about 0.3 % faster
constexpr int kWideRasterGroup = 16;

thread_local int g_last_cuda_error = 0;

gemm_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return GEMM_ERR_CUDA;
}

int elem_bytes(int dt) {
    switch (dt) {
    case GEMM_F16: case GEMM_BF16: return 2;
    case GEMM_E4M3: case GEMM_E5M2: return 1;
    case GEMM_F32: case GEMM_TF32: return 4;
    default: return 0;
    }
}

bool is8(int dt) { return dt == GEMM_E4M3 || dt == GEMM_E5M2; }
bool is4(int dt) { return dt == GEMM_E2M1; }
// Scale modes whose scales the tensor core applies (tiled scale bytes, gemm_run_mx).
bool hw_scaled(int mode) { return mode == GEMM_SCALE_MX_E8M0_32 || mode == GEMM_SCALE_NV_E4M3_16; }
bool known_dtype(int dt) { return elem_bytes(dt) != 0 || is4(dt); }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

int pow2_at_least(int64_t x) {
    int v = 32;
    while (v < x) v <<= 1;
    return v;
}

// Descriptor with every optional field resolved to its documented default.
struct Resolved {
    gemm_desc_t d;
};

gemm_status_t resolve(const gemm_desc_t* in, Resolved* out) {
    if (!in || !out) return GEMM_ERR_INVALID_ARG;
    gemm_desc_t d = *in;
    if (d.M < 0 || d.N < 0 || d.K < 0 || d.batch < 0) return GEMM_ERR_INVALID_ARG;
    if (!known_dtype(d.dtype_a) || !known_dtype(d.dtype_b) || elem_bytes(d.dtype_d) == 0)
        return GEMM_ERR_INVALID_ARG;
    if ((d.major_a != GEMM_K_MAJOR && d.major_a != GEMM_MN_MAJOR) ||
        (d.major_b != GEMM_K_MAJOR && d.major_b != GEMM_MN_MAJOR))
        return GEMM_ERR_INVALID_ARG;
    if (d.scale_mode != GEMM_SCALE_NONE && d.scale_mode != GEMM_SCALE_BLOCK_1x128_128x128 &&
        !hw_scaled(d.scale_mode))
        return GEMM_ERR_INVALID_ARG;
    // tiled scales have a fixed layout: no leading dims
    if (hw_scaled(d.scale_mode) && (d.ld_sa != 0 || d.ld_sb != 0)) return GEMM_ERR_INVALID_ARG;
    if (d.M > INT32_MAX || d.N > INT32_MAX || d.K > INT32_MAX || d.batch > INT32_MAX)
        return GEMM_ERR_UNSUPPORTED;
    const bool ka = d.major_a == GEMM_K_MAJOR, kb = d.major_b == GEMM_K_MAJOR;
    const int64_t min_lda = ka ? d.K : d.M, min_ldb = kb ? d.K : d.N;
    if (d.lda == 0) d.lda = std::max<int64_t>(min_lda, 1);
    if (d.ldb == 0) d.ldb = std::max<int64_t>(min_ldb, 1);
    if (d.ldd == 0) d.ldd = std::max<int64_t>(d.N, 1);
    if (d.lda < min_lda || d.ldb < min_ldb || d.ldd < d.N) return GEMM_ERR_INVALID_ARG;
    const int64_t rows_a = ka ? d.M : d.K, rows_b = kb ? d.N : d.K;
    if (d.stride_a == 0) d.stride_a = rows_a * d.lda;
    if (d.stride_b == 0) d.stride_b = rows_b * d.ldb;
    if (d.stride_d == 0) d.stride_d = d.M * d.ldd;
    if (d.stride_a < 0 || d.stride_b < 0 || d.stride_d < 0) return GEMM_ERR_INVALID_ARG;
    if (d.batch > 1 && d.stride_d < d.M * d.ldd) return GEMM_ERR_INVALID_ARG;  // outputs would overlap
    if (hw_scaled(d.scale_mode)) {
        // bytes of one batch entry's scale tiles: 512 per 128 rows x 4 scale columns
        const int64_t v = d.scale_mode == GEMM_SCALE_MX_E8M0_32 ? 32 : 16;
        const int64_t kq = std::max<int64_t>(ceil_div(ceil_div(d.K, v), 4), 1);
        if (d.stride_sa == 0) d.stride_sa = std::max<int64_t>(ceil_div(d.M, 128), 1) * kq * 512;
        if (d.stride_sb == 0) d.stride_sb = std::max<int64_t>(ceil_div(d.N, 128), 1) * kq * 512;
    } else {
        const int64_t kblk = std::max<int64_t>(ceil_div(d.K, 128), 1);
        if (d.ld_sa == 0) d.ld_sa = kblk;
        if (d.ld_sb == 0) d.ld_sb = kblk;
        if (d.stride_sa == 0) d.stride_sa = d.M * d.ld_sa;
        if (d.stride_sb == 0) d.stride_sb = ceil_div(d.N, 128) * d.ld_sb;
    }
    if (d.wait_timeout_ns == 0) d.wait_timeout_ns = kDefaultTimeoutNs;
    if (d.tile_n < 0 || d.stages < 0 || d.max_ctas < 0) return GEMM_ERR_INVALID_ARG;
    if ((d.flags & GEMM_FLAG_CTA_GROUP_1) && (d.flags & GEMM_FLAG_CTA_GROUP_2)) return GEMM_ERR_INVALID_ARG;
    if ((d.flags & GEMM_FLAG_SINGLE_CTA) && (d.flags & GEMM_FLAG_NO_SINGLE_CTA)) return GEMM_ERR_INVALID_ARG;
    if ((d.flags & GEMM_FLAG_EPILOGUE_DIRECT) && (d.flags & GEMM_FLAG_EPILOGUE_TMA)) return GEMM_ERR_INVALID_ARG;
    if (d.raster_group < 0 || d.reserved0 != 0) return GEMM_ERR_INVALID_ARG;
    out->d = d;
    return GEMM_OK;
}

bool is16(int dt) { return dt == GEMM_F16 || dt == GEMM_BF16; }

gemm_status_t plan_single(const gemm_desc_t& d, const gemm_device_props_t& props, gemm_plan_info_t* info) {
    const int64_t n_pad = std::max<int64_t>(round_up(d.N, 16), 16);
    const int64_t k_pad = std::max<int64_t>(round_up(d.K, 64), 64);
    const int64_t smem = 128 * k_pad * 2 + n_pad * k_pad * 2 + 16 + kAlignSlack;
    if (smem > props.smem_optin_bytes) return GEMM_ERR_RESOURCES;
    info->kernel = GEMM_KERNEL_SINGLE_CTA;
    info->cta_group = 1;
    info->tile_m = 128;
    info->tile_n = (int32_t)n_pad;
    info->tile_k = (int32_t)k_pad;
    info->stages = 1;
    info->tmem_stages = 1;
    info->tmem_cols = pow2_at_least(n_pad);
    info->grid = (int32_t)d.batch;
    info->block_threads = 128;
    info->num_tiles = d.batch;
    info->stage_bytes = 128 * k_pad * 2 + n_pad * k_pad * 2;
    info->pipeline_bytes = info->stage_bytes + 8 + 4;
    info->smem_bytes = smem;
    return GEMM_OK;
}

bool single_fits(const gemm_desc_t& d) {
    return d.M <= 128 && d.N <= 256 && d.K <= 256 && is16(d.dtype_a) && d.scale_mode == GEMM_SCALE_NONE;
}

// Block-scaled e4m3: 256-column tiles (two 128-column halves, each one 128-row
// block of B's scales), 128-deep K stages, two TMEM partial buffers of 256
// columns, 8 promotion/epilogue warps with one 4 KB staging buffer each.
constexpr int kFp8Threads = 384;
constexpr int kFp8DefaultTileN = 256;           // planner default for block-scaled problems
constexpr int64_t kFp8StagingBytes = 8 * 32 * 128;

constexpr int64_t kPairMinKAtoms = 96;   // 128-byte K atoms (K >= 6144 for 16-bit inputs)

int choose_cta_group(const gemm_desc_t& d, const gemm_device_props_t& props, int64_t tile_n) {
    if (d.flags & GEMM_FLAG_CTA_GROUP_1) return 1;
    if (d.flags & GEMM_FLAG_CTA_GROUP_2) return 2;
    // An SM pair halves each SM's B traffic from L2, which pays on long K
    // (measured on GB300: +10 % at 4096^3 and 8192^3).  With short K
    // (batched 256^3) the loads are HBM-bound and single-SM tiles win.  With
    // fewer pair tiles than pairs both forms occupy the same SMs; there pairs
    // won from K = 6144 on (bf16: +3 to +16 %), were even at 4096 and lost
    // at 2048 (-6 %).
    const int64_t pair_tiles = ceil_div(d.M, 256) * ceil_div(d.N, tile_n) * d.batch;
    const int64_t k_atoms = ceil_div(d.K, 128 / elem_bytes(d.dtype_a));
    return (d.M > 128 && d.K >= 1024 && (pair_tiles >= props.sm_count / 2 || k_atoms >= kPairMinKAtoms)) ? 2 : 1;
}

gemm_status_t plan_fp8(const gemm_desc_t& d, const gemm_device_props_t& props, gemm_plan_info_t* info) {
    // Tiles 256 or 128 columns wide (each promotion warp owns half of them, one
    // 128-column block of B's scales at most); 512 / tile_n TMEM partials.
    if (d.tile_n != 0 && d.tile_n != 256 && d.tile_n != 128) return GEMM_ERR_UNSUPPORTED;
    int cg;
    int64_t tile_n;
    if (d.flags & GEMM_FLAG_CTA_GROUP_1) {
        cg = 1;
        tile_n = d.tile_n ? d.tile_n : 256;
    } else if (d.flags & GEMM_FLAG_CTA_GROUP_2) {
        cg = 2;
        tile_n = d.tile_n ? d.tile_n : kFp8DefaultTileN;
    } else {
        // SM pairs whenever they have tiles enough for half the SMs (8192^3 on
        // GB300: 0.386 ms with pairs, 0.404 ms with single-SM tiles)
        tile_n = d.tile_n ? d.tile_n : kFp8DefaultTileN;
        cg = 2;
        if (!(d.M > 128 && ceil_div(d.M, 256) * ceil_div(d.N, tile_n) * d.batch >= props.sm_count / 2)) cg = 1;
    }
    // MN-major B: boxes of 128 contiguous N elements, a whole number per CTA
    if (d.major_b == GEMM_MN_MAJOR && (tile_n / cg) % 128 != 0) return GEMM_ERR_UNSUPPORTED;
    const int tile_k = 128;
    const int partials = (int)(512 / tile_n);
    const int64_t stage_bytes = 128 * tile_k + (tile_n / cg) * tile_k;
    auto smem_for = [&](int64_t s) {
        return s * stage_bytes + kFp8StagingBytes + 8 * (2 * s + 1) + 8 + kAlignSlack;
    };
    int64_t stages = d.stages;
    if (stages == 0) {
        stages = 16;
        while (stages > 2 && smem_for(stages) > props.smem_optin_bytes) --stages;
    }
    // the promotion warps track a block's MMAs through its stage's empty barrier
    // and release partials onto full barriers PB blocks ahead: both stay within
    // one phase of their users only if stages >= partials
    if (stages < 2 || stages > 16 || stages < partials) return GEMM_ERR_UNSUPPORTED;
    if (smem_for(stages) > props.smem_optin_bytes) return GEMM_ERR_RESOURCES;
    const int64_t tiles = ceil_div(d.M, 128 * cg) * ceil_div(d.N, tile_n) * d.batch;
    if (tiles > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    int64_t clusters = props.sm_count / cg;
    if (d.max_ctas > 0) clusters = std::min<int64_t>(clusters, std::max<int64_t>(d.max_ctas / cg, 1));
    clusters = std::min<int64_t>(clusters, tiles);
    // the promotion warps count a CTA's K blocks over all its tiles in an int
    if (ceil_div(tiles, clusters) * ceil_div(d.K, tile_k) > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    info->kernel = GEMM_KERNEL_FP8_BLOCK;
    info->cta_group = cg;
    info->tile_m = 128 * cg;
    info->tile_n = (int32_t)tile_n;
    info->tile_k = tile_k;
    info->stages = (int32_t)stages;
    info->tmem_stages = partials;
    info->tmem_cols = 512;
    info->grid = (int32_t)(clusters * cg);
    info->block_threads = kFp8Threads;
    info->num_tiles = tiles;
    info->stage_bytes = stage_bytes;
    info->pipeline_bytes = stages * stage_bytes + 8 * (2 * stages) + 4;
    info->smem_bytes = smem_for(stages);
    return GEMM_OK;
}

// Hardware block-scaled kernel (MXFP8, MXFP4, NVFP4): 256-column tiles, one
// 128-byte K atom per ring stage (128 8-bit or 256 4-bit elements), scale
// slabs per stage (A's 128 rows, B's two 128-row blocks), one 256-column
// accumulator plus a scale slot per stage in tensor memory, 8 epilogue warps
// with one 4 KB staging buffer each.
constexpr int kMxThreads = 384;
constexpr int kMxTileN = 256;
constexpr int kMxSfColumns = 256;                  // tensor-memory columns left for the scale slots

// 1 = mxf8f6f4, 2 = mxf4, 3 = mxf4nvf4 (the kernel's KIND)
int mx_kind(const gemm_desc_t& d) {
    if (d.scale_mode == GEMM_SCALE_NV_E4M3_16) return 3;
    return is4(d.dtype_a) ? 2 : 1;
}

// 512-byte scale slabs per 128 rows per ring stage: MXFP8 4 scales of 32
// (128 elements), MXFP4 8 of 32 (256 elements), NVFP4 16 of 16.
int mx_chunks(const gemm_desc_t& d) {
    const int kind = mx_kind(d);
    return kind == 1 ? 1 : (kind == 2 ? 2 : 4);
}

gemm_status_t plan_mx(const gemm_desc_t& d, const gemm_device_props_t& props, gemm_plan_info_t* info) {
    // MN-major operands: 8-bit elements only (packed E2M1 is K-major), loaded as
    // boxes of 128 contiguous M/N elements x 128 k-rows
    if ((d.major_a != GEMM_K_MAJOR || d.major_b != GEMM_K_MAJOR) && !is8(d.dtype_a)) return GEMM_ERR_UNSUPPORTED;
    if (d.tile_n != 0 && d.tile_n != kMxTileN) return GEMM_ERR_UNSUPPORTED;
    if (d.flags & (GEMM_FLAG_SINGLE_CTA | GEMM_FLAG_ACCUM_F16 | GEMM_FLAG_STAGE_K2 | GEMM_FLAG_EPILOGUE_DIRECT))
        return GEMM_ERR_UNSUPPORTED;
    const bool fp4 = is4(d.dtype_a);
    if (fp4 && (d.K % 2 != 0)) return GEMM_ERR_UNSUPPORTED;     // whole bytes of packed elements
    int cg;
    if (d.flags & GEMM_FLAG_CTA_GROUP_1) cg = 1;
    else if (d.flags & GEMM_FLAG_CTA_GROUP_2) cg = 2;
    else cg = (d.M > 128 && ceil_div(d.M, 256) * ceil_div(d.N, kMxTileN) * d.batch >= props.sm_count / 2) ? 2 : 1;
    const int chunks = mx_chunks(d);
    const int64_t stage_a = 128 * 128, stage_b = (kMxTileN / cg) * 128;
    const int64_t sf_stage = 3 * chunks * 512;
    // the staging buffers after the scale ring start on a 1024-byte boundary (128-byte swizzle)
    auto smem_for = [&](int64_t s) {
        return round_up(s * (stage_a + stage_b + sf_stage), 1024) + kStagingBytes + 8 * (2 * s + 3) + 8 + kAlignSlack;
    };
    // tensor memory: 12 columns per slab and stage (A 4, B 8) after the accumulator
    const int64_t max_by_tmem = kMxSfColumns / (12 * chunks);
    int64_t stages = d.stages;
    if (stages == 0) {
        stages = std::min<int64_t>(16, max_by_tmem);
        while (stages > 2 && smem_for(stages) > props.smem_optin_bytes) --stages;
    }
    if (stages < 2 || stages > 16 || stages > max_by_tmem) return GEMM_ERR_UNSUPPORTED;
    if (smem_for(stages) > props.smem_optin_bytes) return GEMM_ERR_RESOURCES;
    const int64_t tiles = ceil_div(d.M, 128 * cg) * ceil_div(d.N, kMxTileN) * d.batch;
    if (tiles > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    int64_t clusters = props.sm_count / cg;
    if (d.max_ctas > 0) clusters = std::min<int64_t>(clusters, std::max<int64_t>(d.max_ctas / cg, 1));
    clusters = std::min<int64_t>(clusters, tiles);
    info->kernel = GEMM_KERNEL_MX;
    info->cta_group = cg;
    info->tile_m = 128 * cg;
    info->tile_n = kMxTileN;
    info->tile_k = fp4 ? 256 : 128;                   // elements of K per ring stage (one 128-byte atom)
    info->stages = (int32_t)stages;
    info->tmem_stages = 1;
    info->tmem_cols = 512;
    info->grid = (int32_t)(clusters * cg);
    info->block_threads = kMxThreads;
    info->num_tiles = tiles;
    info->stage_bytes = stage_a + stage_b + sf_stage;
    info->pipeline_bytes = stages * info->stage_bytes + 8 * (2 * stages + 2) + 4;
    info->smem_bytes = smem_for(stages);
    return GEMM_OK;
}

void plan_stream_k(const gemm_desc_t& d, gemm_plan_info_t* info);

// 512-wide tiles only from this many 128-byte K atoms on (K >= 3072 for 16-bit inputs)
constexpr int64_t kWideMinKAtoms = 48;
// Fewer output tiles than clusters: split each tile along K into s ranges on
// s clusters, so that the otherwise idle SMs share the tiles' K loops.  The
// finisher of a tile adds the other s - 1 clusters' fp32 partials, which
// costs about as much as a short K loop: on GB300 (bf16, 128 x 256 tiles) a
// range pays for its fix-up from 32 K atoms on (512^2 x 8192: 4 ranges of 32
// beat 8 of 16 by 14 %), and an uneven spread of about 1.2 clusters per tile
// (64 tiles on 76 pairs, 128 on 152 SMs) ran 12-13 % slower than no split.
// So s = min(clusters / tiles, K atoms / 32, 8), whole ranges per tile, and
// no split below two.
constexpr int64_t kSplitMinKAtoms = 32;
constexpr int64_t kMaxSplit = 8;

int64_t few_tile_split(const gemm_desc_t& d, int64_t tiles, int64_t k_atoms, int64_t clusters) {
    if (tiles >= clusters || (d.flags & (GEMM_FLAG_NO_STREAM_K | GEMM_FLAG_ACCUM_F16))) return 1;
    const int64_t s = std::min(std::min(clusters / tiles, k_atoms / kSplitMinKAtoms), kMaxSplit);
    return s >= 2 ? s : 1;
}

gemm_status_t plan(const gemm_desc_t& d, const gemm_device_props_t& props, gemm_plan_info_t* info) {
    std::memset(info, 0, sizeof(*info));
    if (d.dtype_d != GEMM_F32 && d.dtype_d != GEMM_BF16 && d.dtype_d != GEMM_F16) return GEMM_ERR_UNSUPPORTED;
    const bool hw = hw_scaled(d.scale_mode);
    if (hw) {
        // MX: E4M3/E5M2 in any pairing, or E2M1 with E2M1; NV: E2M1 with E2M1
        const bool f8 = is8(d.dtype_a) && is8(d.dtype_b), f4 = is4(d.dtype_a) && is4(d.dtype_b);
        if (!(f4 || (f8 && d.scale_mode == GEMM_SCALE_MX_E8M0_32))) return GEMM_ERR_UNSUPPORTED;
    } else if (is4(d.dtype_a) || is4(d.dtype_b)) {
        return GEMM_ERR_UNSUPPORTED;     // E2M1 only with hardware block scales
    } else if (is8(d.dtype_a) && is8(d.dtype_b)) {
        // e4m3 / e5m2 in any pairing, block-scaled only
        if (d.scale_mode != GEMM_SCALE_BLOCK_1x128_128x128) return GEMM_ERR_UNSUPPORTED;
    } else if (d.dtype_a != d.dtype_b) {
        return GEMM_ERR_UNSUPPORTED;
    } else if (is16(d.dtype_a) || d.dtype_a == GEMM_TF32) {
        if (d.scale_mode != GEMM_SCALE_NONE) return GEMM_ERR_UNSUPPORTED;
    } else {
        return GEMM_ERR_UNSUPPORTED;
    }
    if (props.sm_count <= 0 || props.smem_optin_bytes <= 0) return GEMM_ERR_INVALID_ARG;

    if (d.M == 0 || d.N == 0 || d.batch == 0 || d.K == 0) {
        info->kernel = (d.K == 0 && d.M > 0 && d.N > 0 && d.batch > 0) ? GEMM_KERNEL_ZERO_FILL : 0;
        info->cta_group = 1;
        return GEMM_OK;
    }

    if (hw) return plan_mx(d, props, info);

    // fp16 accumulation: f16 inputs, persistent kernel, data-parallel tiles
    const bool acc16 = (d.flags & GEMM_FLAG_ACCUM_F16) != 0;
    if (acc16 && (d.dtype_a != GEMM_F16 || d.dtype_b != GEMM_F16 || (d.flags & GEMM_FLAG_SINGLE_CTA)))
        return GEMM_ERR_UNSUPPORTED;
    const bool want_single = (d.flags & GEMM_FLAG_SINGLE_CTA) != 0;
    const bool allow_single = !acc16 && (d.flags & GEMM_FLAG_NO_SINGLE_CTA) == 0 &&
                              (d.flags & (GEMM_FLAG_CTA_GROUP_1 | GEMM_FLAG_CTA_GROUP_2)) == 0 &&
                              d.tile_n == 0 && d.stages == 0;
    if (want_single) {
        if (!single_fits(d)) return GEMM_ERR_UNSUPPORTED;
        return plan_single(d, props, info);
    }
    if (allow_single && single_fits(d)) return plan_single(d, props, info);

    // ------------------------------------------------ persistent pipelines
    // MN-major operands: 16-bit inputs only (tf32 needs K-major operands; the
    // block-scaled kernel is K-major).
    const bool mn_a = d.major_a == GEMM_MN_MAJOR, mn_b = d.major_b == GEMM_MN_MAJOR;
    if ((mn_a || mn_b) && !is16(d.dtype_a) && !is8(d.dtype_a)) return GEMM_ERR_UNSUPPORTED;
    if (is8(d.dtype_a)) return plan_fp8(d, props, info);
    const int out_bytes = elem_bytes(d.dtype_d);
    const int chunk_cols = 128 / out_bytes;
    const int cg = choose_cta_group(d, props, d.N >= 256 ? 256 : std::max<int64_t>(round_up(d.N, 64), 64));
    int64_t tile_n = d.tile_n;
    if (tile_n == 0) {
        tile_n = d.N >= 256 ? 256 : std::max<int64_t>(round_up(d.N, 64), 64);
        // SM pairs on long K take 512-wide tiles: each SM then loads 48 instead of
        // 64 bytes of operands per 1024 MMA cycles, which its TMA path sustains
        // (8192^3 bf16 on GB300: 20 % fewer cycles), unless they pad N more
        // than 256-wide tiles do or the operands are MN-major.  On short K the
        // single accumulator's drain, once per tile, costs more than that
        // saves (K <= 2048 bf16 on GB300: 2-34 % slower than 256-wide tiles),
        // and with tiles for fewer than half of the pairs the narrower tiles
        // keep more SMs busy (2048^2 x 8192: 28 % faster).
        const int64_t pad256 = round_up(d.N, 256) - d.N, pad512 = round_up(d.N, 512) - d.N;
        const int64_t k_atoms = ceil_div(d.K, 128 / elem_bytes(d.dtype_a));
        const int64_t wide_tiles = ceil_div(d.M, 256) * ceil_div(d.N, 512) * d.batch;
        if (cg == 2 && !mn_a && !mn_b && !(d.flags & GEMM_FLAG_STAGE_K2) && d.N >= 1024 &&
            (pad512 - pad256) * 20 <= d.N && k_atoms >= kWideMinKAtoms && wide_tiles >= props.sm_count / 4)
            tile_n = 512;
        // 256-wide tiles for fewer than half of the clusters: 128-wide tiles
        // occupy twice the SMs before any split along K, and a split's fix-up
        // is the kernel's tail (bf16 on GB300: 10-35 % faster on 14 such
        // shapes from 128 x 8192 x 8192 to 1536^2 x 6144; from two thirds of
        // the clusters on, 256-wide tiles were faster again).
        const int64_t tiles256 = ceil_div(d.M, 128 * cg) * ceil_div(d.N, 256) * d.batch;
        if (tile_n == 256 && 2 * tiles256 < props.sm_count / cg) tile_n = 128;
    }
    // 512-wide tiles: two N = 256 MMAs per K step into one 512-column
    // accumulator (K-major operands, one K atom per stage)
    const bool wide = tile_n == 512;
    if (wide && (mn_a || mn_b || (d.flags & GEMM_FLAG_STAGE_K2))) return GEMM_ERR_UNSUPPORTED;
    if (!wide && (tile_n % 16 != 0 || tile_n < 16 || tile_n > 256)) return GEMM_ERR_UNSUPPORTED;
    if (tile_n % chunk_cols != 0) return GEMM_ERR_UNSUPPORTED;     // epilogue writes 128-byte column chunks
    if ((tile_n / cg) % 8 != 0) return GEMM_ERR_UNSUPPORTED;      // B half-tile rows form 8-row swizzle atoms
    if (mn_b && (tile_n / cg) % 64 != 0) return GEMM_ERR_UNSUPPORTED;  // MN-major B: 64-column boxes
    const int tmem_stages = wide ? 1 : 2;
    const int64_t tmem_need = tmem_stages * tile_n;
    if (tmem_need > 512) return GEMM_ERR_RESOURCES;
    const int tmem_cols = pow2_at_least(tmem_need);

    // Ring stage depth: one or two 128-byte swizzle atoms of K (64 or 128
    // 16-bit elements, 32 or 64 tf32).  Two atoms halve the MMA thread's
    // barrier waits per MMA (its issue loop is the bottleneck at one atom:
    // 8192^3 bf16 runs 5.9 % faster on GB300); default whenever both operands
    // are K-major, K spans more than one atom and three stages still fit.
    if ((d.flags & GEMM_FLAG_STAGE_K1) && (d.flags & GEMM_FLAG_STAGE_K2)) return GEMM_ERR_INVALID_ARG;
    if ((d.flags & GEMM_FLAG_STAGE_K2) && (mn_a || mn_b)) return GEMM_ERR_UNSUPPORTED;
    const int64_t atom_k = 128 / elem_bytes(d.dtype_a);
    const int64_t atom_bytes = 128 * 128 + (tile_n / cg) * 128;   // A and B, one atom of K
    const int64_t fixed_bytes = kStagingBytes + 8 * (4 * tmem_stages + 1) + 8 + kAlignSlack;
    int atoms = 1;
    if (d.flags & GEMM_FLAG_STAGE_K2) {
        atoms = 2;
    } else if (!(d.flags & GEMM_FLAG_STAGE_K1) && !wide && !mn_a && !mn_b && d.K > atom_k &&
               3 * (2 * atom_bytes + 16) + fixed_bytes <= props.smem_optin_bytes) {
        atoms = 2;
    }
    const int tile_k = (int)(atoms * atom_k);
    const int64_t stage_a = atoms * 128 * 128;      // 128 rows x 128 B per atom
    const int64_t stage_b = atoms * (tile_n / cg) * 128;
    const int64_t stage_bytes = stage_a + stage_b;
    // Epilogue: TMA stores through a 32 KB staging area (default), or direct
    // row stores with no staging (on request).  On GB300 the staging area's
    // smem buys nothing as a 7th ring stage at 8192^3 (within 1 %), and TMA
    // stores are faster at 4096^3 (+2 %) and on batched problems (+23 %).
    auto smem_for_mode = [&](int64_t s, bool direct) {
        return s * stage_bytes + (direct ? 0 : kStagingBytes) + 8 * (2 * s + 4 * tmem_stages + 1) + 8 + kAlignSlack;
    };
    auto max_stages = [&](bool direct) {
        int64_t s = 16;
        while (s > 2 && smem_for_mode(s, direct) > props.smem_optin_bytes) --s;
        return s;
    };
    bool direct;
    if (d.flags & GEMM_FLAG_EPILOGUE_DIRECT) direct = true;
    else if (d.flags & GEMM_FLAG_EPILOGUE_TMA) direct = false;
    else direct = false;
    auto smem_for = [&](int64_t s) { return smem_for_mode(s, direct); };
    int64_t stages = d.stages;
    if (stages == 0) stages = max_stages(direct);
    if (stages < 2 || stages > 16) return GEMM_ERR_UNSUPPORTED;
    if (smem_for(stages) > props.smem_optin_bytes) return GEMM_ERR_RESOURCES;

    const int64_t num_m = ceil_div(d.M, 128 * cg);
    const int64_t num_n = ceil_div(d.N, tile_n);
    const int64_t tiles = num_m * num_n * d.batch;
    if (tiles > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    int64_t clusters = props.sm_count / cg;
    clusters = std::min<int64_t>(clusters, tiles * few_tile_split(d, tiles, ceil_div(d.K, atom_k), clusters));
    // the cap applies to the grid as planned: below tiles x splits it leaves
    // ranges that straddle tiles, which the schedule handles as well
    if (d.max_ctas > 0) clusters = std::min<int64_t>(clusters, std::max<int64_t>(d.max_ctas / cg, 1));

    info->kernel = GEMM_KERNEL_PERSISTENT;
    info->cta_group = cg;
    info->tile_m = 128 * cg;
    info->tile_n = (int32_t)tile_n;
    info->tile_k = tile_k;
    info->stages = (int32_t)stages;
    info->tmem_stages = tmem_stages;
    info->tmem_cols = tmem_cols;
    info->grid = (int32_t)(clusters * cg);
    info->block_threads = kPersistentThreads;
    info->num_tiles = tiles;
    info->stage_bytes = stage_bytes;
    // the card's accounting (two barriers per stage and per TMEM stage); smem_bytes
    // counts this kernel's barriers: one more per accumulator (two empty halves)
    info->pipeline_bytes = stages * stage_bytes + 8 * (2 * stages + 2 * tmem_stages) + 4;
    info->smem_bytes = smem_for(stages);
    info->epilogue = direct ? 1 : 0;
    plan_stream_k(d, info);
    return GEMM_OK;
}

// ---------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUtensorMapDataType tma_dtype(int dt) {
    switch (dt) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case GEMM_F32: case GEMM_TF32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// Row-major (rows x cols) matrix, `ld` elements between rows, optional batch
// dimension with `bstride` elements; box (box_cols x box_rows), 128-byte swizzle.
bool encode_map(CUtensorMap* m, int dt, const void* base, int64_t cols, int64_t rows, int64_t ld, int64_t batch,
                int64_t bstride, int box_cols, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const int eb = elem_bytes(dt);
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * eb), (cuuint64_t)(bstride * eb)};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const cuuint32_t rank = batch > 1 ? 3 : 2;
    CUresult r = enc(m, tma_dtype(dt), rank, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scale tiles of a matrix with `rows` rows as a 4-D map of 32-bit words: 128
// words (one 512-byte slab of 128 rows x 4 scales), kq slabs along K,
// ceil(rows/128) row blocks, batch entries `batch_stride` bytes apart.  Box
// (128, chunks, 1, 1): one ring stage's slabs of one row block.  Slabs past
// the end along K or past the last row block read as zeros.
bool encode_sf_map(CUtensorMap* m, const void* base, int64_t rows, int64_t kq, int64_t batch, int64_t batch_stride,
                   int chunks) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const int64_t rb = ceil_div(rows, 128);
    cuuint64_t dims[4] = {128, (cuuint64_t)kq, (cuuint64_t)rb, (cuuint64_t)batch};
    cuuint64_t strides[3] = {512, (cuuint64_t)(kq * 512),
                             (cuuint64_t)std::max<int64_t>(batch_stride, rb * kq * 512)};
    cuuint32_t box[4] = {128, (cuuint32_t)chunks, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Stream-K for the 16-bit persistent kernel.  When the tiles do not fill
// whole waves of clusters, the last wave plus one full wave (sk_tiles >=
// clusters) are split evenly along K over all clusters; the rest stays
// data-parallel.  Worth it only for long K: the fix-up moves one fp32 tile
// per split (K <= 2048 bf16 on GB300 ran 2-15 % slower with it).  With fewer
// tiles than clusters (the planner then sizes the grid by few_tile_split),
// every tile is split, over several clusters each.
constexpr int kStreamKMinKBlocks = 48;   // 128-byte K atoms

void plan_stream_k(const gemm_desc_t& d, gemm_plan_info_t* info) {
    info->stream_k_tiles = 0;
    info->workspace_bytes = 0;
    if (info->kernel != GEMM_KERNEL_PERSISTENT || (d.flags & (GEMM_FLAG_NO_STREAM_K | GEMM_FLAG_ACCUM_F16))) return;
    const int64_t clusters = info->grid / info->cta_group;
    if (clusters < 2) return;
    if (info->num_tiles < clusters) {
        // every range holds at least one K block (few_tile_split keeps a cluster's share >= kSplitMinKAtoms)
        if (info->num_tiles * ceil_div(d.K, info->tile_k) < clusters) return;
        info->stream_k_tiles = (int32_t)info->num_tiles;
    } else {
        // the threshold counts 128-byte K atoms, whatever the stage depth
        const int64_t atoms = std::max<int64_t>(info->tile_k * elem_bytes(d.dtype_a) / 128, 1);
        const int64_t nk = ceil_div(d.K, info->tile_k) * atoms;
        if (nk < kStreamKMinKBlocks) return;
        const int64_t rem = info->num_tiles % clusters;
        if (rem == 0) return;
        // 512-wide tiles: a partial is 256 KB per CTA to write and add back;
        // worth it only when the last wave would leave most clusters idle
        if (info->tile_n > 256 && 2 * rem >= clusters) return;
        info->stream_k_tiles = (int32_t)(clusters + rem);
    }
    // one partial slot per cluster: cta_group CTAs x 128 rows x tile_n fp32, plus a flag per epilogue warp
    const int64_t partial_bytes = clusters * info->cta_group * 128 * info->tile_n * 4;
    const int64_t flag_bytes = round_up(clusters * info->cta_group * kSkFlagsPerCta * 4, 256);
    info->workspace_bytes = partial_bytes + flag_bytes;
}

// The fields of the work-unit schedule (units.cuh) for a planned problem.
void fill_schedule(const gemm_desc_t& d, const gemm_plan_info_t& info, dgb::PersistentParams& p) {
    p.num_m_blocks = (int32_t)ceil_div(d.M, info.tile_m);
    p.num_n_blocks = (int32_t)ceil_div(d.N, info.tile_n);
    p.num_k_blocks = (int32_t)ceil_div(d.K, info.tile_k);
    p.tiles_per_batch = p.num_m_blocks * p.num_n_blocks;
    p.num_tiles = (int32_t)info.num_tiles;
    p.group_m = d.raster_group > 0 ? d.raster_group
                                   : (info.tile_n > 256 && p.num_m_blocks >= 2 * kWideRasterGroup ? kWideRasterGroup
                                                                                                : kDefaultRasterGroup);
}

// A persistent grid must be co-resident: cap it by the clusters the device can
// hold at once with the chosen kernel's shared memory.
gemm_status_t cap_resident(const gemm_desc_t& d, gemm_plan_info_t* info) {
    int resident;
    if (info->kernel == GEMM_KERNEL_PERSISTENT)
        resident = dgb::persistent_max_active_clusters(info->cta_group, d.dtype_d, (size_t)info->smem_bytes);
    else if (info->kernel == GEMM_KERNEL_FP8_BLOCK)
        resident = dgb::fp8_max_active_clusters(info->cta_group, info->tile_n, d.dtype_d, (size_t)info->smem_bytes);
    else if (info->kernel == GEMM_KERNEL_MX)
        resident = dgb::mx_max_active_clusters(mx_kind(d), info->cta_group, d.dtype_d, (size_t)info->smem_bytes);
    else
        return GEMM_OK;
    if (resident <= 0) return cuda_fail(cudaGetLastError());
    if (info->grid > resident * info->cta_group) info->grid = resident * info->cta_group;
    return GEMM_OK;
}

}  // namespace

// ---------------------------------------------------------------- allocation-free variant state
//
// gemm_run_noalloc keeps the kernels' device error record in this array
// instead of a cudaMalloc'd one.  It is library-owned device memory: every GPU
// that loads the library holds these bytes until the process exits.  Host code
// must not pass the name itself to a kernel (on the host it is only a stand-in);
// its device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[256];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Zero the first `bytes` of the record in stream order (names the array directly).
__global__ void noalloc_clear_kernel(unsigned bytes) {
    for (unsigned i = threadIdx.x; i < bytes && i < sizeof(g_noalloc_scratch); i += blockDim.x)
        g_noalloc_scratch[i] = 0;
}

// Device address of g_noalloc_scratch on device `dev` (current), looked up on
// the first call for that device.
gemm_status_t noalloc_address(int dev, void** out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return GEMM_OK;
}

// Drop the cached address of device `dev` (looked up again on the next call).
void noalloc_forget(int dev) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    g_noalloc_addr[dev] = nullptr;
}

}  // namespace

constexpr int kHostPanels = 8;    // gemm_run_host: at most this many row (or batch) panels
constexpr int kHostJobs = kHostPanels + 1;

// One GEMM of gemm_run_host's pipeline: rows (or batch entries) [u0, u0+nu)
// of A and D against rows [n0, n0+nn) of B (all of B for batch panels, which
// take their own entries of B).  Before it, the copy-in stream brings that
// many rows of A (unless the previous job of the same panel did) and the
// given range of B.
struct HostJob {
    int64_t u0, nu, n0, nn;
    bool copy_a;
    int64_t b0, bn;                   // rows of B (row panels) to copy before this job; bn = 0: none
    struct gemm_plan_s* sub;
};

// gemm_run_host's pipeline: copy streams, events and one data-parallel plan
// per job (sharing the parent's status record), created on first use.
struct HostPipe {
    bool ready = false;
    int jobs = 0;
    HostJob job[kHostJobs] = {};
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[kHostJobs] = {}, ev_g[kHostJobs] = {};
};

struct gemm_plan_s {
    CUtensorMap maps[3];          // A, B, D tensor maps of the last pointers seen
    const void* map_ptrs[3];
    bool maps_valid;
    gemm_desc_t desc;             // resolved
    gemm_plan_info_t info;
    gemm_device_props_t props;
    int device;
    gemm_device_error_t* status;  // device record; stream-K flags and partials follow it
    uint32_t* sk_flags;
    float* sk_partials;
    HostPipe* pipe = nullptr;     // gemm_run_host's panels (owned; sub-plans share `status`)
    CUtensorMap sf_maps[2];       // MX / NV: scale-tile maps of A and B for sf_ptrs
    const void* sf_ptrs[2] = {nullptr, nullptr};
    bool sf_valid = false;
};

static void host_pipe_free(HostPipe* hp) {
    if (!hp) return;
    for (int i = 0; i < kHostJobs; ++i) {
        if (hp->ev_a[i]) cudaEventDestroy(hp->ev_a[i]);
        if (hp->ev_g[i]) cudaEventDestroy(hp->ev_g[i]);
        delete hp->job[i].sub;
    }
    if (hp->ev_start) cudaEventDestroy(hp->ev_start);
    if (hp->ev_done) cudaEventDestroy(hp->ev_done);
    if (hp->h2d) cudaStreamDestroy(hp->h2d);
    if (hp->d2h) cudaStreamDestroy(hp->d2h);
    delete hp;
}

extern "C" {

gemm_status_t gemm_plan_query(const gemm_desc_t* desc, const gemm_device_props_t* props, gemm_plan_info_t* info) {
    if (!desc || !props || !info) return GEMM_ERR_INVALID_ARG;
    Resolved r;
    gemm_status_t s = resolve(desc, &r);
    if (s != GEMM_OK) return s;
    return plan(r.d, *props, info);
}

gemm_status_t gemm_plan_create(gemm_plan_t* out, const gemm_desc_t* desc) {
    if (!out || !desc) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    Resolved r;
    gemm_status_t s = resolve(desc, &r);
    if (s != GEMM_OK) return s;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { g_last_cuda_error = (int)e; return GEMM_ERR_NO_DEVICE; }
    gemm_device_props_t props{};
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
    props.sm_count = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return cuda_fail(e);
    props.smem_optin_bytes = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
    props.cc_major = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
    props.cc_minor = v;
    if (props.cc_major != 10 || props.cc_minor != 3) return GEMM_ERR_NO_DEVICE;  // built for sm_103a only
    gemm_plan_info_t info;
    s = plan(r.d, props, &info);
    if (s != GEMM_OK) return s;
    if ((s = cap_resident(r.d, &info)) != GEMM_OK) return s;
    plan_stream_k(r.d, &info);
    gemm_plan_s* p = new (std::nothrow) gemm_plan_s();
    if (!p) return GEMM_ERR_RESOURCES;
    p->maps_valid = false;
    p->desc = r.d;
    p->info = info;
    p->props = props;
    p->device = dev;
    p->status = nullptr;
    p->sk_flags = nullptr;
    p->sk_partials = nullptr;
    // One allocation: status record and launch counter (256 B), then stream-K flags, then partials.
    const int64_t flag_bytes = info.stream_k_tiles
                                   ? round_up((int64_t)(info.grid / info.cta_group) * info.cta_group *
                                                  kSkFlagsPerCta * 4, 256) : 0;
    const size_t total = 256 + (size_t)info.workspace_bytes;
    void* mem = nullptr;
    if ((e = cudaMalloc(&mem, total)) != cudaSuccess) {
        delete p;
        return cuda_fail(e);
    }
    if ((e = cudaMemset(mem, 0, 256 + (size_t)flag_bytes)) != cudaSuccess) {
        cudaFree(mem);
        delete p;
        return cuda_fail(e);
    }
    p->status = static_cast<gemm_device_error_t*>(mem);
    if (info.stream_k_tiles) {
        p->sk_flags = reinterpret_cast<uint32_t*>(static_cast<char*>(mem) + 256);
        p->sk_partials = reinterpret_cast<float*>(static_cast<char*>(mem) + 256 + flag_bytes);
    }
    *out = p;
    return GEMM_OK;
}

gemm_status_t gemm_plan_info(gemm_plan_t plan, gemm_plan_info_t* info) {
    if (!plan || !info) return GEMM_ERR_INVALID_ARG;
    *info = plan->info;
    return GEMM_OK;
}

gemm_status_t gemm_plan_work_unit(const gemm_desc_t* desc, const gemm_plan_info_t* info, int32_t cluster,
                                  int32_t index, gemm_work_unit_t* out) {
    if (!desc || !info || !out || index < 0) return GEMM_ERR_INVALID_ARG;
    if (info->kernel != GEMM_KERNEL_PERSISTENT && info->kernel != GEMM_KERNEL_FP8_BLOCK &&
        info->kernel != GEMM_KERNEL_MX)
        return GEMM_ERR_UNSUPPORTED;
    if (info->cta_group < 1 || info->grid < info->cta_group || info->tile_m <= 0 || info->tile_n <= 0 ||
        info->tile_k <= 0 || desc->M < 0 || desc->N < 0 || desc->K < 0)
        return GEMM_ERR_INVALID_ARG;
    const int clusters = info->grid / info->cta_group;
    if (cluster < 0 || cluster >= clusters) return GEMM_ERR_INVALID_ARG;
    dgb::PersistentParams p{};
    fill_schedule(*desc, *info, p);
    p.sk_tiles = info->kernel == GEMM_KERNEL_PERSISTENT ? info->stream_k_tiles : 0;
    // info must be this desc's plan: the tile count and the stream-K region
    // have to agree with the shape, or the raster arithmetic is meaningless
    // (a region narrower than the grid only as every tile, with a K block per cluster at least)
    if (info->num_tiles != (int64_t)p.tiles_per_batch * std::max<int64_t>(desc->batch, 1) || p.sk_tiles < 0 ||
        p.sk_tiles > p.num_tiles ||
        (p.sk_tiles > 0 && p.sk_tiles < clusters &&
         (p.sk_tiles != p.num_tiles || (int64_t)p.num_tiles * p.num_k_blocks < clusters)))
        return GEMM_ERR_INVALID_ARG;
    gemm_work_unit_t r{};
    r.tile = -1;
    dgb::WorkUnit u;
    if (p.num_tiles > 0 && p.num_k_blocks > 0 && dgb::next_unit(p, cluster, clusters, index, u)) {
        int b = 0, mb = 0, nb = 0;
        dgb::tile_coords(p, u.tile, b, mb, nb);
        r.tile = u.tile;
        r.batch = b;
        r.m_block = mb;
        r.n_block = nb;
        r.k_block_begin = u.kb0;
        r.k_block_end = u.kb1;
        r.role = u.role;
        r.slot = u.role == dgb::kUnitWhole ? 0 : u.slot;
        r.slot_first = u.role == dgb::kUnitFinisher ? u.slot0 : r.slot;
    }
    *out = r;
    return GEMM_OK;
}

gemm_status_t gemm_run(gemm_plan_t plan, const void* A, const void* B, void* D, const float* scale_a,
                       const float* scale_b, gemm_stream_t stream_) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const gemm_desc_t& d = plan->desc;
    const gemm_plan_info_t& info = plan->info;
    if (hw_scaled(d.scale_mode)) return GEMM_ERR_INVALID_ARG;     // gemm_run_mx runs these plans
    if (d.M == 0 || d.N == 0 || d.batch == 0) return GEMM_OK;
    if (!D) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(D)) return GEMM_ERR_ALIGNMENT;
    const int eb_d = elem_bytes(d.dtype_d);
    if (((d.ldd * eb_d) & 15) || ((d.batch > 1) && ((d.stride_d * eb_d) & 15))) return GEMM_ERR_ALIGNMENT;
    const bool scaled = d.scale_mode != GEMM_SCALE_NONE;
    if (scaled != (scale_a != nullptr) || scaled != (scale_b != nullptr)) return GEMM_ERR_INVALID_ARG;
    cudaError_t e;
    if (info.kernel == GEMM_KERNEL_ZERO_FILL) {
        e = dgb::launch_zero_fill(D, d.dtype_d, d.M, d.N, d.batch, d.ldd, d.stride_d, plan->props.sm_count, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }
    if (!A || !B) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B)) return GEMM_ERR_ALIGNMENT;
    const int eb_a = elem_bytes(d.dtype_a), eb_b = elem_bytes(d.dtype_b);
    if (((d.lda * eb_a) & 15) || ((d.ldb * eb_b) & 15)) return GEMM_ERR_ALIGNMENT;
    if (d.batch > 1 && (((d.stride_a * eb_a) & 15) || ((d.stride_b * eb_b) & 15))) return GEMM_ERR_ALIGNMENT;

    if (info.kernel == GEMM_KERNEL_SINGLE_CTA) {
        SingleParams p{};
        p.A = A; p.B = B; p.D = D; p.status = plan->status;
        p.lda = d.lda; p.ldb = d.ldb; p.ldd = d.ldd;
        p.stride_a = d.stride_a; p.stride_b = d.stride_b; p.stride_d = d.stride_d;
        p.M = (int32_t)d.M; p.N = (int32_t)d.N; p.K = (int32_t)d.K;
        p.n_pad = info.tile_n; p.k_pad = info.tile_k;
        p.major_a = d.major_a; p.major_b = d.major_b;
        p.tmem_cols = info.tmem_cols;
        p.idesc = dgb::make_idesc(d.dtype_a == GEMM_BF16 ? 1u : 0u, 128u, (uint32_t)info.tile_n);
        p.timeout_ns = d.wait_timeout_ns;
        e = dgb::launch_single_cta(p, d.dtype_d, (int)d.batch, (size_t)info.smem_bytes, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }

    if (scaled && (!aligned16(scale_a) || !aligned16(scale_b))) return GEMM_ERR_ALIGNMENT;

    // persistent pipelines
    PersistentParams p;
    std::memset(&p, 0, sizeof(p));
    const int cg = info.cta_group;
    const int64_t batch_maps = d.batch;
    // Tensor maps depend on the pointers only: re-encode when they change.
    if (!plan->maps_valid || plan->map_ptrs[0] != A || plan->map_ptrs[1] != B || plan->map_ptrs[2] != D) {
        plan->maps_valid = false;
        const bool mn_a = d.major_a == GEMM_MN_MAJOR, mn_b = d.major_b == GEMM_MN_MAJOR;
        // K-major: (K, rows) boxes of one 128-byte atom x rows (k_atoms per
        // stage).  MN-major: (rows, K) boxes of 64 x tile_k.
        const int atom_k = (int)(128 / eb_a);
        const bool ok_a = mn_a ? encode_map(&plan->maps[0], d.dtype_a, A, d.M, d.K, d.lda, batch_maps, d.stride_a,
                                            (int)(128 / eb_a), info.tile_k)
                               : encode_map(&plan->maps[0], d.dtype_a, A, d.K, d.M, d.lda, batch_maps, d.stride_a,
                                            atom_k, 128);
        const bool ok_b = mn_b ? encode_map(&plan->maps[1], d.dtype_b, B, d.N, d.K, d.ldb, batch_maps, d.stride_b,
                                            (int)(128 / eb_b), info.tile_k)
                               : encode_map(&plan->maps[1], d.dtype_b, B, d.K, d.N, d.ldb, batch_maps, d.stride_b,
                                            atom_k, std::min(info.tile_n, 256) / cg);
        if (!ok_a || !ok_b ||
            !encode_map(&plan->maps[2], d.dtype_d, D, d.N, d.M, d.ldd, batch_maps, d.stride_d, 128 / eb_d, 32)) {
            g_last_cuda_error = (int)cudaErrorInvalidValue;
            return GEMM_ERR_CUDA;
        }
        plan->map_ptrs[0] = A;
        plan->map_ptrs[1] = B;
        plan->map_ptrs[2] = D;
        plan->maps_valid = true;
    }
    p.tmap_a = plan->maps[0];
    p.tmap_b = plan->maps[1];
    p.tmap_d = plan->maps[2];
    p.status = plan->status;
    p.M = (int32_t)d.M; p.N = (int32_t)d.N; p.K = (int32_t)d.K; p.batch = (int32_t)d.batch;
    fill_schedule(d, info, p);
    p.tile_n = info.tile_n;
    p.stages = info.stages;
    p.tmem_cols = info.tmem_cols;
    p.tmem_stages = info.tmem_stages;
    p.batched = d.batch > 1 ? 1 : 0;
    p.tile_k = info.tile_k;
    p.k_atoms = (int32_t)(info.tile_k * eb_a / 128);   // 128-byte K atoms per stage
    p.mma_kind = d.dtype_a == GEMM_TF32 ? dgb::kMmaKindTF32 : dgb::kMmaKindF16;
    // A/B formats: kind::f16 0 = f16, 1 = bf16; kind::tf32 2 = tf32
    p.mn_major_a = d.major_a == GEMM_MN_MAJOR;
    p.mn_box_elems = (int32_t)(128 / eb_a);
    p.mn_major_b = d.major_b == GEMM_MN_MAJOR;
    // one MMA covers at most 256 columns (512-wide tiles issue two)
    const uint32_t fmt = d.dtype_a == GEMM_BF16 ? 1u : (d.dtype_a == GEMM_TF32 ? 2u : 0u);
    p.acc_f16 = (d.flags & GEMM_FLAG_ACCUM_F16) ? 1 : 0;
    p.idesc = dgb::make_idesc2(fmt, fmt, (uint32_t)info.tile_m, (uint32_t)std::min(info.tile_n, 256),
                               (uint32_t)p.mn_major_a, (uint32_t)p.mn_major_b, p.acc_f16 ? 0u : 1u);
    p.stage_bytes_a = (uint32_t)(128 * info.tile_k * eb_a);
    p.stage_bytes_b = (uint32_t)((info.tile_n / cg) * info.tile_k * eb_b);
    p.flags = d.flags;
    p.timeout_ns = d.wait_timeout_ns;
    // Single long-K problems revisit A panels across the waves of a raster
    // group and stream D out; batched problems touch every panel once.
    p.l2_hints = (d.batch == 1 && p.num_k_blocks >= 8 && !(d.flags & GEMM_FLAG_NO_L2_HINTS))
                     ? (dgb::kHintKeepA | dgb::kHintStreamD) : 0u;
    p.direct_store = info.epilogue;
    p.d_ptr = D;
    p.ldd = d.ldd;
    p.stride_d = d.stride_d;
    if (info.stream_k_tiles > 0 && plan->sk_flags != nullptr) {
        p.sk_tiles = info.stream_k_tiles;
        p.sk_flags = plan->sk_flags;
        p.sk_epoch = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(plan->status) + kSkEpochOffset);
        p.sk_partials = plan->sk_partials;
    }
    if (info.kernel == GEMM_KERNEL_FP8_BLOCK) {
        p.scale_a = scale_a;
        p.scale_b = scale_b;
        p.ld_sa = d.ld_sa;
        p.ld_sb = d.ld_sb;
        p.stride_sa = d.stride_sa;
        p.stride_sb = d.stride_sb;
        // kind::f8f6f4 formats: 0 = e4m3, 1 = e5m2
        p.idesc = dgb::make_idesc2(d.dtype_a == GEMM_E5M2 ? 1u : 0u, d.dtype_b == GEMM_E5M2 ? 1u : 0u,
                                   (uint32_t)info.tile_m, (uint32_t)info.tile_n, (uint32_t)p.mn_major_a,
                                   (uint32_t)p.mn_major_b);
        e = dgb::launch_fp8_block(p, cg, d.dtype_d, info.grid, (size_t)info.smem_bytes, stream);
    } else {
        e = dgb::launch_persistent(p, cg, d.dtype_d, info.grid, (size_t)info.smem_bytes, stream);
    }
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

gemm_status_t gemm_run_mx(gemm_plan_t plan, const void* A, const void* B, void* D, const void* sf_a,
                          const void* sf_b, const float* tensor_scales, gemm_stream_t stream_) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const gemm_desc_t& d = plan->desc;
    const gemm_plan_info_t& info = plan->info;
    if (!hw_scaled(d.scale_mode)) return GEMM_ERR_INVALID_ARG;     // gemm_run runs the other plans
    const bool nv = d.scale_mode == GEMM_SCALE_NV_E4M3_16;
    if (nv != (tensor_scales != nullptr)) return GEMM_ERR_INVALID_ARG;
    if (d.M == 0 || d.N == 0 || d.batch == 0) return GEMM_OK;
    if (!D) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(D)) return GEMM_ERR_ALIGNMENT;
    const int eb_d = elem_bytes(d.dtype_d);
    if (((d.ldd * eb_d) & 15) || ((d.batch > 1) && ((d.stride_d * eb_d) & 15))) return GEMM_ERR_ALIGNMENT;
    cudaError_t e;
    if (info.kernel == GEMM_KERNEL_ZERO_FILL) {
        e = dgb::launch_zero_fill(D, d.dtype_d, d.M, d.N, d.batch, d.ldd, d.stride_d, plan->props.sm_count, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }
    if (info.kernel != GEMM_KERNEL_MX) return GEMM_ERR_INVALID_ARG;
    if (!A || !B || !sf_a || !sf_b) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(sf_a) || !aligned16(sf_b)) return GEMM_ERR_ALIGNMENT;
    if (nv && (reinterpret_cast<uintptr_t>(tensor_scales) & 3u)) return GEMM_ERR_ALIGNMENT;
    // operands as byte matrices: K bytes per row (E2M1: two elements per byte)
    const bool fp4 = is4(d.dtype_a);
    if (fp4 && ((d.lda | d.ldb | d.stride_a | d.stride_b) & 1)) return GEMM_ERR_INVALID_ARG;
    const int64_t kbytes = fp4 ? d.K / 2 : d.K;
    const bool mn_a = d.major_a == GEMM_MN_MAJOR, mn_b = d.major_b == GEMM_MN_MAJOR;
    const int64_t lda_b = fp4 ? d.lda / 2 : d.lda, ldb_b = fp4 ? d.ldb / 2 : d.ldb;
    const int64_t sta_b = fp4 ? d.stride_a / 2 : d.stride_a, stb_b = fp4 ? d.stride_b / 2 : d.stride_b;
    if ((lda_b & 15) || (ldb_b & 15)) return GEMM_ERR_ALIGNMENT;
    if (d.batch > 1 && ((sta_b & 15) || (stb_b & 15) || (d.stride_sa & 15) || (d.stride_sb & 15)))
        return GEMM_ERR_ALIGNMENT;
    const int cg = info.cta_group;
    const int chunks = mx_chunks(d);
    const int64_t v = nv ? 16 : 32;
    const int64_t kq = std::max<int64_t>(ceil_div(ceil_div(d.K, v), 4), 1);
    if (!plan->maps_valid || plan->map_ptrs[0] != A || plan->map_ptrs[1] != B || plan->map_ptrs[2] != D) {
        plan->maps_valid = false;
        // byte boxes of one 128-byte K atom x 128 rows (A) or 256 / cg rows (B);
        // MN-major: 128 contiguous M (N) bytes x 128 k-rows
        const bool ok_a = mn_a ? encode_map(&plan->maps[0], GEMM_E4M3, A, d.M, d.K, lda_b, d.batch, sta_b, 128, 128)
                               : encode_map(&plan->maps[0], GEMM_E4M3, A, kbytes, d.M, lda_b, d.batch, sta_b, 128, 128);
        const bool ok_b = mn_b ? encode_map(&plan->maps[1], GEMM_E4M3, B, d.N, d.K, ldb_b, d.batch, stb_b, 128, 128)
                               : encode_map(&plan->maps[1], GEMM_E4M3, B, kbytes, d.N, ldb_b, d.batch, stb_b, 128,
                                            kMxTileN / cg);
        if (!ok_a || !ok_b ||
            !encode_map(&plan->maps[2], d.dtype_d, D, d.N, d.M, d.ldd, d.batch, d.stride_d, 128 / eb_d, 32)) {
            g_last_cuda_error = (int)cudaErrorInvalidValue;
            return GEMM_ERR_CUDA;
        }
        plan->map_ptrs[0] = A;
        plan->map_ptrs[1] = B;
        plan->map_ptrs[2] = D;
        plan->maps_valid = true;
    }
    if (!plan->sf_valid || plan->sf_ptrs[0] != sf_a || plan->sf_ptrs[1] != sf_b) {
        plan->sf_valid = false;
        if (!encode_sf_map(&plan->sf_maps[0], sf_a, d.M, kq, d.batch, d.stride_sa, chunks) ||
            !encode_sf_map(&plan->sf_maps[1], sf_b, d.N, kq, d.batch, d.stride_sb, chunks)) {
            g_last_cuda_error = (int)cudaErrorInvalidValue;
            return GEMM_ERR_CUDA;
        }
        plan->sf_ptrs[0] = sf_a;
        plan->sf_ptrs[1] = sf_b;
        plan->sf_valid = true;
    }
    dgb::MxParams q;
    std::memset(&q, 0, sizeof(q));
    PersistentParams& p = q.base;
    p.tmap_a = plan->maps[0];
    p.tmap_b = plan->maps[1];
    p.tmap_d = plan->maps[2];
    p.status = plan->status;
    p.M = (int32_t)d.M; p.N = (int32_t)d.N; p.K = (int32_t)d.K; p.batch = (int32_t)d.batch;
    fill_schedule(d, info, p);              // K blocks of info.tile_k elements (one 128-byte atom)
    p.tile_n = info.tile_n;
    p.stages = info.stages;
    p.tmem_cols = info.tmem_cols;
    p.tmem_stages = 1;
    p.batched = d.batch > 1 ? 1 : 0;
    p.tile_k = 128;                         // the producers' K coordinate counts bytes
    p.k_atoms = 1;
    p.mn_box_elems = 128;
    p.mn_major_a = mn_a ? 1 : 0;
    p.mn_major_b = mn_b ? 1 : 0;
    // element formats: mxf8f6f4 0 = E4M3, 1 = E5M2; mxf4 / mxf4nvf4 1 = E2M1; scales UE8M0 (MX) or UE4M3 (NV)
    const uint32_t fa = fp4 ? 1u : (d.dtype_a == GEMM_E5M2 ? 1u : 0u);
    const uint32_t fb = fp4 ? 1u : (d.dtype_b == GEMM_E5M2 ? 1u : 0u);
    p.idesc = dgb::make_idesc_block_scaled(fa, fb, (uint32_t)info.tile_m, (uint32_t)info.tile_n, nv ? 0u : 1u,
                                           (uint32_t)p.mn_major_a, (uint32_t)p.mn_major_b);
    p.stage_bytes_a = 128u * 128u;
    p.stage_bytes_b = (uint32_t)((info.tile_n / cg) * 128);
    p.flags = d.flags;
    p.timeout_ns = d.wait_timeout_ns;
    p.l2_hints = (d.batch == 1 && p.num_k_blocks >= 8 && !(d.flags & GEMM_FLAG_NO_L2_HINTS))
                     ? (dgb::kHintKeepA | dgb::kHintStreamD) : 0u;
    p.d_ptr = D;
    p.ldd = d.ldd;
    p.stride_d = d.stride_d;
    q.tmap_sfa = plan->sf_maps[0];
    q.tmap_sfb = plan->sf_maps[1];
    q.tensor_scales = nv ? tensor_scales : nullptr;
    q.chunks = chunks;
    q.sf_stage_bytes = (uint32_t)(3 * chunks * 512);
    q.sf_ring_offset = (uint32_t)info.stages * (p.stage_bytes_a + p.stage_bytes_b);
    e = dgb::launch_mx(q, mx_kind(d), cg, d.dtype_d, info.grid, (size_t)info.smem_bytes, stream);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

// Panels for gemm_run_host: rows of A and D (one batch entry), or batch
// entries; each panel large enough that its GEMM keeps the GPU busy.
static int host_panels(const gemm_desc_t& d, int64_t* unit0) {
    const int64_t units = d.batch > 1 ? d.batch : d.M;
    int64_t want = d.batch > 1 ? d.batch / 64 : d.M / 1024;
    if (want > kHostPanels) want = kHostPanels;
    if (want < 2 || d.K == 0) return 1;
    const int64_t align = d.batch > 1 ? 1 : 256;          // whole pair-tile row bands
    int n = 0;
    unit0[0] = 0;
    for (int i = 1; i <= want; ++i) {
        int64_t u = std::min(units, round_up(ceil_div(units * i, want), align));
        if (u > unit0[n]) unit0[++n] = u;
    }
    unit0[n] = units;
    return n;
}

static gemm_status_t host_pipe_setup(gemm_plan_t plan) {
    HostPipe* hp = new (std::nothrow) HostPipe();
    if (!hp) return GEMM_ERR_RESOURCES;
    cudaError_t e;
    const gemm_desc_t& d = plan->desc;
    int64_t unit0[kHostPanels + 1];
    const int panels = host_panels(d, unit0);
    auto fail = [&](cudaError_t err) { host_pipe_free(hp); return cuda_fail(err); };
    if (panels > 1) {
        const bool by_batch = d.batch > 1;
        int n = 0;
        if (!by_batch && d.M >= 4096 && d.N >= 2048) {
            // The copy-out is the long pole (D is the largest operand in and out
            // of the GPU).  Keep it busy from early on: a first block of 40 % of
            // A's rows, multiplied against B's four column quarters as each
            // lands (while B streams in, each quarter yields a block of D about
            // as large as the next quarter of B), then the remaining rows in
            // panels against all of B.
            const int64_t r0 = std::min(d.M, round_up(d.M * 2 / 5, 256));
            int64_t q_prev = 0;
            for (int q = 1; q <= 4; ++q) {
                const int64_t qe = q == 4 ? d.N : std::min(d.N, round_up(ceil_div(d.N * q, 4), 256));
                if (qe > q_prev) hp->job[n++] = HostJob{0, r0, q_prev, qe - q_prev, q_prev == 0, q_prev, qe - q_prev, nullptr};
                q_prev = qe;
            }
            const int64_t rest = d.M - r0;
            const int64_t np = std::min<int64_t>(kHostJobs - n, std::max<int64_t>(1, ceil_div(rest, 1024)));
            int64_t u_prev = r0;
            for (int64_t i = 1; i <= np && rest > 0; ++i) {
                const int64_t ue = i == np ? d.M : std::min(d.M, r0 + round_up(ceil_div(rest * i, np), 256));
                if (ue > u_prev) hp->job[n++] = HostJob{u_prev, ue - u_prev, 0, d.N, true, 0, 0, nullptr};
                u_prev = ue;
            }
        } else {
            // Row panels: the first panel multiplies against the two halves of B's
            // rows separately, so that its first half of D starts copying out once
            // A's first rows and half of B are in, not all of B.
            const int64_t ns = round_up(d.N / 2, 256);
            const bool split = !by_batch && d.N >= 1024 && ns < d.N;
            for (int i = 0; i < panels; ++i) {
                const int64_t u0 = unit0[i], nu = unit0[i + 1] - u0;
                if (split && i == 0) {
                    hp->job[n++] = HostJob{u0, nu, 0, ns, true, 0, ns, nullptr};
                    hp->job[n++] = HostJob{u0, nu, ns, d.N - ns, false, ns, d.N - ns, nullptr};
                } else {
                    hp->job[n++] = HostJob{u0, nu, 0, d.N, true, 0, (!by_batch && !split && i == 0) ? d.N : 0,
                                           nullptr};
                }
            }
        }
        hp->jobs = n;
        if ((e = cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking)) != cudaSuccess) return fail(e);
        if ((e = cudaEventCreateWithFlags(&hp->ev_start, cudaEventDisableTiming)) != cudaSuccess) return fail(e);
        if ((e = cudaEventCreateWithFlags(&hp->ev_done, cudaEventDisableTiming)) != cudaSuccess) return fail(e);
        for (int i = 0; i < hp->jobs; ++i) {
            HostJob& jb = hp->job[i];
            if ((e = cudaEventCreateWithFlags(&hp->ev_a[i], cudaEventDisableTiming)) != cudaSuccess) return fail(e);
            if ((e = cudaEventCreateWithFlags(&hp->ev_g[i], cudaEventDisableTiming)) != cudaSuccess) return fail(e);
            gemm_desc_t pd = d;
            if (by_batch) pd.batch = jb.nu; else pd.M = jb.nu;
            pd.N = jb.nn;
            pd.flags |= GEMM_FLAG_NO_STREAM_K;       // no workspace: data-parallel tiles
            Resolved r;
            gemm_status_t s = resolve(&pd, &r);
            gemm_plan_s* sp = s == GEMM_OK ? new (std::nothrow) gemm_plan_s() : nullptr;
            if (s == GEMM_OK && !sp) s = GEMM_ERR_RESOURCES;
            if (s == GEMM_OK) {
                jb.sub = sp;
                sp->maps_valid = false;
                sp->desc = r.d;
                sp->props = plan->props;
                sp->device = plan->device;
                sp->status = plan->status;           // shared: gemm_sync_status sees every job
                s = ::plan(r.d, plan->props, &sp->info);
            }
            if (s == GEMM_OK) s = cap_resident(r.d, &sp->info);
            if (s != GEMM_OK) { host_pipe_free(hp); return s; }
            sp->info.stream_k_tiles = 0;
            sp->info.workspace_bytes = 0;
        }
    }
    hp->ready = true;
    plan->pipe = hp;
    return GEMM_OK;
}

gemm_status_t gemm_run_host(gemm_plan_t plan, const void* hA, const void* hB, void* hD, const float* hsa,
                            const float* hsb, void* dA, void* dB, void* dD, float* dsa, float* dsb,
                            gemm_stream_t stream_) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const gemm_desc_t& d = plan->desc;
    if (hw_scaled(d.scale_mode)) return GEMM_ERR_UNSUPPORTED;
    if (d.M == 0 || d.N == 0 || d.batch == 0) return GEMM_OK;
    if (!hD || !dD) return GEMM_ERR_INVALID_ARG;
    const bool ka = d.major_a == GEMM_K_MAJOR, kb = d.major_b == GEMM_K_MAJOR;
    const bool scaled = d.scale_mode != GEMM_SCALE_NONE;
    const int64_t eb_a = elem_bytes(d.dtype_a), eb_b = elem_bytes(d.dtype_b), eb_d = elem_bytes(d.dtype_d);
    // extent in elements of one batch entry of each operand: last element index + 1
    const int64_t one_a = ka ? (d.M - 1) * d.lda + d.K : (d.K - 1) * d.lda + d.M;
    const int64_t one_b = kb ? (d.N - 1) * d.ldb + d.K : (d.K - 1) * d.ldb + d.N;
    const int64_t one_d = (d.M - 1) * d.ldd + d.N;
    const int64_t ext_b = (d.batch - 1) * d.stride_b + one_b;
    const int64_t kblk = ceil_div(d.K, 128);
    const int64_t one_sa = (d.M - 1) * d.ld_sa + kblk;
    const int64_t ext_sb = (d.batch - 1) * d.stride_sb + (ceil_div(d.N, 128) - 1) * d.ld_sb + kblk;
    cudaError_t e;
    if (d.K > 0) {
        if (!hA || !hB || !dA || !dB) return GEMM_ERR_INVALID_ARG;
        if (scaled && (!hsa || !hsb || !dsa || !dsb)) return GEMM_ERR_INVALID_ARG;
    }
    if (!plan->pipe) {
        gemm_status_t s = host_pipe_setup(plan);
        if (s != GEMM_OK) return s;
    }
    HostPipe& hp = *plan->pipe;

    if (hp.jobs == 0) {
        // One piece: copy in, multiply, copy out, in stream order.
        if (d.K > 0) {
            const int64_t ext_a = (d.batch - 1) * d.stride_a + one_a;
            if ((e = cudaMemcpyAsync(dA, hA, (size_t)(ext_a * eb_a), cudaMemcpyHostToDevice, stream)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = cudaMemcpyAsync(dB, hB, (size_t)(ext_b * eb_b), cudaMemcpyHostToDevice, stream)) != cudaSuccess)
                return cuda_fail(e);
            if (scaled) {
                const int64_t ext_sa = (d.batch - 1) * d.stride_sa + one_sa;
                if ((e = cudaMemcpyAsync(dsa, hsa, (size_t)ext_sa * 4, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
                    return cuda_fail(e);
                if ((e = cudaMemcpyAsync(dsb, hsb, (size_t)ext_sb * 4, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
                    return cuda_fail(e);
            }
        }
        gemm_status_t s = gemm_run(plan, dA, dB, dD, scaled ? dsa : nullptr, scaled ? dsb : nullptr, stream_);
        if (s != GEMM_OK) return s;
        const int64_t ext_d = (d.batch - 1) * d.stride_d + one_d;
        if ((e = cudaMemcpyAsync(hD, dD, (size_t)(ext_d * eb_d), cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
            return cuda_fail(e);
        return GEMM_OK;
    }

    // Jobs (row or batch-entry panels): the copy-in stream brings, ahead of
    // each job, the rows of B and of A it is the first to need; the job's GEMM
    // runs on `stream` once they landed, and its block of D goes back on the
    // copy-out stream while later jobs still copy in or multiply.  Events keep
    // the whole call ordered on `stream`.
    const bool by_batch = d.batch > 1;
    auto cu = [](const void* p, int64_t bytes) { return static_cast<const char*>(p) + bytes; };
    auto mu = [](void* p, int64_t bytes) { return static_cast<char*>(p) + bytes; };
    auto h2d = [&](void* dst, const void* src, int64_t bytes) {
        return cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyHostToDevice, hp.h2d);
    };
    // rows [r0, r0+nr) of a row-per-M/N operand with leading dim ld (K-major) or
    // columns of a [K][ld] operand (MN-major)
    auto h2d_rows = [&](void* dbase, const void* hbase, bool kmaj, int64_t ld, int64_t eb, int64_t r0,
                        int64_t nr) -> cudaError_t {
        if (kmaj)
            return cudaMemcpy2DAsync(mu(dbase, r0 * ld * eb), (size_t)(ld * eb), cu(hbase, r0 * ld * eb),
                                     (size_t)(ld * eb), (size_t)(d.K * eb), (size_t)nr, cudaMemcpyHostToDevice,
                                     hp.h2d);
        return cudaMemcpy2DAsync(mu(dbase, r0 * eb), (size_t)(ld * eb), cu(hbase, r0 * eb), (size_t)(ld * eb),
                                 (size_t)(nr * eb), (size_t)d.K, cudaMemcpyHostToDevice, hp.h2d);
    };
    const int64_t one_sb = (ceil_div(d.N, 128) - 1) * d.ld_sb + kblk;
    if ((e = cudaEventRecord(hp.ev_start, stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(hp.h2d, hp.ev_start, 0)) != cudaSuccess) return cuda_fail(e);
    for (int k = 0; k < hp.jobs; ++k) {
        const HostJob& jb = hp.job[k];
        int64_t off_a, off_b, off_d, off_sa, off_sb;   // element offsets of the job's operands
        if (by_batch) {
            off_a = jb.u0 * d.stride_a;
            off_b = jb.u0 * d.stride_b;
            off_d = jb.u0 * d.stride_d;
            off_sa = jb.u0 * d.stride_sa;
            off_sb = jb.u0 * d.stride_sb;
            if ((e = h2d(mu(dA, off_a * eb_a), cu(hA, off_a * eb_a), ((jb.nu - 1) * d.stride_a + one_a) * eb_a)) !=
                cudaSuccess)
                return cuda_fail(e);
            if ((e = h2d(mu(dB, off_b * eb_b), cu(hB, off_b * eb_b), ((jb.nu - 1) * d.stride_b + one_b) * eb_b)) !=
                cudaSuccess)
                return cuda_fail(e);
            if (scaled) {
                if ((e = h2d(dsa + off_sa, hsa + off_sa, ((jb.nu - 1) * d.stride_sa + one_sa) * 4)) != cudaSuccess)
                    return cuda_fail(e);
                if ((e = h2d(dsb + off_sb, hsb + off_sb, ((jb.nu - 1) * d.stride_sb + one_sb) * 4)) != cudaSuccess)
                    return cuda_fail(e);
            }
        } else {
            off_a = ka ? jb.u0 * d.lda : jb.u0;
            off_b = kb ? jb.n0 * d.ldb : jb.n0;
            off_d = jb.u0 * d.ldd + jb.n0;
            off_sa = jb.u0 * d.ld_sa;
            off_sb = (jb.n0 / 128) * d.ld_sb;
            if (jb.bn > 0) {
                if ((e = h2d_rows(dB, hB, kb, d.ldb, eb_b, jb.b0, jb.bn)) != cudaSuccess) return cuda_fail(e);
                if (scaled) {
                    const int64_t q0 = jb.b0 / 128, nq = ceil_div(jb.b0 + jb.bn, 128) - q0;
                    if ((e = h2d(dsb + q0 * d.ld_sb, hsb + q0 * d.ld_sb, ((nq - 1) * d.ld_sb + kblk) * 4)) !=
                        cudaSuccess)
                        return cuda_fail(e);
                }
            }
            if (jb.copy_a) {
                if ((e = h2d_rows(dA, hA, ka, d.lda, eb_a, jb.u0, jb.nu)) != cudaSuccess) return cuda_fail(e);
                if (scaled &&
                    (e = h2d(dsa + off_sa, hsa + off_sa, ((jb.nu - 1) * d.ld_sa + kblk) * 4)) != cudaSuccess)
                    return cuda_fail(e);
            }
        }
        if ((e = cudaEventRecord(hp.ev_a[k], hp.h2d)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(stream, hp.ev_a[k], 0)) != cudaSuccess) return cuda_fail(e);
        gemm_status_t s = gemm_run(jb.sub, cu(dA, off_a * eb_a), cu(dB, off_b * eb_b), mu(dD, off_d * eb_d),
                                   scaled ? dsa + off_sa : nullptr, scaled ? dsb + off_sb : nullptr, stream_);
        if (s != GEMM_OK) return s;
        if ((e = cudaEventRecord(hp.ev_g[k], stream)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(hp.d2h, hp.ev_g[k], 0)) != cudaSuccess) return cuda_fail(e);
        if (by_batch)
            e = cudaMemcpyAsync(mu(hD, off_d * eb_d), cu(dD, off_d * eb_d), (size_t)(((jb.nu - 1) * d.stride_d + one_d) * eb_d),
                                cudaMemcpyDeviceToHost, hp.d2h);
        else
            e = cudaMemcpy2DAsync(mu(hD, off_d * eb_d), (size_t)(d.ldd * eb_d), cu(dD, off_d * eb_d),
                                  (size_t)(d.ldd * eb_d), (size_t)(jb.nn * eb_d), (size_t)jb.nu,
                                  cudaMemcpyDeviceToHost, hp.d2h);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if ((e = cudaEventRecord(hp.ev_done, hp.d2h)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(stream, hp.ev_done, 0)) != cudaSuccess) return cuda_fail(e);
    return GEMM_OK;
}

gemm_status_t gemm_sync_status(gemm_plan_t plan, gemm_stream_t stream_, gemm_device_error_t* out) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    gemm_device_error_t rec;
    cudaError_t e;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpy(&rec, plan->status, sizeof(rec), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if (rec.code != 0 && (e = cudaMemset(plan->status, 0, sizeof(rec))) != cudaSuccess) return cuda_fail(e);
    if (out) *out = rec;
    return rec.code == 0 ? GEMM_OK : (gemm_status_t)rec.code;
}

gemm_status_t gemm_run_noalloc(const gemm_desc_t* desc, const void* A, const void* B, void* D,
                               const float* scale_a, const float* scale_b, gemm_stream_t stream_,
                               gemm_device_error_t* status_out) {
    if (!desc) return GEMM_ERR_INVALID_ARG;
    Resolved r;
    gemm_status_t s = resolve(desc, &r);
    if (s != GEMM_OK) return s;
    if (hw_scaled(r.d.scale_mode)) return GEMM_ERR_UNSUPPORTED;
    // The only device memory the kernels use beyond A, B, D and the scales is
    // their error record; it must fit the static array.
    if (sizeof(gemm_device_error_t) > sizeof(g_noalloc_scratch)) return GEMM_ERR_RESOURCES;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { g_last_cuda_error = (int)e; return GEMM_ERR_NO_DEVICE; }
    gemm_plan_s p{};
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
    p.props.sm_count = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return cuda_fail(e);
    p.props.smem_optin_bytes = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
    p.props.cc_major = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
    p.props.cc_minor = v;
    if (p.props.cc_major != 10 || p.props.cc_minor != 3) return GEMM_ERR_NO_DEVICE;
    r.d.flags |= GEMM_FLAG_NO_STREAM_K;   // no workspace here: data-parallel tiles only, one cluster per tile at most
    s = plan(r.d, p.props, &p.info);
    if (s != GEMM_OK) return s;
    if ((s = cap_resident(r.d, &p.info)) != GEMM_OK) return s;
    p.info.stream_k_tiles = 0;
    p.info.workspace_bytes = 0;
    void* record = nullptr;
    if ((s = noalloc_address(dev, &record)) != GEMM_OK) return s;
    p.desc = r.d;
    p.device = dev;
    p.status = static_cast<gemm_device_error_t*>(record);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    noalloc_clear_kernel<<<1, 32, 0, stream>>>((unsigned)sizeof(gemm_device_error_t));
    if ((e = cudaGetLastError()) != cudaSuccess) {
        noalloc_forget(dev);
        return cuda_fail(e);
    }
    s = gemm_run(&p, A, B, D, scale_a, scale_b, stream_);
    if (s == GEMM_ERR_CUDA) noalloc_forget(dev);      // e.g. a context reset moved the array
    if (s != GEMM_OK || status_out == nullptr) return s;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpy(status_out, record, sizeof(*status_out), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    return status_out->code == 0 ? GEMM_OK : (gemm_status_t)status_out->code;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
    if (!plan) return GEMM_OK;
    cudaError_t e = cudaSuccess;
    host_pipe_free(plan->pipe);
    if (plan->status) e = cudaFree(plan->status);   // one allocation holds the workspace too
    delete plan;
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE";
    case GEMM_ERR_RESOURCES: return "GEMM_ERR_RESOURCES";
    default: return "GEMM_ERR_UNKNOWN";
    }
}

int gemm_last_cuda_error(void) { return g_last_cuda_error; }

int gemm_version(void) { return kVersion; }

}  // extern "C"
