// kernels_fp8.cu -- persistent tcgen05 GEMM for block-scaled e4m3 inputs.
//
//   D[m][n] = sum_kb  sA[m][kb] * sB[n/128][kb] * sum_{k in block kb} qA[m][k] * qB[n][k]
//
// Every 1x128 block of a row of A and every 128x128 block of B carries its own
// fp32 scale ("Hopper and Blackwell GEMM", concept "FP8 and FP4, with block
// scaling").  Those scales are arbitrary fp32 values, which the hardware's
// block-scaled MMA kinds (E8M0 scales per 32 elements) cannot express, so the
// scales are applied in software, once per 128-deep K block:
//
//   warps 0 and 2    : TMA producers (shared loop), one 128-deep K block per
//                      ring stage (one 128-byte swizzle row of e4m3): warp 0
//                      copies A and posts the stage's expected bytes, warp 2
//                      copies B.
//   warp 1           : allocates tensor memory; the pair leader's warp runs the
//                      MMA loop, one elected lane issuing four K32 tcgen05.mma
//                      kind::f8f6f4 per block into a
//                      fresh partial P[j mod PB] (j counts blocks over all tiles)
//                      and commits them to the stage's empty barrier.
//   warp 3           : idle.
//   warps 4..11      : promotion and epilogue.  Warp w owns TMEM lanes
//                      32*(w mod 4).. (its 32 rows) and 128 of the tile's 256
//                      columns (half (w-4)/4, exactly one 128-row block of B).
//                      Per block: read its 32x128 slice of P with tcgen05.ld,
//                      give the partial back, and accumulate
//                      acc += P * (sA[row][kb] * sB[col/128][kb]) in registers.
//                      After the tile's last block: convert, stage in swizzled
//                      shared memory, TMA store.
//
// Two or four partial buffers let the tensor core compute block j+1 while the
// epilogue warps promote block j.  Waits are bounded as in the 16-bit kernel.
//
// Registers: a promotion thread holds its row's 128 fp32 accumulators, and the
// read-back of a partial is only fast with several tcgen05.ld in flight per
// warp (one 16-column load at a time leaves the tensor core idle about half of
// each block on GB300).  Twelve warps launch with 168 registers each; the first
// warpgroup (producers, MMA) gives registers back (setmaxnreg) down to
// kFp8RegsLow and the two promotion warpgroups take them up to kFp8RegsHigh.
//
// One barrier wait per block in the MMA thread.  In a thread with tcgen05.mma
// in flight every mbarrier probe costs about 230 cycles (22 in a thread
// without; measured on GB300), and four K32 MMAs of a 128 x 256 block take
// 512 cycles, so the MMA thread cannot afford to wait for both the stage's
// data and the partial's release.  Block j's full barrier therefore carries
// both: the producer's arrival with the expected bytes, plus one arrival from
// every promotion warp of the pair once it has read partial j mod PB back for
// block j - PB (the first PB blocks get theirs up front).  The promotion warps
// learn that a block's MMAs completed from the stage's empty barrier (the
// MMA's single commit per block).  With the ring at least as deep as the
// partial count, neither barrier can run a phase ahead of the warps that use it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace dgb {

// acc[0..1] += x[0..1] * s with one packed fp32 FMA (round to nearest, as two fmaf)
__device__ __forceinline__ void fma2_rn(float& a0, float& a1, uint32_t x0, uint32_t x1, float s) {
    asm("{\n\t.reg .b64 a, x, s;\n\t"
        "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\tmov.b64 s, {%4, %4};\n\t"
        "fma.rn.f32x2 a, x, s, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(x0), "r"(x1), "f"(s));
}

constexpr int kFp8TileK = 128;              // e4m3 elements per ring stage (128 B)
constexpr int kFp8EpiWarps = 8;
constexpr int kFp8EpiWarp0 = 4;                  // first promotion warp: warpgroups 1 and 2
constexpr int kFp8Threads = 32 * (kFp8EpiWarp0 + kFp8EpiWarps);
constexpr int kFp8LaunchRegs = 168;              // what 12 warps get: 3 per sub-partition's 16K registers
constexpr int kFp8RegsLow = 72;                  // producers and MMA warpgroup
constexpr int kFp8RegsHigh = 216;                // promotion warpgroups
static_assert(128 * kFp8RegsLow + 32 * kFp8EpiWarps * kFp8RegsHigh <= kFp8Threads * kFp8LaunchRegs,
              "register shares exceed the launch's pool");
constexpr uint32_t kFp8StagingBytes = 32 * 128;   // one buffer per epilogue warp

// COLS: columns of the tile each promotion warp owns (tile_n / 2): 128 for
// 256-wide tiles, 64 for 128-wide tiles.  The tile has 512 / tile_n partial
// buffers in TMEM (2 or 4), so the MMA can run that many blocks minus one
// ahead of the promotion.
template <int CG, int OUT, int COLS>
__global__ void __launch_bounds__(kFp8Threads, 1) fp8_block_kernel(const __grid_constant__ PersistentParams p) {
    constexpr int kOutBytes = (OUT == GEMM_F32) ? 4 : 2;
    constexpr int kChunkCols = 128 / kOutBytes;          // columns per 128-byte staging row
    constexpr int kChunks = COLS / kChunkCols;           // chunks per warp's columns
    // hand a partial back before the last FMAs (with 128 columns per warp the
    // compiler then spills)
    constexpr bool kEarlyRelease = COLS == 64;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int S = p.stages;
    const uint32_t stage_bytes = p.stage_bytes_a + p.stage_bytes_b;
    uint8_t* ring = smem;
    uint8_t* staging = ring + (size_t)S * stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + kFp8EpiWarps * kFp8StagingBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8u * S;
    const int PB = p.tmem_stages;                // partial buffers (2 or 4), PB <= S
    const uint32_t drain_bar = empty0 + 8u * S;

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1 + CG * kFp8EpiWarps);   // producer + partial released
            mbar_init(empty0 + 8u * s, 1);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&p.tmap_a);
        prefetch_tensormap(&p.tmap_b);
        prefetch_tensormap(&p.tmap_d);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the previous kernel of the stream; its results are
    // visible from here on.  The next GEMM may be launched now: its CTAs take
    // SMs as this grid's CTAs leave and wait in griddep_wait.
    griddep_wait();
    griddep_launch_dependents();

    const int cluster_id = blockIdx.x / CG;
    const int num_clusters = gridDim.x / CG;
    const uint64_t tmo = p.timeout_ns;

    // Each role raises or lowers its registers first thing, so that the code
    // that follows is compiled against its own share.
    if (warp < kFp8EpiWarp0) {
        setmaxnreg_dec<kFp8RegsLow>();
        if (warp == 0) {
            producer_loop<CG, 1, 1, kPartA>(p, ring, stage_bytes, kFp8TileK, full0, empty0, abort_flag, rank,
                                            cluster_id, num_clusters);
            __syncwarp();
        } else if (warp == 2) {
            producer_loop<CG, 1, 1, kPartB0>(p, ring, stage_bytes, kFp8TileK, full0, empty0, abort_flag, rank,
                                             cluster_id, num_clusters);
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp runs the loop and waits; one lane, elected once, issues
            // every MMA and commit (a commit tracks only its own thread's MMAs).
            if (leader) {
                int stage = 0;
                uint32_t phase = 0;
                int pb = 0;
                bool aborted = false;
                bool issued_any = false;
                const bool issuer = elect_one();
                for (int t = cluster_id; t < p.num_tiles && !aborted; t += num_clusters) {
                    for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                        // completes once the block's bytes landed and its partial is free
                        if (!wait_phase_warp<false>(full0 + 8u * stage, phase, abort_flag, tmo, p.status, kRoleMma,
                                                    stage, t)) {
                            aborted = true;
                            break;
                        }
                        if (issuer) {
                            tc_fence_after();
                            const uint32_t sa = smem_u32(ring + (size_t)stage * stage_bytes);
                            const uint32_t sb = sa + p.stage_bytes_a;
                            // K-major: the next K32 is 32 bytes along the row (+2 in the
                            // address field); MN-major: 32 k-rows of 128 B on (+256), atoms
                            // along M/N one 16 KB box apart
                            constexpr uint32_t kBox = 128u * kFp8TileK;
                            const uint64_t da = p.mn_major_a ? smem_desc_sw128_mn_lbo(sa, kBox) : smem_desc_sw128(sa);
                            const uint64_t db = p.mn_major_b ? smem_desc_sw128_mn_lbo(sb, kBox) : smem_desc_sw128(sb);
                            const uint64_t step_a = p.mn_major_a ? 256u : 2u;
                            const uint64_t step_b = p.mn_major_b ? 256u : 2u;
                            const uint32_t d_tmem = tmem_base + (uint32_t)(pb * p.tile_n);
    #pragma unroll
                            for (int kk = 0; kk < kFp8TileK / 32; ++kk)
                                mma_f8<CG>(d_tmem, da + step_a * kk, db + step_b * kk, p.idesc, kk != 0);
                            issued_any = true;
                            commit_to<CG>(empty0 + 8u * stage);   // stage free, partial written
                        }
                        __syncwarp();
                        if (++stage == S) { stage = 0; phase ^= 1u; }
                        if (++pb == PB) pb = 0;
                    }
                }
                if (aborted && issuer && issued_any) {
                    commit_local<CG>(drain_bar);
                    wait_phase_drain(drain_bar, 0, tmo);
                }
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kFp8RegsHigh>();
        // ------------------------------------------------------------ promotion + epilogue
        // D is written once and never read back here: let it leave L2 first.
        const bool stream_d = (p.l2_hints & kHintStreamD) != 0;
        const uint64_t pol_d = l2_policy_evict_first();
        const int wq = warp & 3;                  // TMEM lane quarter
        const int half = (warp - kFp8EpiWarp0) >> 2;   // which COLS columns of the tile
        uint8_t* buf = staging + (warp - kFp8EpiWarp0) * kFp8StagingBytes;
        int pb = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        // blocks this CTA has still to promote, over all its tiles (the plan
        // keeps the count within int)
        const int my_tiles = cluster_id < p.num_tiles ? (p.num_tiles - 1 - cluster_id) / num_clusters + 1 : 0;
        int left = my_tiles * p.num_k_blocks;
        // the first PB blocks find their partials free
        if (lane == 0)
            for (int i = 0; i < PB && i < left; ++i) arrive_leader<CG>(full0 + 8u * i);
        for (int t = cluster_id; t < p.num_tiles && !aborted; t += num_clusters) {
            int b, mb, nb;
            tile_coords(p, t, b, mb, nb);
            const int m_warp = mb * (128 * CG) + (int)rank * 128 + wq * 32;
            const int row = m_warp + lane;
            const int col0 = nb * p.tile_n + half * COLS;   // inside one 128-column block of B's scales
            const bool row_ok = row < p.M;
            const bool cols_ok = col0 < p.N;
            const float* sa_row = p.scale_a + (size_t)b * p.stride_sa + (size_t)(row_ok ? row : 0) * p.ld_sa;
            const float* sb_blk = p.scale_b + (size_t)b * p.stride_sb + (size_t)(cols_ok ? col0 / 128 : 0) * p.ld_sb;
            float acc[COLS];
#pragma unroll
            for (int i = 0; i < COLS; ++i) acc[i] = 0.0f;
            // Scales are loaded two blocks ahead so that their L2 latency hides
            // behind the promotion of the blocks in between.
            const bool scaled = row_ok && cols_ok;
            const int nkb = p.num_k_blocks;
            float sa0 = scaled ? __ldg(sa_row) : 0.0f, sb0 = scaled ? __ldg(sb_blk) : 0.0f;
            float sa1 = (scaled && nkb > 1) ? __ldg(sa_row + 1) : 0.0f;
            float sb1 = (scaled && nkb > 1) ? __ldg(sb_blk + 1) : 0.0f;
            for (int kb = 0; kb < nkb; ++kb) {
                const float s = sa0 * sb0;
                sa0 = sa1;
                sb0 = sb1;
                sa1 = (scaled && kb + 2 < nkb) ? __ldg(sa_row + kb + 2) : 0.0f;
                sb1 = (scaled && kb + 2 < nkb) ? __ldg(sb_blk + kb + 2) : 0.0f;
                const bool ok = wait_phase_warp<false>(empty0 + 8u * stage, phase, abort_flag, tmo, p.status,
                                                       kRoleEpilogue, stage, t);
                if (!ok) { aborted = true; break; }
                tc_fence_after();
                // partial pb is free again once this warp's last tcgen05.ld of it
                // completed: count towards block j + PB's full barrier (64-column
                // warps before their last FMAs, which block j + PB need not wait for)
                if (cols_ok) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(pb * p.tile_n + half * COLS);
                    // two 16-column loads in flight, one wait per pair: on GB300
                    // faster than four in flight
#pragma unroll
                    for (int c = 0; c < COLS / 16; c += 2) {
                        uint32_t r0[16], r1[16];
                        tmem_ld_32x32b_x16(taddr + c * 16, r0);
                        tmem_ld_32x32b_x16(taddr + c * 16 + 16, r1);
                        tmem_wait_ld();
                        tmem_reg_fence16(r0);
                        tmem_reg_fence16(r1);
                        if (kEarlyRelease && c + 2 == COLS / 16) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0 && left > PB)
                                arrive_leader<CG>(full0 + 8u * (stage + PB < S ? stage + PB : stage + PB - S));
                        }
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            fma2_rn(acc[c * 16 + i], acc[c * 16 + i + 1], r0[i], r0[i + 1], s);
                            fma2_rn(acc[c * 16 + 16 + i], acc[c * 16 + 17 + i], r1[i], r1[i + 1], s);
                        }
                    }
                }
                if (!kEarlyRelease || !cols_ok) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0 && left > PB)
                        arrive_leader<CG>(full0 + 8u * (stage + PB < S ? stage + PB : stage + PB - S));
                }
                --left;
                if (++pb == PB) pb = 0;
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
            if (aborted || !cols_ok || m_warp >= p.M) continue;
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int x = col0 + c * kChunkCols;
                if (x >= p.N) break;
                // 16-byte piece j of this thread's row, packed straight from the accumulators
                auto piece = [&](int j) -> uint4 {
                    if constexpr (OUT == GEMM_F32) {
                        const int e = c * 32 + 4 * j;
                        return make_uint4(__float_as_uint(acc[e]), __float_as_uint(acc[e + 1]),
                                          __float_as_uint(acc[e + 2]), __float_as_uint(acc[e + 3]));
                    } else {
                        const int e = c * 64 + 8 * j;
                        return make_uint4(pack2<OUT>(acc[e], acc[e + 1]), pack2<OUT>(acc[e + 2], acc[e + 3]),
                                          pack2<OUT>(acc[e + 4], acc[e + 5]), pack2<OUT>(acc[e + 6], acc[e + 7]));
                    }
                };
                if (chunk_needs_clipped_store<kOutBytes>(x, kChunkCols, p.N)) {
                    // ragged right edge inside a 16-byte granule: plain stores up to N
                    const int row = m_warp + lane;
                    if (row < p.M)
                        store_segment_clipped<kOutBytes>(static_cast<uint8_t*>(p.d_ptr) +
                                                             ((size_t)b * p.stride_d + (size_t)row * p.ldd + x) *
                                                                 kOutBytes,
                                                         p.N - x, piece);
                    continue;
                }
                // single staging buffer: the previous store must have read it
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = piece(j);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (stream_d) {
                        if (p.batched) tma_store_3d_hint(&p.tmap_d, smem_u32(buf), x, m_warp, b, pol_d);
                        else tma_store_2d_hint(&p.tmap_d, smem_u32(buf), x, m_warp, pol_d);
                    } else {
                        if (p.batched) tma_store_3d(&p.tmap_d, smem_u32(buf), x, m_warp, b);
                        else tma_store_2d(&p.tmap_d, smem_u32(buf), x, m_warp);
                    }
                    bulk_commit_group();
                }
            }
        }
        // Abort while waiting for block j (at `stage`, `left` blocks to go):
        // give this warp's arrival to the blocks it has not released yet that
        // the ring can hold, j + PB .. j + S - 1, so that a stage whose copies
        // are in flight still completes and the producer's drain sees them
        // land.  Their previous phases (blocks < j) are complete, and the warp
        // arrives at most once per phase: no barrier is over-arrived (a phase
        // still waiting for bytes must get no arrival beyond its count).
        if (aborted && lane == 0)
            for (int x = PB; x < S && x < left; ++x) {
                const int rs = stage + x < S ? stage + x : stage + x - S;
                arrive_leader<CG>(full0 + 8u * rs);
            }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, (uint32_t)p.tmem_cols);
    }
}

template <int CG>
static cudaLaunchConfig_t fp8_config(size_t smem, int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kFp8Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// The kernel's setmaxnreg shares assume it was built with kFp8LaunchRegs
// registers per thread: with fewer the promotion warps' increase could never
// be granted, so such a build is refused rather than launched.
template <typename Kern>
static bool fp8_regs_ok(Kern kern) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kern) != cudaSuccess) return false;
    return a.numRegs == kFp8LaunchRegs;
}

template <int CG, int OUT, int COLS>
static cudaError_t fp8_launch_typed(const PersistentParams& p, int grid, size_t smem, cudaStream_t stream) {
    auto kern = fp8_block_kernel<CG, OUT, COLS>;
    if (!fp8_regs_ok(kern)) return cudaErrorInvalidConfiguration;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = fp8_config<CG>(smem, grid, stream, attr);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CG, int OUT, int COLS>
static int fp8_clusters_typed(size_t smem) {
    auto kern = fp8_block_kernel<CG, OUT, COLS>;
    if (!fp8_regs_ok(kern)) return 0;
    static std::atomic<int> smem_set[kMaxDevices];
    if (ensure_smem_limit(kern, smem, smem_set) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = fp8_config<CG>(smem, CG, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

#define DGB_FP8_DISPATCH_OUT(FN, CGV, COLSV, ...)                                        \
    switch (dtype_d) {                                                                   \
    case GEMM_F32: return FN<CGV, GEMM_F32, COLSV>(__VA_ARGS__);                         \
    case GEMM_BF16: return FN<CGV, GEMM_BF16, COLSV>(__VA_ARGS__);                       \
    case GEMM_F16: return FN<CGV, GEMM_F16, COLSV>(__VA_ARGS__);                         \
    default: break;                                                                      \
    }
#define DGB_FP8_DISPATCH(FN, ...)                                                        \
    if (cta_group == 1 && tile_n == 256) { DGB_FP8_DISPATCH_OUT(FN, 1, 128, __VA_ARGS__) } \
    if (cta_group == 1 && tile_n == 128) { DGB_FP8_DISPATCH_OUT(FN, 1, 64, __VA_ARGS__) }  \
    if (cta_group == 2 && tile_n == 256) { DGB_FP8_DISPATCH_OUT(FN, 2, 128, __VA_ARGS__) } \
    if (cta_group == 2 && tile_n == 128) { DGB_FP8_DISPATCH_OUT(FN, 2, 64, __VA_ARGS__) }

cudaError_t launch_fp8_block(const PersistentParams& p, int cta_group, int dtype_d, int grid, size_t smem_bytes,
                             cudaStream_t stream) {
    const int tile_n = p.tile_n;
    DGB_FP8_DISPATCH(fp8_launch_typed, p, grid, smem_bytes, stream)
    return cudaErrorInvalidValue;
}

int fp8_max_active_clusters(int cta_group, int tile_n, int dtype_d, size_t smem_bytes) {
    DGB_FP8_DISPATCH(fp8_clusters_typed, smem_bytes)
    return 0;
}

}  // namespace dgb
