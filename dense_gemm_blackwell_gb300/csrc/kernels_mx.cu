// kernels_mx.cu -- persistent tcgen05 GEMM with hardware block scaling:
// MXFP8 (E4M3 / E5M2 elements, one E8M0 scale per 32 K elements), MXFP4 (E2M1
// elements packed two per byte, E8M0 per 32) and NVFP4 (E2M1, one E4M3 scale
// per 16 and one fp32 scale per tensor).
//
//   D[m][n] = tA * tB * sum_k (qA[m][k] * sA[m][k/V]) * (qB[n][k] * sB[n][k/V])
//
// ("Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling":
// the tensor core applies the block scales inside tcgen05.mma .kind::mxf8f6f4,
// .kind::mxf4 or .kind::mxf4nvf4; tA = tB = 1 for the MX formats.)
//
// Roles (12 warps):
//   warp 0     : TMA producer of A; posts the operand bytes of each stage
//   warp 1     : allocates tensor memory; the pair leader's warp runs the MMA
//                loop: per ring stage it copies the stage's scale slabs into
//                tensor memory (tcgen05.cp) and issues four block-scaled MMAs
//                per 128-byte K atom, then commits the stage back
//   warp 2     : TMA producer of B
//   warp 3     : TMA producer of the scale tiles (A's 128 rows and all of B's
//                256 rows; every CTA of a pair holds B's scales in full, since
//                each SM's tensor core applies them to its 128 rows of D);
//                posts the scale bytes on the same full barrier
//   warps 4..11: epilogue: tcgen05.ld of all of a warp's accumulator columns,
//                hand-back, convert (times tA * tB for NVFP4), stage, TMA store
//
// Tensor memory: one 256-column fp32 accumulator (columns [0, 256)) and, from
// column 256, one scale slot per ring stage (A's slabs, then B's, 4 columns
// per slab).  Two accumulators would fill all 512 columns and leave the scales
// no room, so the next tile's MMAs wait for the epilogue's read-back.  A
// stage's scale slot is rewritten only after the MMAs that read it completed
// (the stage's empty barrier), and tcgen05.cp and the MMAs that read its
// result are issued by the same thread, which orders them.
//
// Every wait is bounded, as in the 16-bit kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"
#include "mx_ptx.cuh"
#include "pipeline.cuh"

namespace dgb {

constexpr int kMxEpiWarps = 8;
constexpr int kMxEpiWarp0 = 4;
constexpr int kMxThreads = 32 * (kMxEpiWarp0 + kMxEpiWarps);
constexpr uint32_t kMxStagingBytes = 32 * 128;   // one warp's output chunk: 32 rows x 128 B
constexpr int kMxTileN = 256;
constexpr int kMxSfCol0 = 256;                   // first tensor-memory column of the scale slots
// Registers: an epilogue warp reads all its columns of the accumulator (128
// per thread) before handing it back, so the next tile's MMAs wait only for
// the tcgen05.ld, not for the TMA stores behind it.  Twelve warps launch with
// 168 registers each; the first warpgroup (producers, MMA) gives registers
// back (setmaxnreg) down to kMxRegsLow and the two epilogue warpgroups take
// them up to kMxRegsHigh.
constexpr int kMxLaunchRegs = 168;
constexpr int kMxRegsLow = 56;
constexpr int kMxRegsHigh = 224;
static_assert(128 * kMxRegsLow + 32 * kMxEpiWarps * kMxRegsHigh <= kMxThreads * kMxLaunchRegs,
              "register shares exceed the launch's pool");

// Scale slab and scale-factor id of MMA kk (0..3) of a 128-byte K atom.
// mxf8f6f4: K32 per MMA, one E8M0 per 32 -> slab 0, byte kk.
// mxf4: K64 per MMA (32 bytes of packed E2M1), two E8M0 per MMA -> slab kk/2, bytes 2(kk%2), +1.
// mxf4nvf4: K64 per MMA, four E4M3 per MMA -> slab kk, the whole word.
template <int KIND>
__device__ __forceinline__ void mx_slab_of(int kk, int& slab, uint32_t& sf_id) {
    if constexpr (KIND == kMxF8) { slab = 0; sf_id = (uint32_t)kk; }
    else if constexpr (KIND == kMxF4) { slab = kk >> 1; sf_id = (uint32_t)(kk & 1) * 2u; }
    else { slab = kk; sf_id = 0u; }
}

// Producer of the scale tiles: for every ring stage, the 512-byte slabs of
// A's 128 rows and of B's two 128-row blocks that cover the stage's K atom.
template <int CG>
__device__ void mx_scale_producer(const MxParams& q, uint8_t* sf_ring, uint32_t full0, uint32_t empty0,
                                  volatile uint32_t* abort_flag, uint32_t rank, int cluster_id, int num_clusters) {
    const PersistentParams& p = q.base;
    const int S = p.stages;
    const bool leader = rank == 0;
    const uint64_t tmo = p.timeout_ns;
    const uint32_t fb0 = (CG == 2) ? map_to_cta(full0, 0) : full0;
    const uint32_t slab_bytes = 512u * (uint32_t)q.chunks;
    const uint32_t tx = (uint32_t)CG * q.sf_stage_bytes;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;
    WorkUnit u;
    for (int idx = 0; !aborted && next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
        int b, mb, nb;
        tile_coords(p, u.tile, b, mb, nb);
        const int rb_a = mb * CG + (int)rank;          // A's 128-row block
        const int rb_b = nb * 2;                         // B's first 128-row block of the tile
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
            if (!wait_phase_warp<false, true>(empty0 + 8u * stage, phase ^ 1u, abort_flag, tmo, p.status,
                                              kRoleProducer, stage, u.tile)) {
                aborted = true;
                break;
            }
            if (elect_one()) {
                if (leader) mbar_arrive_expect_tx(full0 + 8u * stage, tx);
                const uint32_t dst = smem_u32(sf_ring + (size_t)stage * q.sf_stage_bytes);
                const uint32_t fb = fb0 + 8u * stage;
                const int y = kb * q.chunks;
                if constexpr (CG == 1) {
                    tma_load_4d(dst, &q.tmap_sfa, fb, 0, y, rb_a, b);
                    tma_load_4d(dst + slab_bytes, &q.tmap_sfb, fb, 0, y, rb_b, b);
                    tma_load_4d(dst + 2 * slab_bytes, &q.tmap_sfb, fb, 0, y, rb_b + 1, b);
                } else {
                    tma_load_4d_pair(dst, &q.tmap_sfa, fb, 0, y, rb_a, b);
                    tma_load_4d_pair(dst + slab_bytes, &q.tmap_sfb, fb, 0, y, rb_b, b);
                    tma_load_4d_pair(dst + 2 * slab_bytes, &q.tmap_sfb, fb, 0, y, rb_b + 1, b);
                }
            }
            __syncwarp();
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    }
    // On abort the copies this warp issued land on the stages' full barriers,
    // whose phases the A producer drains (bounded) before the CTA exits.
    if (!aborted) {
        // tail: every slot released, so no commit lands on an exited CTA
        for (int i = 0; i < S; ++i) {
            if (!wait_phase_warp<false>(empty0 + 8u * stage, phase ^ 1u, abort_flag, tmo, p.status, kRoleProducer,
                                        stage, 0xFFFFFFFFu))
                break;
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    }
}

// MMA issuer (the pair leader's warp 1; one elected lane issues).
template <int CG, int KIND>
__device__ void mx_mma_issuer(const MxParams& q, uint8_t* ring, uint8_t* sf_ring, uint32_t stage_bytes,
                              uint32_t tmem_base, uint32_t full0, uint32_t empty0, uint32_t tfull, uint32_t tempty,
                              uint32_t drain_bar, volatile uint32_t* abort_flag, int cluster_id, int num_clusters) {
    const PersistentParams& p = q.base;
    const int S = p.stages;
    const uint64_t tmo = p.timeout_ns;
    const int C = q.chunks;
    const uint32_t slot_cols = (uint32_t)(12 * C);        // per stage: A's C slabs (4 cols each), B's 2C
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool aborted = false;
    bool issued_any = false;
    const bool issuer = elect_one();
    WorkUnit u;
    for (int idx = 0; !aborted && next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
        if (!wait_phase_warp<CG == 2>(tempty, acc_phase ^ 1u, abort_flag, tmo, p.status, kRoleMma, 0, u.tile)) {
            aborted = true;
            break;
        }
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
            if (!wait_phase_warp<false>(full0 + 8u * stage, phase, abort_flag, tmo, p.status, kRoleMma, stage,
                                        u.tile)) {
                aborted = true;
                break;
            }
            if (issuer) {
                tc_fence_after();
                const uint32_t sa = smem_u32(ring + (size_t)stage * stage_bytes);
                const uint32_t sb = sa + p.stage_bytes_a;
                const uint32_t sf = smem_u32(sf_ring + (size_t)stage * q.sf_stage_bytes);
                const uint32_t t_sfa = tmem_base + (uint32_t)kMxSfCol0 + (uint32_t)stage * slot_cols;
                const uint32_t t_sfb = t_sfa + 4u * (uint32_t)C;
                // scales of this stage: A's slabs, then B's row blocks 0 and 1 of
                // each slab side by side (the MMA reads B's 256 rows from 8
                // consecutive columns, row r at column r / 32)
                for (int c = 0; c < C; ++c) {
                    tmem_cp_scales<CG>(t_sfa + 4u * c, smem_desc_scale_slab(sf + 512u * c));
                    tmem_cp_scales<CG>(t_sfb + 8u * c, smem_desc_scale_slab(sf + 512u * (C + c)));
                    tmem_cp_scales<CG>(t_sfb + 8u * c + 4u, smem_desc_scale_slab(sf + 512u * (2 * C + c)));
                }
                // K-major: the next MMA is 32 bytes further along the 128-byte row (+2
                // in the address field).  MN-major (8-bit only): 32 k-rows of 128 B on
                // (+256), atoms along M/N one 128 x 128 box (16 KB) apart.
                constexpr uint32_t kBox = 128u * 128u;
                const uint64_t da = p.mn_major_a ? smem_desc_sw128_mn_lbo(sa, kBox) : smem_desc_sw128(sa);
                const uint64_t db = p.mn_major_b ? smem_desc_sw128_mn_lbo(sb, kBox) : smem_desc_sw128(sb);
                const uint64_t step_a = p.mn_major_a ? 256u : 2u;
                const uint64_t step_b = p.mn_major_b ? 256u : 2u;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    int slab;
                    uint32_t sf_id;
                    mx_slab_of<KIND>(kk, slab, sf_id);
                    mma_block_scaled<CG, KIND>(tmem_base, da + step_a * kk, db + step_b * kk,
                                               idesc_with_scale_ids(p.idesc, sf_id), t_sfa + 4u * slab,
                                               t_sfb + 8u * slab, (kb != u.kb0 || kk != 0) ? 1u : 0u);
                }
                issued_any = true;
                commit_to<CG>(empty0 + 8u * stage);
            }
            __syncwarp();
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        if (issuer) commit_to<CG>(tfull);
        __syncwarp();
        acc_phase ^= 1u;
    }
    if (aborted && issuer && issued_any) {
        commit_local<CG>(drain_bar);
        wait_phase_drain(drain_bar, 0, tmo);
    }
    __syncwarp();
}

template <int CG, int OUT, int KIND>
__global__ void __launch_bounds__(kMxThreads, 1) mx_kernel(const __grid_constant__ MxParams q) {
    const PersistentParams& p = q.base;
    constexpr int kOutBytes = (OUT == GEMM_F32) ? 4 : 2;
    constexpr int kChunkCols = 128 / kOutBytes;           // output columns per 128-byte staging row
    constexpr int kChunks = kMxTileN / kChunkCols;        // chunks per tile row: 8 (fp32) or 4
    constexpr int kWarpChunks = kChunks / 2;              // per epilogue warp (two warps per lane quarter)
    constexpr int kSub = kChunkCols / 32;                 // 32-column TMEM loads per chunk
    constexpr int kBatchChunks = kWarpChunks;             // a warp's chunks, all held in registers at once

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int S = p.stages;
    const uint32_t stage_bytes = p.stage_bytes_a + p.stage_bytes_b;
    uint8_t* ring = smem;
    uint8_t* sf_ring = ring + q.sf_ring_offset;
    // staging buffers: 1024-byte aligned, as the D map's 128-byte swizzle requires
    uint8_t* staging = smem + ((q.sf_ring_offset + (size_t)S * q.sf_stage_bytes + 1023) & ~size_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + kMxEpiWarps * kMxStagingBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 3);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8u * S;
    const uint32_t tfull = empty0 + 8u * S;
    const uint32_t tempty = tfull + 8u;
    const uint32_t drain_bar = tempty + 8u;

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 2);      // operand producer's and scale producer's expect_tx
            mbar_init(empty0 + 8u * s, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, CG * kMxEpiWarps);
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&p.tmap_a);
        prefetch_tensormap(&p.tmap_b);
        prefetch_tensormap(&p.tmap_d);
        prefetch_tensormap(&q.tmap_sfa);
        prefetch_tensormap(&q.tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();
    griddep_launch_dependents();

    const int cluster_id = blockIdx.x / CG;
    const int num_clusters = gridDim.x / CG;
    const uint64_t tmo = p.timeout_ns;

    // Each role raises or lowers its registers first thing, so that the code
    // that follows is compiled against its own share.
    if (warp < kMxEpiWarp0) {
        setmaxnreg_dec<kMxRegsLow>();
        if (warp == 0) {
            producer_loop<CG, 1, 1, kPartA>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                            cluster_id, num_clusters);
            __syncwarp();
        } else if (warp == 2) {
            producer_loop<CG, 1, 1, kPartB0>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                             cluster_id, num_clusters);
            __syncwarp();
        } else if (warp == 3) {
            mx_scale_producer<CG>(q, sf_ring, full0, empty0, abort_flag, rank, cluster_id, num_clusters);
            __syncwarp();
        } else {
            if (leader)
                mx_mma_issuer<CG, KIND>(q, ring, sf_ring, stage_bytes, tmem_base, full0, empty0, tfull, tempty,
                                        drain_bar, abort_flag, cluster_id, num_clusters);
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kMxRegsHigh>();
        // ------------------------------------------------------------ epilogue
        const bool stream_d = (p.l2_hints & kHintStreamD) != 0;
        const uint64_t pol_d = l2_policy_evict_first();
        const int wq = warp & 3;
        const int half = (warp - kMxEpiWarp0) >> 2;
        uint8_t* buf = staging + (warp - kMxEpiWarp0) * kMxStagingBytes;
        float alpha = 1.0f;
        if (KIND == kNvF4 && q.tensor_scales != nullptr) alpha = __ldg(q.tensor_scales) * __ldg(q.tensor_scales + 1);
        uint32_t acc_phase = 0;
        WorkUnit u;
        for (int idx = 0; next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
            int b, mb, nb;
            tile_coords(p, u.tile, b, mb, nb);
            if (!wait_phase_warp<false>(tfull, acc_phase, abort_flag, tmo, p.status, kRoleEpilogue, 0, u.tile)) break;
            tc_fence_after();
            acc_phase ^= 1u;
            const uint32_t t_lane = tmem_base + ((uint32_t)(wq * 32) << 16);
            const int m0 = mb * (128 * CG) + (int)rank * 128 + wq * 32;
            const int n0 = nb * kMxTileN;
            const int c_lo = half * kWarpChunks;
            // chunks with an in-range column of an in-range row; the rest is padding
            const int n_valid = (m0 < p.M) ? min(kChunks, (p.N - n0 + kChunkCols - 1) / kChunkCols) : 0;
            const int c_end = min(c_lo + kWarpChunks, n_valid);
            if (c_lo >= c_end) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader<CG>(tempty);
                continue;
            }
            for (int c0 = c_lo; c0 < c_end; c0 += kBatchChunks) {
                const int nc = min(kBatchChunks, c_end - c0);
                uint32_t r[kBatchChunks * kSub][32];
#pragma unroll
                for (int i = 0; i < kBatchChunks * kSub; ++i)
                    if (i < nc * kSub) tmem_ld_32x32b_x32(t_lane + (uint32_t)((c0 * kSub + i) * 32), r[i]);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < kBatchChunks * kSub; ++i)
                    if (i < nc * kSub) tmem_reg_fence(r[i]);
                if (c0 + nc >= c_end) {
                    // this warp's last read of the accumulator: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_leader<CG>(tempty);
                }
                if (KIND == kNvF4) {
#pragma unroll
                    for (int i = 0; i < kBatchChunks * kSub; ++i)
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[i][j] = __float_as_uint(__uint_as_float(r[i][j]) * alpha);
                }
#pragma unroll
                for (int cc = 0; cc < kBatchChunks; ++cc) {
                    if (cc >= nc) break;
                    auto piece = [&](int j) -> uint4 {
                        if constexpr (OUT == GEMM_F32) {
                            return make_uint4(r[cc][4 * j], r[cc][4 * j + 1], r[cc][4 * j + 2], r[cc][4 * j + 3]);
                        } else {
                            const int i = cc * kSub + (j >> 2), o = 8 * (j & 3);
                            return make_uint4(pack2<OUT>(__uint_as_float(r[i][o]), __uint_as_float(r[i][o + 1])),
                                              pack2<OUT>(__uint_as_float(r[i][o + 2]), __uint_as_float(r[i][o + 3])),
                                              pack2<OUT>(__uint_as_float(r[i][o + 4]), __uint_as_float(r[i][o + 5])),
                                              pack2<OUT>(__uint_as_float(r[i][o + 6]), __uint_as_float(r[i][o + 7])));
                        }
                    };
                    const int x = n0 + (c0 + cc) * kChunkCols;
                    if (chunk_needs_clipped_store<kOutBytes>(x, kChunkCols, p.N)) {
                        // ragged right edge inside a 16-byte granule: plain stores up to N
                        const int row = m0 + lane;
                        if (row < p.M)
                            store_segment_clipped<kOutBytes>(static_cast<uint8_t*>(p.d_ptr) +
                                                                 ((size_t)b * p.stride_d + (size_t)row * p.ldd + x) *
                                                                     kOutBytes,
                                                             p.N - x, piece);
                        continue;
                    }
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = piece(j);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (stream_d) {
                            if (p.batched) tma_store_3d_hint(&p.tmap_d, smem_u32(buf), x, m0, b, pol_d);
                            else tma_store_2d_hint(&p.tmap_d, smem_u32(buf), x, m0, pol_d);
                        } else {
                            if (p.batched) tma_store_3d(&p.tmap_d, smem_u32(buf), x, m0, b);
                            else tma_store_2d(&p.tmap_d, smem_u32(buf), x, m0);
                        }
                        bulk_commit_group();
                    }
                }
            }
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
static cudaLaunchConfig_t mx_config(size_t smem, int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kMxThreads, 1, 1);
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

// The kernel's setmaxnreg shares assume it was built with kMxLaunchRegs
// registers per thread: with fewer the epilogue warps' increase could never
// be granted, so such a build is refused rather than launched.
template <typename Kern>
static bool mx_regs_ok(Kern kern) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kern) != cudaSuccess) return false;
    return a.numRegs == kMxLaunchRegs;
}

template <int CG, int OUT, int KIND>
static cudaError_t mx_launch_typed(const MxParams& q, int grid, size_t smem, cudaStream_t stream) {
    auto kern = mx_kernel<CG, OUT, KIND>;
    if (!mx_regs_ok(kern)) return cudaErrorInvalidConfiguration;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = mx_config<CG>(smem, grid, stream, attr);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, q);
}

template <int CG, int OUT, int KIND>
static int mx_clusters_typed(size_t smem) {
    auto kern = mx_kernel<CG, OUT, KIND>;
    if (!mx_regs_ok(kern)) return 0;
    static std::atomic<int> smem_set[kMaxDevices];
    if (ensure_smem_limit(kern, smem, smem_set) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = mx_config<CG>(smem, CG, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

#define DGB_MX_DISPATCH_KIND(FN, CGV, OUTV, ...)                                     \
    switch (kind) {                                                                  \
    case kMxF8: return FN<CGV, OUTV, kMxF8>(__VA_ARGS__);                            \
    case kMxF4: return FN<CGV, OUTV, kMxF4>(__VA_ARGS__);                            \
    case kNvF4: return FN<CGV, OUTV, kNvF4>(__VA_ARGS__);                            \
    default: break;                                                                  \
    }
#define DGB_MX_DISPATCH_OUT(FN, CGV, ...)                                            \
    switch (dtype_d) {                                                               \
    case GEMM_F32: DGB_MX_DISPATCH_KIND(FN, CGV, GEMM_F32, __VA_ARGS__) break;       \
    case GEMM_BF16: DGB_MX_DISPATCH_KIND(FN, CGV, GEMM_BF16, __VA_ARGS__) break;     \
    case GEMM_F16: DGB_MX_DISPATCH_KIND(FN, CGV, GEMM_F16, __VA_ARGS__) break;       \
    default: break;                                                                  \
    }
#define DGB_MX_DISPATCH(FN, ...)                                                     \
    if (cta_group == 1) { DGB_MX_DISPATCH_OUT(FN, 1, __VA_ARGS__) }                  \
    if (cta_group == 2) { DGB_MX_DISPATCH_OUT(FN, 2, __VA_ARGS__) }

cudaError_t launch_mx(const MxParams& q, int kind, int cta_group, int dtype_d, int grid, size_t smem_bytes,
                      cudaStream_t stream) {
    DGB_MX_DISPATCH(mx_launch_typed, q, grid, smem_bytes, stream)
    return cudaErrorInvalidValue;
}

int mx_max_active_clusters(int kind, int cta_group, int dtype_d, size_t smem_bytes) {
    DGB_MX_DISPATCH(mx_clusters_typed, smem_bytes)
    return 0;
}

}  // namespace dgb
