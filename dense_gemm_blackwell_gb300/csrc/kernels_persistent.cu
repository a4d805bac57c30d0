// kernels_persistent.cu -- warp-specialised persistent tcgen05 GEMM, D = A * B^T.
//
// Structure ("Hopper and Blackwell GEMM", concepts on warp specialisation and
// stage count; cuBLASDx "API Card: Blackwell Pipeline (tcgen05)", sections
// "Depth and shared memory" and "Device side"):
//
//   warps 0 and 10    : TMA producers.  For every ring stage of every tile
//                       both wait for the slot to be empty; warp 0 sets the
//                       expected bytes on the slot's full barrier and copies
//                       A, warp 10 copies B (one or two 128-byte K atoms
//                       each; for 512-wide tiles warp 0 also takes B's first
//                       half), all completing on that barrier.
//   warp 1            : allocates tensor memory (whole warp); the pair
//                       leader's warp runs the MMA loop: waits for a full slot,
//                       issues four K16 (K8 for tf32) tcgen05.mma per K atom
//                       and accumulator half (the tile's first starts a fresh
//                       accumulator), commits to the slot's empty barrier;
//                       after the tile's last stage commits to the
//                       accumulator's full barrier.
//   warps 2..9        : epilogue.  Wait for a full accumulator, read it with
//                       tcgen05.ld (one row per thread; two warps per 32-lane
//                       quarter, sharing the chunks of each part), hand the
//                       part back, convert, stage 32x128 B chunks in swizzled
//                       shared memory and write D with TMA stores (coalesced
//                       lines).
//
// Tiles up to 256 wide keep two accumulators in tensor memory, so the
// epilogue of tile t overlaps the MMAs of tile t+1.  512-wide tiles (two
// N = 256 MMAs per K step) fill all 512 columns with one accumulator, handed
// back in two 256-column halves.  A long enough tile runs its first K blocks
// on the left half alone and repeats them on the right half alone at its end
// (split units, units.cuh), so each half drains while MMAs run on the other;
// otherwise the MMAs of tile t+1 start on the left half and wait for the
// right one after kWideLeadStages stages.  The grid is
// persistent: CTA (pair) c takes tiles c, c+G, ... in a grouped raster that
// keeps a wave's A and B panels in L2; when the tiles do not fill whole waves,
// a stream-K region split along K comes first (units.cuh).  Every thread
// follows the same unit sequence and leaves the loop together.
//
// cta_group::2: a cluster of two CTAs on neighbouring SMs computes a
// (256 x tile_n) tile with one MMA stream issued by the even CTA.  Each CTA
// loads its own 128 rows of A and its own half of B's tile_n rows into its own
// shared memory; both CTAs' copies complete on the leader's full barrier.  The
// leader's commits arrive on the empty / accumulator-full barriers of both
// CTAs; each CTA's epilogue reads its own TMEM (its 128 rows) and both arrive on
// the leader's accumulator-empty barriers.
//
// Every wait is bounded (wait_phase): on expiry the kernel records
// GEMM_ERR_TIMEOUT, raises a CTA-wide abort flag, drains what it has in flight
// (copies, MMAs, stores), frees tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace dgb {

constexpr uint32_t kStagingBytes = 32 * 128;  // one warp's output chunk: 32 rows x 128 B
constexpr int kEpilogueWarps = 8;             // two per TMEM lane quarter, one half of the chunks each
constexpr int kThreads = 96 + 32 * kEpilogueWarps;   // + producer, MMA and second producer warps
constexpr int kProducerBWarp = 2 + kEpilogueWarps;
constexpr int kWideLeadStages = 2;            // 512-wide tiles: left-half stages issued before the right half is free
// 32-column TMEM loads an epilogue warp holds in registers at once: as many as
// fit the 168 registers a thread of an 11-warp CTA can have (3 warps share a
// sub-partition's 16K registers) without spilling
template <int OUT>
__host__ __device__ constexpr int batch_loads() { return OUT == GEMM_F32 ? 3 : 2; }

// MMA issuer (the pair leader's MMA warp).  Per ring stage: wait for the
// stage's data, issue four MMAs per 128-byte K atom (K16 of 16-bit elements
// or K8 of tf32; ATOMS atoms per stage, rows x 128 B apart), commit the
// stage back to the producer.  Per tile: wait for an empty accumulator
// buffer first, commit it to the epilogue after the tile's last stage.
// Issuing costs about 45 cycles per MMA and, from a lone divergent lane, 230
// per barrier wait (measured on GB300): at one atom per stage that is ~450 of
// the 512 cycles the four MMAs of a 256 x 256 pair tile take.  So the whole
// warp runs the loop and waits, and one lane, elected once, issues every MMA
// and commit (a commit tracks only its own thread's MMAs).
// HALVES = 2 (512-wide tiles): each K step is two N = 256 MMAs, into
// accumulator columns [0, 256) and [256, 512), B rows of the second half
// 256 / CG rows further on in the stage.  The two column halves are handed
// back separately, so a tile starts with the left halves of its first
// kWideLeadStages stages before it waits for the right half.
template <int CG, int ATOMS, int HALVES>
__device__ __forceinline__ void mma_issuer(const PersistentParams& p, uint8_t* ring, uint32_t stage_bytes,
                                           uint32_t tmem_base, uint32_t full0, uint32_t empty0, uint32_t tfull0,
                                           uint32_t tempty0, uint32_t drain_bar, volatile uint32_t* abort_flag,
                                           int cluster_id, int num_clusters) {
    const int S = p.stages;
    const int TS = p.tmem_stages;
    const uint64_t tmo = p.timeout_ns;
    auto full = [&](int s) { return full0 + 8u * s; };
    auto empty = [&](int s) { return empty0 + 8u * s; };
    auto tfull = [&](int a, int part) { return tfull0 + 8u * (2 * a + part); };
    auto tempty = [&](int a, int part) { return tempty0 + 8u * (2 * a + part); };
    const uint64_t b_atom = (uint64_t)(p.tile_n / CG) * 8u;   // B atom stride in descriptor units
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool aborted = false;
    bool issued_any = false;
    const bool issuer = elect_one();
    WorkUnit u;
    for (int idx = 0; !aborted && next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
        const int t = u.tile;
        if (!wait_phase_warp<CG == 2>(tempty(acc, 0), acc_phase ^ 1u, abort_flag, tmo, p.status, kRoleMma, acc,
                                      t)) {
            aborted = true;
            break;
        }
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.tile_n);
        // The MMAs of one ring stage for accumulator halves [h0, h1), the first
        // of the left (right) half's MMAs overwriting it if first_l (first_r);
        // issuer lane only.
        auto issue_stage = [&](int st, int h0, int h1, bool first_l, bool first_r) {
            tc_fence_after();
            const uint32_t sa = smem_u32(ring + (size_t)st * stage_bytes);
            const uint32_t sb = sa + p.stage_bytes_a;
            // K-major: next MMA's K is 32 bytes along the row (+2 in the
            // descriptor's address field); MN-major: 16 k-rows on (+128).
            const uint64_t da = p.mn_major_a ? smem_desc_sw128_mn(sa) : smem_desc_sw128(sa);
            const uint64_t db = p.mn_major_b ? smem_desc_sw128_mn(sb) : smem_desc_sw128(sb);
            const uint64_t step_a = p.mn_major_a ? 128u : 2u;
            const uint64_t step_b = p.mn_major_b ? 128u : 2u;
#pragma unroll
            for (int at = 0; at < ATOMS; ++at) {
                // next atom: 128 rows (A) or tile_n / CG rows (B) x 128 B on
                const uint64_t da_at = da + (uint64_t)at * (128u * 8u);
                const uint64_t db_at = db + (uint64_t)at * b_atom;
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    if (h < h0 || h >= h1) continue;
                    const bool first = (h == 0 ? first_l : first_r) && at == 0;
                    const uint32_t d_h = d_tmem + (uint32_t)(h * 256);
                    const uint64_t db_h = db_at + (uint64_t)(h * (256 / CG) * 8);
                    if (p.mma_kind == kMmaKindTF32) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_tf32<CG>(d_h, da_at + 2u * kk, db_h + 2u * kk, p.idesc, !first || (kk != 0));
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16<CG>(d_h, da_at + step_a * kk, db_h + step_b * kk, p.idesc, !first || (kk != 0));
                    }
                }
            }
            issued_any = true;
        };
        int kb = u.kb0;
        if constexpr (HALVES == 2) {
            const int n = u.kb1 - u.kb0;
            const int L = split_stages(u, true);
            if (L > 0) {
                // Split unit (units.cuh): left-only stages, then both halves once
                // the right one is free, then right-only stages; the left half is
                // complete (and handed to the epilogue) after the last two-half stage.
                for (int i = 0; i < n + L; ++i) {
                    int walk, halves;
                    stage_of(i, n, L, walk, halves);
                    if (i == L && !wait_phase_warp<CG == 2>(tempty(acc, 1), acc_phase ^ 1u, abort_flag, tmo, p.status,
                                                           kRoleMma, acc, t)) {
                        aborted = true;
                        break;
                    }
                    if (!wait_phase_warp<false>(full(stage), phase, abort_flag, tmo, p.status, kRoleMma, stage, t)) {
                        aborted = true;
                        break;
                    }
                    if (issuer) {
                        issue_stage(stage, (halves & kHalfLeft) ? 0 : 1, (halves & kHalfRight) ? 2 : 1, i == 0, i == L);
                        commit_to<CG>(empty(stage));
                        if (i == n - 1) commit_to<CG>(tfull(acc, 0));
                    }
                    __syncwarp();
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (aborted) break;
                if (issuer) commit_to<CG>(tfull(acc, 1));
                __syncwarp();
                if (++acc == TS) { acc = 0; acc_phase ^= 1u; }
                continue;
            }
            // The epilogue hands back columns [0, 256) first: run the first
            // stages' left-half MMAs while it still reads [256, 512).
            const int lead = min(kWideLeadStages, n);
            int st = stage;
            uint32_t ph = phase;
            for (int i = 0; i < lead; ++i) {
                if (!wait_phase_warp<false>(full(st), ph, abort_flag, tmo, p.status, kRoleMma, st, t)) {
                    aborted = true;
                    break;
                }
                if (issuer) issue_stage(st, 0, 1, i == 0, false);
                __syncwarp();
                if (++st == S) { st = 0; ph ^= 1u; }
            }
            if (aborted) break;
            if (!wait_phase_warp<CG == 2>(tempty(acc, 1), acc_phase ^ 1u, abort_flag, tmo, p.status, kRoleMma, acc,
                                          t)) {
                aborted = true;
                break;
            }
            if (issuer) {
                for (int i = 0, st2 = stage; i < lead; ++i) {
                    issue_stage(st2, 1, 2, false, i == 0);
                    commit_to<CG>(empty(st2));
                    if (++st2 == S) st2 = 0;
                }
            }
            __syncwarp();
            for (int i = 0; i < lead; ++i)
                if (++stage == S) { stage = 0; phase ^= 1u; }
            kb = u.kb0 + lead;
        }
        for (; kb < u.kb1; ++kb) {
            if (!wait_phase_warp<false>(full(stage), phase, abort_flag, tmo, p.status, kRoleMma, stage, t)) {
                aborted = true;
                break;
            }
            if (issuer) {
                issue_stage(stage, 0, HALVES, kb == u.kb0, kb == u.kb0);
                commit_to<CG>(empty(stage));
            }
            __syncwarp();
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        if (issuer) {
            commit_to<CG>(tfull(acc, 0));
            if (HALVES == 2) commit_to<CG>(tfull(acc, 1));
        }
        __syncwarp();
        if (++acc == TS) { acc = 0; acc_phase ^= 1u; }
    }
    if (aborted && issuer && issued_any) {
        // Abort: make sure every MMA issued so far has finished before TMEM is freed.
        commit_local<CG>(drain_bar);
        wait_phase_drain(drain_bar, 0, tmo);
    }
    __syncwarp();
}

template <int CG, int OUT>
__global__ void __launch_bounds__(kThreads, 1) persistent_kernel(const __grid_constant__ PersistentParams p) {
    constexpr int kOutBytes = (OUT == GEMM_F32) ? 4 : 2;
    constexpr int kChunkCols = 128 / kOutBytes;   // output columns per 128-byte staging row

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int S = p.stages;
    const int TS = p.tmem_stages;
    const uint32_t stage_bytes = p.stage_bytes_a + p.stage_bytes_b;
    uint8_t* ring = smem;
    uint8_t* staging = ring + (size_t)S * stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + (p.direct_store ? 0 : kEpilogueWarps * kStagingBytes));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4 * TS + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8u * S;
    // accumulator full / empty: two of each per accumulator, one per part
    // (columns [0, 256) and [256, 512); tiles up to 256 wide use part 0 only)
    const uint32_t tfull0 = empty0 + 8u * S;
    const uint32_t tempty0 = tfull0 + 16u * TS;
    const uint32_t drain_bar = tempty0 + 16u * TS;
    auto full = [&](int s) { return full0 + 8u * s; };
    auto empty = [&](int s) { return empty0 + 8u * s; };
    auto tfull = [&](int a, int part) { return tfull0 + 8u * (2 * a + part); };
    auto tempty = [&](int a, int part) { return tempty0 + 8u * (2 * a + part); };

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < TS; ++a) {
            mbar_init(tfull(a, 0), 1);
            mbar_init(tfull(a, 1), 1);
            mbar_init(tempty(a, 0), CG * kEpilogueWarps);
            mbar_init(tempty(a, 1), CG * kEpilogueWarps);
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

    if (warp == 0 || warp == kProducerBWarp) {
        // ------------------------------------------------------------ TMA producers
        // warp 0: A (+ B's first half of a 512-wide tile); the second producer: the rest of B
        const bool first = warp == 0;
        if (p.tile_n > 256) {
            if (first)
                producer_loop<CG, 1, 2, kPartA | kPartB0, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag,
                                                          rank, cluster_id, num_clusters);
            else
                producer_loop<CG, 1, 2, kPartB1, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                                 cluster_id, num_clusters);
        } else if (p.k_atoms == 2) {
            if (first)
                producer_loop<CG, 2, 1, kPartA, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                                cluster_id, num_clusters);
            else
                producer_loop<CG, 2, 1, kPartB0, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                                 cluster_id, num_clusters);
        } else {
            if (first)
                producer_loop<CG, 1, 1, kPartA, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                                cluster_id, num_clusters);
            else
                producer_loop<CG, 1, 1, kPartB0, true>(p, ring, stage_bytes, p.tile_k, full0, empty0, abort_flag, rank,
                                                 cluster_id, num_clusters);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (leader) {
            // the stage depth is a template argument: this warp runs the
            // kernel's tightest loop, so no per-stage branching on it
            if (p.tile_n > 256)
                mma_issuer<CG, 1, 2>(p, ring, stage_bytes, tmem_base, full0, empty0, tfull0, tempty0, drain_bar,
                                     abort_flag, cluster_id, num_clusters);
            else if (p.k_atoms == 2)
                mma_issuer<CG, 2, 1>(p, ring, stage_bytes, tmem_base, full0, empty0, tfull0, tempty0, drain_bar,
                                     abort_flag, cluster_id, num_clusters);
            else
                mma_issuer<CG, 1, 1>(p, ring, stage_bytes, tmem_base, full0, empty0, tfull0, tempty0, drain_bar,
                                     abort_flag, cluster_id, num_clusters);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Eight warps: warp w reads TMEM lanes [32 (w mod 4), +32) (its 32 rows).
        // A tile's columns form one part, or two 256-column parts for 512-wide
        // tiles, each handed back on its own barrier; the two warps of a lane
        // quarter split every part's output chunks.  A warp loads its chunks
        // of a part in register batches (the first batch takes the remainder,
        // so the last is full) and hands the part back right after its last
        // tcgen05.ld of it, before staging and storing that batch: with a
        // single 512-column accumulator the next tile's MMAs wait for these
        // hand-backs, the left part's first.
        // D is written once and never read back here: let it leave L2 first.
        const bool stream_d = (p.l2_hints & kHintStreamD) != 0;
        const uint64_t pol_d = l2_policy_evict_first();
        const int wq = warp & 3;                 // TMEM lanes [32*wq, 32*wq+32) are this warp's
        const int half = (warp - 2) >> 2;       // which of the lane quarter's two warps
        uint8_t* buf = staging + (warp - 2) * kStagingBytes;
        // this warp's share of the operand ring, used by the last unit's stream-K fix-up
        const uint32_t slice_bytes = ((uint32_t)S * stage_bytes / kEpilogueWarps) & ~15u;
        const uint32_t slice = smem_u32(ring) + (uint32_t)(warp - 2) * slice_bytes;
        const float4* slice_f4 = reinterpret_cast<const float4*>(ring + (size_t)(warp - 2) * slice_bytes);
        int acc = 0;
        uint32_t acc_phase = 0;
        const int nchunks = p.tile_n / kChunkCols;
        const int parts = p.tile_n > 256 ? 2 : 1;
        const int cpp = nchunks / parts;         // chunks per part
        const int split = (cpp + 1) / 2;         // a part's chunks [0, split) for warp half 0
        constexpr int kSub = kChunkCols / 32;    // 32-column TMEM loads per output chunk
        constexpr int kBatchLoads = batch_loads<OUT>();
        constexpr int kBatchChunks = kBatchLoads / kSub;
        WorkUnit u;
        for (int idx = 0; next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
            const int t = u.tile;
            int b, mb, nb;
            tile_coords(p, t, b, mb, nb);
            const bool ok = wait_phase_warp<false>(tfull(acc, 0), acc_phase, abort_flag, tmo, p.status,
                                                   kRoleEpilogue, acc, t);
            if (!ok) break;
            tc_fence_after();
            // A 512-wide tile's right part may complete after its left one
            // (split units, units.cuh): wait for it before reading it.
            auto wait_part = [&](int pt) {
                if (pt == 0) return true;
                const bool got = wait_phase_warp<false>(tfull(acc, pt), acc_phase, abort_flag, tmo, p.status,
                                                        kRoleEpilogue, acc, t);
                tc_fence_after();
                return got;
            };
            bool lost = false;
            const uint32_t t_lane = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * p.tile_n);
            const int m0 = mb * (128 * CG) + (int)rank * 128 + wq * 32;
            const int n0 = nb * p.tile_n;
            auto release = [&](int part) {
                // Every TMEM read of this part by this warp is complete: hand it back.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader<CG>(tempty(acc, part));
            };
            auto release_all = [&]() {
                for (int q = 0; q < parts; ++q) release(q);
            };
            // slot s's partial of this CTA (in float4) and this warp's flag of it
            auto part_base_of = [&](int s) { return (size_t)(s * CG + (int)rank) * 128 * p.tile_n / 4; };
            auto flag_of = [&](int s) { return p.sk_flags + (s * CG + (int)rank) * kEpilogueWarps + half * 4 + wq; };
            const size_t part_base = part_base_of(u.slot);
            uint32_t* flag = flag_of(u.slot);

            if (u.role == kUnitContributor) {
                // Leave this K range's fp32 partial for the finisher, then publish it.
                // Each accumulator part goes back to the MMA warp right after
                // this warp's last TMEM load of it, before that load's stores.
                float4* part = reinterpret_cast<float4*>(p.sk_partials) + part_base;
                for (int pt = 0; pt < parts; ++pt) {
                    if (!wait_part(pt)) {
                        lost = true;
                        break;
                    }
                    const int q_lo = (pt * cpp + (half == 0 ? 0 : split)) * kSub;   // this warp's 32-column loads
                    const int q_hi = (pt * cpp + (half == 0 ? split : cpp)) * kSub;
                    if (q_lo >= q_hi) release(pt);
                    for (int q = q_lo; q < q_hi; ++q) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(t_lane + q * 32, r);
                        tmem_wait_ld();
                        tmem_reg_fence(r);
                        if (q + 1 == q_hi) release(pt);
                        float4* dst = part + sk_partial_index(p.tile_n, wq, q, 0, lane);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[32 * j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                      __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    }
                }
                if (lost) break;
                __threadfence();
                __syncwarp();
                if (lane == 0) store_release_gpu(flag, sk_launch_epoch(p.sk_epoch));
                if (++acc == TS) { acc = 0; acc_phase ^= 1u; }
                continue;
            }

            const bool adds = u.role == kUnitFinisher;
            bool staged = false;    // partial gathered into this warp's slice of the ring
            if (adds) {
                // the tile's contributors: slots u.slot (the latest K range) down to u.slot0
                int got = 1;
                if (lane == 0)
                    for (int s = u.slot; s >= u.slot0 && got; --s)
                        got = wait_flag(flag_of(s), sk_launch_epoch(p.sk_epoch), abort_flag, tmo, p.status,
                                        kRoleEpilogue, s, t);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    release_all();
                    break;
                }
                for (int s = u.slot; s >= u.slot0; --s) {
                    uint32_t v;   // every lane acquires the flags before reading the partials
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag_of(s)) : "memory");
                    (void)v;
                }
                // A finisher is its cluster's last unit: with its accumulator
                // full, no copy or MMA touches the operand ring again, so the
                // partial is gathered there by asynchronous copies (a whole part
                // in flight per thread) rather than by register loads.
                WorkUnit nxt;
                staged = (uint32_t)(split * kSub) * 4096u <= slice_bytes &&
                         !next_unit(p, cluster_id, num_clusters, idx + 1, nxt);
                if (staged) fence_proxy_async_smem();
            }
            const float4* part = reinterpret_cast<const float4*>(p.sk_partials) + part_base;
            // Chunks that hold at least one in-range column of an in-range row; the
            // rest of the tile (padding beyond M or N) is neither read nor stored.
            const int n_valid = (m0 < p.M) ? min(nchunks, (p.N - n0 + kChunkCols - 1) / kChunkCols) : 0;
            for (int pt = 0; pt < parts; ++pt) {
                if (!wait_part(pt)) {
                    lost = true;
                    break;
                }
                const int c_lo = pt * cpp + (half == 0 ? 0 : split);          // this warp's chunks of the part
                const int c_end = min(pt * cpp + (half == 0 ? split : cpp), n_valid);
                if (c_lo >= c_end) release(pt);
                if (staged) {
                    // thread-private layout: this lane's float4 i of the part at i * 32 + lane
                    for (int c = c_lo; c < c_end; ++c)
                        for (int h = 0; h < kSub; ++h)
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                cp_async_16(slice + (uint32_t)(((((c - c_lo) * kSub + h) * 8 + j) * 32 + lane) * 16),
                                            part + sk_partial_index(p.tile_n, wq, c * kSub + h, j, lane));
                }
                bool pending = staged;
                const int first_nc = (c_end - c_lo) % kBatchChunks;
                for (int c0 = c_lo; c0 < c_end;) {
                    const int nc = (c0 == c_lo && first_nc) ? first_nc : kBatchChunks;   // chunks in this batch
                    uint32_t r[kBatchLoads][32];
#pragma unroll
                    for (int q = 0; q < kBatchLoads; ++q)
                        if (q < nc * kSub) tmem_ld_32x32b_x32(t_lane + (c0 * kSub + q) * 32, r[q]);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < kBatchLoads; ++q)
                        if (q < nc * kSub) tmem_reg_fence(r[q]);
                    if (c0 + nc == c_end) release(pt);
                    if (pending) {
                        cp_async_wait_all();
                        pending = false;
                    }
                    if (p.acc_f16) {
                        // fp16 accumulator: the value is the low half of each 32-bit cell
#pragma unroll
                        for (int q = 0; q < kBatchLoads; ++q)
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                r[q][i] = __float_as_uint(__half2float(__ushort_as_half((unsigned short)(r[q][i] & 0xFFFFu))));
                    }
#pragma unroll
                    for (int cc = 0; cc < kBatchChunks; ++cc) {
                        if (cc >= nc) break;
                        const int c = c0 + cc;
                        if (adds) {
                            // own part (later K) + the contributors' partials, latest K range first:
                            // one fixed order
                            for (int sl = u.slot; sl >= u.slot0; --sl) {
                                const bool from_slice = staged && sl == u.slot;
                                const float4* ps = reinterpret_cast<const float4*>(p.sk_partials) + part_base_of(sl);
#pragma unroll
                                for (int h = 0; h < kSub; ++h) {
#pragma unroll
                                    for (int j = 0; j < 8; ++j) {
                                        const float4 qv =
                                            from_slice ? slice_f4[(((c - c_lo) * kSub + h) * 8 + j) * 32 + lane]
                                                       : __ldcg(ps + sk_partial_index(p.tile_n, wq, c * kSub + h, j, lane));
                                        const int q = cc * kSub + h;
                                        r[q][4 * j] = __float_as_uint(__uint_as_float(r[q][4 * j]) + qv.x);
                                        r[q][4 * j + 1] = __float_as_uint(__uint_as_float(r[q][4 * j + 1]) + qv.y);
                                        r[q][4 * j + 2] = __float_as_uint(__uint_as_float(r[q][4 * j + 2]) + qv.z);
                                        r[q][4 * j + 3] = __float_as_uint(__uint_as_float(r[q][4 * j + 3]) + qv.w);
                                    }
                                }
                            }
                        }
                        // 16-byte piece j (0..7) of this thread's 128-byte row segment
                        auto piece = [&](int j) -> uint4 {
                            if constexpr (OUT == GEMM_F32) {
                                return make_uint4(r[cc][4 * j], r[cc][4 * j + 1], r[cc][4 * j + 2], r[cc][4 * j + 3]);
                            } else {
                                const int q = cc * kSub + (j >> 2), o = 8 * (j & 3);
                                return make_uint4(pack2<OUT>(__uint_as_float(r[q][o]), __uint_as_float(r[q][o + 1])),
                                                  pack2<OUT>(__uint_as_float(r[q][o + 2]), __uint_as_float(r[q][o + 3])),
                                                  pack2<OUT>(__uint_as_float(r[q][o + 4]), __uint_as_float(r[q][o + 5])),
                                                  pack2<OUT>(__uint_as_float(r[q][o + 6]), __uint_as_float(r[q][o + 7])));
                            }
                        };
                        const int x = n0 + c * kChunkCols;
                        if (p.direct_store || chunk_needs_clipped_store<kOutBytes>(x, kChunkCols, p.N)) {
                            // This thread's row: 128 contiguous bytes, streaming stores
                            // (element by element past N at a ragged right edge).
                            const int row = m0 + lane;
                            if (row < p.M) {
                                uint8_t* dst = static_cast<uint8_t*>(p.d_ptr) +
                                               ((size_t)b * p.stride_d + (size_t)row * p.ldd + x) * kOutBytes;
                                if (x + kChunkCols <= p.N) {
#pragma unroll
                                    for (int j = 0; j < 8; ++j) __stcs(reinterpret_cast<uint4*>(dst) + j, piece(j));
                                } else {
                                    store_segment_clipped<kOutBytes>(dst, p.N - x, piece);
                                }
                            }
                            continue;
                        }
                        // The staging buffer's previous store must have read it.
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
                    c0 += nc;
                }
            }
            if (lost) break;
            if (++acc == TS) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, (uint32_t)p.tmem_cols);
    }
    if (p.sk_tiles > 0 && threadIdx.x == 0) sk_finish_launch(p.sk_epoch, sk_launch_epoch(p.sk_epoch));
}

template <int CG, int OUT>
static cudaError_t launch_typed(const PersistentParams& p, int grid, size_t smem, cudaStream_t stream) {
    auto kern = persistent_kernel<CG, OUT>;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CG, int OUT>
static int max_clusters_typed(size_t smem) {
    auto kern = persistent_kernel<CG, OUT>;
    static std::atomic<int> smem_set[kMaxDevices];
    if (ensure_smem_limit(kern, smem, smem_set) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CG, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

int persistent_max_active_clusters(int cta_group, int dtype_d, size_t smem_bytes) {
    if (cta_group == 1) {
        switch (dtype_d) {
        case GEMM_F32: return max_clusters_typed<1, GEMM_F32>(smem_bytes);
        case GEMM_BF16: return max_clusters_typed<1, GEMM_BF16>(smem_bytes);
        case GEMM_F16: return max_clusters_typed<1, GEMM_F16>(smem_bytes);
        default: return 0;
        }
    }
    switch (dtype_d) {
    case GEMM_F32: return max_clusters_typed<2, GEMM_F32>(smem_bytes);
    case GEMM_BF16: return max_clusters_typed<2, GEMM_BF16>(smem_bytes);
    case GEMM_F16: return max_clusters_typed<2, GEMM_F16>(smem_bytes);
    default: return 0;
    }
}

cudaError_t launch_persistent(const PersistentParams& p, int cta_group, int dtype_d, int grid,
                              size_t smem_bytes, cudaStream_t stream) {
    if (cta_group == 1) {
        switch (dtype_d) {
        case GEMM_F32: return launch_typed<1, GEMM_F32>(p, grid, smem_bytes, stream);
        case GEMM_BF16: return launch_typed<1, GEMM_BF16>(p, grid, smem_bytes, stream);
        case GEMM_F16: return launch_typed<1, GEMM_F16>(p, grid, smem_bytes, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (dtype_d) {
    case GEMM_F32: return launch_typed<2, GEMM_F32>(p, grid, smem_bytes, stream);
    case GEMM_BF16: return launch_typed<2, GEMM_BF16>(p, grid, smem_bytes, stream);
    case GEMM_F16: return launch_typed<2, GEMM_F16>(p, grid, smem_bytes, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dgb
