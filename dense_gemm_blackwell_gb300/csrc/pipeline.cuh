// pipeline.cuh -- pieces shared by the persistent kernels: tile raster, the TMA
// producer loop, MMA commits and output packing.
//
// The producer follows the main loop of "Hopper and Blackwell GEMM" (warp
// specialisation): a producer warp walks every K slice of every tile the CTA
// (pair) owns, waits for the ring slot to be empty, announces the slot's
// expected bytes on its full barrier and issues tensor copies that complete on
// it (a kernel may run two such warps, one for A and one for B).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "common.cuh"
#include "units.cuh"

namespace dgb {

// Float4 index, inside one (slot, rank) partial, of 16-byte piece j (0..7) of
// thread `lane` of epilogue warp wq for 32-column chunk c32: a warp's pieces
// j are 512 contiguous bytes, so partial stores and loads are coalesced.
__device__ __forceinline__ size_t sk_partial_index(int tile_n, int wq, int c32, int j, int lane) {
    return ((size_t)(wq * (tile_n / 32) + c32) * 8 + j) * 32 + lane;
}

// Commit every MMA issued so far to `bar` (in both CTAs of a pair).
template <int CG>
__device__ __forceinline__ void commit_to(uint32_t bar) {
    if constexpr (CG == 1) mma_commit(bar);
    else mma_commit_pair(bar, 0x3);
}

// Commit to `bar` of this CTA only (drain on the abort path).
template <int CG>
__device__ __forceinline__ void commit_local(uint32_t bar) {
    if constexpr (CG == 1) mma_commit(bar);
    else mma_commit_pair(bar, 0x1);
}

// Hand an accumulator (or partial) buffer back to the pair leader's MMA thread.
template <int CG>
__device__ __forceinline__ void arrive_leader(uint32_t bar) {
    if constexpr (CG == 1) mbar_arrive(bar);
    else mbar_arrive_remote(map_to_cta(bar, 0));
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (OUT == GEMM_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Whether an output chunk is written with plain stores rather than a TMA
// store: a TMA store writes whole 16-byte granules of a row, so a chunk that
// ends inside one (N x element bytes not a multiple of 16, with the caller's
// padding columns behind column N) would also overwrite that padding.
template <int kOutBytes>
__device__ __forceinline__ bool chunk_needs_clipped_store(int x, int chunk_cols, int N) {
    return x + chunk_cols > N && ((N * kOutBytes) & 15) != 0;
}

// One thread's 128-byte segment of an output row (eight 16-byte pieces,
// piece(j)) at dst, of which the first `valid` elements lie inside D: whole
// pieces while they fit, then element by element up to column N.  dst is
// 16-byte aligned.
template <int kOutBytes, typename Piece>
__device__ __forceinline__ void store_segment_clipped(uint8_t* dst, int valid, Piece&& piece) {
    constexpr int kPer = 16 / kOutBytes;   // elements per piece
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j * kPer >= valid) break;
        const uint4 q = piece(j);
        if ((j + 1) * kPer <= valid) {
            *reinterpret_cast<uint4*>(dst + 16 * j) = q;
        } else {
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                if (j * kPer + e >= valid) break;
                if constexpr (kOutBytes == 4) reinterpret_cast<uint32_t*>(dst + 16 * j)[e] = w[e];
                else reinterpret_cast<uint16_t*>(dst + 16 * j)[e] = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
            }
        }
    }
}

// Copy one operand's slice for one ring stage: `rows` rows (M or N) of
// `tile_k` K elements.  K-major: ATOMS boxes of (tile_k / ATOMS) x rows, one
// 128-byte swizzle atom column each, `atom_stride` bytes apart (default
// rows x 128 B).  MN-major (ATOMS == 1): boxes of `mn_elems` contiguous M/N
// elements (128 bytes) x tile_k k-rows, one per `mn_elems` rows, `mn_box_bytes`
// apart.
template <int CG, int ATOMS = 1>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar, bool mn_major,
                                             int rows, int row0, int kx, int b, bool batched, bool hint,
                                             uint64_t policy, int atom_k = 0, uint32_t atom_stride = 0,
                                             int mn_elems = 64, uint32_t mn_box_bytes = kMNMajorBoxBytes) {
    const int boxes = mn_major ? rows / mn_elems : ATOMS;
    const uint32_t a_stride = atom_stride ? atom_stride : (uint32_t)rows * 128u;
    for (int j = 0; j < boxes; ++j) {
        const int x = mn_major ? row0 + mn_elems * j : (ATOMS == 1 ? kx : kx + j * atom_k);
        const int y = mn_major ? kx : row0;
        const uint32_t d = dst + (uint32_t)j * (mn_major ? mn_box_bytes : a_stride);
        if constexpr (CG == 1) {
            if (batched) {
                if (hint) tma_load_3d_hint(d, map, bar, x, y, b, policy);
                else tma_load_3d(d, map, bar, x, y, b);
            } else {
                if (hint) tma_load_2d_hint(d, map, bar, x, y, policy);
                else tma_load_2d(d, map, bar, x, y);
            }
        } else {
            if (batched) {
                if (hint) tma_load_3d_pair_hint(d, map, bar, x, y, b, policy);
                else tma_load_3d_pair(d, map, bar, x, y, b);
            } else {
                if (hint) tma_load_2d_pair_hint(d, map, bar, x, y, policy);
                else tma_load_2d_pair(d, map, bar, x, y);
            }
        }
    }
}

// TMA producer (one warp: every lane runs the loop and waits, one elected
// lane issues).  `tile_k` is the ring stage depth in elements of
// A/B: ATOMS 128-byte swizzle rows (one row: 64 for 16-bit, 128 for 8-bit
// types).  HALVES = 2 for 512-wide tiles: B's tile rows are two 256-row
// halves (one MMA each), every CTA loads its 256 / CG rows of each half; the
// stage holds B as [atom][half][rows of the half].  Like the MMA issuer, this
// warp's loop is near its per-stage budget, so both are template arguments.
//
// PARTS selects the copies this warp issues: kPartA (A, and the leader
// CTA's expect_tx for the whole stage), kPartB0 (B, or B's first half),
// kPartB1 (B's second half).  On GB300 a thread's TMA issue slows to about
// 290 cycles a box when the SM's copies back up, so a 128 x 256 stage (two
// boxes) issued by one warp takes longer than its 512 cycles of MMA; two
// warps issuing A and B side by side each stay inside it.  Bytes of B may
// land before A's warp posts the expect_tx: the barrier's pending arrival
// keeps the phase open meanwhile (its tx-count may go below zero).
constexpr uint32_t kPartA = 1u, kPartB0 = 2u, kPartB1 = 4u, kPartsAll = 7u;
//
// kSerpentine: a cluster's odd-numbered whole tiles sweep K backwards.  The
// clusters move through their tiles in step, one wave at a time, and a wave
// touches more A and B (plus the D it writes) than L2 holds, so in a forward
// sweep each wave finds its first K slices evicted.  Backwards, a wave starts
// on the slices the previous one read last (8192^3 on GB300: 845 -> 694 MB
// read from DRAM, 1.2 % faster at the power cap).  Only the summation order
// of the tile changes; a kernel that applies per-K-block scales keeps it off.
template <int CG, int ATOMS = 1, int HALVES = 1, uint32_t PARTS = kPartsAll, bool kSerpentine = false>
__device__ void producer_loop(const PersistentParams& p, uint8_t* ring, uint32_t stage_bytes, int tile_k,
                              uint32_t full0, uint32_t empty0, volatile uint32_t* abort_flag, uint32_t rank,
                              int cluster_id, int num_clusters) {
    constexpr uint32_t parts = PARTS;
    const int S = p.stages;
    const bool leader = rank == 0;
    const uint64_t tmo = p.timeout_ns;
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool aborted = false;
    const uint32_t tx_bytes = (uint32_t)CG * stage_bytes;
    const int b_rows = p.tile_n / CG;
    const int atom_k = tile_k / ATOMS;
    const int mn_elems = p.mn_box_elems > 0 ? p.mn_box_elems : 64;
    const uint32_t mn_box_bytes = 128u * (uint32_t)tile_k;     // one MN-major box: tile_k rows of 128 B
    // Consecutive waves of a raster group reuse its A panels: keep them in L2.
    const bool keep_a = (p.l2_hints & kHintKeepA) != 0;
    const uint64_t pol_a = l2_policy_evict_last();
    // pair: every CTA's copies complete on the leader's barrier
    const uint32_t fb0 = (CG == 2) ? map_to_cta(full0, 0) : full0;
    const bool drop_any = (p.flags & GEMM_FLAG_TEST_DROP_LOAD) && blockIdx.x == 0;
    WorkUnit u;
    for (int idx = 0; !aborted && next_unit(p, cluster_id, num_clusters, idx, u); ++idx) {
        const int t = u.tile;
        int b, mb, nb;
        tile_coords(p, t, b, mb, nb);
        const int a_row = mb * (128 * CG) + (int)rank * 128;
        const int b_row = nb * p.tile_n + (int)rank * b_rows;
        // 512-wide tiles: the unit's stages, split ones included (units.cuh)
        const int n = u.kb1 - u.kb0;
        const int L = split_stages(u, HALVES == 2);
        for (int i = 0; i < n + L; ++i) {
            int walk, halves;
            stage_of(i, n, L, walk, halves);
            const int kb = u.kb0 + walk;
            if (!wait_phase_warp<false, true>(empty0 + 8u * stage, phase ^ 1u, abort_flag, tmo, p.status,
                                              kRoleProducer, stage, t)) {
                aborted = true;
                break;
            }
            const uint32_t fb = fb0 + 8u * stage;
            const bool drop = drop_any && issued == 0;
            if (elect_one()) {
                if (leader && (parts & kPartA) != 0) {
                    // a split stage carries one of B's two halves
                    const uint32_t tx = halves == kHalvesBoth ? tx_bytes
                                                              : tx_bytes - (uint32_t)CG * (p.stage_bytes_b / 2u);
                    mbar_arrive_expect_tx(full0 + 8u * stage, tx);
                }
                if (!drop) {
                    const uint32_t sa = smem_u32(ring + (size_t)stage * stage_bytes);
                    const uint32_t sb = sa + p.stage_bytes_a;
                    // the K block loaded: backwards on a cluster's odd whole tiles (kSerpentine)
                    const bool back = kSerpentine && u.role == kUnitWhole && (idx & 1);
                    const int kx = (back ? u.kb0 + u.kb1 - 1 - kb : kb) * tile_k;
                    if constexpr ((parts & kPartA) != 0)
                        load_operand<CG, ATOMS>(sa, &p.tmap_a, fb, p.mn_major_a != 0, 128, a_row, kx, b,
                                                p.batched != 0, keep_a, pol_a, atom_k, 0, mn_elems, mn_box_bytes);
                    if constexpr (HALVES == 1) {
                        if constexpr ((parts & kPartB0) != 0)
                            load_operand<CG, ATOMS>(sb, &p.tmap_b, fb, p.mn_major_b != 0, b_rows, b_row, kx, b,
                                                    p.batched != 0, false, pol_a, atom_k, 0, mn_elems, mn_box_bytes);
                    } else {
                        constexpr int kHalfRows = 256 / CG;
#pragma unroll
                        for (int h = 0; h < HALVES; ++h)
                            if ((parts & (kPartB0 << h)) != 0 && (halves & (1 << h)) != 0)
                                load_operand<CG, ATOMS>(sb + (uint32_t)(h * kHalfRows * 128), &p.tmap_b, fb, false,
                                                        kHalfRows, nb * p.tile_n + h * 256 + (int)rank * kHalfRows,
                                                        kx, b, p.batched != 0, false, pol_a, atom_k,
                                                        (uint32_t)b_rows * 128u);
                    }
                }
            }
            __syncwarp();
            ++issued;
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    }
    if (!aborted) {
        // Tail: wait until the MMA released every slot, so that no commit
        // arrives on this CTA's barriers after it exits.
        for (int i = 0; i < S; ++i) {
            if (!wait_phase_warp<false>(empty0 + 8u * stage, phase ^ 1u, abort_flag, tmo, p.status,
                                        kRoleProducer, stage, 0xFFFFFFFFu))
                break;
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    } else if (leader && (parts & kPartA) != 0) {
        // Abort: wait (bounded) for the copies still in flight into the ring
        // (a stage's barrier counts the bytes of every warp's copies).
        int s = stage;
        uint32_t ph = phase;
        const int n = issued < S ? issued : S;
        for (int i = 0; i < n; ++i) {
            if (s == 0) { s = S - 1; ph ^= 1u; } else { --s; }
            wait_phase_drain(full0 + 8u * s, ph, tmo);
        }
    }
}

}  // namespace dgb
