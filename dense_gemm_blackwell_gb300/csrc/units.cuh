// units.cuh -- which output tile, and which K blocks of it, each cluster of a
// persistent kernel works on, in order.  Host and device compile the same
// functions: the kernels call them per unit, and gemm_plan_work_unit exposes
// them to the host so that the schedule can be checked without a GPU.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dgb {

// Linear tile index -> (batch, m block, n block); tiles of one batch entry are
// visited in groups of `group_m` m blocks, m fastest inside a group, so that
// the CTAs of one wave share A and B panels and consecutive waves of a group
// share its A panels in L2.
__host__ __device__ __forceinline__ void tile_coords(const PersistentParams& p, int t, int& b, int& mb, int& nb) {
    b = t / p.tiles_per_batch;
    const int r = t - b * p.tiles_per_batch;
    const int span = p.group_m * p.num_n_blocks;
    const int g = r / span;
    const int first_m = g * p.group_m;
    const int gm = p.num_m_blocks - first_m < p.group_m ? p.num_m_blocks - first_m : p.group_m;
    const int rr = r - g * span;
    mb = first_m + rr % gm;
    nb = rr / gm;
}

// One piece of work of a cluster: K blocks [kb0, kb1) of one output tile.
struct WorkUnit {
    int tile;
    int kb0, kb1;
    int role;    // kUnitWhole, kUnitContributor or kUnitFinisher
    int slot;    // partial slot written (contributor) or the last one read (finisher)
    int slot0;   // finisher: the first partial slot read; it adds slots slot, slot-1, ..., slot0
};
constexpr int kUnitWhole = 0, kUnitContributor = 1, kUnitFinisher = 2;

// The idx-th unit of cluster c (of G) in processing order.
//  1. Stream-K region (tiles [T - sk_tiles, T)): its sk_tiles * nk K blocks
//     are cut into G contiguous ranges, one per cluster, and each range into
//     segments at tile boundaries.  A segment that ends its tile but does not
//     start it is a finisher; one that does not end its tile is a contributor
//     and leaves its fp32 partial in slot c (only a range's last segment can
//     be one); the rest are whole tiles.  With ranges at least one tile long
//     (sk_tiles >= G) a tile is split between clusters c-1 and c.  With fewer
//     tiles than clusters (sk_tiles == T < G) ranges are shorter, and the
//     contributors of a tile are all the clusters slot0 .. c-1 before its
//     finisher c.  A cluster walks its range from the last segment to the
//     first: it publishes its contributor partial before anything else and
//     reaches its finisher segment last, so a finisher waits only on
//     clusters that wait on no one.
//  2. Data-parallel tiles c, c+G, ... of [0, T - sk_tiles).  Run after the
//     stream-K region, they hide a finisher's fix-up behind the MMAs of the
//     cluster's next tile; without them the finisher is the cluster's last
//     unit and its fix-up the kernel's tail.
__host__ __device__ __forceinline__ bool next_unit(const PersistentParams& p, int c, int G, int idx, WorkUnit& u) {
    const int nk = p.num_k_blocks;
    const int dp_tiles = p.num_tiles - p.sk_tiles;
    if (p.sk_tiles > 0) {
        const int64_t total = (int64_t)p.sk_tiles * nk;
        const int64_t it0 = total * c / G;
        int64_t hi = total * (c + 1) / G;
        int k = 0;
        while (hi > it0) {
            const int64_t j = (hi - 1) / nk;
            const int64_t lo = it0 > j * nk ? it0 : j * nk;
            if (k == idx) {
                u.tile = dp_tiles + (int)j;
                u.kb0 = (int)(lo - j * nk);
                u.kb1 = (int)(hi - j * nk);
                const bool starts = u.kb0 == 0, ends = u.kb1 == nk;
                u.role = ends ? (starts ? kUnitWhole : kUnitFinisher) : kUnitContributor;
                u.slot = ends ? (starts ? 0 : c - 1) : c;
                // the cluster whose range holds the tile's first K block:
                // the largest c0 with floor(total * c0 / G) <= j * nk
                u.slot0 = (u.role == kUnitFinisher) ? (int)(((j * nk + 1) * G + total - 1) / total - 1) : u.slot;
                return true;
            }
            ++k;
            hi = lo;
        }
        idx -= k;
    }
    const int t = c + idx * G;
    if (t >= dp_tiles) return false;
    u.tile = t;
    u.kb0 = 0;
    u.kb1 = nk;
    u.role = kUnitWhole;
    u.slot = 0;
    u.slot0 = 0;
    return true;
}

// 512-wide tiles hold one accumulator of two 256-column halves, and the next
// tile can start only on a half the epilogue has drained.  A whole unit of
// such a tile therefore runs its first kSplitStages K blocks for the left half
// alone and repeats them for the right half alone after its last K block: the
// left half is complete kSplitStages stages before the right one, so it
// drains while the tile's right-only stages run, and the right half drains
// while the next tile's left-only stages run.  Those stages carry A and one
// half of B.  Units with fewer than 4 x kSplitStages K blocks run every stage
// on both halves.  Six split stages measured best on GB300 (8192^3 and 4096^3
// bf16, 2 % faster than none; from eight on, the extra half-stages, which take
// in A and half of B per 512 MMA cycles, cost more than the hidden drain).
constexpr int kSplitStages = 6;

__host__ __device__ __forceinline__ int split_stages(const WorkUnit& u, bool wide) {
    return (wide && u.role == kUnitWhole && u.kb1 - u.kb0 >= 4 * kSplitStages) ? kSplitStages : 0;
}

// Stage i (0 <= i < n + L) of a unit of n K blocks with L split stages: the
// position of its K block in the unit's walk, and the accumulator halves it
// feeds (bit 0: left, bit 1: right).
constexpr int kHalfLeft = 1, kHalfRight = 2, kHalvesBoth = 3;
__host__ __device__ __forceinline__ void stage_of(int i, int n, int L, int& walk, int& halves) {
    if (i < L) {
        walk = i;
        halves = kHalfLeft;
    } else if (i < n) {
        walk = i;
        halves = kHalvesBoth;
    } else {
        walk = i - n;
        halves = kHalfRight;
    }
}

}  // namespace dgb
