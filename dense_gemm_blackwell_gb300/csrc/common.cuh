// common.cuh -- descriptors, launch parameters and bounded waits shared by the
// GEMM kernels (host and device).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm.h"
#include "ptx.cuh"

namespace dgb {

// ---------------------------------------------------------------- descriptors
//
// Shared-memory matrix descriptor for tcgen05.mma (public PTX ISA, "Shared
// memory descriptor"; the pages do not print its bits):
//   [0,14)  start address >> 4         [16,30) leading-dim byte offset >> 4
//   [32,46) stride-dim byte offset >> 4 [46,48) version = 1
//   [49,52) base offset                 [52]    LBO mode (0 = relative)
//   [61,64) swizzle: 0 none, 1 128B/32B-atom, 2 128B, 4 64B, 6 32B
//
// Operand tiles are K-major with the 128-byte swizzle (TVM TIRx "Blackwell
// Tensor Cores": swizzle mode 3 = 128 B, 1024-byte period, hence 1024-byte
// tile alignment).  Each row of a tile is 128 bytes of K; eight rows form one
// 1024-byte swizzle atom, so the stride between 8-row groups is 1024 bytes.
// The leading-dim offset is unused when one MMA's K (32 bytes) lies inside
// the 128-byte swizzle row.  Advancing K by 32 bytes inside the row is a +2
// on the start-address field: the swizzle is applied to absolute address
// bits, so a 1024-aligned tile keeps matching what TMA wrote.
constexpr uint64_t kSmemDescSw128KMajorBase =
    (uint64_t(1) << 16) |            // LBO (unused), 16 bytes
    (uint64_t(1024 >> 4) << 32) |    // SBO: 8 rows x 128 B
    (uint64_t(1) << 46) |            // descriptor version for tcgen05
    (uint64_t(2) << 61);             // 128-byte swizzle

__host__ __device__ constexpr uint64_t smem_desc_sw128(uint32_t smem_addr) {
    return kSmemDescSw128KMajorBase | uint64_t((smem_addr >> 4) & 0x3FFFu);
}

// MN-major operand (M or N contiguous in memory) with the 128-byte swizzle:
// each 128-byte row holds 128 bytes of consecutive M (or N) elements of one k
// (64 16-bit or 128 8-bit elements), eight k-rows form a 1024-byte atom.  The
// tile is stored as TMA boxes of one such row width x tile_k k-rows, side by
// side along M/N.  Leading-dim offset = the box size (8 KB for 16-bit,
// 64 k-rows; 16 KB for 8-bit, 128 k-rows) between atoms along M/N; stride-dim
// offset = 1024 B between groups of 8 k-rows.  One MMA spans 16 (K16) or 32
// (K32) k-rows: +2048 or +4096 B per MMA.
constexpr uint32_t kMNMajorBoxBytes = 64 * 128;
constexpr uint64_t kSmemDescSw128MNMajorBase =
    (uint64_t(kMNMajorBoxBytes >> 4) << 16) |   // LBO: next 64 elements of M/N
    (uint64_t(1024 >> 4) << 32) |                // SBO: next 8 k-rows
    (uint64_t(1) << 46) |
    (uint64_t(2) << 61);

__host__ __device__ constexpr uint64_t smem_desc_sw128_mn(uint32_t smem_addr) {
    return kSmemDescSw128MNMajorBase | uint64_t((smem_addr >> 4) & 0x3FFFu);
}

// Same with a given leading-dim offset (the MN-major box size in bytes).
__host__ __device__ constexpr uint64_t smem_desc_sw128_mn_lbo(uint32_t smem_addr, uint32_t lbo_bytes) {
    return (uint64_t(lbo_bytes >> 4) << 16) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) |
           (uint64_t(2) << 61) | uint64_t((smem_addr >> 4) & 0x3FFFu);
}

// Instruction descriptor of tcgen05.mma kind::f16 / kind::f8f6f4 (public PTX ISA):
//   [4,6) D format (0 = f16, 1 = f32)   [7,10) A format   [10,13) B format
//   [15] A major (0 = K)       [16] B major      [17,23) N >> 3   [24,29) M >> 4
// A/B format for kind::f16: 0 = f16, 1 = bf16; for kind::f8f6f4: 0 = e4m3.
// kind::tf32: 2 = tf32.  kind::f8f6f4: 0 = e4m3, 1 = e5m2 (A and B independently).
__host__ __device__ constexpr uint32_t make_idesc2(uint32_t a_format, uint32_t b_format, uint32_t m, uint32_t n,
                                                   uint32_t a_mn_major = 0, uint32_t b_mn_major = 0,
                                                   uint32_t d_format = 1) {
    return (d_format << 4) | (a_format << 7) | (b_format << 10) | (a_mn_major << 15) |
           (b_mn_major << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, uint32_t m, uint32_t n,
                                                  uint32_t a_mn_major = 0, uint32_t b_mn_major = 0) {
    return make_idesc2(ab_format, ab_format, m, n, a_mn_major, b_mn_major);
}
constexpr uint32_t kMmaKindF16 = 0, kMmaKindTF32 = 1;

// ---------------------------------------------------------------- parameters

enum Role : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleSingle = 4 };

// Persistent warp-specialised kernel: one CTA (or CTA pair) per SM, loops over
// output tiles.  Passed by value as a __grid_constant__ parameter.
struct PersistentParams {
    CUtensorMap tmap_a;   // A: (K, M[, batch]) box (tile_k, 128[, 1])
    CUtensorMap tmap_b;   // B: (K, N[, batch]) box (tile_k, tile_n / cta_group[, 1])
    CUtensorMap tmap_d;   // D: (N, M[, batch]) box (128 B of columns, 32[, 1])
    gemm_device_error_t* status;
    const float* scale_a; // block-scaled kernels only: [b][m][k/128] and [b][n/128][k/128]
    const float* scale_b;
    int64_t ld_sa, ld_sb;
    int64_t stride_sa, stride_sb;
    int32_t M, N, K, batch;
    int32_t num_m_blocks, num_n_blocks, num_k_blocks;
    int32_t tiles_per_batch, num_tiles;
    int32_t tile_n, stages, tmem_cols, tmem_stages;
    int32_t group_m;
    int32_t batched;          // 1 = 3-D tensor maps
    int32_t tile_k;           // elements of K per ring stage (k_atoms 128-byte swizzle rows)
    int32_t k_atoms;          // 128-byte K atoms per stage (1 or 2; 2 only with K-major operands)
    uint32_t mma_kind;        // kMmaKindF16 or kMmaKindTF32 (16-bit kernel only)
    int32_t mn_major_a;       // 1: A is M-contiguous (loaded as 64x64 boxes, MN-major descriptor)
    int32_t mn_major_b;       // 1: B is N-contiguous
    int32_t acc_f16;          // 1: the accumulator is fp16 (one per 32-bit TMEM column, low half)
    int32_t mn_box_elems;     // MN-major boxes: elements along M/N per 128-byte row (64 or 128)
    uint32_t idesc;
    uint32_t stage_bytes_a;   // per CTA
    uint32_t stage_bytes_b;   // per CTA
    uint32_t flags;
    uint32_t l2_hints;        // bit 0: A loads evict_last; bit 1: D stores evict_first
    uint64_t timeout_ns;
    // Stream-K: the last sk_tiles tiles of the raster are split into equal K
    // ranges over all clusters and processed first.  A contributor (a part of
    // a tile that does not end it) leaves its fp32 partial in
    // sk_partials[slot] and publishes sk_flags = the launch's epoch; the
    // finisher (the part that ends the tile) adds every contributor's
    // partial before storing D.
    int32_t sk_tiles;
    // Epilogue without shared-memory staging: each thread writes its row's
    // 128-byte chunks straight to D (frees the staging area for a ring stage).
    int32_t direct_store;
    void* d_ptr;
    int64_t ldd, stride_d;
    float* sk_partials;       // [slot][cta rank][128 rows x tile_n], layout of sk_partial_index
    uint32_t* sk_flags;       // [slot][cta rank][8 epilogue warps]
    // Launch counter in device memory, so that a launch replayed from a CUDA
    // graph (same parameters) still gets a fresh epoch: [0] the epoch of the
    // last launch that completed, [1] CTAs of the running launch that finished.
    uint32_t* sk_epoch;
};

// The epoch of this launch: one past the last completed one (never 0, the
// flags' initial value).  A CTA reads the same value whenever it asks before
// its own finish, since the counter moves only once every CTA has finished.
__device__ __forceinline__ uint32_t sk_launch_epoch(const uint32_t* sk_epoch) {
    uint32_t last;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(last) : "l"(sk_epoch) : "memory");
    return last + 1u == 0u ? 1u : last + 1u;
}

// Called by one thread of each CTA after all of its threads are done: the
// last CTA to finish publishes the launch's epoch for the next launch.
__device__ __forceinline__ void sk_finish_launch(uint32_t* sk_epoch, uint32_t epoch) {
    __threadfence();
    if (atomicAdd(sk_epoch + 1, 1u) == gridDim.x - 1) {
        sk_epoch[1] = 0u;
        sk_epoch[0] = epoch;
        __threadfence();
    }
}

constexpr uint32_t kHintKeepA = 1u;
constexpr uint32_t kHintStreamD = 2u;

// Single-CTA kernel: one CTA per batch entry, threads stage the operands.
struct SingleParams {
    const void* A;
    const void* B;
    void* D;
    gemm_device_error_t* status;
    int64_t lda, ldb, ldd, stride_a, stride_b, stride_d;
    int32_t M, N, K;
    int32_t n_pad, k_pad;     // N rounded up to 16, K rounded up to 64
    int32_t major_a, major_b;
    int32_t tmem_cols;
    uint32_t idesc;
    uint64_t timeout_ns;
};

// ---------------------------------------------------------------- host helpers

// Raise a kernel's dynamic shared-memory limit only when a launch needs more
// than any earlier launch on this device did (the attribute call costs a
// driver round trip; launches reuse the raised limit).
constexpr int kMaxDevices = 64;
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, size_t smem, std::atomic<int> (&done)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (done[dev].load(std::memory_order_acquire) >= (int)smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
        int prev = done[dev].load();
        while (prev < (int)smem && !done[dev].compare_exchange_weak(prev, (int)smem)) {}
    }
    return e;
}

// ---------------------------------------------------------------- bounded waits

// Record the first device-side timeout of a launch in the plan's status record.
__device__ __forceinline__ void report_timeout(gemm_device_error_t* st, uint32_t role,
                                               uint32_t stage, uint32_t tile) {
    if (st == nullptr) return;
    if (atomicCAS(&st->code, 0u, (uint32_t)GEMM_ERR_TIMEOUT) == 0u) {
        st->role = role;
        st->stage = stage;
        st->tile = tile;
        st->block = blockIdx.x;
        __threadfence();
    }
}

// Bounded wait on an mbarrier phase.  Returns true when the phase completed,
// false when the CTA's abort flag was raised or `timeout_ns` elapsed (the
// timeout is recorded and the abort flag raised).  Callers leave their loops
// on false; every wait in the kernels goes through this function.
template <bool kClusterScope>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                           uint64_t timeout_ns, gemm_device_error_t* st,
                                           uint32_t role, uint32_t stage, uint32_t tile) {
    auto probe = [&]() {
        return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (probe()) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            report_timeout(st, role, stage, tile);
            *abort_flag = 1u;
            return false;
        }
    }
}

// Same, called by every lane of a warp, with the same result in every lane.
// The issuing warps (TMA producer, MMA) run their loops warp-uniformly and let
// one elected lane issue: on GB300 an MMA issue loop whose single divergent
// lane also waits spends about 460 cycles per barrier wait and four MMAs,
// against about 330 this way.
template <bool kClusterScope, bool kRelaxed = false>
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                uint64_t timeout_ns, gemm_device_error_t* st,
                                                uint32_t role, uint32_t stage, uint32_t tile) {
    auto probe = [&]() {
        if constexpr (kRelaxed) return mbar_try_wait_relaxed(bar, parity);
        else return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (__all_sync(0xffffffffu, probe())) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, probe())) return true;
        if (__shfl_sync(0xffffffffu, *abort_flag ? 1 : 0, 0)) return false;
        if (__shfl_sync(0xffffffffu, (globaltimer_ns() - t0 > timeout_ns) ? 1 : 0, 0)) {
            if ((threadIdx.x & 31) == 0) {
                report_timeout(st, role, stage, tile);
                *abort_flag = 1u;
            }
            __syncwarp();
            return false;
        }
    }
}

// Bounded wait until a flag in global memory equals `value` (acquire, GPU
// scope).  Same abort/timeout behaviour as wait_phase.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t value, volatile uint32_t* abort_flag,
                                          uint64_t timeout_ns, gemm_device_error_t* st, uint32_t role,
                                          uint32_t stage, uint32_t tile) {
    auto probe = [&]() {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        return v == value;
    };
    if (probe()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (probe()) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            report_timeout(st, role, stage, tile);
            *abort_flag = 1u;
            return false;
        }
    }
}

__device__ __forceinline__ void store_release_gpu(uint32_t* flag, uint32_t value) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(flag), "r"(value) : "memory");
}

// Wait that ignores the abort flag (used while draining in-flight copies on
// the abort path); bounded by `timeout_ns`, result not reported.
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

}  // namespace dgb
