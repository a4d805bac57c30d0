// kernels_single.cu -- one-CTA tcgen05 GEMM for small problems, and the K == 0 fill.
//
// The single-CTA kernel follows the life of one accumulator in the TVM TIRx
// "Blackwell Tensor Cores" guide (section "The Accumulator's Lifetime"):
// warp 0 allocates tensor memory; thread 0 initialises an mbarrier; all 128
// threads stage A and B into 128-byte-swizzled shared memory; a proxy fence
// and a CTA barrier hand the tiles to the tensor core; thread 0 issues one
// tcgen05.mma per 16-deep K slice (the first starts a fresh accumulator) and
// commits them to the mbarrier; every thread waits for phase 0, fences, and
// each warp reads its 32 TMEM lanes (one output row per thread); a final CTA
// barrier keeps TMEM alive until warp 0 frees it.
//
// Generalised from the guide's 128x64 . (64x64)^T: M <= 128 rows (padded with
// zero rows), N <= 256 (padded to a multiple of 16 -- the MMA's N step for
// M = 128), K <= 256 (padded to 64-deep swizzle rows), either majorness (the
// threads read any stride), one CTA per batch entry.  The wait on the MMA is
// bounded; on expiry the kernel records GEMM_ERR_TIMEOUT and skips its stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace dgb {

template <int OUT>
__device__ __forceinline__ void store_out(void* D, int64_t idx, float v) {
    if constexpr (OUT == GEMM_F32) {
        static_cast<float*>(D)[idx] = v;
    } else if constexpr (OUT == GEMM_BF16) {
        static_cast<__nv_bfloat16*>(D)[idx] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half*>(D)[idx] = __float2half_rn(v);
    }
}

// One 64-deep swizzle row block (K elements kbase .. kbase + 63) of an operand
// row, zero past K or past the last row: chunk j (8 elements, 16 bytes) lands
// at 16-byte position j ^ (row mod 8) of the row's 128 bytes.  A K-major row
// whose block lies inside K takes eight 16-byte loads, all in flight before the
// stores (rows start on 16-byte boundaries: leading dimensions are multiples of
// 16 bytes); other rows go element by element.
__device__ __forceinline__ void stage_row(uint8_t* block, int row, const uint16_t* src, int64_t row_stride,
                                          int64_t k_stride, int kbase, int K, bool row_ok) {
    uint8_t* dst = block + row * 128;
    if (row_ok && k_stride == 1 && kbase + 64 <= K) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + row * row_stride + kbase);
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldg(s4 + j);
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(dst + ((j ^ (row & 7)) << 4)) = v[j];
        return;
    }
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k_lo = kbase + 8 * j + 2 * e, k_hi = k_lo + 1;
            const uint32_t lo = (row_ok && k_lo < K) ? src[row * row_stride + k_lo * k_stride] : 0u;
            const uint32_t hi = (row_ok && k_hi < K) ? src[row * row_stride + k_hi * k_stride] : 0u;
            w[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(dst + ((j ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 32 consecutive outputs of one row (columns col0 ..), 16 bytes per store when
// all of them are in range (D's rows start on 16-byte boundaries and col0 is a
// multiple of 32), element by element at the ragged right edge.
template <int OUT>
__device__ __forceinline__ void store_row32(void* D, int64_t base, int col0, int N, const uint32_t (&r)[32]) {
    if (col0 + 32 <= N) {
        if constexpr (OUT == GEMM_F32) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(D) + base + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(D) + base + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack2<OUT>(__uint_as_float(r[8 * q + 2 * e]), __uint_as_float(r[8 * q + 2 * e + 1]));
                dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < N) store_out<OUT>(D, base + col0 + i, __uint_as_float(r[i]));
    }
}

template <int OUT>
__global__ void __launch_bounds__(128, 1) single_cta_kernel(const __grid_constant__ SingleParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int kblocks = p.k_pad / 64;
    uint8_t* sa = smem;                                   // kblocks x (128 rows x 128 B)
    uint8_t* sb = sa + kblocks * 128 * 128;               // kblocks x (n_pad rows x 128 B)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sb + kblocks * p.n_pad * 128);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t b = blockIdx.x;

    if (warp == 0) {
        tmem_alloc<1>(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish<1>();
    }
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // the previous kernel of the stream may still be running up to here
    griddep_wait();
    griddep_launch_dependents();

    // Stage A (row = tid) and B (rows tid, tid+128) into the swizzled layout.
    const uint16_t* A = static_cast<const uint16_t*>(p.A) + b * p.stride_a;
    const uint16_t* B = static_cast<const uint16_t*>(p.B) + b * p.stride_b;
    const int64_t a_rs = p.major_a == GEMM_K_MAJOR ? p.lda : 1, a_ks = p.major_a == GEMM_K_MAJOR ? 1 : p.lda;
    const int64_t b_rs = p.major_b == GEMM_K_MAJOR ? p.ldb : 1, b_ks = p.major_b == GEMM_K_MAJOR ? 1 : p.ldb;
    for (int kb = 0; kb < kblocks; ++kb) {
        stage_row(sa + kb * 128 * 128, tid, A, a_rs, a_ks, kb * 64, p.K, tid < p.M);
        for (int r = tid; r < p.n_pad; r += 128)
            stage_row(sb + kb * p.n_pad * 128, r, B, b_rs, b_ks, kb * 64, p.K, r < p.N);
    }
    // Generic-proxy writes -> async proxy (the tensor core), then publish to thread 0.
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint32_t a0 = smem_u32(sa + kb * 128 * 128);
            const uint32_t b0 = smem_u32(sb + kb * p.n_pad * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16<1>(tmem, smem_desc_sw128(a0 + 32 * kk), smem_desc_sw128(b0 + 32 * kk), p.idesc,
                           (kb | kk) != 0);
        }
        mma_commit(smem_u32(bar));
    }
    __syncwarp();

    bool ok = wait_phase<false>(smem_u32(bar), 0, abort_flag, p.timeout_ns, p.status, kRoleSingle, 0,
                                blockIdx.x);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
        const int row = warp * 32 + lane;
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        for (int c = 0; c * 32 < p.n_pad; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(lane_base + c * 32, r);
            tmem_wait_ld();
            tmem_reg_fence(r);
            if (row < p.M) store_row32<OUT>(p.D, b * p.stride_d + (int64_t)row * p.ldd, c * 32, p.N, r);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, (uint32_t)p.tmem_cols);
    }
}

template <int OUT>
__global__ void zero_fill_kernel(void* D, int64_t M, int64_t N, int64_t batch, int64_t ldd, int64_t stride_d) {
    const int64_t total = M * N * batch;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / (M * N), r = i % (M * N);
        store_out<OUT>(D, b * stride_d + (r / N) * ldd + (r % N), 0.0f);
    }
}

template <int OUT>
static cudaError_t launch_single_typed(const SingleParams& p, int batch, size_t smem, cudaStream_t stream) {
    auto kern = single_cta_kernel<OUT>;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_single_cta(const SingleParams& p, int dtype_d, int batch, size_t smem_bytes,
                              cudaStream_t stream) {
    switch (dtype_d) {
    case GEMM_F32: return launch_single_typed<GEMM_F32>(p, batch, smem_bytes, stream);
    case GEMM_BF16: return launch_single_typed<GEMM_BF16>(p, batch, smem_bytes, stream);
    case GEMM_F16: return launch_single_typed<GEMM_F16>(p, batch, smem_bytes, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_zero_fill(void* D, int dtype_d, int64_t M, int64_t N, int64_t batch, int64_t ldd,
                             int64_t stride_d, int sm_count, cudaStream_t stream) {
    const int64_t total = M * N * batch;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    if (blocks < 1) blocks = 1;
    switch (dtype_d) {
    case GEMM_F32: zero_fill_kernel<GEMM_F32><<<(unsigned)blocks, threads, 0, stream>>>(D, M, N, batch, ldd, stride_d); break;
    case GEMM_BF16: zero_fill_kernel<GEMM_BF16><<<(unsigned)blocks, threads, 0, stream>>>(D, M, N, batch, ldd, stride_d); break;
    case GEMM_F16: zero_fill_kernel<GEMM_F16><<<(unsigned)blocks, threads, 0, stream>>>(D, M, N, batch, ldd, stride_d); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace dgb
