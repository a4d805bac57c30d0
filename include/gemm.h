/*
 * gemm.h -- C ABI of a dense GEMM for one NVIDIA GB300 (sm_103a).
 *
 * Computes, for every batch entry b:
 *
 *     D[b] = A[b] * B[b]^T          (fp32 accumulation, one rounding to D's type)
 *
 * "Out = A @ B.T" is the product of the TVM TIRx "Blackwell Tensor Cores"
 * guide (section "The Accumulator's Lifetime"); accumulation starts fresh on
 * the first K slice and there is no alpha/beta -- scaling belongs to the
 * caller (TVM TIRx "mma.sync", section "Accumulation, transpose and
 * alpha/beta").  Block-scaled 8-bit inputs multiply every 1x128 block of a
 * row of A and every 128x128 block of B by its own fp32 scale ("Hopper and
 * Blackwell GEMM", concept "FP8 and FP4, with block scaling").
 *
 * Element addressing (elements, not bytes):
 *   A, K-major  : A[b*stride_a + m*lda + k]    A, MN-major : A[b*stride_a + k*lda + m]
 *   B, K-major  : B[b*stride_b + n*ldb + k]    B, MN-major : B[b*stride_b + k*ldb + n]
 *   D (row-major): D[b*stride_d + m*ldd + n]
 *   scale_a     : scale_a[b*stride_sa + m*ld_sa + k/128]           (fp32 block scales only)
 *   scale_b     : scale_b[b*stride_sb + (n/128)*ld_sb + k/128]     (fp32 block scales only)
 * "row-major A, column-major B" in BLAS terms is K-major A and K-major B (TN).
 * GEMM_E2M1 elements are packed two per byte, element k of a row in the low
 * nibble of byte k/2 when k is even and in the high nibble when k is odd;
 * leading dims and batch strides still count elements.
 *
 * Hardware block scaling (GEMM_SCALE_MX_E8M0_32, GEMM_SCALE_NV_E4M3_16; the
 * formats of "Hopper and Blackwell GEMM", concept "FP8 and FP4, with block
 * scaling"): each row of A and each row of B (K-major) is cut along K into
 * blocks of V elements (V = 32 for MX, 16 for NV), every block with one scale
 * byte (MX: E8M0, 2^(e-127), 0xFF is NaN; NV: E4M3 with sign bit 0).  For a
 * matrix with R rows and KB = ceil(K/V) scale columns the scale bytes are
 * tiled as the tensor core reads them ("TMEM -- the accumulator's new home",
 * section "Block-scaled MMA": lane = row mod 32, column = row / 32): 512-byte
 * tiles of 128 rows x 4 scale columns,
 *   tile (r/128, kb/4) at byte  ((r/128) * ceil(KB/4) + kb/4) * 512
 *   inside a tile      at byte  (r mod 32) * 16 + ((r/32) mod 4) * 4 + kb mod 4
 * from the batch entry's start (stride_sa / stride_sb bytes apart; 0 = packed,
 * ceil(R/128) * ceil(KB/4) * 512).  Entries past R or KB must hold finite
 * codes (they meet zero-filled operands).  NV additionally multiplies D by
 * one fp32 scale per tensor, tA * tB.
 *
 * Ownership: the caller owns every device buffer and the stream; the library
 * never frees or retains them past the call that uses them.  A plan owns its
 * host state, one small device status record and, when the planner splits
 * the last wave's tiles along K (stream-K), a workspace for fp32 partial
 * tiles (all allocated by gemm_plan_create, freed by gemm_plan_destroy;
 * gemm_plan_info reports its size).
 *
 * Errors: every call returns a gemm_status_t; nothing throws across the ABI.
 * Unsupported combinations fail with GEMM_ERR_UNSUPPORTED -- never a silent
 * fallback to another kernel or to the CPU.
 *
 * Threading: calls on different plans are independent.  One plan may be run
 * on one stream, from one host thread, at a time (its status record and its
 * cached tensor maps are shared by its launches).
 */
#ifndef DENSE_GEMM_BLACKWELL_GB300_GEMM_H
#define DENSE_GEMM_BLACKWELL_GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, bad leading dim */
    GEMM_ERR_UNSUPPORTED = 2,  /* valid request this library does not implement */
    GEMM_ERR_ALIGNMENT = 3,    /* pointer or stride not a multiple of 16 bytes */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (see gemm_last_cuda_error) */
    GEMM_ERR_TIMEOUT = 5,      /* a device-side wait ran out; reported by gemm_sync_status */
    GEMM_ERR_NO_DEVICE = 6,    /* no sm_103 device is current */
    GEMM_ERR_RESOURCES = 7     /* shared/tensor memory budget cannot hold the requested tile */
} gemm_status_t;

/* Element types.  GEMM_TF32 is fp32 storage multiplied at tf32 precision (the
 * tensor core reads the top 19 bits of each fp32 value); GEMM_F32 is an output type. */
typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_E4M3 = 2, GEMM_F32 = 3, GEMM_E5M2 = 4, GEMM_TF32 = 5,
               GEMM_E2M1 = 6 } gemm_dtype_t;
typedef enum { GEMM_K_MAJOR = 0, GEMM_MN_MAJOR = 1 } gemm_major_t;
typedef enum {
    GEMM_SCALE_NONE = 0,
    GEMM_SCALE_BLOCK_1x128_128x128 = 1,  /* fp32 scale per 1x128 block of A and 128x128 block of B (gemm_run) */
    GEMM_SCALE_MX_E8M0_32 = 2,           /* MXFP8 (E4M3/E5M2) or MXFP4 (E2M1): E8M0 per 32, tiled (gemm_run_mx) */
    GEMM_SCALE_NV_E4M3_16 = 3            /* NVFP4 (E2M1): E4M3 per 16, tiled, times fp32 tA * tB (gemm_run_mx) */
} gemm_scale_mode_t;

/* Kernel families a plan can select. */
typedef enum {
    GEMM_KERNEL_SINGLE_CTA = 1,   /* one CTA per problem, threads stage operands (small problems) */
    GEMM_KERNEL_PERSISTENT = 2,   /* warp-specialised persistent TMA/tcgen05 pipeline */
    GEMM_KERNEL_FP8_BLOCK = 3,    /* persistent pipeline with per-block scale promotion */
    GEMM_KERNEL_ZERO_FILL = 4,    /* K == 0: D is written with zeros */
    GEMM_KERNEL_MX = 5            /* persistent pipeline with hardware block-scaled MMA (MX / NVFP4) */
} gemm_kernel_t;

/* gemm_desc_t.flags */
#define GEMM_FLAG_CTA_GROUP_1     (1u << 0)  /* force the single-SM MMA form */
#define GEMM_FLAG_CTA_GROUP_2     (1u << 1)  /* force the SM-pair (cta_group::2) MMA form */
#define GEMM_FLAG_NO_SINGLE_CTA   (1u << 2)  /* never choose GEMM_KERNEL_SINGLE_CTA */
#define GEMM_FLAG_SINGLE_CTA      (1u << 3)  /* require GEMM_KERNEL_SINGLE_CTA */
#define GEMM_FLAG_NO_L2_HINTS     (1u << 4)  /* issue copies without L2 eviction-priority hints */
#define GEMM_FLAG_NO_STREAM_K     (1u << 5)  /* data-parallel tiles only (no stream-K workspace) */
#define GEMM_FLAG_EPILOGUE_DIRECT (1u << 6)  /* force direct row stores of D (no staging area) */
#define GEMM_FLAG_EPILOGUE_TMA    (1u << 7)  /* force TMA stores of D through shared-memory staging */
#define GEMM_FLAG_STAGE_K1        (1u << 8)  /* 16-bit/tf32 persistent kernel: one 128-byte K atom per ring stage */
#define GEMM_FLAG_STAGE_K2        (1u << 9)  /* ... two 128-byte K atoms per ring stage (K-major operands only) */
#define GEMM_FLAG_ACCUM_F16       (1u << 10) /* f16 A and B only: accumulate in fp16 in tensor memory ("half inputs
                                                with a half or float accumulator", cuBLASDx "API Card: Blackwell
                                                Pipeline (tcgen05)", precision list); persistent kernel, no
                                                stream-K; partial sums must stay within fp16's range */
#define GEMM_FLAG_TEST_DROP_LOAD  (1u << 30) /* test only: the producer skips one stage's load so
                                                the consumer's bounded wait expires (GEMM_ERR_TIMEOUT) */

/* One GEMM problem.  Zero-valued optional fields take the documented default. */
typedef struct {
    int64_t M, N, K;        /* D is M x N per batch entry; K is the contraction length */
    int64_t batch;          /* number of independent problems (>= 1; 0 = no-op) */
    int32_t dtype_a, dtype_b;   /* gemm_dtype_t: F16+F16, BF16+BF16, TF32+TF32 (K-major), any pair of
                                   E4M3/E5M2 (fp32 block scales or MX), E2M1+E2M1 (MX or NV, K-major) */
    int32_t dtype_d;            /* gemm_dtype_t: F32, BF16 or F16 */
    int32_t major_a, major_b;   /* gemm_major_t */
    int32_t scale_mode;         /* gemm_scale_mode_t; BLOCK and MX require 8-bit or E2M1 inputs as listed */
    int64_t lda, ldb, ldd;      /* leading dims in elements; 0 = packed (K or M/N, and N for D) */
    int64_t stride_a, stride_b, stride_d;  /* elements between batch entries; 0 = packed */
    int64_t ld_sa, ld_sb;       /* fp32 block scales: leading dims in floats, 0 = ceil(K/128); MX/NV: must be 0 */
    int64_t stride_sa, stride_sb;  /* between batch entries of the scales: floats (fp32 block scales) or bytes
                                      (MX/NV tiles); 0 = packed */
    uint32_t flags;             /* GEMM_FLAG_* */
    int32_t tile_n;             /* N extent of one output tile: a multiple of 16 in 16..256, or 512 (16-bit/tf32
                                   K-major operands: two N = 256 MMAs per K step, one 512-column accumulator);
                                   block-scaled fp8: 128 or 256; MX/NV: 256; 0 = planner */
    int32_t stages;             /* shared-memory ring depth (2..16); 0 = planner */
    int32_t max_ctas;           /* cap on persistent CTAs; 0 = all SMs */
    uint64_t wait_timeout_ns;   /* bound on every device-side wait; 0 = 2 s */
    int32_t raster_group;       /* m blocks per raster group of the tile schedule; 0 = planner */
    int32_t reserved0;          /* must be 0 */
} gemm_desc_t;

/* The planner's decisions, as gemm_plan_query / gemm_plan_info report them. */
typedef struct {
    int32_t kernel;          /* gemm_kernel_t */
    int32_t cta_group;       /* 1 or 2 SMs per MMA */
    int32_t tile_m;          /* M extent of one MMA tile (128 per SM) */
    int32_t tile_n;          /* N extent of one output tile (512: two N = 256 MMAs per K step) */
    int32_t tile_k;          /* K depth of one ring stage (64 for 16-bit, 128 for 8-bit inputs) */
    int32_t stages;          /* shared-memory ring depth */
    int32_t tmem_stages;     /* accumulator buffers in tensor memory */
    int32_t tmem_cols;       /* tensor-memory columns allocated per CTA (power of two, <= 512) */
    int32_t grid;            /* CTAs launched */
    int32_t block_threads;   /* threads per CTA */
    int64_t num_tiles;       /* output tiles over all batch entries */
    int64_t stage_bytes;     /* bytes of one ring stage per CTA */
    int64_t pipeline_bytes;  /* ring + 8 B per barrier (2 per stage, 2 per TMEM stage) + 4 B TMEM handle */
    int64_t smem_bytes;      /* dynamic shared memory per CTA, all included */
    int32_t stream_k_tiles;  /* tiles whose K range is split between clusters (0 = data-parallel only) */
    int32_t epilogue;        /* 0 = TMA stores through shared-memory staging, 1 = direct row stores */
    int64_t workspace_bytes; /* device scratch the plan holds for stream-K partials and flags */
} gemm_plan_info_t;

/* Device properties the planner depends on (gemm_plan_query takes them explicitly). */
typedef struct {
    int32_t sm_count;            /* streaming multiprocessors */
    int32_t smem_optin_bytes;    /* cudaDevAttrMaxSharedMemoryPerBlockOptin */
    int32_t cc_major, cc_minor;  /* compute capability; this library runs on 10.3 only */
} gemm_device_props_t;

/* Device-side error record (gemm_sync_status). */
typedef struct {
    uint32_t code;    /* GEMM_OK or GEMM_ERR_TIMEOUT */
    uint32_t role;    /* 1 = TMA producer, 2 = MMA issuer, 3 = epilogue, 4 = single-CTA kernel */
    uint32_t stage;   /* ring stage or accumulator buffer being waited on */
    uint32_t tile;    /* linear output tile index */
    uint32_t block;   /* blockIdx.x of the CTA that timed out */
    uint32_t reserved[3];
} gemm_device_error_t;

typedef struct gemm_plan_s* gemm_plan_t;

/*
 * gemm_plan_query -- plan a problem for the given device properties without
 * touching any GPU (host arithmetic only).  Checks the descriptor's gates --
 * supported element types, tile shape legality (tcgen05: N a multiple of 16
 * up to 256, the accumulator within 512 tensor-memory columns), ring depth
 * within the shared-memory budget -- and fills *info.  The budget arithmetic
 * follows the cuBLASDx "API Card: Blackwell Pipeline (tcgen05)", section
 * "Depth and shared memory": one stage holds an A and a B tile, plus 8 bytes
 * per barrier and a 4-byte tensor-memory handle.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED or GEMM_ERR_RESOURCES.
 */
gemm_status_t gemm_plan_query(const gemm_desc_t* desc, const gemm_device_props_t* props,
                              gemm_plan_info_t* info);

/*
 * gemm_plan_create -- plan a problem on the current CUDA device and allocate
 * the plan's device status record.  *plan receives an opaque handle.
 * Returns GEMM_OK, or the gemm_plan_query codes, GEMM_ERR_NO_DEVICE (current
 * device is not compute capability 10.3) or GEMM_ERR_CUDA.
 */
gemm_status_t gemm_plan_create(gemm_plan_t* plan, const gemm_desc_t* desc);

/* gemm_plan_info -- copy the plan's decisions into *info. */
gemm_status_t gemm_plan_info(gemm_plan_t plan, gemm_plan_info_t* info);

/* One unit of a persistent kernel's work (see gemm_plan_work_unit). */
typedef struct {
    int32_t tile;            /* linear output tile, or -1: the cluster has no unit of that index */
    int32_t batch;           /* the tile's batch entry */
    int32_t m_block;         /* the tile covers D rows [m_block * tile_m, + tile_m) ... */
    int32_t n_block;         /* ... and columns [n_block * tile_n, + tile_n), clipped to M and N */
    int32_t k_block_begin;   /* contraction range [k_block_begin * tile_k, k_block_end * tile_k), */
    int32_t k_block_end;     /* clipped to K */
    int32_t role;            /* 0 whole tile; 1 stream-K contributor (leaves an fp32 partial);
                                2 stream-K finisher (adds the tile's partials and writes D) */
    int32_t slot;            /* partial slot written (role 1), or the last one read (role 2); 0 for role 0 */
    int32_t slot_first;      /* role 2: the first slot read -- the finisher adds the partials of slots
                                slot, slot - 1, ..., slot_first in that order; otherwise equal to slot */
} gemm_work_unit_t;

/*
 * gemm_plan_work_unit -- the index-th unit (0-based, in processing order) of
 * cluster `cluster` of a persistent plan; `desc` and `info` are the problem and
 * its plan (gemm_plan_query or gemm_plan_info).  A cluster is info->cta_group
 * CTAs sharing one MMA stream; there are info->grid / info->cta_group.  Host
 * arithmetic only, touching no GPU: the same schedule functions the kernels
 * run, compiled for the host, so a caller can check which tiles and K ranges
 * each SM (pair) takes.  Order: first the stream-K region's segments (the last
 * wave plus one full wave, or every tile when there are fewer tiles than
 * clusters, cut into equal K ranges, each cluster walking its range from the
 * end), then data-parallel tiles, raster groups of m blocks
 * first (the L2 reuse across a wave that the "Hopper and Blackwell GEMM" page
 * asks for next to its table of ridges).  The block-scaled kernel has no
 * stream-K region (its producers call the same functions; its MMA and
 * promotion loops step through the same tiles c, c + G, ... directly).
 * Past the cluster's last unit, out->tile is -1.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (null pointer, cluster outside
 * [0, grid / cta_group), negative index, or an info whose tile count or
 * stream-K region does not fit desc) or GEMM_ERR_UNSUPPORTED (a single-CTA
 * plan, which has no persistent schedule).
 */
gemm_status_t gemm_plan_work_unit(const gemm_desc_t* desc, const gemm_plan_info_t* info, int32_t cluster,
                                  int32_t index, gemm_work_unit_t* out);

/*
 * gemm_run -- enqueue D = A * B^T on `stream` (asynchronous, stream-ordered).
 * A, B, D are device pointers laid out as described at the top of this file;
 * scale_a / scale_b are device pointers for GEMM_SCALE_BLOCK_1x128_128x128 and
 * must be NULL otherwise.  A, B, D (and scales) must be 16-byte aligned and
 * every leading dimension / batch stride a multiple of 16 bytes
 * (GEMM_ERR_ALIGNMENT).  M, N or batch equal to 0 is a no-op; K equal to 0
 * writes zeros to D.  Tensor maps are encoded on the host from the pointers
 * (kept while the pointers stay the same).
 * The call only enqueues kernels (no allocation, no synchronisation), so it
 * may be captured into a CUDA graph and replayed: a plan whose tiles are
 * split along K (stream-K, gemm_plan_info_t.stream_k_tiles > 0) takes each
 * launch's epoch from a counter in its device memory, so replays stay
 * correct.  Launches of one plan must be ordered (one stream, or streams
 * joined by events): concurrent launches would share its status record,
 * stream-K workspace and launch counter.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (also for an MX / NV plan, which
 * gemm_run_mx runs), GEMM_ERR_ALIGNMENT or GEMM_ERR_CUDA.
 * Device-side wait expiry is not visible here; see gemm_sync_status.
 */
gemm_status_t gemm_run(gemm_plan_t plan, const void* A, const void* B, void* D,
                       const float* scale_a, const float* scale_b, gemm_stream_t stream);

/*
 * gemm_run_mx -- enqueue D = tA*tB * (A . SA) * (B . SB)^T on `stream` for a
 * plan whose scale_mode is GEMM_SCALE_MX_E8M0_32 or GEMM_SCALE_NV_E4M3_16
 * (kernel GEMM_KERNEL_MX): the tensor core applies the block scales inside
 * tcgen05.mma (.kind::mxf8f6f4 for 8-bit elements, .kind::mxf4 for MXFP4,
 * .kind::mxf4nvf4 for NVFP4), fp32 accumulation, one rounding to D's type.
 * A, B, D: device pointers laid out as at the top of this file (E4M3/E5M2 A
 * and B in either majorness; E2M1 K-major, rows a multiple of 32 elements
 * apart, K even).  sf_a, sf_b: device
 * pointers to the tiled scale bytes (16-byte aligned).  tensor_scales: NV: a
 * device pointer to two fp32 values {tA, tB}, read by the kernel when it runs;
 * MX: NULL.  Asynchronous and stream-ordered like gemm_run.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (a plan of another kind, a missing or
 * superfluous pointer), GEMM_ERR_ALIGNMENT or GEMM_ERR_CUDA; device-side wait
 * expiry is reported by gemm_sync_status.
 */
gemm_status_t gemm_run_mx(gemm_plan_t plan, const void* A, const void* B, void* D, const void* sf_a,
                          const void* sf_b, const float* tensor_scales, gemm_stream_t stream);

/*
 * gemm_run_host -- the same product for operands that live in host memory.
 * Copies hA, hB (and the scales) into the caller's device buffers dA, dB
 * (dsa, dsb), runs the product into dD and copies dD back into hD.  Host and
 * device buffers share the plan's layout (leading dims and batch strides) and
 * each must span that layout's extent; host memory should be pinned, or the
 * copies are not asynchronous.
 * Problems with at least 2048 rows (or 128 batch entries) are split into up
 * to 9 GEMMs over row (or batch-entry) panels: operands are copied in on an
 * internal stream while earlier GEMMs run on `stream` and copy their block of
 * D out on a second internal stream.  With M >= 4096 and N >= 2048 a first
 * block of 40 % of the rows is multiplied against B's four column quarters as
 * they land, then the remaining rows in panels against all of B; otherwise the
 * first row panel is multiplied in two column halves.  Events order everything after prior work on `stream`
 * and before later work on it; the panels' GEMMs report device timeouts to
 * the plan's record like gemm_run.  The internal streams, events and panel
 * plans are created on the first call and freed by gemm_plan_destroy; calls
 * on one plan must not run concurrently from several host threads.
 * The call returns once the work is enqueued; synchronise `stream` before
 * reading hD.  MX / NV plans are not offered here (GEMM_ERR_UNSUPPORTED).
 */
gemm_status_t gemm_run_host(gemm_plan_t plan, const void* hA, const void* hB, void* hD,
                            const float* hscale_a, const float* hscale_b,
                            void* dA, void* dB, void* dD, float* dscale_a, float* dscale_b,
                            gemm_stream_t stream);

/*
 * gemm_sync_status -- synchronise `stream`, read the plan's device error
 * record into *out (may be NULL), reset it, and return its code: GEMM_OK, or
 * GEMM_ERR_TIMEOUT when a bounded device-side wait ran out in a launch since
 * the last call (the kernel then released its resources and returned).
 */
gemm_status_t gemm_sync_status(gemm_plan_t plan, gemm_stream_t stream, gemm_device_error_t* out);

/*
 * gemm_run_noalloc -- D = A * B^T without any device allocation.  The pages
 * have no counterpart to this call; it exists for callers that cannot call
 * cudaMalloc, which gemm_plan_create does for its error record: code whose
 * device memory is entirely owned by a framework's caching pool (an allocation
 * behind the pool's back can fail for lack of memory or fragment it), and
 * latency-critical loops that cannot afford the device-wide synchronisation a
 * cudaMalloc or cudaFree may imply.
 *
 * Arguments are those of gemm_plan_create followed by those of gemm_run; the
 * problem is planned on the current device on every call (host arithmetic and
 * device-attribute queries, nothing allocated).  The kernels' device error
 * record lives in a library-owned static device array of 256 bytes (the
 * record needs 32), which every GPU that loads the library holds until the
 * process exits; no problem size needs more, and a build whose record did not
 * fit would return GEMM_ERR_RESOURCES.  The first call on each device looks up
 * the array's device address; make that first call before any stream capture.
 * A reset of the device's primary context (cudaDeviceReset) reloads the
 * library's device code and moves the array: a call that then fails with
 * GEMM_ERR_CUDA drops the cached address, and the next call looks it up again.
 * Each call clears the record on `stream`, then enqueues the product; the
 * record keeps the last call's contents.  All calls share this one record, so
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race on it.
 *
 * status_out: NULL returns once the work is enqueued; otherwise the call
 * synchronises `stream`, copies the record into *status_out and returns its
 * code (GEMM_OK or GEMM_ERR_TIMEOUT).  Other returns: the codes of
 * gemm_plan_create and gemm_run (MX / NV problems: GEMM_ERR_UNSUPPORTED).
 */
gemm_status_t gemm_run_noalloc(const gemm_desc_t* desc, const void* A, const void* B, void* D,
                               const float* scale_a, const float* scale_b, gemm_stream_t stream,
                               gemm_device_error_t* status_out);

/* Inputs of the pipeline schedule model (time units are arbitrary but common). */
typedef struct {
    int32_t tiles;          /* T: output tiles one CTA runs in sequence */
    int32_t k_slices;       /* K: ring stages (K slices) per tile */
    int32_t stages;         /* S: shared-memory ring depth */
    int32_t accumulators;   /* A: accumulator buffers (TMEM stages) */
    double t_issue;         /* producer time to issue one slice's copies */
    double t_load;          /* copy latency of one slice */
    double t_mma;           /* tensor-core time of one slice */
    double t_epi;           /* epilogue time of one tile */
} gemm_sched_params_t;

typedef struct {
    double run_length;      /* end of the last tile's epilogue */
    double tensor_busy;     /* T*K*t_mma / run_length */
    double steady_period;   /* M_{g+S} - M_g over the last tile's last S slices (0 if K <= S) */
    int32_t stages_needed;  /* ceil((t_load + t_mma) / t_mma): fewest stages that never starve */
    int32_t reserved;
} gemm_sched_result_t;

/*
 * gemm_schedule_model -- evaluate the max-plus schedule of a warp-specialised
 * main loop ("Hopper and Blackwell GEMM", section "Maths"): with slices
 * numbered g = t*K + k,
 *   L_g = max(L_{g-1} + t_issue, D_{g-S}),
 *   M_g = max(L_g + t_load, D_{g-1}, E_{t-A} if k = 0),
 *   D_g = M_g + t_mma,  E_t = max(D_{tK+K-1}, E_{t-1}) + t_epi.
 * Host arithmetic only.  Returns GEMM_OK or GEMM_ERR_INVALID_ARG (counts below
 * 1, T*K above 2^24, negative times, t_mma <= 0).
 */
gemm_status_t gemm_schedule_model(const gemm_sched_params_t* in, gemm_sched_result_t* out);

/*
 * gemm_schedule_choose -- the fewest accumulators, then the fewest stages,
 * whose modelled run is within `tolerance` (relative) of the run with
 * max_stages and max_accumulators; in->stages and in->accumulators are ignored.
 */
gemm_status_t gemm_schedule_choose(const gemm_sched_params_t* in, int32_t max_stages, int32_t max_accumulators,
                                   double tolerance, int32_t* stages, int32_t* accumulators);

/* Unit costs of one SM, in SM clock cycles, from which gemm_plan_schedule
 * derives the schedule model's times for a plan. */
typedef struct {
    double mma_flops_per_cycle;       /* tensor core, kind::f16 (bf16/f16 inputs); tf32 runs at half, 8-bit
                                         inputs at twice this rate */
    double stage_fixed_cycles;        /* copy path: cost of one ring stage beyond its bytes */
    double ingest_bytes_per_cycle;    /* copy path: operand bytes per cycle into one SM's shared memory */
    double load_latency_cycles;       /* from a stage's copies being issued to its first bytes landing */
    double tmem_read_bytes_per_cycle; /* epilogue: tcgen05.ld bytes per cycle per SM */
    double handback_cycles;           /* epilogue: fixed cost of handing an accumulator back to the MMA warp */
} gemm_machine_t;

/*
 * gemm_plan_schedule -- the schedule model ("Hopper and Blackwell GEMM",
 * section "Maths"; see gemm_schedule_model) applied to a planned persistent
 * 16-bit/tf32 problem.  From the plan's tile, stage depth and accumulator count
 * and a machine's unit costs (NULL: the GB300 figures this library measured,
 * see gemm_machine_gb300) it derives, per SM (pair):
 *   tiles      T = ceil(output tiles / clusters) (stream-K plans: the K slices of
 *                  one cluster's share, in whole tiles, or 1 when that share is
 *                  less than a tile)
 *   k_slices   K = ceil(K / tile_k) (a share less than a tile: its K slices)
 *   t_mma      = 2 * 128 * tile_n * tile_k / mma rate
 *   t_issue    = stage_fixed + stage_bytes / ingest      (the copy path's throughput)
 *   t_load     = load_latency + stage_bytes / ingest     (one stage's data in)
 *   t_epi      = 128 * tile_n * 4 / tmem_read + handback (an accumulator's read-back)
 * fills *params (may be NULL) and evaluates the model into *result (may be
 * NULL), in cycles.  *model_stages / *model_accumulators (may be NULL) receive
 * gemm_schedule_choose's pick, tolerance 0.5 %, within the plan's limits:
 * the ring depth the shared memory of `props` holds and the accumulators its
 * tensor memory and kernel support (two up to 256 columns, one for 512-wide
 * tiles).  Host arithmetic only.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, or GEMM_ERR_UNSUPPORTED for plans
 * other than GEMM_KERNEL_PERSISTENT.
 */
gemm_status_t gemm_plan_schedule(const gemm_desc_t* desc, const gemm_plan_info_t* info,
                                 const gemm_device_props_t* props, const gemm_machine_t* machine,
                                 gemm_sched_params_t* params, gemm_sched_result_t* result,
                                 int32_t* model_stages, int32_t* model_accumulators);

/* gemm_machine_gb300 -- the unit costs measured on GB300 with this library's
 * kernels and probes (clock64 and CUDA events; values in cycles at the SM clock). */
gemm_status_t gemm_machine_gb300(gemm_machine_t* out);

/* gemm_plan_destroy -- free the plan and its status record (NULL is allowed). */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* gemm_status_string -- static, human-readable name of a status code. */
const char* gemm_status_string(gemm_status_t status);

/* gemm_last_cuda_error -- the cudaError_t of the most recent GEMM_ERR_CUDA on this thread. */
int gemm_last_cuda_error(void);

/* gemm_version -- library version, major*10000 + minor*100 + patch. */
int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_BLACKWELL_GB300_GEMM_H */
