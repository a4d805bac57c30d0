/*
 * oracle.c -- plain, slow, obviously correct CPU reference for D = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (the plain definition, nothing blocked, fused or
 * reordered):
 *
 *   D_ref[b,m,n] = sum_{k=0}^{K-1} a(b,m,k) * b(b,n,k)      (fp64, ascending k)
 *   S[b,m,n]     = sum_{k=0}^{K-1} |a(b,m,k) * b(b,n,k)|    (fp64)
 *
 * "Out = A @ B.T", checked against a.float() @ b.float().T
 *   -- TVM TIRx "Blackwell Tensor Cores", section "The Accumulator's Lifetime"
 *      and its closing check.
 * Accumulation in a wide type with the first product starting a fresh sum
 *   -- TVM TIRx "mma.sync", sections "Data representation" and
 *      "Accumulation, transpose and alpha/beta".
 * Block scaling multiplies each block's values by that block's scale
 *   -- "Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling".
 *
 * For block-scaled 8-bit inputs with fp32 block scales the element values are
 *   a(b,m,k) = q_a(b,m,k) * sA[b][m][floor(k/128)]
 *   b(b,n,k) = q_b(b,n,k) * sB[b][floor(n/128)][floor(k/128)]
 * (one fp32 scale per 1x128 block of A and per 128x128 block of B).
 *
 * Hardware block scaling ("Hopper and Blackwell GEMM", table of MXFP8, MXFP4
 * and NVFP4: every row of A and of B is cut into blocks of V consecutive K
 * elements, each block carrying one scale):
 *   MX (V = 32, E8M0 scale):  a(b,m,k) = q_a(b,m,k) * 2^(eA(b,m,floor(k/32)) - 127)
 *   NV (V = 16, E4M3 scale, plus one fp32 per tensor):
 *                             a(b,m,k) = q_a(b,m,k) * e4m3(sA(b,m,floor(k/16))) * tA
 *   and the same for b(b,n,k) with B's scales.
 * The scale bytes of a matrix with R rows and KB = ceil(K/V) scale columns
 * are stored in 512-byte tiles of 128 rows x 4 scale columns, tile (r/128,
 * kb/4) at ((r/128) * ceil(KB/4) + kb/4) * 512 bytes from the batch entry's
 * start, and inside a tile at (r mod 32)*16 + ((r/32) mod 4)*4 + (kb mod 4):
 * the folding "TMEM -- the accumulator's new home" (section "Block-scaled
 * MMA") describes, lane = r mod 32 and column = r/32, 4 scales per column.
 *
 * Element addressing (elements, not bytes):
 *   A K-major : A[b*stride_a + m*lda + k]     A MN-major : A[b*stride_a + k*lda + m]
 *   B K-major : B[b*stride_b + n*ldb + k]     B MN-major : B[b*stride_b + k*ldb + n]
 *
 * Element formats are decoded from their IEEE-754 / OCP definitions:
 *   fp16  : 1 sign, 5 exponent (bias 15), 10 mantissa bits, IEEE inf/NaN
 *   bf16  : 1 sign, 8 exponent (bias 127), 7 mantissa bits, IEEE inf/NaN
 *   e4m3  : 1 sign, 4 exponent (bias 7), 3 mantissa bits, no inf,
 *           S.1111.111 is NaN, largest finite 448 (OCP 8-bit FP, "E4M3FN")
 *   e5m2  : 1 sign, 5 exponent (bias 15), 2 mantissa bits, IEEE inf/NaN,
 *           largest finite 57344 (OCP 8-bit FP, "E5M2")
 *   fp32  : 1 sign, 8 exponent (bias 127), 23 mantissa bits (also as an input)
 *   e2m1  : 1 sign, 2 exponent (bias 1), 1 mantissa bit, no inf or NaN,
 *           largest 6 (OCP MX "FP4"); two per byte, element 2i in the low
 *           nibble of byte i
 *   e8m0  : 8 exponent bits, no sign or mantissa: 2^(e - 127), 0xFF is NaN
 *           (OCP MX scale)
 * Rounding to an output format is round-to-nearest, ties to even, from the
 * exact fp64 value (one rounding).  e4m3 encoding saturates to +-448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element type codes used by this file's callers (the Python test wrapper). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F32 = 3, ORC_E5M2 = 4, ORC_E2M1 = 5, ORC_E8M0 = 6 };

/* Scale kinds of orc_problem.scaled. */
enum { ORC_SCALE_NONE = 0, ORC_SCALE_FP32_BLOCK = 1, ORC_SCALE_MX = 2, ORC_SCALE_NV = 3 };

/* Parameters of one binary floating-point format. */
typedef struct {
    int mbits;    /* explicit mantissa bits */
    int ebits;    /* exponent bits */
    int bias;     /* exponent bias */
    int has_inf;  /* IEEE-style all-ones exponent = inf/NaN */
    int has_nan;  /* without inf: the all-ones code (sign aside) is NaN (E4M3FN); 0 = every code finite */
    int satfinite;/* encoder clamps to the largest finite value */
} orc_format;

static int orc_format_of(int dtype, orc_format* f) {
    switch (dtype) {
    case ORC_F16:  f->mbits = 10; f->ebits = 5; f->bias = 15;  f->has_inf = 1; f->has_nan = 1; f->satfinite = 0; return 0;
    case ORC_BF16: f->mbits = 7;  f->ebits = 8; f->bias = 127; f->has_inf = 1; f->has_nan = 1; f->satfinite = 0; return 0;
    case ORC_F32:  f->mbits = 23; f->ebits = 8; f->bias = 127; f->has_inf = 1; f->has_nan = 1; f->satfinite = 0; return 0;
    case ORC_E4M3: f->mbits = 3;  f->ebits = 4; f->bias = 7;   f->has_inf = 0; f->has_nan = 1; f->satfinite = 1; return 0;
    case ORC_E5M2: f->mbits = 2;  f->ebits = 5; f->bias = 15;  f->has_inf = 1; f->has_nan = 1; f->satfinite = 0; return 0;
    case ORC_E2M1: f->mbits = 1;  f->ebits = 2; f->bias = 1;   f->has_inf = 0; f->has_nan = 0; f->satfinite = 1; return 0;
    default: return -1;
    }
}

/* Largest finite magnitude of a format. */
static double orc_max_finite(const orc_format* f) {
    int emax_field = (1 << f->ebits) - 1;
    if (f->has_inf) {
        /* all-ones exponent is reserved: largest normal has field emax_field-1 and all-ones mantissa */
        return ldexp(2.0 - ldexp(1.0, -f->mbits), (emax_field - 1) - f->bias);
    }
    /* OCP E4M3: all-ones exponent is a normal binade, only mantissa all-ones is NaN */
    if (f->has_nan) return ldexp(2.0 - ldexp(1.0, -(f->mbits - 1)), emax_field - f->bias);
    /* OCP E2M1: every code is a number, the largest has all ones */
    return ldexp(2.0 - ldexp(1.0, -f->mbits), emax_field - f->bias);
}

/* Decode one code of width 8/16/32 bits into its exact real value. */
double orc_decode(int dtype, uint32_t code) {
    if (dtype == ORC_E8M0) {
        /* a bare exponent: 2^(e - 127); the all-ones code is NaN */
        code &= 0xFFu;
        return code == 0xFFu ? NAN : ldexp(1.0, (int)code - 127);
    }
    orc_format f;
    if (orc_format_of(dtype, &f)) return NAN;
    int total = 1 + f.ebits + f.mbits;
    uint32_t sign = (code >> (total - 1)) & 1u;
    uint32_t efield = (code >> f.mbits) & ((1u << f.ebits) - 1u);
    uint32_t mfield = code & ((1u << f.mbits) - 1u);
    uint32_t eall = (1u << f.ebits) - 1u;
    double v;
    if (f.has_inf && efield == eall) {
        v = (mfield == 0) ? INFINITY : NAN;
    } else if (!f.has_inf && f.has_nan && efield == eall && mfield == ((1u << f.mbits) - 1u)) {
        v = NAN;
    } else if (efield == 0) {
        /* subnormal: 0.m * 2^(1-bias) */
        v = ldexp((double)mfield, 1 - f.bias - f.mbits);
    } else {
        /* normal: 1.m * 2^(e-bias) */
        v = ldexp((double)((1u << f.mbits) + mfield), (int)efield - f.bias - f.mbits);
    }
    return sign ? -v : v;
}

/* Round x to the nearest value of the format, ties to even.  Returns the
 * rounded value (inf on overflow for IEEE formats, +-max for saturating ones). */
double orc_round(int dtype, double x) {
    orc_format f;
    if (orc_format_of(dtype, &f)) return NAN;
    if (isnan(x)) return NAN;
    double maxf = orc_max_finite(&f);
    int neg = signbit(x) ? 1 : 0;
    double ax = fabs(x);
    if (isinf(ax)) return f.satfinite ? (neg ? -maxf : maxf) : x;
    int emin = 1 - f.bias;                     /* exponent of the smallest normal */
    double r;
    if (ax < ldexp(1.0, emin)) {
        double q = ldexp(1.0, emin - f.mbits);  /* subnormal spacing */
        r = rint(ax / q) * q;                   /* rint: ties to even in the default mode */
    } else {
        int e2;
        frexp(ax, &e2);                          /* ax = fr * 2^e2, fr in [0.5,1) */
        double q = ldexp(1.0, (e2 - 1) - f.mbits);
        r = rint(ax / q) * q;
    }
    if (r > maxf) r = f.satfinite ? maxf : INFINITY;
    return neg ? -r : r;
}

/* Encode x (RNE, saturating for e4m3) into the format's bit pattern. */
uint32_t orc_encode(int dtype, double x) {
    orc_format f;
    if (orc_format_of(dtype, &f)) return 0;
    int total = 1 + f.ebits + f.mbits;
    uint32_t eall = (1u << f.ebits) - 1u;
    if (isnan(x) && !f.has_nan) return 0;   /* a format without NaN has no code for it */
    if (isnan(x)) {
        /* canonical quiet NaN: all-ones exponent, top mantissa bit (e4m3: all ones) */
        uint32_t m = f.has_inf ? (1u << (f.mbits - 1)) : ((1u << f.mbits) - 1u);
        return (eall << f.mbits) | m;
    }
    double r = orc_round(dtype, x);
    uint32_t sign = signbit(r) ? 1u : 0u;
    double ar = fabs(r);
    uint32_t efield, mfield;
    if (isinf(ar)) {
        efield = eall; mfield = 0;
    } else if (ar == 0.0) {
        efield = 0; mfield = 0;
    } else if (ar < ldexp(1.0, 1 - f.bias)) {
        efield = 0;
        mfield = (uint32_t)ldexp(ar, -(1 - f.bias - f.mbits));
    } else {
        int e2;
        frexp(ar, &e2);
        int e = e2 - 1;
        efield = (uint32_t)(e + f.bias);
        mfield = (uint32_t)(ldexp(ar, f.mbits - e) - ldexp(1.0, f.mbits));
    }
    return (sign << (total - 1)) | (efield << f.mbits) | mfield;
}

/* Bulk forms for the test wrapper. */
void orc_decode_array(int dtype, const uint32_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode(dtype, codes[i]);
}
void orc_round_array(int dtype, const double* x, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round(dtype, x[i]);
}
void orc_encode_array(int dtype, const double* x, int64_t n, uint32_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode(dtype, x[i]);
}

static int orc_elem_bytes(int dtype) {
    switch (dtype) {
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_E4M3: case ORC_E5M2: case ORC_E8M0: return 1;
    case ORC_E2M1: return 1;   /* two elements per byte, see orc_load_elem */
    case ORC_F32: return 4;
    default: return 0;
    }
}

static uint32_t orc_load_code(const void* base, int bytes, int64_t idx) {
    if (bytes == 1) return ((const uint8_t*)base)[idx];
    if (bytes == 2) return ((const uint16_t*)base)[idx];
    return ((const uint32_t*)base)[idx];
}

/* Code of element `idx` (in elements) of an operand: 4-bit E2M1 elements sit
 * two per byte, element 2i in the low nibble of byte i. */
static uint32_t orc_load_elem(int dtype, const void* base, int64_t idx) {
    if (dtype == ORC_E2M1) {
        uint8_t byte = ((const uint8_t*)base)[idx / 2];
        return (idx % 2 == 0) ? (uint32_t)(byte & 0xFu) : (uint32_t)(byte >> 4);
    }
    return orc_load_code(base, orc_elem_bytes(dtype), idx);
}

/* One GEMM problem as the oracle sees it. */
typedef struct {
    int64_t M, N, K, batch;
    int32_t dtype_a, dtype_b;
    int32_t major_a, major_b;       /* 0 = K contiguous, 1 = M (resp. N) contiguous */
    int64_t lda, ldb;
    int64_t stride_a, stride_b;
    int32_t scaled;                  /* ORC_SCALE_*: 1 = fp32 scales per 1x128 (A) and 128x128 (B) block,
                                        2 = MX (E8M0 per 32 K elements), 3 = NV (E4M3 per 16, times tA / tB) */
    int32_t pad_;
    int64_t ld_sa, ld_sb;            /* fp32 blocks: floats between scale rows */
    int64_t stride_sa, stride_sb;    /* fp32 blocks: floats between batches of scales; MX / NV: bytes
                                        between batches of the tiled scales (0 = whole tiles, packed) */
    double tensor_scale_a, tensor_scale_b;   /* NV: the per-tensor fp32 scales tA and tB */
} orc_problem;

/* Byte offset of the scale of (batch b, row r, scale column kb) in the tiled
 * layout of a matrix with R rows and KB scale columns (see the file header). */
static int64_t orc_tiled_offset(int64_t b, int64_t r, int64_t kb, int64_t R, int64_t KB, int64_t batch_stride) {
    const int64_t row_tiles = (R + 127) / 128, col_tiles = (KB + 3) / 4;
    const int64_t per_batch = batch_stride ? batch_stride : row_tiles * col_tiles * 512;
    return b * per_batch + ((r / 128) * col_tiles + kb / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4;
}

/* Real value of one block scale of row r of a matrix with R rows (MX / NV). */
static double orc_block_scale(const orc_problem* p, const uint8_t* sf, int64_t b, int64_t r, int64_t R, int64_t k,
                              int64_t batch_stride) {
    const int64_t V = p->scaled == ORC_SCALE_MX ? 32 : 16;
    const int64_t KB = (p->K + V - 1) / V;
    const uint8_t code = sf[orc_tiled_offset(b, r, k / V, R, KB, batch_stride)];
    return p->scaled == ORC_SCALE_MX ? orc_decode(ORC_E8M0, code) : orc_decode(ORC_E4M3, code);
}

static int64_t orc_index_a(const orc_problem* p, int64_t b, int64_t m, int64_t k) {
    return b * p->stride_a + (p->major_a == 0 ? m * p->lda + k : k * p->lda + m);
}
static int64_t orc_index_b(const orc_problem* p, int64_t b, int64_t n, int64_t k) {
    return b * p->stride_b + (p->major_b == 0 ? n * p->ldb + k : k * p->ldb + n);
}

/* Decode table for every code of an 8- or 16-bit format (filled from orc_decode);
 * NULL for 32-bit formats, which are decoded element by element. */
static double* orc_make_table(int dtype) {
    int bytes = orc_elem_bytes(dtype);
    if (bytes > 2) return NULL;
    int64_t n = (int64_t)1 << (8 * bytes);
    double* t = (double*)malloc(sizeof(double) * (size_t)n);
    if (!t) return NULL;
    for (int64_t c = 0; c < n; ++c) t[c] = orc_decode(dtype, (uint32_t)c);
    return t;
}

/* Real value of A(b,m,k) and B(b,n,k), scales applied when the problem is block-scaled. */
static double orc_lookup(int dtype, const double* lut, uint32_t code) {
    return lut ? lut[code] : orc_decode(dtype, code);
}

static double orc_value_a(const orc_problem* p, const double* lut, const void* A, const void* sA,
                          int64_t b, int64_t m, int64_t k) {
    double v = orc_lookup(p->dtype_a, lut, orc_load_elem(p->dtype_a, A, orc_index_a(p, b, m, k)));
    if (p->scaled == ORC_SCALE_FP32_BLOCK)
        v *= (double)((const float*)sA)[b * p->stride_sa + m * p->ld_sa + k / 128];
    else if (p->scaled == ORC_SCALE_MX)
        v *= orc_block_scale(p, (const uint8_t*)sA, b, m, p->M, k, p->stride_sa);
    else if (p->scaled == ORC_SCALE_NV)
        v *= orc_block_scale(p, (const uint8_t*)sA, b, m, p->M, k, p->stride_sa) * p->tensor_scale_a;
    return v;
}
static double orc_value_b(const orc_problem* p, const double* lut, const void* B, const void* sB,
                          int64_t b, int64_t n, int64_t k) {
    double v = orc_lookup(p->dtype_b, lut, orc_load_elem(p->dtype_b, B, orc_index_b(p, b, n, k)));
    if (p->scaled == ORC_SCALE_FP32_BLOCK)
        v *= (double)((const float*)sB)[b * p->stride_sb + (n / 128) * p->ld_sb + k / 128];
    else if (p->scaled == ORC_SCALE_MX)
        v *= orc_block_scale(p, (const uint8_t*)sB, b, n, p->N, k, p->stride_sb);
    else if (p->scaled == ORC_SCALE_NV)
        v *= orc_block_scale(p, (const uint8_t*)sB, b, n, p->N, k, p->stride_sb) * p->tensor_scale_b;
    return v;
}

/*
 * Reference product for a list of output rows.  rows[i] = b*M + m names one
 * row of D; row i of the outputs holds D_ref[b,m,0..N) and S[b,m,0..N).
 * rows == NULL means every row of every batch, in order.  Rows are spread
 * over OpenMP threads; each output element is one ascending-k fp64 sum.
 * Inputs are 8-, 16- or 32-bit codes.  Returns 0, or -1 on a bad argument.
 */
int orc_gemm_rows(const orc_problem* p, const void* A, const void* B,
                  const void* sA, const void* sB,
                  int64_t nrows, const int64_t* rows, double* dref, double* sabs) {
    if (!p || p->M < 0 || p->N < 0 || p->K < 0 || p->batch < 0) return -1;
    int ba = orc_elem_bytes(p->dtype_a), bb = orc_elem_bytes(p->dtype_b);
    if (ba < 1 || bb < 1) return -1;
    if (p->scaled < ORC_SCALE_NONE || p->scaled > ORC_SCALE_NV) return -1;
    if (p->scaled && (!sA || !sB)) return -1;
    /* 4-bit elements: K-major only, each row a whole number of bytes */
    if ((p->dtype_a == ORC_E2M1 && (p->major_a != 0 || p->lda % 2 || p->stride_a % 2)) ||
        (p->dtype_b == ORC_E2M1 && (p->major_b != 0 || p->ldb % 2 || p->stride_b % 2)))
        return -1;
    if (rows == NULL) nrows = p->batch * p->M;
    double* lut_a = orc_make_table(p->dtype_a);
    double* lut_b = orc_make_table(p->dtype_b);
    if ((ba <= 2 && !lut_a) || (bb <= 2 && !lut_b)) { free(lut_a); free(lut_b); return -1; }
    const int64_t N = p->N, K = p->K;
#pragma omp parallel
    {
        double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t r = rows ? rows[i] : i;
            int64_t b = p->M ? r / p->M : 0, m = p->M ? r % p->M : 0;
            for (int64_t k = 0; k < K; ++k) arow[k] = orc_value_a(p, lut_a, A, sA, b, m, k);
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0, s = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double prod = arow[k] * orc_value_b(p, lut_b, B, sB, b, n, k);
                    acc += prod;
                    s += fabs(prod);
                }
                dref[i * N + n] = acc;
                if (sabs) sabs[i * N + n] = s;
            }
        }
        free(arow);
    }
    free(lut_a);
    free(lut_b);
    return 0;
}

/* Number of OpenMP threads the oracle's parallel loops use. */
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
