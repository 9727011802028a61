/*
 * nvfp4_oracle.c -- plain CPU oracle for the NVFP4 block-scaled grouped GEMM.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check of the entry module and
 * the CPU-baseline leg of the benchmark may load or call this code. The GPU
 * library never links it, and it shares no code, table or helper with the GPU
 * library (csrc/). It is slow on purpose: every step is the definition,
 * written out.
 *
 * What it computes (the three "nvfp4 group gemm" submissions on
 * kernelindex.com agree on it):
 *   - the block-scaled MMA accumulates the product of A, its scale, B and its
 *     scale (submission 499344, kernel main loop, at the gemm call);
 *   - element types Float4E2M1FN for A/B, Float8E4M3FN for the scales, one
 *     scale per 16 K-elements (sf_vec_size = 16), Float16 for C
 *     (submission 506336, the module-level kernel configuration);
 *   - the fp32 accumulator is converted to the C type once, in the epilogue
 *     (submission 506336, epilogue warps).
 * So, per group with m, n > 0:
 *     C[i][j] = fp16_rne( sum_k e2m1(A[i][k]) * e4m3(SFA[i][k/16])
 *                                * e2m1(B[j][k]) * e4m3(SFB[j][k/16]) )
 * accumulated here in fp64 and rounded once to fp16 (round to nearest even,
 * overflow to +-inf).
 *
 * Data layouts read by the oracle (submission 499344, custom_kernel docstring):
 *   A  [m][k/2]  bytes, two e2m1 codes per byte, K-major; B [n][k/2] likewise.
 *      Reading: the low nibble holds the even k, the high nibble the odd k.
 *   SFA [m][k/16], SFB [n][k/16]: e4m3fn codes, row-major (the plain form of
 *      the scales; the GPU path consumes the reordered atom layout instead).
 *   C  [m][n]    fp16 bit patterns, row-major.
 * The problem sizes are (m, n, k, l) per group; l is always 1 here.
 *
 * The atom-layout packer below (nvfp4_oracle_pack_scales) is the CPU
 * statement of the reordered scale layout of submission 385043 (kernel body,
 * where the scale tensors are built): atom shape ((32,4),(16,4)), stride
 * ((16,4),(0,1)), tiled over (rows, k) with the K atoms fastest.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- element formats ---------------------------------------------------- */

/* e2m1 (OCP MX FP4): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent field 0 is subnormal: value = mantissa * 2^-1. */
double nvfp4_oracle_e2m1_value(uint32_t code)
{
    code &= 0xFu;
    uint32_t sign = (code >> 3) & 1u;
    uint32_t expo = (code >> 1) & 3u;
    uint32_t mant = code & 1u;
    double mag;
    if (expo == 0)
        mag = 0.5 * (double)mant;
    else
        mag = ldexp(1.0 + 0.5 * (double)mant, (int)expo - 1);
    return sign ? -mag : mag;
}

/* e4m3fn (OCP FP8 E4M3): sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0. Exponent field 0 is subnormal: value = mantissa/8 * 2^-6.
 * S.1111.111 is NaN; there is no infinity. */
double nvfp4_oracle_e4m3fn_value(uint32_t code)
{
    code &= 0xFFu;
    uint32_t sign = code >> 7;
    uint32_t expo = (code >> 3) & 0xFu;
    uint32_t mant = code & 7u;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, (int)expo - 7);
    return sign ? -mag : mag;
}

/* IEEE-754 binary16 bit pattern of x, round to nearest, ties to even.
 * Subnormal results keep the 2^-24 quantum; |x| that rounds past 65504
 * becomes infinity; NaN becomes the quiet NaN 0x7E00. */
uint16_t nvfp4_oracle_fp16_bits(double x)
{
    if (isnan(x))
        return 0x7E00u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);
    int e2;
    (void)frexp(a, &e2);      /* a = f * 2^e2 with f in [0.5, 1)   */
    int binade = e2 - 1;      /* a in [2^binade, 2^(binade+1))       */
    if (binade < -14)
        binade = -14;         /* below 2^-14 the quantum stays 2^-24 */
    if (binade > 15)
        return (uint16_t)(sign | 0x7C00u);
    double quantum = ldexp(1.0, binade - 10);
    double r = nearbyint(a / quantum); /* exact scaling, then RNE */
    if (r >= 2048.0) {                 /* rounded up into the next binade */
        r = 1024.0;
        binade += 1;
    }
    if (r < 1024.0)                    /* only reachable when binade == -14 */
        return (uint16_t)(sign | (uint16_t)r);
    if (binade + 15 >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((binade + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* ---- operand access ----------------------------------------------------- */

/* e2m1 code of element kk of a K-major packed row (low nibble = even kk). */
static uint32_t fp4_code(const uint8_t *row, int kk)
{
    uint8_t byte = row[kk / 2];
    return (kk % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
}

/* One term of the sum: a * sfa * b * sfb for row i of A and row j of B. */
static double term(const uint8_t *a_row, const uint8_t *sfa_row,
                   const uint8_t *b_row, const uint8_t *sfb_row, int kk)
{
    double a = nvfp4_oracle_e2m1_value(fp4_code(a_row, kk)) *
               nvfp4_oracle_e4m3fn_value(sfa_row[kk / 16]);
    double b = nvfp4_oracle_e2m1_value(fp4_code(b_row, kk)) *
               nvfp4_oracle_e4m3fn_value(sfb_row[kk / 16]);
    return a * b;
}

static double dot(int k, const uint8_t *A, const uint8_t *SFA, const uint8_t *B,
                  const uint8_t *SFB, int i, int j)
{
    const uint8_t *a_row = A + (size_t)i * (size_t)(k / 2);
    const uint8_t *b_row = B + (size_t)j * (size_t)(k / 2);
    const uint8_t *sfa_row = SFA + (size_t)i * (size_t)(k / 16);
    const uint8_t *sfb_row = SFB + (size_t)j * (size_t)(k / 16);
    double s = 0.0;
    for (int kk = 0; kk < k; ++kk)
        s += term(a_row, sfa_row, b_row, sfb_row, kk);
    return s;
}

static void set_threads(int num_threads)
{
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
}

int nvfp4_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- the grouped GEMM --------------------------------------------------- */

/* Full C for every group with m, n > 0; groups with m == 0 or n == 0 are not
 * touched. k == 0 gives the empty sum, +0. problem_sizes is [G][4] =
 * (m, n, k, l). If C64 is non-null, C64[g] receives the fp64 sums before
 * rounding ([m][n] doubles) and C[g] may be null. */
void nvfp4_oracle_grouped_gemm(int group_count, const int32_t *problem_sizes,
                               const uint8_t *const *A, const uint8_t *const *B,
                               const uint8_t *const *SFA, const uint8_t *const *SFB,
                               uint16_t *const *C, double *const *C64, int num_threads)
{
    set_threads(num_threads);
    for (int g = 0; g < group_count; ++g) {
        int m = problem_sizes[4 * g + 0];
        int n = problem_sizes[4 * g + 1];
        int k = problem_sizes[4 * g + 2];
        if (m <= 0 || n <= 0)
            continue;
        const uint8_t *a = A[g], *b = B[g], *sfa = SFA[g], *sfb = SFB[g];
        uint16_t *c = C ? C[g] : NULL;
        double *c64 = C64 ? C64[g] : NULL;
#pragma omp parallel for schedule(dynamic, 1)
        for (int i = 0; i < m; ++i) {
            for (int j = 0; j < n; ++j) {
                double s = dot(k, a, sfa, b, sfb, i, j);
                if (c)
                    c[(size_t)i * (size_t)n + (size_t)j] = nvfp4_oracle_fp16_bits(s);
                if (c64)
                    c64[(size_t)i * (size_t)n + (size_t)j] = s;
            }
        }
    }
}

/* Selected outputs of one group: out[s] = C[rows[s]][cols[s]] (fp16 bits). */
void nvfp4_oracle_gemm_sampled(int m, int n, int k, const uint8_t *A, const uint8_t *B,
                               const uint8_t *SFA, const uint8_t *SFB, int num_samples,
                               const int32_t *rows, const int32_t *cols, uint16_t *out,
                               int num_threads)
{
    set_threads(num_threads);
    (void)m;
    (void)n;
#pragma omp parallel for schedule(static)
    for (int s = 0; s < num_samples; ++s)
        out[s] = nvfp4_oracle_fp16_bits(dot(k, A, SFA, B, SFB, rows[s], cols[s]));
}

/* ---- the reordered scale layout ---------------------------------------- */

/* Bytes of the atom layout for a [rows][k/16] scale matrix: rows padded to a
 * multiple of 128, scale columns padded to a multiple of 4. */
size_t nvfp4_oracle_scale_atom_bytes(int rows, int k)
{
    size_t row_blocks = (size_t)((rows + 127) / 128);
    size_t k_atoms = (size_t)((k + 63) / 64);
    return row_blocks * k_atoms * 512u;
}

/* Byte offset of scale (r, kb) -- row r, 16-element K block kb -- in the atom
 * layout. Inside a 512-byte atom (128 rows x 4 K blocks) the shape
 * ((32,4),(16,4)) with stride ((16,4),(0,1)) puts row r at 16*(r%32) +
 * 4*((r/32)%4) and K block kb at +kb%4; the atoms are laid out K-atom fastest,
 * then 128-row block. */
size_t nvfp4_oracle_scale_atom_offset(int r, int kb, int k)
{
    size_t k_atoms = (size_t)((k + 63) / 64);
    size_t atom = (size_t)(r / 128) * k_atoms + (size_t)(kb / 4);
    return atom * 512u + (size_t)(16 * (r % 32) + 4 * ((r / 32) % 4) + kb % 4);
}

/* Row-major [rows][k/16] scales -> atom layout; padding bytes are 0x00. */
void nvfp4_oracle_pack_scales(const uint8_t *sf_rowmajor, int rows, int k, uint8_t *sf_atoms)
{
    memset(sf_atoms, 0, nvfp4_oracle_scale_atom_bytes(rows, k));
    int kbs = k / 16;
    for (int r = 0; r < rows; ++r)
        for (int kb = 0; kb < kbs; ++kb)
            sf_atoms[nvfp4_oracle_scale_atom_offset(r, kb, k)] =
                sf_rowmajor[(size_t)r * (size_t)kbs + (size_t)kb];
}

/* ---- NVFP4 quantisation of activations ---------------------------------- */
/*
 * The quantiser that turns real-valued operands into the NVFP4 pair (e2m1
 * codes, one e4m3fn scale per 16 K-elements). The submissions receive their
 * operands already in this form; the quantisation itself is the one the
 * grouped-GEMM task states for its inputs: per row and 16-element K block,
 *     amax  = max |x|
 *     sf    = e4m3fn(amax / 6), round to nearest, ties to the even code,
 *             saturating at 448
 *     code  = e2m1(x / dec(sf)), round to nearest, ties to the even code,
 *             saturating at 6, the sign of x kept (a negative x that rounds
 *             to zero gives -0, code 8)
 *     every code is +0 when dec(sf) == 0.
 * Both quotients are taken in double precision here. For inputs that are
 * bf16 or fp16 values this decides the same codes as the quotients rounded
 * to fp32 (neither quotient can land within an fp32 rounding of a rounding
 * boundary without being on it); the pin tests check that claim exhaustively
 * over bf16 and fp16.
 */

/* e4m3fn code nearest to s >= 0 (ties to the even code), 0x7E (448) for
 * s >= 448. */
uint32_t nvfp4_oracle_e4m3fn_round(double s)
{
    if (!(s < 448.0))
        return 0x7Eu;
    uint32_t best = 0;
    double best_d = INFINITY;
    for (uint32_t c = 0; c <= 0x7Eu; ++c) {
        double d = fabs(nvfp4_oracle_e4m3fn_value(c) - s);
        if (d < best_d || (d == best_d && (c & 1u) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* e2m1 code nearest to q (ties to the even code), magnitude saturating at 6,
 * sign bit from q. */
uint32_t nvfp4_oracle_e2m1_round(double q)
{
    uint32_t sign = signbit(q) ? 8u : 0u;
    double a = fabs(q);
    if (a >= 6.0)
        return sign | 7u;
    uint32_t best = 0;
    double best_d = INFINITY;
    for (uint32_t c = 0; c <= 7u; ++c) {
        double d = fabs(nvfp4_oracle_e2m1_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1u) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;
}

/* Quantise x [rows][k] (k % 16 == 0) into codes [rows][k/2] (low nibble = even
 * k) and row-major scales sf [rows][k/16]. */
void nvfp4_oracle_quantize(const float *x, int rows, int k, uint8_t *codes, uint8_t *sf)
{
    int kbs = k / 16;
    for (int r = 0; r < rows; ++r) {
        const float *xr = x + (size_t)r * (size_t)k;
        uint8_t *cr = codes + (size_t)r * (size_t)(k / 2);
        for (int b = 0; b < kbs; ++b) {
            double amax = 0.0;
            for (int j = 0; j < 16; ++j)
                amax = fmax(amax, fabs((double)xr[16 * b + j]));
            uint32_t s = nvfp4_oracle_e4m3fn_round(amax / 6.0);
            double dec = nvfp4_oracle_e4m3fn_value(s);
            sf[(size_t)r * (size_t)kbs + (size_t)b] = (uint8_t)s;
            for (int j = 0; j < 16; j += 2) {
                uint32_t lo = dec == 0.0 ? 0u : nvfp4_oracle_e2m1_round((double)xr[16 * b + j] / dec);
                uint32_t hi = dec == 0.0 ? 0u : nvfp4_oracle_e2m1_round((double)xr[16 * b + j + 1] / dec);
                cr[8 * b + j / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}
