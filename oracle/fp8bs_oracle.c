/*
 * CPU oracle for the FP8 block-scaled GEMM and the MXFP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA library shares
 * no code, header, table or helper with it.
 *
 * What it computes is the plain definition, evaluated in fp64 and rounded to
 * bf16 once:
 *
 *   blockscale (skill card "FlyDSL fp8 blockscale GEMM", sections "When to use"
 *   and "Mechanism A": fp32 scales per 128-wide K block of A rows and per
 *   128x128 block of B, the scale applied to the fp8 products in fp32
 *   arithmetic outside the matrix unit; "Procedure" step 1: the oracle is
 *   dequantise -> matmul -> bf16):
 *
 *     C[m,n] = bf16( sum_k  (e4m3(A[m,k]) * sa[m, k/128]) * (e4m3(B[n,k]) * sb[n/128, k/128]) )
 *
 *   mxfp8 (PR "1x32 ue8m0 (MXFP8) 8-wave FlyDSL GEMM for gfx950", sections
 *   "Why it is faster" and "Correctness": one ue8m0 power-of-two scale per
 *   32-wide K group on both operands, applied exactly):
 *
 *     C[m,n] = bf16( sum_k  (e4m3(A[m,k]) * 2^(ea[m,k/32]-127)) * (e4m3(B[n,k]) * 2^(eb[n,k/32]-127)) )
 *
 * Readings where the pages are silent: E4M3 is the OCP E4M3FN format the
 * skill card names (bias 7, max 448, no infinities, S.1111.111 is NaN); bf16
 * rounding is IEEE round-to-nearest-even with overflow to infinity; a partial
 * last N block of B uses its own scale row.
 *
 * Every function is pinned by the tests (tests/test_oracle_pins.py): the
 * decoders against torch's float8_e4m3fn decode and golden anchor codes, the
 * bf16 rounding against exact rational rounding, the GEMMs against exact
 * rational brute force on tiny inputs, a plain fp64 matmul at unit scales,
 * linearity in one block scale, power-of-two exactness, integer inputs with a
 * known exact product, the block-partial form and the blockscale/MXFP8 cross case.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* OCP E4M3FN code -> value, from the bit definition: sign bit 7, exponent
 * bits 6..3 (bias 7), mantissa bits 2..0; exponent 0 is subnormal
 * (m * 2^-9); exponent 15 with mantissa 7 is NaN. */
double oracle_e4m3_decode(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* ue8m0 byte -> 2^(byte-127); 0xFF is NaN. */
double oracle_ue8m0_decode(uint8_t code)
{
    if (code == 0xFF)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Round a double to bf16 (8 significant bits, 8 exponent bits, bias 127)
 * once, to nearest with ties to even; overflow -> +-inf; NaN -> quiet NaN.
 * The value is scaled by a power of two so that its bf16 quantum becomes 1,
 * rounded to an integer by hand (independent of the FP environment), and
 * scaled back; the rounded value is then exactly representable in fp32 and
 * bf16 is the top half of that fp32 word. */
uint16_t oracle_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    if (isinf(x))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1): leading bit 2^(e2-1) */
    int lead = e2 - 1;
    int qexp = (lead >= -126 ? lead : -126) - 7; /* bf16 quantum at this magnitude */
    double s = ldexp(a, -qexp);   /* exact: power-of-two scaling, s < 256 */
    double fl = floor(s);
    double rem = s - fl;          /* exact: s has at most 53 bits, fl < 256 */
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) == 1.0))
        fl += 1.0;
    double v = ldexp(fl, qexp);
    const double bf16_max = ldexp(255.0, 127 - 7); /* (2 - 2^-7) * 2^127 */
    if (v > bf16_max)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;           /* exact */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | ((bits >> 16) & 0x7FFFu));
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void decode_table(double t[256])
{
    for (int c = 0; c < 256; ++c)
        t[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Blockscale GEMM, definition form: dequantise every operand element with its
 * scale to fp64, then the naive triple loop, then one bf16 rounding.
 *   A       uint8 [M][K]      E4M3 codes, row-major
 *   a_scale fp32  [M][K/128]  logical a_scale[m][kb]
 *   B       uint8 [N][K]      E4M3 codes, row-major
 *   b_scale fp32  [ceil(N/128)][K/128]
 * Rows [row_begin, row_end) of C are computed; C (bf16 bits) and C_exact
 * (the fp64 value before rounding, may be NULL) are indexed
 * [(m-row_begin)*N + n]. Returns 0, or -1 on bad arguments / no memory. */
int oracle_blockscale(const uint8_t *A, const float *a_scale, const uint8_t *B, const float *b_scale,
                      int M, int N, int K, int row_begin, int row_end, uint16_t *C, double *C_exact)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    const int KB = K / 128;
    double lut[256];
    decode_table(lut);
    double *Bd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)(K ? K : 1));
    if (!Bd)
        return -1;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            Bd[(size_t)n * K + k] = lut[B[(size_t)n * K + k]] * (double)b_scale[(size_t)(n / 128) * KB + k / 128];
    int err = 0;
#pragma omp parallel
    {
        double *Ad = (double *)malloc(sizeof(double) * (size_t)(K ? K : 1));
        if (!Ad) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int m = row_begin; m < row_end; ++m) {
            if (!Ad)
                continue;
            for (int k = 0; k < K; ++k)
                Ad[k] = lut[A[(size_t)m * K + k]] * (double)a_scale[(size_t)m * KB + k / 128];
            for (int n = 0; n < N; ++n) {
                const double *b = Bd + (size_t)n * K;
                double acc = 0.0;
                for (int k = 0; k < K; ++k)
                    acc += Ad[k] * b[k];
                size_t o = (size_t)(m - row_begin) * N + n;
                C[o] = oracle_bf16_rne(acc);
                if (C_exact)
                    C_exact[o] = acc;
            }
        }
        free(Ad);
    }
    free(Bd);
    return err ? -1 : 0;
}

/* Blockscale GEMM, block-partial form (the order the skill card's software
 * promote uses, section "Mechanism A"): for each 128-wide K block, the
 * unscaled fp8 partial sum S_kb = sum_{k in kb} e4m3(A)*e4m3(B) (exact in
 * fp64), times sa*sb, summed over blocks. Used only to cross-check the
 * definition form. Same arguments as oracle_blockscale. */
int oracle_blockscale_blockpartial(const uint8_t *A, const float *a_scale, const uint8_t *B,
                                   const float *b_scale, int M, int N, int K, int row_begin,
                                   int row_end, uint16_t *C, double *C_exact)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    const int KB = K / 128;
    double lut[256];
    decode_table(lut);
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = row_begin; m < row_end; ++m) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int kb = 0; kb < KB; ++kb) {
                double part = 0.0;
                for (int k = kb * 128; k < kb * 128 + 128; ++k)
                    part += lut[A[(size_t)m * K + k]] * lut[B[(size_t)n * K + k]];
                double s = (double)a_scale[(size_t)m * KB + kb] * (double)b_scale[(size_t)(n / 128) * KB + kb];
                acc += s * part;
            }
            size_t o = (size_t)(m - row_begin) * N + n;
            C[o] = oracle_bf16_rne(acc);
            if (C_exact)
                C_exact[o] = acc;
        }
    }
    return 0;
}

/* MXFP8 GEMM, definition form.
 *   A      uint8 [M][K]     E4M3 codes;  a_e8m0 uint8 [M][K/32]
 *   B      uint8 [N][K]     E4M3 codes;  b_e8m0 uint8 [N][K/32]
 * Output as for oracle_blockscale. K must be a multiple of 32. */
int oracle_mxfp8(const uint8_t *A, const uint8_t *a_e8m0, const uint8_t *B, const uint8_t *b_e8m0,
                 int M, int N, int K, int row_begin, int row_end, uint16_t *C, double *C_exact)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    const int G = K / 32;
    double lut[256];
    decode_table(lut);
    double *Bd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)(K ? K : 1));
    if (!Bd)
        return -1;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            Bd[(size_t)n * K + k] = lut[B[(size_t)n * K + k]] * oracle_ue8m0_decode(b_e8m0[(size_t)n * G + k / 32]);
    int err = 0;
#pragma omp parallel
    {
        double *Ad = (double *)malloc(sizeof(double) * (size_t)(K ? K : 1));
        if (!Ad) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int m = row_begin; m < row_end; ++m) {
            if (!Ad)
                continue;
            for (int k = 0; k < K; ++k)
                Ad[k] = lut[A[(size_t)m * K + k]] * oracle_ue8m0_decode(a_e8m0[(size_t)m * G + k / 32]);
            for (int n = 0; n < N; ++n) {
                const double *b = Bd + (size_t)n * K;
                double acc = 0.0;
                for (int k = 0; k < K; ++k)
                    acc += Ad[k] * b[k];
                size_t o = (size_t)(m - row_begin) * N + n;
                C[o] = oracle_bf16_rne(acc);
                if (C_exact)
                    C_exact[o] = acc;
            }
        }
        free(Ad);
    }
    free(Bd);
    return err ? -1 : 0;
}
