/*
 * oracle.c -- plain, slow CPU reference for block-scaled FP4 (MXFP4 / NVFP4).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA library: every value here is derived from the
 * format definitions written out below.
 *
 * Sources (web pages, cited by title and section):
 *   [DG]  "Packed MXFP4 & NVFP4 GEMM + mega-MoE (SM100, true 2-CTA multicast)"
 *         (DeepGEMM pull request), section "Summary": both operands are packed
 *         E2M1, two elements per byte; MXFP4 carries one UE8M0 scale per 32
 *         K-elements, NVFP4 one E4M3/UE4M3 scale per 16 K-elements plus
 *         per-tensor fp32 global scales, dequantised as acc * gs_act * gs_weight;
 *         the GEMM is [M,K] @ [N,K]^T -> [M,N].
 *   [MJ]  "fp4_quantization" (Mojo kernel module API), section "Functions":
 *         dynamic BF16 -> NVFP4/MXFP4 quantisation with per-block scale factors
 *         (quantize_dynamic_scaled_fp4fp8) and the re-interleave of rank-2
 *         scale factors into the 5D TCGEN layout (block_scales_interleave).
 *   [QB]  "quadbit" README, section "Accuracy (real models)": per-16 ue4m3
 *         local scale with an fp32 global scale (NVFP4), ue8m0 (MXFP4); the
 *         two-level recipe with a per-row fp32 global scale, and a per-row
 *         and per-column fp32 global rescale in the MMA epilogue.
 *   [QG]  "qgemm-mx" project page, section "The gap": MXFP4 moves ~1.88x fewer
 *         bytes per weight than FP8.
 * The pages do not print the bit layouts.  Those are taken from the public
 * OCP Microscaling Formats (MX) v1.0 specification (E2M1 element, E8M0 scale)
 * and the OCP 8-bit floating point specification (E4M3), as stated at each
 * function.  Readings of what the pages leave open are marked READING.
 *
 * Precision: decoding and the GEMM are done in fp64 (every product is exact);
 * the quantiser is done in IEEE fp32 with round-to-nearest-even, because the
 * quantised bytes are defined by fp32 arithmetic.  Build without -ffast-math
 * and with -ffp-contract=off.
 *
 * Parity pins: every function below is checked in the CPU test suite against
 * closed forms, library conversions, brute-force searches or invariants.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MXFP4 0
#define ORACLE_NVFP4 1
/* NVFP4 with one UE4M3 scale per 32 K-elements (plus the fp32 global
 * scales): the scale blocks of the 2:4-sparse path.  [QB] "Accuracy (real
 * models)": the deployed two-level sparse kernel is trained "per-32 matched"
 * (weights and activations quantised with 32-element blocks).
 * READING: that is this format, for both operands of a sparse GEMM. */
#define ORACLE_NVFP4_B32 2

/* ------------------------------------------------------------------------ */
/* Element and scale decoding                                                */
/* ------------------------------------------------------------------------ */

/* E2M1 (OCP MX v1.0, FP4 E2M1): bits s e1 e0 m, exponent bias 1.
 * e == 0: subnormal, value m * 0.5; else (1 + m/2) * 2^(e-1).
 * Codes 0..7 give 0, 0.5, 1, 1.5, 2, 3, 4, 6; codes 8..15 their negatives. */
double oracle_e2m1_value(int code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return s ? -mag : mag;
}

/* UE8M0 (OCP MX v1.0, E8M0 scale): value 2^(e-127) for e in 0..254; 255 is NaN. */
double oracle_ue8m0_value(int byte)
{
    if (byte < 0 || byte > 254) return NAN;
    return ldexp(1.0, byte - 127);
}

/* UE4M3: the E4M3 format (OCP 8-bit FP spec, bias 7) with the sign bit fixed
 * at zero.  e = bits[6:3], m = bits[2:0]; e == 0 is subnormal m * 2^-9,
 * otherwise (1 + m/8) * 2^(e-7).  0x7F is NaN; bit 7 set is not a UE4M3 code.
 * Largest finite value 0x7E = 448. */
double oracle_ue4m3_value(int byte)
{
    if (byte < 0 || byte > 0x7E) return NAN;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    if (e == 0) return ldexp((double)m, -9);
    return (1.0 + m / 8.0) * ldexp(1.0, e - 7);
}

/* Scale decoding keyed on the format: MXFP4 -> UE8M0, NVFP4 -> UE4M3 [DG]. */
double oracle_scale_value(int fmt, int byte)
{
    return fmt == ORACLE_MXFP4 ? oracle_ue8m0_value(byte) : oracle_ue4m3_value(byte);
}

int oracle_block_size(int fmt) { return fmt == ORACLE_NVFP4 ? 16 : 32; }

/* ------------------------------------------------------------------------ */
/* Rounding to the formats (round to nearest, ties to even code)            */
/* ------------------------------------------------------------------------ */

/* Nearest entry of a table of ncodes non-negative values that increase with
 * the code, for a >= 0: the two codes that bracket a are compared (their
 * distances to a are exact in fp64), ties go to the even code, and anything
 * at or above the last value gives the last code (saturation).  The first
 * code whose value is >= a is found by bisection, which the increasing
 * values allow. */
static int nearest_even_code(double a, double (*value)(int), int ncodes)
{
    if (a >= value(ncodes - 1)) return ncodes - 1;
    int hi = 0, top = ncodes - 1;          /* value(top) > a */
    while (hi < top) {
        int mid = (hi + top) / 2;
        if (value(mid) < a) hi = mid + 1;
        else top = mid;
    }
    if (hi == 0) return 0;
    int lo = hi - 1;
    double dlo = a - value(lo), dhi = value(hi) - a;
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return (lo & 1) ? hi : lo;
}

static double e2m1_magnitude(int code) { return oracle_e2m1_value(code & 7); }

/* E2M1 rounding of an fp32 value q, written as the definition: the nearest
 * of the eight magnitudes, ties to the code whose mantissa bit is 0 (the even
 * code), saturating (|q| > 6 -> 6, E2M1 has no Inf/NaN).  The sign bit is
 * copied from q, so a negative q that rounds to zero gives code 8 (-0).
 * READING: the pages fix neither the tie rule nor the sign of zero; round to
 * nearest even is the RNE rule applied to the element, and keeping the sign
 * matches a sign-preserving conversion. */
int oracle_e2m1_round(float q)
{
    int mag = nearest_even_code(fabs((double)q), e2m1_magnitude, 8);
    return signbit(q) ? (mag | 8) : mag;
}

/* UE4M3 rounding of t >= 0: nearest finite UE4M3 value, ties to the even
 * code, saturating to 0x7E (448) for anything larger ("satfinite"). */
int oracle_ue4m3_round(float t)
{
    double a = (double)t;
    /* zero, and NaN: t = (0/6)/0 for the all-zero tensor, whose global
     * scale is 0 (READING: the pages do not cover that tensor; code 0 makes
     * s = 0 and the block encode as zeros, as for any zero block) */
    if (!(a > 0.0)) return 0;
    return nearest_even_code(a, oracle_ue4m3_value, 0x7F);
}

/* UE8M0 rounding of t >= 0: nearest value 2^(c-127), c in 0..254, ties to
 * the even code, clamped to 254.  UE8M0 has no zero: t == 0 gives code 0.
 * READING: the scale rule is round-to-nearest-even of amax/6 (divided by the
 * global scale); OCP MX v1.0 itself derives the shared exponent as
 * floor(log2(amax)) - 2, which differs at ties and near the top of a binade. */
int oracle_ue8m0_round(float t)
{
    double a = (double)t;
    if (!(a > 0.0)) return 0;
    return nearest_even_code(a, oracle_ue8m0_value, 255);
}

int oracle_scale_round(int fmt, float t)
{
    return fmt == ORACLE_MXFP4 ? oracle_ue8m0_round(t) : oracle_ue4m3_round(t);
}

/* ------------------------------------------------------------------------ */
/* Quantiser                                                                  */
/* ------------------------------------------------------------------------ */

/* Global scale of a tensor for NVFP4: gs = amax / (6 * 448), one fp32
 * division (6 * 448 = 2688 is exact).  The largest block amax then lands on
 * the top of the UE4M3 range.  [DG] "Summary" (per-tensor fp32 global scale);
 * READING: the value amax/(6*448) is the usual NVFP4 choice. */
float oracle_global_scale(const float *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    return amax / 2688.0f;
}

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float oracle_global_scale_bf16(const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16_bits_to_float(x[i]));
        if (a > amax) amax = a;
    }
    return amax / 2688.0f;
}

/* One block of g fp32 values -> g nibbles (one per byte, low 4 bits) and the
 * scale byte.  Steps, in fp32 with round-to-nearest-even at each operation:
 *   amax = max |x_i|
 *   t    = (amax / 6) / gs           two divisions, in that order
 *   sf   = round-to-format(t)        UE8M0 (MXFP4) or UE4M3 (NVFP4)
 *   s    = decode(sf) * gs           one multiply
 *   q_i  = x_i / s                   one division per element
 *   nib_i = E2M1-round(q_i)
 * READING: if s is zero (UE4M3 code 0, or the product underflows) every
 * element is encoded as +0 instead of dividing by zero.
 * [DG] "Summary"; [MJ] quantize_dynamic_scaled_fp4fp8: block amax -> scale
 * -> E2M1; MXFP4 uses gs = 1. */
static int quantize_block(int fmt, const float *x, int g, float gs,
                          uint8_t *nib, uint8_t *sf)
{
    float amax = 0.0f;
    for (int i = 0; i < g; ++i) {
        if (isnan(x[i]) || isinf(x[i])) return -1;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float t = (amax / 6.0f) / gs;
    int code = oracle_scale_round(fmt, t);
    float s = (float)oracle_scale_value(fmt, code) * gs;
    *sf = (uint8_t)code;
    for (int i = 0; i < g; ++i) {
        if (s == 0.0f) {
            nib[i] = 0;
        } else {
            float q = x[i] / s;
            nib[i] = (uint8_t)oracle_e2m1_round(q);
        }
    }
    return 0;
}

/* X fp32 row-major [M, K] -> Q packed [M, K/2] and SF row-major [M, K/g].
 * Packing: element k of a row lives in byte k/2, even k in bits [3:0], odd k
 * in bits [7:4].  READING: the pages say only "2 elems/byte" ([DG]); the
 * low-nibble-first order is the one the tensor-core GEMM in this library is
 * pinned to by one-hot probes.  Returns 0, or -1 on bad arguments/inputs. */
int oracle_quantize_f32(int fmt, const float *X, int64_t M, int64_t K, float gs,
                        uint8_t *Q, uint8_t *SF)
{
    int g = oracle_block_size(fmt);
    if (M < 0 || K < 0 || K % g != 0) return -1;
    if (fmt == ORACLE_MXFP4) gs = 1.0f;
    int64_t kg = K / g;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t m = 0; m < M; ++m) {
        uint8_t nib[32];
        for (int64_t j = 0; j < kg; ++j) {
            const float *x = X + m * K + j * g;
            if (quantize_block(fmt, x, g, gs, nib, &SF[m * kg + j]) != 0) {
                bad = 1;
                continue;
            }
            for (int i = 0; i < g; i += 2)
                Q[m * (K / 2) + (j * g + i) / 2] = (uint8_t)(nib[i] | (nib[i + 1] << 4));
        }
    }
    return bad ? -1 : 0;
}

/* Same, from bf16 bit patterns (each converts to fp32 exactly). */
int oracle_quantize_bf16(int fmt, const uint16_t *X, int64_t M, int64_t K, float gs,
                         uint8_t *Q, uint8_t *SF)
{
    int g = oracle_block_size(fmt);
    if (M < 0 || K < 0 || K % g != 0) return -1;
    if (fmt == ORACLE_MXFP4) gs = 1.0f;
    int64_t kg = K / g;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t m = 0; m < M; ++m) {
        float x[32];
        uint8_t nib[32];
        for (int64_t j = 0; j < kg; ++j) {
            for (int i = 0; i < g; ++i) x[i] = bf16_bits_to_float(X[m * K + j * g + i]);
            if (quantize_block(fmt, x, g, gs, nib, &SF[m * kg + j]) != 0) {
                bad = 1;
                continue;
            }
            for (int i = 0; i < g; i += 2)
                Q[m * (K / 2) + (j * g + i) / 2] = (uint8_t)(nib[i] | (nib[i + 1] << 4));
        }
    }
    return bad ? -1 : 0;
}

/* Two-level NVFP4 ([QB] "Accuracy (real models)"): every row m has its own
 * fp32 global scale gs_rows[m] = amax over row m / (6 * 448), and row m is
 * quantised exactly as oracle_quantize_bf16 quantises it alone with that
 * scale.  READING: "per-row fp32 global" is taken as the same amax / (6*448)
 * rule applied to each row instead of the whole tensor. */
int oracle_global_scale_rows_bf16(const uint16_t *X, int64_t M, int64_t K, float *gs_out)
{
    if (M < 0 || K < 0) return -1;
    for (int64_t m = 0; m < M; ++m) gs_out[m] = oracle_global_scale_bf16(X + m * K, K);
    return 0;
}

int oracle_quantize_bf16_rows(int fmt, const uint16_t *X, int64_t M, int64_t K, const float *gs_rows,
                              uint8_t *Q, uint8_t *SF)
{
    int g = oracle_block_size(fmt);
    if (M < 0 || K < 0 || K % g != 0) return -1;
    int bad = 0;
    for (int64_t m = 0; m < M; ++m)
        if (oracle_quantize_bf16(fmt, X + m * K, 1, K, gs_rows[m], Q + m * (K / 2), SF + m * (K / g)) != 0)
            bad = 1;
    return bad ? -1 : 0;
}

/* Dequantise packed codes back to fp64: x[m,k] = E2M1(Q[m,k]) * SF[m,k/g] * gs. */
int oracle_dequantize(int fmt, const uint8_t *Q, const uint8_t *SF, int64_t M, int64_t K,
                      float gs, double *X)
{
    int g = oracle_block_size(fmt);
    if (K % g != 0) return -1;
    double gsd = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            int byte = Q[m * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            X[m * K + k] = oracle_e2m1_value(code) *
                           oracle_scale_value(fmt, SF[m * (K / g) + k / g]) * gsd;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout for the tensor cores                                  */
/* ------------------------------------------------------------------------ */

/* [MJ] block_scales_interleave: rank-2 scale factors [rows, cols] are
 * re-interleaved into the "5D TCGEN layout".  The pages do not print the
 * layout; the one used here is the public Blackwell block-scaled layout:
 * tiles of 128 rows x 4 scale columns, each tile 512 contiguous bytes in
 * which row r and column c sit at byte (r % 32) * 16 + (r / 32) * 4 + c;
 * tiles ordered row-tile-major, i.e. a 5D array
 * [ceil(rows/128)][ceil(cols/4)][32][4][4].  Padding bytes are 0. */
int64_t oracle_sf_mma_bytes(int64_t rows, int64_t cols)
{
    return ((rows + 127) / 128) * ((cols + 3) / 4) * 512;
}

int oracle_sf_to_mma(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t ctiles = (cols + 3) / 4;
    memset(out, 0, (size_t)oracle_sf_mma_bytes(rows, cols));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t tile = (r / 128) * ctiles + c / 4;
            int64_t rr = r % 128;
            int64_t off = tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
            out[off] = in[r * cols + c];
        }
    return 0;
}

int oracle_sf_from_mma(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t ctiles = (cols + 3) / 4;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t tile = (r / 128) * ctiles + c / 4;
            int64_t rr = r % 128;
            out[r * cols + c] = in[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4)];
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                       */
/* ------------------------------------------------------------------------ */

/* One output element, the definition written out ([DG] "Summary"):
 *   D[m,n] = gs_a * gs_b * sum_k e2m1(A[m,k]) sfA[m,k/g] * e2m1(B[n,k]) sfB[n,k/g]
 * Every product is exact in fp64 (at most 12 significant bits, exponents far
 * inside the fp64 range); the sum is accumulated in fp64 in k order.  Also
 * returns T = |gs_a gs_b| * sum_k |a_k b_k| for the error bound.
 * SF are row-major [rows, K/g]. */
static void gemm_entry(int fmt, int64_t K, const uint8_t *A, const uint8_t *Asf,
                       const uint8_t *B, const uint8_t *Bsf, double gsab,
                       int64_t m, int64_t n, double *d_out, double *t_out)
{
    int g = oracle_block_size(fmt);
    int64_t kg = K / g;
    double acc = 0.0, tacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        int ab = A[m * (K / 2) + k / 2];
        int bb = B[n * (K / 2) + k / 2];
        int ca = (k & 1) ? (ab >> 4) : (ab & 15);
        int cb = (k & 1) ? (bb >> 4) : (bb & 15);
        double a = oracle_e2m1_value(ca) * oracle_scale_value(fmt, Asf[m * kg + k / g]);
        double b = oracle_e2m1_value(cb) * oracle_scale_value(fmt, Bsf[n * kg + k / g]);
        acc += a * b;
        tacc += fabs(a * b);
    }
    *d_out = gsab * acc;
    *t_out = fabs(gsab) * tacc;
}

/* Full NT GEMM: A packed [M, K/2], B packed [N, K/2], SF row-major; D and T
 * fp64 [M, N].  MXFP4 ignores gs (1.0).  Returns 0 or -1. */
int oracle_gemm_nt(int fmt, int64_t M, int64_t N, int64_t K,
                   const uint8_t *A, const uint8_t *Asf, const uint8_t *B, const uint8_t *Bsf,
                   float gs_a, float gs_b, double *D, double *T)
{
    int g = oracle_block_size(fmt);
    if (K % g != 0 || K % 2 != 0) return -1;
    double gsab = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs_a * (double)gs_b;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            gemm_entry(fmt, K, A, Asf, B, Bsf, gsab, m, n, &D[m * N + n], &T[m * N + n]);
    return 0;
}

/* Sampled entries (m_i, n_i), for checks at sizes the full product would take
 * too long on the CPU. */
int oracle_gemm_nt_entries(int fmt, int64_t K,
                           const uint8_t *A, const uint8_t *Asf, const uint8_t *B, const uint8_t *Bsf,
                           float gs_a, float gs_b, int64_t count, const int64_t *mi, const int64_t *ni,
                           double *D, double *T)
{
    int g = oracle_block_size(fmt);
    if (K % g != 0 || K % 2 != 0) return -1;
    double gsab = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs_a * (double)gs_b;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        gemm_entry(fmt, K, A, Asf, B, Bsf, gsab, mi[i], ni[i], &D[i], &T[i]);
    return 0;
}

/* Two-level GEMM ([QB] "Accuracy (real models)": a per-row and per-column
 * fp32 global rescale in the MMA epilogue):
 *   D[m,n] = gs_a gs_b row_scale[m] col_scale[n] sum_k a[m,k] b[n,k]
 * with T scaled alike.  A NULL row_scale or col_scale stands for all ones.
 * MXFP4 ignores gs_a, gs_b (1.0) but not the row and column scales. */
static double rc_scale(const float *rs, const float *cs, int64_t m, int64_t n)
{
    return (rs ? (double)rs[m] : 1.0) * (cs ? (double)cs[n] : 1.0);
}

int oracle_gemm_nt_scaled(int fmt, int64_t M, int64_t N, int64_t K,
                          const uint8_t *A, const uint8_t *Asf, const uint8_t *B, const uint8_t *Bsf,
                          float gs_a, float gs_b, const float *row_scale, const float *col_scale,
                          double *D, double *T)
{
    int g = oracle_block_size(fmt);
    if (K % g != 0 || K % 2 != 0) return -1;
    double gsab = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs_a * (double)gs_b;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            gemm_entry(fmt, K, A, Asf, B, Bsf, gsab * rc_scale(row_scale, col_scale, m, n), m, n,
                       &D[m * N + n], &T[m * N + n]);
    return 0;
}

int oracle_gemm_nt_scaled_entries(int fmt, int64_t K,
                                  const uint8_t *A, const uint8_t *Asf, const uint8_t *B, const uint8_t *Bsf,
                                  float gs_a, float gs_b, const float *row_scale, const float *col_scale,
                                  int64_t count, const int64_t *mi, const int64_t *ni, double *D, double *T)
{
    int g = oracle_block_size(fmt);
    if (K % g != 0 || K % 2 != 0) return -1;
    double gsab = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs_a * (double)gs_b;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        gemm_entry(fmt, K, A, Asf, B, Bsf, gsab * rc_scale(row_scale, col_scale, mi[i], ni[i]), mi[i], ni[i],
                   &D[i], &T[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* SwiGLU of the MoE up-projection's output, before its requantisation       */
/* ------------------------------------------------------------------------ */

/* H = silu(G) * U = G * U / (1 + exp(-G)), elementwise in fp64, from the
 * exact gate and up outputs G and U of the up-projection.  [QB] "Accuracy
 * (real models)": a fused SwiGLU quantiser between the GEMMs; [DG] "Summary":
 * the MoE L1 output is requantised with the L2 activations' global scale
 * (that step is the a2 quantiser applied to H, see oracle/__init__.py).
 * READING: silu(x) = x * sigmoid(x) = x / (1 + exp(-x)), the gate being the
 * first half of the pair.  exp(-G) may overflow to +inf for G < -709; the
 * quotient is then a signed zero, the limit of the expression. */
int oracle_swiglu_f64(const double *G, const double *U, int64_t n, double *H)
{
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) H[i] = G[i] * U[i] / (1.0 + exp(-G[i]));
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Residual add and RMSNorm in front of a quantiser                         */
/* ------------------------------------------------------------------------ */

/* Round an fp32 value to the nearest bf16 bit pattern, ties to even (the
 * bf16 format is the top 16 bits of fp32).  NaN stays NaN. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
    const uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* [QB] "Accuracy (real models)": fused RMSNorm and residual-add quantisers
 * around the GEMMs of a transformer block.  Row m of the bf16 inputs:
 *   y[k] = bf16(x[k] + r[k])            one fp32 addition, rounded to bf16
 *                                       (the new residual stream; r may be
 *                                       NULL, then y = x)
 *   z[k] = y[k] / sqrt(mean_k y[k]^2 + eps) * gamma[k]       in fp64
 * READING: the pages name the fusion only; this is the usual RMSNorm with a
 * learned bf16 weight gamma, on the bf16 sum that the residual path keeps.
 * Writes y (bf16 bits), z (fp64) and 1/rms per row (fp64). */
int oracle_residual_rmsnorm(const uint16_t *x, const uint16_t *r, const uint16_t *gamma, int64_t M, int64_t K,
                            double eps, uint16_t *y, double *z, double *inv_rms)
{
    if (M < 0 || K <= 0 || !(eps >= 0.0)) return -1;
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const float xv = bf16_bits_to_float(x[m * K + k]);
            const float s = r ? xv + bf16_bits_to_float(r[m * K + k]) : xv;
            y[m * K + k] = float_to_bf16_rne(s);
            const double yv = (double)bf16_bits_to_float(y[m * K + k]);
            ss += yv * yv;
        }
        const double inv = 1.0 / sqrt(ss / (double)K + eps);
        inv_rms[m] = inv;
        for (int64_t k = 0; k < K; ++k)
            z[m * K + k] = (double)bf16_bits_to_float(y[m * K + k]) * inv * (double)bf16_bits_to_float(gamma[k]);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 2:4 pair-granular sparse operand                                          */
/* ------------------------------------------------------------------------ */

/* [QB] "Accuracy (real models)": Blackwell FP4 2:4 sparsity is pair-granular,
 * the MMA keeping 2 of every 4 consecutive fp4 pairs along K.
 * READING: a pair is the two E2M1 elements of one packed byte, so each group
 * of four bytes (eight elements) of a row keeps two bytes, at pair indices
 * i0 < i1, stored in that order in the compressed row [K/4 bytes].  The
 * group's metadata nibble is i0 | (i1 << 2); two groups per metadata byte,
 * the even group in the low nibble ([K/16] bytes per row).  The scale
 * factors are indexed by the dense K; for NVFP4 they are the per-32 blocks of
 * ORACLE_NVFP4_B32 (one scale per 16 stored elements of the sparse operand).
 * A pair is zero when both of its elements decode to 0 (codes 0 or 8). */
static int pair_is_zero(uint8_t b) { return (b & 7) == 0 && ((b >> 4) & 7) == 0; }

int oracle_sparse24_decompress(const uint8_t *Wc, const uint8_t *meta, int64_t rows, int64_t K, uint8_t *W)
{
    if (rows < 0 || K < 0 || K % 16 != 0) return -1;
    const int64_t groups = K / 8;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < groups; ++j) {
            const int nib = (meta[r * (K / 16) + j / 2] >> (4 * (j & 1))) & 15;
            const int i0 = nib & 3, i1 = nib >> 2;
            if (i0 >= i1) return -1;
            uint8_t *w = W + r * (K / 2) + 4 * j;
            for (int i = 0; i < 4; ++i) w[i] = 0;
            w[i0] = Wc[r * (K / 4) + 2 * j];
            w[i1] = Wc[r * (K / 4) + 2 * j + 1];
        }
    return 0;
}

/* The inverse for a dense packed matrix with at most two non-zero pairs per
 * group: the non-zero pairs are kept, and a group with fewer keeps its
 * lowest-indexed zero pairs as well, so that i0 < i1 always.  -1 if a group
 * has more than two non-zero pairs. */
int oracle_sparse24_compress(const uint8_t *W, int64_t rows, int64_t K, uint8_t *Wc, uint8_t *meta)
{
    if (rows < 0 || K < 0 || K % 16 != 0) return -1;
    const int64_t groups = K / 8;
    memset(meta, 0, (size_t)(rows * (K / 16)));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < groups; ++j) {
            const uint8_t *w = W + r * (K / 2) + 4 * j;
            int keep[4] = {0, 0, 0, 0}, n = 0;
            for (int i = 0; i < 4; ++i)
                if (!pair_is_zero(w[i])) { keep[i] = 1; ++n; }
            if (n > 2) return -1;
            for (int i = 0; i < 4 && n < 2; ++i)
                if (!keep[i]) { keep[i] = 1; ++n; }
            int idx[2], c = 0;
            for (int i = 0; i < 4; ++i)
                if (keep[i]) idx[c++] = i;
            Wc[r * (K / 4) + 2 * j] = w[idx[0]];
            Wc[r * (K / 4) + 2 * j + 1] = w[idx[1]];
            meta[r * (K / 16) + j / 2] |= (uint8_t)((idx[0] | (idx[1] << 2)) << (4 * (j & 1)));
        }
    return 0;
}

/* The format roundings over an array (one call of the scalar rule per
 * element), for checks over many values at once. */
int oracle_e2m1_round_n(const float *q, int64_t n, uint8_t *code)
{
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) code[i] = (uint8_t)oracle_e2m1_round(q[i]);
    return 0;
}

int oracle_scale_round_n(int fmt, const float *t, int64_t n, uint8_t *code)
{
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) code[i] = (uint8_t)oracle_scale_round(fmt, t[i]);
    return 0;
}

/* The quantiser's two rounding steps over ranges of fp32 bit patterns, for
 * checks against every fp32 input: x_i is the float whose bit pattern is
 * first + i, for i < n (the caller keeps NaN and Inf patterns out).
 *   oracle_scale_codes_bits:   the scale step of quantize_block with
 *                              amax = x_i >= 0: t = (x_i / 6) / gs, two fp32
 *                              divisions, rounded to the format (gs = 1 for
 *                              MXFP4);
 *   oracle_element_codes_bits: the element step for a block scale s > 0:
 *                              E2M1-round(x_i / s), one fp32 division. */
static float float_of_bits(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

int oracle_scale_codes_bits(int fmt, uint32_t first, int64_t n, float gs, uint8_t *code)
{
    if (n < 0 || (uint64_t)first + (uint64_t)n > ((uint64_t)1 << 32)) return -1;
    if (fmt == ORACLE_MXFP4) gs = 1.0f;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float amax = float_of_bits(first + (uint32_t)i);
        float t = (amax / 6.0f) / gs;
        code[i] = (uint8_t)oracle_scale_round(fmt, t);
    }
    return 0;
}

int oracle_element_codes_bits(uint32_t first, int64_t n, float s, uint8_t *code)
{
    if (n < 0 || (uint64_t)first + (uint64_t)n > ((uint64_t)1 << 32) || !(s > 0.0f)) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float q = float_of_bits(first + (uint32_t)i) / s;
        code[i] = (uint8_t)oracle_e2m1_round(q);
    }
    return 0;
}

/* Thread count of the OpenMP loops above (n > 0), for timing the oracle on
 * a given number of host cores. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
