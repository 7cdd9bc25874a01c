/*
 * q8ref.c -- plain, slow CPU oracle for the Q8_0 W8A16 decode matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or constant with the CUDA
 * library; it is compiled with plain gcc, -O2, no fast-math, no FP contraction.
 *
 * What it follows (page titles are those of the web pages the method is
 * taken from):
 *
 *  - "MODEL-BASELINE-RESULTS" (fak), ACT 3, "How it was closed", item 1:
 *    weights are cut into 32-element blocks; each block carries one scale
 *    d = maxabs/127 and 32 int8 codes (about 1.06 bytes per weight, which is
 *    a 2-byte scale per 32 codes: the scale is stored as IEEE binary16).
 *  - same page, ACT 4, "Correctness": codes are rounded half away from zero
 *    (the result must equal math.Round; adding 0.5 and truncating is wrong,
 *    e.g. 0.49999997 must give 0, not 1).
 *  - same page, ACT 5, "What moved", item 3: the quantizer must stay exact on
 *    zeros, denormals and exact halves.
 *  - "Frigg" README, Finding 8: W8A16 means int8 weights times bf16
 *    activations, each weight read once per matmul; accumulation is wide.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes):
 *  - the scale is computed in binary32 (d32 = amax/127, IEEE division, round
 *    to nearest even), then rounded once more to binary16 (nearest even,
 *    subnormals kept); the code divides the weight by the STORED scale and the
 *    exact quotient is rounded half away from zero, then clamped to +-127;
 *  - a zero scale gives all-zero codes;
 *  - a block holding a NaN or an infinity, or whose scale overflows binary16,
 *    is flagged and stored as zero codes with a zero scale;
 *  - the matmul reference dequantises every weight to s*q and forms the dot
 *    product in binary64, k in increasing order, and also returns the bound
 *    B = sum_k |s*q*x| used by the tolerance |y - y_ref| <= 2e-3*B + 1e-6.
 *
 * Parity pins: every function below is checked by the CPU test suite against
 * values fixed by the pages or by mathematics (exhaustive binary16 checks
 * against numpy, an integer-exact rounding comparator, exact-half blocks with
 * closed-form codes, brute-force rational dot products on tiny inputs).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define Q8REF_FLAG_NONFINITE 1u
#define Q8REF_FLAG_SCALE_OVF 2u

/* ---------------------------------------------------------------------- */
/* IEEE-754 binary16 from binary32: round to nearest, ties to even.        */
/* Written from the definition: find the spacing of binary16 numbers at    */
/* the magnitude of v, divide (exact, a power of two), round the quotient  */
/* to an integer with ties to even, multiply back, then encode.            */
/* ---------------------------------------------------------------------- */
uint16_t q8ref_f32_to_f16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);

    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    if (isinf(f)) return (uint16_t)(sign | 0x7c00u);

    double v = fabs((double)f);          /* exact */
    if (v == 0.0) return sign;

    /* spacing of binary16 values around v */
    int e2;
    (void)frexp(v, &e2);                 /* v = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                      /* v in [2^e, 2^(e+1)) */
    if (e < -14) e = -14;                /* subnormal range has fixed spacing 2^-24 */
    double ulp = ldexp(1.0, e - 10);

    double t = v / ulp;                  /* exact: scaling by a power of two */
    double fl = floor(t);
    double frac = t - fl;                /* exact */
    double r;
    if (frac > 0.5) r = fl + 1.0;
    else if (frac < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: to even */
    double rv = r * ulp;                 /* exact */

    if (rv >= 65536.0) return (uint16_t)(sign | 0x7c00u);   /* overflow -> inf */

    if (rv < ldexp(1.0, -14)) {
        /* subnormal (or zero): value = n * 2^-24, n < 1024 */
        uint16_t n = (uint16_t)(rv / ldexp(1.0, -24));
        return (uint16_t)(sign | n);
    }
    int e2r;
    double mr = frexp(rv, &e2r);         /* rv = mr * 2^e2r */
    int er = e2r - 1;                    /* rv = (1 + frac) * 2^er */
    double fracr = mr * 2.0 - 1.0;       /* in [0, 1) */
    uint16_t mant = (uint16_t)(fracr * 1024.0);   /* exact: 10 fraction bits */
    uint16_t expo = (uint16_t)(er + 15);
    return (uint16_t)(sign | (expo << 10) | mant);
}

/* binary16 bits -> exact binary64 value */
double q8ref_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0x1f) v = mant ? NAN : INFINITY;
    else if (expo == 0) v = ldexp((double)mant, -24);
    else v = ldexp(1.0 + mant / 1024.0, expo - 15);
    return sign ? -v : v;
}

/* bfloat16 bits -> exact binary64 value (bf16 is the top half of binary32) */
double q8ref_bf16_to_f64(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------- */
/* The code of one weight given the stored scale s (> 0, finite):          */
/* exact quotient |w|/s rounded half away from zero, clamped to 127.       */
/* The binary64 quotient decides ties exactly: w has 24 significant bits   */
/* and s has 11, so a quotient below 128 that is not a half-integer sits   */
/* at least 2^-35 away from one, far beyond binary64 rounding (2^-46).     */
/* ---------------------------------------------------------------------- */
int8_t q8ref_code(float w, double s)
{
    if (s == 0.0) return 0;
    double t = (double)w / s;
    double a = fabs(t);
    double k = floor(a + 0.5);           /* exact for a < 2^52 */
    if (k > 127.0) k = 127.0;
    return (int8_t)(t < 0.0 ? -k : k);
}

/* ---------------------------------------------------------------------- */
/* Compatibility codes: the binary32 quotient w / d32 (IEEE division,      */
/* round to nearest even; d32 = amax/127 in binary32, before the binary16  */
/* rounding of the stored scale) rounded half away from zero and clamped   */
/* to 127 -- the binary32 quotient that "MODEL-BASELINE-RESULTS" (fak),    */
/* ACT 4 "Correctness", rounds with q8round.  The half-away rounding of a  */
/* binary32 value is exact in binary64 (24 significant bits + 0.5).        */
/* ---------------------------------------------------------------------- */
int8_t q8ref_code_fl32(float w, float d32)
{
    if (d32 == 0.0f) return 0;
    volatile float t = w / d32;
    double a = fabs((double)t);
    double k = floor(a + 0.5);
    if (k > 127.0) k = 127.0;
    return (int8_t)(t < 0.0f ? -k : k);
}

/* ---------------------------------------------------------------------- */
/* Quantize rows x K binary32 weights into Q8_0 blocks along K.            */
/*   q      : int8  [rows][K]                                              */
/*   s_bits : binary16 bits [rows][K/32]                                   */
/*   flags  : uint32 [rows][K/32] (may be NULL), per-block flag bits        */
/* Returns the OR of all flags.  K must be a multiple of 32.               */
/* ---------------------------------------------------------------------- */
uint32_t q8ref_quantize_rows(const float *w, int64_t rows, int64_t K,
                             int8_t *q, uint16_t *s_bits, uint32_t *flags)
{
    uint32_t all = 0;
    int64_t nb = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = w + r * K + b * 32;
            int8_t *qb = q + r * K + b * 32;
            uint32_t fl = 0;

            /* step 1: amax over the block (exact in binary32) */
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                if (!isfinite(blk[i])) fl |= Q8REF_FLAG_NONFINITE;
                else if (fabsf(blk[i]) > amax) amax = fabsf(blk[i]);
            }
            uint16_t sb = 0;
            if (!fl) {
                /* step 2: d = amax / 127 in binary32 */
                volatile float d32 = amax / 127.0f;
                /* step 3: stored scale = binary16(d) */
                sb = q8ref_f32_to_f16(d32);
                if ((sb & 0x7c00u) == 0x7c00u) fl |= Q8REF_FLAG_SCALE_OVF;
            }
            if (fl) {
                for (int i = 0; i < 32; ++i) qb[i] = 0;
                s_bits[r * nb + b] = 0;
            } else {
                /* step 4: codes from the stored scale */
                double sd = q8ref_f16_to_f64(sb);
                for (int i = 0; i < 32; ++i) qb[i] = q8ref_code(blk[i], sd);
                s_bits[r * nb + b] = sb;
            }
            if (flags) flags[r * nb + b] = fl;
            all |= fl;
        }
    }
    return all;
}

/* ---------------------------------------------------------------------- */
/* Dequantise-then-dot in binary64 for output rows [n_begin, n_end):       */
/*   y[m][n]   = sum_k (s[n][k/32] * q[n][k]) * x[m][k]                    */
/*   bnd[m][n] = sum_k |(s[n][k/32] * q[n][k]) * x[m][k]|                  */
/* q int8 [N][K], s_bits binary16 [N][K/32], x_bf16 bf16 bits [M][ldx],    */
/* y and bnd binary64 [M][ldy] (bnd may be NULL).                          */
/* ---------------------------------------------------------------------- */
/* ---------------------------------------------------------------------- */
/* As q8ref_quantize_rows, with the compatibility codes: the same scale    */
/* d32, the same stored binary16 scale and flags, but each code is         */
/* q8ref_code_fl32(w, d32); a stored scale of zero still gives zero codes. */
/* ---------------------------------------------------------------------- */
uint32_t q8ref_quantize_rows_fl32(const float *w, int64_t rows, int64_t K,
                                  int8_t *q, uint16_t *s_bits, uint32_t *flags)
{
    uint32_t all = 0;
    int64_t nb = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = w + r * K + b * 32;
            int8_t *qb = q + r * K + b * 32;
            uint32_t fl = 0;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                if (!isfinite(blk[i])) fl |= Q8REF_FLAG_NONFINITE;
                else if (fabsf(blk[i]) > amax) amax = fabsf(blk[i]);
            }
            uint16_t sb = 0;
            volatile float d32 = 0.0f;
            if (!fl) {
                d32 = amax / 127.0f;
                sb = q8ref_f32_to_f16(d32);
                if ((sb & 0x7c00u) == 0x7c00u) fl |= Q8REF_FLAG_SCALE_OVF;
            }
            if (fl || sb == 0) {
                for (int i = 0; i < 32; ++i) qb[i] = 0;
                s_bits[r * nb + b] = fl ? 0 : sb;
            } else {
                for (int i = 0; i < 32; ++i) qb[i] = q8ref_code_fl32(blk[i], d32);
                s_bits[r * nb + b] = sb;
            }
            if (flags) flags[r * nb + b] = fl;
            all |= fl;
        }
    }
    return all;
}

void q8ref_code_fl32_array(const float *w, int64_t n, float d32, int8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q8ref_code_fl32(w[i], d32);
}

void q8ref_matmul(const int8_t *q, const uint16_t *s_bits, int64_t N, int64_t K,
                  const uint16_t *x_bf16, int64_t ldx, int64_t M,
                  int64_t n_begin, int64_t n_end,
                  double *y, double *bnd, int64_t ldy)
{
    (void)N;
    int64_t nb = K / 32;
    for (int64_t n = n_begin; n < n_end; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, b = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double wd = q8ref_f16_to_f64(s_bits[n * nb + k / 32]) * (double)q[n * K + k];
                double xd = q8ref_bf16_to_f64(x_bf16[m * ldx + k]);
                double p = wd * xd;
                acc += p;
                b += fabs(p);
            }
            y[m * ldy + n] = acc;
            if (bnd) bnd[m * ldy + n] = b;
        }
    }
}

/* Elementwise helpers for exhaustive checks from Python. */
void q8ref_f32_to_f16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q8ref_f32_to_f16(in[i]);
}

void q8ref_f16_to_f64_array(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q8ref_f16_to_f64(in[i]);
}

void q8ref_code_array(const float *w, int64_t n, uint16_t s_bits, int8_t *out)
{
    double sd = q8ref_f16_to_f64(s_bits);
    for (int64_t i = 0; i < n; ++i) out[i] = q8ref_code(w[i], sd);
}
