/*
 * fp8_oracle.c -- plain, slow CPU definition of the Float8 linear layer's hot
 * path: per-tensor scaling (dynamic, delayed, static), row-wise scaling and
 * block scaling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library; it includes no CUDA header.
 *
 * Sources (page titles; sections):
 *  - "TorchTitan: a one-stop PyTorch-native solution for production LLM
 *    pre-training" (zenmind.me paper analysis), section 3.3 "Memory and compute
 *    optimisations", bullet "Mixed precision and Float8": Float8 is a derived
 *    dtype applied to linear layers, with dynamic / delayed / static per-tensor
 *    scaling, composable with autograd.
 *  - "Lecture 9 exercises" (juanwang-buaa tutorials), answer on fp16 loss
 *    scaling versus FP8 scaling: FP8 scaling is one factor per tensor (or per
 *    block); what FP8 saves is only what is stored in FP8.
 * The pages do not fix the formats or the arithmetic.  The readings used here
 * (e4m3 for X and W, e5m2 for dY; scale = fmt_max / amax with fmt_max = 448;
 * fp32 product then one saturating round-to-nearest-even into the format;
 * amax floored at 1e-12; the three GEMMs of a linear's forward and backward
 * with the inverse scales applied after the fp32 sum) are listed with their
 * reasons in the design notes.
 *
 * FP8 formats follow their published bit-level definitions (OCP 8-bit
 * floating point, "FP8 formats for deep learning"):
 *   e4m3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 *        no infinities, S.1111.111 is NaN, largest finite 448 (0x7E).
 *   e5m2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits, IEEE-like:
 *        exponent 31 holds Inf (mantissa 0) and NaN, largest finite 57344 (0x7B).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fno-fast-math -shared.
 * fp-contract is off so that no product is fused into an add on any host.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_E4M3 0
#define ORC_E5M2 1

/* ------------------------------------------------------------------ bits */

static float f32_from_bits(uint32_t b) {
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f) {
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return b;
}

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* ------------------------------------------------------- format params */

typedef struct {
    int ebits;      /* exponent field width          */
    int mbits;      /* mantissa field width          */
    int bias;       /* exponent bias                 */
    int max_code;   /* largest finite magnitude code */
    int ieee_inf;   /* 1: all-ones exponent is Inf/NaN (e5m2); 0: only S.1111.111 is NaN (e4m3fn) */
} fp8_fmt;

static fp8_fmt fmt_params(int fmt) {
    fp8_fmt f;
    if (fmt == ORC_E4M3) {
        f.ebits = 4; f.mbits = 3; f.bias = 7; f.max_code = 0x7E; f.ieee_inf = 0;
    } else {
        f.ebits = 5; f.mbits = 2; f.bias = 15; f.max_code = 0x7B; f.ieee_inf = 1;
    }
    return f;
}

/* --------------------------------------------------------------- decode */

/* Value of one FP8 code, straight from the sign/exponent/mantissa definition.
 * Returns NaN for NaN codes and +-Inf for e5m2's infinities. */
double orc_fp8_decode(int fmt, uint8_t code) {
    fp8_fmt f = fmt_params(fmt);
    int sign = code >> 7;
    int e = (code >> f.mbits) & ((1 << f.ebits) - 1);
    int m = code & ((1 << f.mbits) - 1);
    int emax_field = (1 << f.ebits) - 1;
    double v;
    if (f.ieee_inf && e == emax_field) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (!f.ieee_inf && e == emax_field && m == (1 << f.mbits) - 1) {
        v = NAN;
    } else if (e == 0) {
        /* subnormal: 0.m x 2^(1-bias) */
        v = ldexp((double)m, 1 - f.bias - f.mbits);
    } else {
        /* normal: 1.m x 2^(e-bias) */
        v = ldexp((double)((1 << f.mbits) + m), e - f.bias - f.mbits);
    }
    return sign ? -v : v;
}

/* ------------------------------------------------------------- encode */

/* x / 2^s rounded to the nearest integer, ties to the even integer. */
static uint64_t shift_rne(uint64_t x, int s) {
    if (s <= 0) return x;
    if (s >= 64) return 0;
    uint64_t q = x >> s;
    uint64_t r = x & ((1ull << s) - 1);
    uint64_t half = 1ull << (s - 1);
    if (r > half || (r == half && (q & 1))) q += 1;
    return q;
}

/* Saturating round-to-nearest-even of one fp32 value into an FP8 code,
 * by integer manipulation of the binary32 fields:
 *  - NaN, of either sign and any payload, gives 0x7F: the one NaN code the
 *    sm_103a conversion emits (positive, mantissa all ones; reading adopted
 *    from the hardware, the pages being silent on NaN);
 *  - |v| at or above the largest finite value (Inf included) gives the
 *    largest finite code with v's sign (saturation);
 *  - otherwise the significand is rounded to the format's mantissa width at
 *    v's exponent, or at the format's subnormal spacing when v lies below the
 *    smallest normal; ties go to the even code; the sign of zero is kept. */
uint8_t orc_fp8_encode(int fmt, float v) {
    fp8_fmt f = fmt_params(fmt);
    uint32_t u = bits_from_f32(v);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) /* NaN */
        return 0x7F;
    double max_val = orc_fp8_decode(fmt, (uint8_t)f.max_code);
    if ((double)f32_from_bits(a) >= max_val) /* saturate, Inf included */
        return (uint8_t)(sign | f.max_code);

    int exp32 = (int)(a >> 23);             /* biased binary32 exponent */
    uint64_t sig = a & 0x7FFFFFu;           /* 23-bit fraction           */
    if (exp32 == 0) {
        /* binary32 subnormal: below 2^-126, far under half the smallest
         * FP8 subnormal (2^-10 for e4m3, 2^-17 for e5m2): rounds to zero. */
        return sign;
    }
    sig |= 1u << 23;                        /* implicit leading one      */
    int e = exp32 - 127;                    /* unbiased exponent         */
    int emin = 1 - f.bias;                  /* smallest normal exponent  */
    uint32_t mag;
    if (e >= emin) {
        uint64_t r = shift_rne(sig, 23 - f.mbits);   /* 1.m with mbits bits */
        if (r == (1ull << (f.mbits + 1))) {          /* carried into next binade */
            r >>= 1;
            e += 1;
        }
        mag = (uint32_t)(((e + f.bias) << f.mbits) | (int)(r & ((1u << f.mbits) - 1)));
    } else {
        /* subnormal target: count units of 2^(emin - mbits).  A carry to
         * 2^mbits units is exactly the smallest normal code. */
        int s = (23 - f.mbits) + (emin - e);
        mag = (uint32_t)shift_rne(sig, s);
    }
    return (uint8_t)(sign | mag);
}

/* encode() applied to an array of binary32 values. */
void orc_encode_f32(const float *v, int64_t n, int fmt, uint8_t *q) {
    for (int64_t i = 0; i < n; ++i) q[i] = orc_fp8_encode(fmt, v[i]);
}

/* ---------------------------------------------------------------- amax */

/* amax = max_i |x_i| over a bf16 tensor (fp32 result, exact: the maximum of
 * bf16 magnitudes is itself a bf16 value).  Magnitudes are ordered by the
 * IEEE 754 totalOrder predicate: for finite values that is the ordinary
 * order, +Inf lies above every finite value and NaNs lie above +Inf, ordered
 * by payload.  An empty tensor gives 0. */
float orc_amax_bf16(const uint16_t *x, int64_t n) {
    float best = 0.0f;
    uint16_t nan_mag = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint16_t mag = (uint16_t)(x[i] & 0x7FFF);
        if (mag > 0x7F80) {                 /* NaN */
            if (mag > nan_mag) nan_mag = mag;
            continue;
        }
        float v = fabsf(orc_bf16_to_f32(x[i]));
        if (v > best) best = v;
    }
    if (nan_mag) return orc_bf16_to_f32(nan_mag);
    return best;
}

/* --------------------------------------------------------------- scale */

/* A binary32 operation whose result is NaN gives, on the GPU, the one NaN
 * 0x7FFFFFFF (sign clear, every significand bit set), where x86 keeps an
 * operand's sign and payload.  The scale arithmetic below stores its NaN
 * results in that form (reading adopted from the hardware; the pages say
 * nothing of NaN). */
static float canonical_nan(float v) {
    return (bits_from_f32(v) & 0x7FFFFFFFu) > 0x7F800000u ? f32_from_bits(0x7FFFFFFFu) : v;
}

/* scale = fmt_max / max(amax, 1e-12) and inv_scale = 1 / scale, both as
 * binary32 round-to-nearest operations.  A NaN amax gives the canonical NaN
 * for both. */
void orc_scale(float amax, float fmt_max, float *scale, float *inv_scale) {
    volatile float a = (amax < 1e-12f) ? 1e-12f : amax;
    volatile float s = fmt_max / a;
    volatile float inv = 1.0f / s;
    *scale = canonical_nan(s);
    *inv_scale = canonical_nan(inv);
}

/* orc_scale applied to n amax values. */
void orc_scales(const float *amax, int64_t n, float fmt_max, float *scale, float *inv_scale) {
    for (int64_t i = 0; i < n; ++i) orc_scale(amax[i], fmt_max, &scale[i], &inv_scale[i]);
}

/* 1 / s as one binary32 round-to-nearest division (static scaling's
 * inverse scale). */
float orc_reciprocal(float s) {
    volatile float r = 1.0f / s;
    return canonical_nan(r);
}

/* Largest entry of an amax history h[0..n), leaving out index `skip` (the
 * slot the current step writes): delayed scaling takes its statistic from
 * earlier steps.  Entries are non-negative; ordered like orc_amax_bf16
 * (totalOrder: a NaN ranks above every number).  No entry gives 0. */
float orc_history_max(const float *h, int64_t n, int64_t skip) {
    float best = 0.0f;
    uint32_t nan_bits = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (i == skip) continue;
        uint32_t b = bits_from_f32(h[i]) & 0x7FFFFFFFu;
        if (b > 0x7F800000u) {
            if (b > nan_bits) nan_bits = b;
            continue;
        }
        float v = f32_from_bits(b);
        if (v > best) best = v;
    }
    if (nan_bits) return f32_from_bits(nan_bits);
    return best;
}

/* ---------------------------------------------------------------- cast */

/* q_i = encode(fp32(x_i) * scale): the product is one binary32 multiply
 * (round to nearest even), then one saturating RNE into the FP8 format. */
void orc_cast_bf16(const uint16_t *x, int64_t n, int fmt, float scale, uint8_t *q) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        volatile float v = orc_bf16_to_f32(x[i]) * scale;
        q[i] = orc_fp8_encode(fmt, v);
    }
}

/* Row-wise scaling ("per block", one block = one row of the operand, the
 * finest block that stays constant along the GEMM's contraction):
 * amax of every row of a row-major bf16 [rows x cols] matrix. */
void orc_amax_rows_bf16(const uint16_t *x, int64_t rows, int64_t cols, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) out[r] = orc_amax_bf16(x + r * cols, cols);
}

/* amax of every column (column c's elements are x[r][c], r = 0..rows-1). */
void orc_amax_cols_bf16(const uint16_t *x, int64_t rows, int64_t cols, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        float best = 0.0f;
        uint16_t nan_mag = 0;
        for (int64_t r = 0; r < rows; ++r) {
            uint16_t h = x[r * cols + c];
            uint16_t mag = (uint16_t)(h & 0x7FFF);
            if (mag > 0x7F80) {
                if (mag > nan_mag) nan_mag = mag;
                continue;
            }
            float v = fabsf(orc_bf16_to_f32(h));
            if (v > best) best = v;
        }
        out[c] = nan_mag ? orc_bf16_to_f32(nan_mag) : best;
    }
}

/* q[r][c] = encode(fp32(x[r][c]) * scale[r]): the cast with one scale per row. */
void orc_cast_rows_bf16(const uint16_t *x, int64_t rows, int64_t cols, int fmt, const float *scale,
                        uint8_t *q) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            volatile float v = orc_bf16_to_f32(x[r * cols + c]) * scale[r];
            q[r * cols + c] = orc_fp8_encode(fmt, v);
        }
}

/* Block scaling ("per block", block = br x bc elements of the row-major
 * [rows x cols] source; blocks at the right and bottom edges are cut short):
 * amax of block (i, j) = max |x[r][c]| over r in [i br, (i+1) br) and
 * c in [j bc, (j+1) bc), same ordering as orc_amax_bf16 (a NaN magnitude
 * above every number).  out is [ceil(rows/br) x ceil(cols/bc)]. */
void orc_amax_blocks_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t br, int64_t bc, float *out) {
    const int64_t nbr = (rows + br - 1) / br, nbc = (cols + bc - 1) / bc;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < nbr * nbc; ++b) {
        const int64_t bi = b / nbc, bj = b % nbc;
        float best = 0.0f;
        uint16_t nan_mag = 0;
        for (int64_t r = bi * br; r < rows && r < (bi + 1) * br; ++r)
            for (int64_t c = bj * bc; c < cols && c < (bj + 1) * bc; ++c) {
                uint16_t mag = (uint16_t)(x[r * cols + c] & 0x7FFF);
                if (mag > 0x7F80) {
                    if (mag > nan_mag) nan_mag = mag;
                    continue;
                }
                float v = orc_bf16_to_f32(mag);
                if (v > best) best = v;
            }
        out[b] = nan_mag ? orc_bf16_to_f32(nan_mag) : best;
    }
}

/* q[r][c] = encode(fp32(x[r][c]) * scale[r / br][c / bc]): the cast with one
 * scale per block (scale is [ceil(rows/br) x ceil(cols/bc)]). */
void orc_cast_blocks_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t br, int64_t bc, int fmt,
                          const float *scale, uint8_t *q) {
    const int64_t nbc = (cols + bc - 1) / bc;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            volatile float v = orc_bf16_to_f32(x[r * cols + c]) * scale[(r / br) * nbc + c / bc];
            q[r * cols + c] = orc_fp8_encode(fmt, v);
        }
}

/* qT[c][r] = q[r][c] for a row-major [rows x cols] byte matrix. */
void orc_transpose_u8(const uint8_t *q, int64_t rows, int64_t cols, uint8_t *qT) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c)
        for (int64_t r = 0; r < rows; ++r)
            qT[c * rows + r] = q[r * cols + c];
}

/* ---------------------------------------------------------------- GEMM */

/* Reference for one scaled FP8 GEMM written as C = A . B^T, with both
 * operands stored with the contraction index contiguous:
 *     A is [P x R] codes (format fa), B is [Q x R] codes (format fb),
 *     C[p][q] = ( sum_k dec(A[p][k]) * dec(B[q][k]) ) * inv_a * inv_b,
 * the sum taken in binary64 in increasing k, the inverse scales applied
 * after it in binary64.  Only the rows listed in `rows` (nrows of them) are
 * computed; out is [nrows x Q].  The forward pass, input gradient and weight
 * gradient of the linear layer are the three instances
 *     Y  = Xq . Wq^T        (A = Xq,   B = Wq)
 *     dX = dYq . (WqT)^T    (A = dYq,  B = WqT,  i.e. dY . W)
 *     dW = dYqT . (XqT)^T   (A = dYqT, B = XqT,  i.e. dY^T . X). */
void orc_gemm_rows(const uint8_t *A, int fa, const uint8_t *B, int fb,
                   int64_t P, int64_t Q, int64_t R, float inv_a, float inv_b,
                   const int64_t *rows, int64_t nrows, double *out) {
    double da[256], db[256];
    for (int c = 0; c < 256; ++c) {
        da[c] = orc_fp8_decode(fa, (uint8_t)c);
        db[c] = orc_fp8_decode(fb, (uint8_t)c);
    }
    (void)P;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const uint8_t *a = A + rows[i] * R;
        for (int64_t q = 0; q < Q; ++q) {
            const uint8_t *b = B + q * R;
            double s = 0.0;
            for (int64_t k = 0; k < R; ++k)
                s += da[a[k]] * db[b[k]];
            out[i * Q + q] = s * (double)inv_a * (double)inv_b;
        }
    }
}

/* orc_gemm_rows with one inverse scale per row of A and per row of B:
 * C[p][q] = ( sum_k dec(A[p][k]) * dec(B[q][k]) ) * inv_a[p] * inv_b[q]. */
void orc_gemm_rows_vec(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t P, int64_t Q, int64_t R,
                       const float *inv_a, const float *inv_b, const int64_t *rows, int64_t nrows, double *out) {
    double da[256], db[256];
    for (int c = 0; c < 256; ++c) {
        da[c] = orc_fp8_decode(fa, (uint8_t)c);
        db[c] = orc_fp8_decode(fb, (uint8_t)c);
    }
    (void)P;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const uint8_t *a = A + rows[i] * R;
        for (int64_t q = 0; q < Q; ++q) {
            const uint8_t *b = B + q * R;
            double s = 0.0;
            for (int64_t k = 0; k < R; ++k)
                s += da[a[k]] * db[b[k]];
            out[i * Q + q] = s * (double)inv_a[rows[i]] * (double)inv_b[q];
        }
    }
}

/* The GEMM with block scales along the contraction: the contraction is cut
 * into blocks of rb indices (the last one short), and
 *     C[p][q] = sum over blocks j of
 *               ( sum_{k in block j} dec(A[p][k]) * dec(B[q][k]) ) * inv_a[p][j] * inv_b[q][j],
 * each block's sum in binary64 in increasing k, scaled in binary64, the
 * blocks added in increasing j.  inv_a is [P x nb], inv_b is [Q x nb]
 * (nb = ceil(R / rb)): one inverse scale per operand row and contraction
 * block, whatever block shape the operand was quantised with. */
void orc_gemm_blocks(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t P, int64_t Q, int64_t R,
                     int64_t rb, const float *inv_a, const float *inv_b, const int64_t *rows, int64_t nrows,
                     double *out) {
    double da[256], db[256];
    for (int c = 0; c < 256; ++c) {
        da[c] = orc_fp8_decode(fa, (uint8_t)c);
        db[c] = orc_fp8_decode(fb, (uint8_t)c);
    }
    (void)P;
    const int64_t nb = (R + rb - 1) / rb;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t p = rows[i];
        const uint8_t *a = A + p * R;
        for (int64_t q = 0; q < Q; ++q) {
            const uint8_t *b = B + q * R;
            double total = 0.0;
            for (int64_t j = 0; j < nb; ++j) {
                double s = 0.0;
                for (int64_t k = j * rb; k < R && k < (j + 1) * rb; ++k)
                    s += da[a[k]] * db[b[k]];
                total += s * (double)inv_a[p * nb + j] * (double)inv_b[q * nb + j];
            }
            out[i * Q + q] = total;
        }
    }
}

/* ------------------------------------------------ power-of-two block scales */

/* Block scaling with power-of-two scales (the "per block" factor of the
 * Lecture 9 exercises, restricted to powers of two so that the tensor cores'
 * block-scaled MMA can apply it): a block's scale is 2^e, e the largest
 * integer with max(amax, 1e-12) * 2^e <= fmt_max -- the largest power of two
 * not above fmt_max / amax, so the block's largest magnitude lands at or
 * below the format maximum and nothing saturates -- clamped to [-127, 127].
 * The result is the byte 127 - e, the unsigned-exponent (UE8M0) code of the
 * inverse scale 2^-e.  A NaN or infinite amax gives 0xFF (the UE8M0 NaN).
 * Written as a search over e: scaling by a power of two is exact in
 * binary64 for every value reached here, so each comparison is exact. */
uint8_t orc_pow2_scale_byte(float amax, float fmt_max) {
    if (!(amax <= 3.4028234663852886e38f)) return 0xFF;  /* NaN or +Inf */
    const double a = (amax < 1e-12f) ? (double)1e-12f : (double)amax;
    const double f = (double)fmt_max;
    int e = 0;
    while (e > -400 && ldexp(a, e) > f) --e;
    while (e < 400 && ldexp(a, e + 1) <= f) ++e;
    if (e > 127) e = 127;
    if (e < -127) e = -127;
    return (uint8_t)(127 - e);
}

/* The OCP Microscaling (MX) rule for the same blocks: the block's shared
 * scale is X = 2^(floor(log2 amax) - emax_elem), emax_elem the exponent of
 * the element format's largest normal (8 for e4m3, 15 for e5m2), and the
 * elements are x / X cast with saturation -- magnitudes in (fmt_max, 2^(emax+1))
 * saturate.  A zero amax gives the smallest scale (2^-127), a NaN or infinite
 * amax 0xFF.  Returned as the byte 127 + log2 X (the code of X, which is the
 * inverse scale here: the cast multiplies by 1 / X), clamped to [0, 254].
 * floor(log2 amax) is found by search: the largest f with 2^f <= amax. */
uint8_t orc_ocp_scale_byte(float amax, int fmt) {
    if (!(amax <= 3.4028234663852886e38f)) return 0xFF;  /* NaN or +Inf */
    if (amax == 0.0f) return 0;
    const int emax = fmt == ORC_E4M3 ? 8 : 15;
    const double a = (double)amax;
    int f = 0;
    while (f > -400 && ldexp(1.0, f) > a) --f;
    while (f < 400 && ldexp(1.0, f + 1) <= a) ++f;
    int b = 127 + f - emax;
    if (b < 0) b = 0;
    if (b > 254) b = 254;
    return (uint8_t)b;
}

void orc_ocp_scale_bytes(const float *amax, int64_t n, int fmt, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_ocp_scale_byte(amax[i], fmt);
}

/* orc_pow2_scale_byte applied to n amax values. */
void orc_pow2_scale_bytes(const float *amax, int64_t n, float fmt_max, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_pow2_scale_byte(amax[i], fmt_max);
}

/* Number of threads the parallel loops above use. */
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
