/*
 * oref.c -- CPU oracle for the forward FP8 MLP down-projection.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, independent
 * statement of what the GPU path computes.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark load it.  It shares no code,
 * header, table or constant generator with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Every floating-point step is written in double precision and rounded to the
 * precision the method fixes with a single, explicit cast.  Where float32
 * arithmetic decides an FP8 code (the scaled value v = a * s, the scale
 * 448 / (margin * amax)), the oracle forms the product or quotient of two
 * float32 values in double and casts it to float: the double product is exact,
 * and for the quotient 53 >= 2*24 + 2 makes the double rounding innocuous, so
 * the result is the correctly rounded float32 one.  Build with
 * -ffp-contract=off so the compiler fuses nothing.
 *
 * Sources (cited by page title and section):
 *  - "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records",
 *    second paragraph: the fused activation + quantize step, the BF16 copy
 *    kept for backward, running maxima, previous-step amax times a margin.
 *  - "FP8 training: what it is and how it works": Step 1 (formats, max 448 /
 *    57344, gaps 0.125 / 0.25), Step 2 (scale = format max / amax; worked
 *    example 3.2 -> 140, 0.01 -> 1.375), Step 3 (FP8 inputs, wide sums),
 *    Worked example (per-tensor vs 128-value tiles), Trade-offs and edge
 *    cases (1x128 activation tiles, 128x128 weight blocks, delayed scaling
 *    from a stored amax history).
 *  - "FP8 Training & Inference": FP8 Formats: E4M3 vs E5M2; FP8 Training
 *    Recipe (the three GEMMs, dX = dY x W^T); Per-Tensor Scaling for FP8
 *    (scales factored out of the matmul); Delayed Scaling.
 *  - "Pretraining at scale", 4a (float anatomy, bf16 worked example), 4d.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OREF_E4M3 0
#define OREF_E5M2 1

#define OREF_ACT_IDENTITY 0
#define OREF_ACT_RELU 1
#define OREF_ACT_RELU2 2

#define OREF_GROUP 128 /* width of one scale group along the contraction */

/* ------------------------------------------------------------------------ */
/* Float32 / BF16                                                            */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* A BF16 value is the top half of a float32 pattern. */
float oref_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/*
 * Round a float32 to BF16, to nearest, ties to even ("Pretraining at scale",
 * 4a: sign, 8 exponent bits, 7 fraction bits).  Dropping the low 16 bits of
 * the float32 pattern truncates the fraction; adding 0x7FFF plus the kept LSB
 * first rounds to nearest with ties to the even kept fraction.  A carry out of
 * the fraction bumps the exponent, and values past the largest BF16 become
 * infinity, as IEEE rounding does.  NaN stays NaN (quiet bit set, sign kept).
 */
uint16_t oref_f32_to_bf16(float x)
{
    uint32_t u = bits_from_f32(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oref_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oref_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* FP8 formats, from their definitions                                       */
/* ------------------------------------------------------------------------ */
/*
 * E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.  No infinity; the
 * pattern S.1111.111 is NaN, so the largest finite code is 0x7E = 1.75 * 2^8
 * = 448.  E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits, IEEE-like:
 * exponent field 31 is infinity (mantissa 0) or NaN; the largest finite code
 * is 0x7B = 1.75 * 2^15 = 57344.  Exponent field 0 holds zero and the
 * subnormals m * 2^(1 - bias - mbits).  ("FP8 training: what it is and how it
 * works", Step 1; "FP8 Training & Inference", FP8 Formats: E4M3 vs E5M2.)
 */
typedef struct {
    int ebits, mbits, bias;
    int max_code;     /* largest finite non-negative code */
    double max_value; /* its value */
} fmt_desc;

static fmt_desc fmt_of(int fmt)
{
    fmt_desc d;
    if (fmt == OREF_E5M2) {
        d.ebits = 5; d.mbits = 2; d.bias = 15; d.max_code = 0x7B; d.max_value = 57344.0;
    } else {
        d.ebits = 4; d.mbits = 3; d.bias = 7; d.max_code = 0x7E; d.max_value = 448.0;
    }
    return d;
}

double oref_fp8_max(int fmt) { return fmt_of(fmt).max_value; }

/* Value of an FP8 code, straight from the field definitions. */
double oref_fp8_decode(uint8_t code, int fmt)
{
    fmt_desc d = fmt_of(fmt);
    int sign = code >> 7;
    int e = (code >> d.mbits) & ((1 << d.ebits) - 1);
    int m = code & ((1 << d.mbits) - 1);
    int e_all_ones = (1 << d.ebits) - 1;
    double v;
    if (fmt == OREF_E4M3 && e == e_all_ones && m == (1 << d.mbits) - 1)
        return NAN;
    if (fmt == OREF_E5M2 && e == e_all_ones) {
        if (m != 0) return NAN;
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, 1 - d.bias - d.mbits);
    } else {
        v = ldexp(1.0 + ldexp((double)m, -d.mbits), e - d.bias);
    }
    return sign ? -v : v;
}

/*
 * Encode a float32 to FP8: the representable value nearest to |v|, ties to the
 * code whose last mantissa bit is even (round to nearest even); values beyond
 * the largest finite value, and infinities, saturate to it with v's sign (the
 * method saturates at +-448 instead of overflowing).  Values at or below half
 * the smallest subnormal round to a zero of v's sign.  NaN gives the NaN code
 * 0x7F (its sign is not part of the contract).
 *
 * The search runs over the decoded values of the non-negative finite codes,
 * which increase strictly with the code; no bit manipulation of v is used.
 */
uint8_t oref_fp8_encode(float v, int fmt)
{
    fmt_desc d = fmt_of(fmt);
    if (v != v) return 0x7F;
    uint8_t sign = (bits_from_f32(v) >> 31) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= d.max_value) return (uint8_t)(sign | d.max_code);
    int lo = 0, hi = d.max_code; /* invariant: decode(lo) <= a < decode(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oref_fp8_decode((uint8_t)mid, fmt) <= a) lo = mid; else hi = mid;
    }
    double vlo = oref_fp8_decode((uint8_t)lo, fmt);
    double vhi = oref_fp8_decode((uint8_t)hi, fmt);
    double midpoint = 0.5 * (vlo + vhi); /* exact: both are short dyadics */
    int code;
    if (a < midpoint) code = lo;
    else if (a > midpoint) code = hi;
    else code = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | code);
}

void oref_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oref_fp8_encode(v[i], fmt);
}

void oref_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oref_fp8_decode(c[i], fmt);
}

/* ------------------------------------------------------------------------ */
/* Activation and float32 helpers                                            */
/* ------------------------------------------------------------------------ */
/*
 * The down-projection consumes act(H) for the pre-activation H.  ReLU(h) is h
 * when h > 0, else +0 (so -0 and NaN give +0).  ReLU^2 squares that; the
 * square of a BF16 value has at most 16 significant bits, so it is exact in
 * float32 unless it overflows to infinity.
 */
float oref_act(float h, int act)
{
    if (act == OREF_ACT_IDENTITY) return h;
    double r = (h > 0.0f) ? (double)h : 0.0;
    if (act == OREF_ACT_RELU) return (float)r;
    return (float)(r * r);
}

/* Correctly rounded float32 product and quotient (see the file header). */
static float mul_f32(float x, float y) { return (float)((double)x * (double)y); }
static float div_f32(float x, float y) { return (float)((double)x / (double)y); }

/* |x| as an ordered key: for non-negative floats the bit pattern orders them,
 * and a NaN magnitude sorts above infinity, so the maximum is total. */
static uint32_t mag_key(float x) { return bits_from_f32(x) & 0x7FFFFFFFu; }

/* ------------------------------------------------------------------------ */
/* Scales                                                                    */
/* ------------------------------------------------------------------------ */
/*
 * Delayed per-tensor scale ("Paradigma Details FP8 ...", second paragraph:
 * the previous step's maximum multiplied by a safety margin; "FP8 training:
 * what it is and how it works", Step 2: scale = format max / amax):
 *     s = float32( fmt_max / float32(margin * amax_ref) ).
 * Returns 0 when amax_ref is not a positive finite number or the scale is not
 * finite and positive; the caller then keeps its previous scale.
 */
float oref_delayed_scale(float amax_ref, float margin, int fmt)
{
    if (!(amax_ref > 0.0f) || isinf(amax_ref)) return 0.0f;
    float denom = mul_f32(margin, amax_ref);
    float s = div_f32((float)fmt_of(fmt).max_value, denom);
    if (!(s > 0.0f) || isinf(s)) return 0.0f;
    return s;
}

/*
 * The amax history ("FP8 training: what it is and how it works", Trade-offs:
 * delayed scaling needs a stored history; "FP8 Training & Inference", Delayed
 * Scaling: use the previous iteration's statistics).  history[0..L-1] is a
 * ring whose newest entry is history[*head].  One update pushes amax_new into
 * the next slot, takes amax_ref = max over all L entries, and sets
 * *scale = oref_delayed_scale(amax_ref, margin, fmt) when that is valid.
 * Returns 0 on success, 1 when the scale was kept because the reference
 * amax (or the scale it gives) is not usable.
 */
int oref_history_update(float* history, int L, int* head, float amax_new,
                        float margin, int fmt, float* scale)
{
    int h = (*head + 1) % L;
    history[h] = amax_new;
    *head = h;
    uint32_t ref = 0;
    for (int i = 0; i < L; ++i)
        if (mag_key(history[i]) > ref) ref = mag_key(history[i]);
    float s = oref_delayed_scale(f32_from_bits(ref), margin, fmt);
    if (s == 0.0f) return 1;
    *scale = s;
    return 0;
}

/*
 * Online scale of one group ("FP8 training: what it is and how it works",
 * Trade-offs: amax computed online for each 1x128 activation tile and each
 * 128x128 weight block):  s_g = float32(fmt_max / amax_g), no margin.  An
 * all-zero group gets s_g = 1; a quotient that overflows float32 is clamped
 * to FLT_MAX.
 */
float oref_group_scale(float amax_g, int fmt)
{
    if (!(amax_g > 0.0f)) return 1.0f;
    float s = div_f32((float)fmt_of(fmt).max_value, amax_g);
    if (s > FLT_MAX) s = FLT_MAX;
    return s;
}

/* ------------------------------------------------------------------------ */
/* Fused activation + quantize                                               */
/* ------------------------------------------------------------------------ */
/*
 * One element of the fused step ("Paradigma Details FP8 ...", second
 * paragraph): a = act(h); abf = BF16(a) (the copy kept for backward);
 * v = float32(abf * s); q = FP8(v).
 */
static void quant_one(uint16_t h, int act, int fmt, float s,
                      uint16_t* abf_out, float* v_out, uint8_t* q_out)
{
    float a = oref_act(oref_bf16_to_f32(h), act);
    uint16_t abf = oref_f32_to_bf16(a);
    float v = mul_f32(oref_bf16_to_f32(abf), s);
    *abf_out = abf;
    *v_out = v;
    *q_out = oref_fp8_encode(v, fmt);
}

/*
 * Per-tensor mode.  For the row-major [M,K] BF16 tensor h, with one scale:
 *   act_out[i,k] = BF16(act(h[i,k]))          (NULL: not written)
 *   q_out[i,k]   = FP8(float32(act_out * scale))
 *   q_t_out[k,i] = q_out[i,k]                 (transposed copy, [K,M])
 *   *amax_out    = max |act_out|
 *   *sat_out     = #{ |float32(act_out * scale)| > fmt_max }
 * Rows are independent; per-row maxima and counts are reduced serially.
 */
void oref_quant(const uint16_t* h, int64_t M, int64_t K, int act, int fmt, float scale,
                uint16_t* act_out, uint8_t* q_out, uint8_t* q_t_out,
                float* amax_out, uint64_t* sat_out, int nthreads)
{
    double fmax = fmt_of(fmt).max_value;
    uint32_t* row_amax = (uint32_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint32_t));
    uint64_t* row_sat = (uint64_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint64_t));
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t k = 0; k < K; ++k) {
            uint16_t abf; float v; uint8_t q;
            quant_one(h[i * K + k], act, fmt, scale, &abf, &v, &q);
            if (act_out) act_out[i * K + k] = abf;
            if (q_out) q_out[i * K + k] = q;
            if (q_t_out) q_t_out[k * M + i] = q;
            if (mag_key(oref_bf16_to_f32(abf)) > row_amax[i]) row_amax[i] = mag_key(oref_bf16_to_f32(abf));
            if (fabs((double)v) > fmax) row_sat[i] += 1;
        }
    }
    uint32_t am = 0;
    uint64_t sat = 0;
    for (int64_t i = 0; i < M; ++i) {
        if (row_amax[i] > am) am = row_amax[i];
        sat += row_sat[i];
    }
    if (amax_out) *amax_out = f32_from_bits(am);
    if (sat_out) *sat_out = sat;
    free(row_amax);
    free(row_sat);
}

/*
 * Group mode.  The [M,K] tensor is cut into blocks of group_rows rows x 128
 * columns (group_rows = 1: the 1x128 activation tiles; 128: the 128x128 weight
 * blocks).  K must be a multiple of 128; a last block of rows may be short.
 * For block (r, c):
 *   amax_g = max |BF16(act(h))| over the block
 *   s_g    = oref_group_scale(amax_g)            -> scales[r * (K/128) + c]
 *   q      = FP8(float32(BF16(act(h)) * s_g))
 * act_out, q_out, q_t_out, amax_out and sat_out are as in per-tensor mode
 * (amax over the whole tensor, sat against each element's own group scale).
 */
void oref_quant_group(const uint16_t* h, int64_t M, int64_t K, int act, int fmt, int group_rows,
                      uint16_t* act_out, uint8_t* q_out, uint8_t* q_t_out, float* scales,
                      float* amax_out, uint64_t* sat_out, int nthreads)
{
    double fmax = fmt_of(fmt).max_value;
    int64_t kg = K / OREF_GROUP;
    int64_t nbr = (M + group_rows - 1) / group_rows;
    uint32_t* blk_amax = (uint32_t*)calloc((size_t)(nbr * kg > 0 ? nbr * kg : 1), sizeof(uint32_t));
    uint32_t* row_amax = (uint32_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint32_t));
    uint64_t* row_sat = (uint64_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint64_t));
    (void)nthreads;
    /* pass 1: block maxima of the BF16 activation */
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            float a = oref_act(oref_bf16_to_f32(h[i * K + k]), act);
            uint32_t m = mag_key(oref_bf16_to_f32(oref_f32_to_bf16(a)));
            int64_t b = (i / group_rows) * kg + k / OREF_GROUP;
            if (m > blk_amax[b]) blk_amax[b] = m;
        }
    for (int64_t b = 0; b < nbr * kg; ++b)
        if (scales) scales[b] = oref_group_scale(f32_from_bits(blk_amax[b]), fmt);
    /* pass 2: quantize each element with its block's scale */
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t k = 0; k < K; ++k) {
            float s = oref_group_scale(f32_from_bits(blk_amax[(i / group_rows) * kg + k / OREF_GROUP]), fmt);
            uint16_t abf; float v; uint8_t q;
            quant_one(h[i * K + k], act, fmt, s, &abf, &v, &q);
            if (act_out) act_out[i * K + k] = abf;
            if (q_out) q_out[i * K + k] = q;
            if (q_t_out) q_t_out[k * M + i] = q;
            if (mag_key(oref_bf16_to_f32(abf)) > row_amax[i]) row_amax[i] = mag_key(oref_bf16_to_f32(abf));
            if (fabs((double)v) > fmax) row_sat[i] += 1;
        }
    }
    uint32_t am = 0;
    uint64_t sat = 0;
    for (int64_t i = 0; i < M; ++i) {
        if (row_amax[i] > am) am = row_amax[i];
        sat += row_sat[i];
    }
    if (amax_out) *amax_out = f32_from_bits(am);
    if (sat_out) *sat_out = sat;
    free(blk_amax);
    free(row_amax);
    free(row_sat);
}

/* ------------------------------------------------------------------------ */
/* Microscaling (MX): 32-value blocks with power-of-two scales                */
/* ------------------------------------------------------------------------ */
/*
 * "FP8 training: what it is and how it works", Trade-offs and edge cases: the
 * microscaling FP8 recipe gives every block of 32 adjacent values its own
 * scale, and the scales are powers of two.  The pages do not say which power
 * of two; the reading taken here is Step 2's scale (format max / amax) rounded
 * down to a power of two, so that no value of the block saturates:
 *   s_b = 2^e with e the largest integer such that amax_b * 2^e <= fmt_max,
 *   clamped to [-127, 127] (the range of an 8-bit power-of-two exponent);
 *   an all-zero block gets s_b = 1.
 * The comparison amax_b * 2^e <= fmt_max is exact (scaling by a power of two
 * is exact in double), so e is found without any rounded logarithm.
 */
float oref_mx_scale(float amax_b, int fmt)
{
    if (!(amax_b > 0.0f)) return 1.0f;
    double fmax = fmt_of(fmt).max_value;
    int e = 0;
    (void)frexp(fmax / (double)amax_b, &e); /* a first guess near log2 */
    while (ldexp((double)amax_b, e) > fmax) --e;
    while (ldexp((double)amax_b, e + 1) <= fmax) ++e;
    if (e > 127) e = 127;
    if (e < -127) e = -127;
    return (float)ldexp(1.0, e);
}

/*
 * MX quantize of the row-major [M,K] BF16 tensor h (K a multiple of 32): for
 * the 32-value block b of row i (columns 32b .. 32b + 31),
 *   amax_b = max |BF16(act(h))| over the block
 *   s_b    = oref_mx_scale(amax_b)         -> scales[i * (K/32) + b]
 *   e8m0   = 127 - log2(s_b)               -> exps[i * (K/32) + b]: the biased
 *            exponent byte of the dequantisation factor 1 / s_b
 *   q      = FP8(float32(BF16(act(h)) * s_b))
 * act_out, q_out, amax_out and sat_out as in per-tensor mode (sat against
 * each element's own block scale; 0 for finite inputs by the choice of s_b).
 */
void oref_quant_mx(const uint16_t* h, int64_t M, int64_t K, int act, int fmt,
                   uint16_t* act_out, uint8_t* q_out, float* scales, uint8_t* exps,
                   float* amax_out, uint64_t* sat_out, int nthreads)
{
    const int64_t B = 32, nb = K / B;
    double fmax = fmt_of(fmt).max_value;
    uint32_t* row_amax = (uint32_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint32_t));
    uint64_t* row_sat = (uint64_t*)calloc((size_t)(M > 0 ? M : 1), sizeof(uint64_t));
    (void)nthreads;
    /* rows are independent: they are split over host threads, each row's
       maximum and count kept apart and combined below */
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t b = 0; b < nb; ++b) {
            uint32_t m = 0;
            for (int64_t k = b * B; k < (b + 1) * B; ++k) {
                float a = oref_act(oref_bf16_to_f32(h[i * K + k]), act);
                uint32_t mk = mag_key(oref_bf16_to_f32(oref_f32_to_bf16(a)));
                if (mk > m) m = mk;
            }
            float s = oref_mx_scale(f32_from_bits(m), fmt);
            int e = 0;
            (void)frexp((double)s, &e); /* s = 2^(e - 1) */
            if (scales) scales[i * nb + b] = s;
            if (exps) exps[i * nb + b] = (uint8_t)(127 - (e - 1));
            if (m > row_amax[i]) row_amax[i] = m;
            for (int64_t k = b * B; k < (b + 1) * B; ++k) {
                uint16_t abf; float v; uint8_t q;
                quant_one(h[i * K + k], act, fmt, s, &abf, &v, &q);
                if (act_out) act_out[i * K + k] = abf;
                if (q_out) q_out[i * K + k] = q;
                if (fabs((double)v) > fmax) row_sat[i] += 1;
            }
        }
    }
    uint32_t am = 0;
    uint64_t sat = 0;
    for (int64_t i = 0; i < M; ++i) {
        if (row_amax[i] > am) am = row_amax[i];
        sat += row_sat[i];
    }
    if (amax_out) *amax_out = f32_from_bits(am);
    if (sat_out) *sat_out = sat;
    free(row_amax);
    free(row_sat);
}

/* amax only: max |BF16(act(h))| over the tensor (the calibration pass). */
float oref_amax(const uint16_t* h, int64_t n, int act)
{
    uint32_t am = 0;
    for (int64_t i = 0; i < n; ++i) {
        float a = oref_act(oref_bf16_to_f32(h[i]), act);
        uint32_t m = mag_key(oref_bf16_to_f32(oref_f32_to_bf16(a)));
        if (m > am) am = m;
    }
    return f32_from_bits(am);
}

/* ------------------------------------------------------------------------ */
/* GEMMs over the dequantised FP8 values, in double                          */
/* ------------------------------------------------------------------------ */
/*
 * Forward ("FP8 Training & Inference", FP8 Training Recipe: Y = X x W, both
 * E4M3; Per-Tensor Scaling: the scales are factored out of the matmul and the
 * output is rescaled; "FP8 training: what it is and how it works", Step 3:
 * FP8 inputs, a wider running sum):
 *   Y[i,j] = sum_k dec(X[i,k]) * dec(W[k,j]) / (s_x * s_w)
 * X is [M,K] row-major, W is [K,N] row-major.  Group mode (group != 0):
 * s_x is [M, K/128] (one scale per 1x128 tile of X) and s_w is
 * [K/128, ceil(N/128)] (one per 128x128 block of W), and each 128-long slice
 * of the sum is divided by its own pair of scales.  S[i,j] is the same sum of
 * |terms|, the scale of the rounding error.  Only the output rows listed in
 * rows[0..nrows-1] are computed; Y and S are [nrows, N].
 */
void oref_gemm_fwd(const uint8_t* X, int fmt_x, const uint8_t* W, int fmt_w,
                   int64_t M, int64_t N, int64_t K,
                   const float* s_x, const float* s_w, int group,
                   const int64_t* rows, int64_t nrows, double* Y, double* S, int nthreads)
{
    double dx[256], dw[256];
    for (int c = 0; c < 256; ++c) {
        dx[c] = oref_fp8_decode((uint8_t)c, fmt_x);
        dw[c] = oref_fp8_decode((uint8_t)c, fmt_w);
    }
    int64_t kg = K / OREF_GROUP;
    int64_t ng = (N + OREF_GROUP - 1) / OREF_GROUP;
    (void)M; (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        for (int64_t j = 0; j < N; ++j) {
            double y = 0.0, s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = dx[X[i * K + k]] * dw[W[k * N + j]];
                double d = group ? (double)s_x[i * kg + k / OREF_GROUP] *
                                   (double)s_w[(k / OREF_GROUP) * ng + j / OREF_GROUP]
                                 : (double)s_x[0] * (double)s_w[0];
                y += t / d;
                s += fabs(t) / d;
            }
            Y[r * N + j] = y;
            S[r * N + j] = s;
        }
    }
}

/*
 * MX forward: the same sum with one scale per 32-value block on each side,
 *   Y[i,j] = sum_k dec(X[i,k]) * dec(W[k,j]) / (s_x[i, k/32] * s_w[j, k/32])
 * X [M,K] and W [K,N] row-major; s_x is [M, K/32] (the blocks of X's rows),
 * s_w is [N, K/32] (the blocks of W's columns, i.e. of the rows of W^T, the
 * contraction-major operand).  S is the sum of |terms|.  Rows as above.
 */
void oref_gemm_mx(const uint8_t* X, int fmt_x, const uint8_t* W, int fmt_w,
                  int64_t M, int64_t N, int64_t K, const float* s_x, const float* s_w,
                  const int64_t* rows, int64_t nrows, double* Y, double* S, int nthreads)
{
    double dx[256], dw[256];
    for (int c = 0; c < 256; ++c) {
        dx[c] = oref_fp8_decode((uint8_t)c, fmt_x);
        dw[c] = oref_fp8_decode((uint8_t)c, fmt_w);
    }
    const int64_t nb = K / 32;
    (void)M; (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        for (int64_t j = 0; j < N; ++j) {
            double y = 0.0, s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = dx[X[i * K + k]] * dw[W[k * N + j]];
                double d = (double)s_x[i * nb + k / 32] * (double)s_w[j * nb + k / 32];
                y += t / d;
                s += fabs(t) / d;
            }
            Y[r * N + j] = y;
            S[r * N + j] = s;
        }
    }
}

/*
 * Activation gradient ("FP8 Training & Inference", FP8 Training Recipe:
 * dX = dY x W^T, dY in E5M2, W in E4M3):
 *   dX[i,k] = sum_n dec(dY[i,n]) * dec(W[k,n]) / (s_dy * s_w)
 * dY is [M,N] row-major, W is [K,N] row-major (the same W as the forward).
 * Only the rows listed are computed; dX and S are [nrows, K].
 */
void oref_gemm_dgrad(const uint8_t* dY, int fmt_dy, const uint8_t* W, int fmt_w,
                     int64_t M, int64_t N, int64_t K, float s_dy, float s_w,
                     const int64_t* rows, int64_t nrows, double* dX, double* S, int nthreads)
{
    double dd[256], dw[256];
    for (int c = 0; c < 256; ++c) {
        dd[c] = oref_fp8_decode((uint8_t)c, fmt_dy);
        dw[c] = oref_fp8_decode((uint8_t)c, fmt_w);
    }
    double denom = (double)s_dy * (double)s_w;
    (void)M; (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        for (int64_t k = 0; k < K; ++k) {
            double y = 0.0, s = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double t = dd[dY[i * N + n]] * dw[W[k * N + n]];
                y += t;
                s += fabs(t);
            }
            dX[r * K + k] = y / denom;
            S[r * K + k] = s / denom;
        }
    }
}

int oref_openmp_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
