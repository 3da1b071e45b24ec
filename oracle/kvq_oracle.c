/*
 * kvq_oracle.c -- plain, slow, obviously correct CPU reference for the FP4 KV
 * cache and the decode attention that reads it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant with the CUDA
 * library; it is written from the format definitions and the method's steps.
 *
 * Sources (page title, section):
 *   "Quantising the KV cache", section "Code": the per-16-channel quantiser --
 *       scale = RNE_e4m3(amax/6) saturating, a zero scale replaced by the E4M3
 *       minimum subnormal, then each value rounded to E2M1 (RNE, saturating)
 *       after division by the scale; the quantised K and V replace the real
 *       ones between projection and an otherwise unchanged attention.
 *   "Quantising the KV cache", section "FP4 with a fine-grained scale": E2M1
 *       elements with one FP8 E4M3 scale per 16 channels.
 *   "Quantising the KV cache", section "Maths": b + s/g bits per number.
 *   "Week 6 -- FP4 KV Caches and Bounded Replay", "Overview" and "Lecture
 *       notes": the sliding-window (SWA) KV stays FP8.
 *   "Quantising the KV cache", table row "FP8 E4M3, one scale per tensor".
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - E2M1 is the OCP MX FP4 format: sign bit 3, exponent bits 2..1 (bias 1),
 *     mantissa bit 0; magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   - E4M3 is OCP FP8 E4M3FN: bias 7, no infinities, 0x7F/0xFF are NaN,
 *     max finite 448 (0x7E), min subnormal 2^-9 (0x01).
 *   - "rne" is round-to-nearest, ties to the even code (mantissa LSB 0);
 *     "saturating" clamps magnitudes above the largest finite value to it.
 *   - amax/6 and v/s are IEEE fp32 divisions (correctly rounded).
 *   - The sign bit of a value is kept even when its magnitude rounds to zero
 *     (-0.0 and small negatives encode as nibble 0x8), as IEEE rounding keeps
 *     the sign of zero.
 *   - Packing: byte j of a block holds channel 2j in its low nibble and
 *     channel 2j+1 in its high nibble.
 *   - FP8 SWA: x / s_h in fp32, RNE to E4M3 saturating; dequantised value is
 *     the fp32 product e4m3(c) * s_h.  s_h = amax/448 in fp32 (1 if amax == 0).
 *   - Attention: softmax(q.k * scale) v per query head, all positions attended,
 *     no mask, no rotary embedding; computed in fp64.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in single precision"
#endif

/* ------------------------------------------------------------------ */
/* Format definitions                                                  */
/* ------------------------------------------------------------------ */

/* Value of one E2M1 nibble (bits 3..0 = s e1 e0 m). */
double oq_e2m1_value(uint8_t nib)
{
    int s = (nib >> 3) & 1;
    int e = (nib >> 1) & 3;
    int m = nib & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Value of one E4M3FN byte (bits 7..0 = s e3 e2 e1 e0 m2 m1 m0). */
double oq_e4m3_value(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9); /* m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round a non-negative exact value q to an integer, ties to even. */
static int rne_int(double q)
{
    double f = floor(q);
    double r = q - f;
    int k = (int)f;
    if (r > 0.5)
        return k + 1;
    if (r < 0.5)
        return k;
    return (k & 1) ? k + 1 : k;
}

/* ------------------------------------------------------------------ */
/* Encoders, direct form: exponent, then the mantissa rounded (RNE).   */
/* ------------------------------------------------------------------ */

/* E2M1 magnitude code (0..7) of m >= 0, RNE, saturating. */
static uint8_t e2m1_mag_direct(double m)
{
    int e, E, k, code;
    double f, q;
    if (!(m < 6.0))
        return 7; /* saturate (and +inf) */
    if (m < 1.0) /* subnormal binade: spacing 0.5; k == 2 is 1.0 = code 2 */
        return (uint8_t)rne_int(m * 2.0);
    f = frexp(m, &e); /* m = f * 2^e, f in [0.5, 1) */
    E = e - 1;        /* m = 2^E * (2f), 2f in [1, 2); E in 0..2 */
    q = (2.0 * f - 1.0) * 2.0; /* mantissa in halves, exact */
    k = rne_int(q);
    if (k == 2) {
        E += 1;
        k = 0;
    }
    code = ((E + 1) << 1) | k;
    return (uint8_t)(code > 7 ? 7 : code);
}

/* E4M3 magnitude code (0..0x7E) of m >= 0, RNE, saturating. */
static uint8_t e4m3_mag_direct(double m)
{
    int e, E, k, code;
    double f, q;
    if (!(m < 448.0))
        return 0x7E;
    if (m < 0x1p-6) /* subnormal binade: spacing 2^-9; k == 8 is 2^-6 = 0x08 */
        return (uint8_t)rne_int(m * 512.0);
    f = frexp(m, &e);
    E = e - 1;                 /* -6 .. 8 */
    q = (2.0 * f - 1.0) * 8.0; /* mantissa in eighths, exact */
    k = rne_int(q);
    if (k == 8) {
        E += 1;
        k = 0;
    }
    code = ((E + 7) << 3) | k;
    return (uint8_t)(code > 0x7E ? 0x7E : code);
}

/* E2M1 nibble of a float: sign bit of y, magnitude RNE saturating.
 * NaN maps to 0x7 with the sign bit of the NaN (callers flag it). */
uint8_t oq_e2m1_encode(float y)
{
    uint8_t sign = signbit(y) ? 0x8 : 0x0;
    if (isnan(y))
        return sign | 0x7;
    return sign | e2m1_mag_direct(fabs((double)y));
}

/* E4M3 byte of a float: sign bit of t, magnitude RNE saturating; NaN -> 0x7F. */
uint8_t oq_e4m3_encode(float t)
{
    uint8_t sign = signbit(t) ? 0x80 : 0x00;
    if (isnan(t))
        return 0x7F;
    return sign | e4m3_mag_direct(fabs((double)t));
}

/* ------------------------------------------------------------------ */
/* Encoders, brute-force form: nearest finite candidate, ties to the   */
/* candidate whose mantissa LSB (code LSB) is 0.  Used to pin the      */
/* direct encoders.                                                    */
/* ------------------------------------------------------------------ */

uint8_t oq_e2m1_encode_brute(float y)
{
    double m = fabs((double)y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 7; c++) {
        double d = fabs(oq_e2m1_value((uint8_t)c) - m);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    if (isnan(y) || m >= 6.0)
        best = 7; /* NaN is flagged by callers; beyond the grid saturates
                     (huge m would make every distance round to the same double) */
    return (uint8_t)((signbit(y) ? 0x8 : 0) | best);
}

uint8_t oq_e4m3_encode_brute(float t)
{
    double m = fabs((double)t);
    int best = 0;
    double bestd = INFINITY;
    if (isnan(t))
        return 0x7F;
    for (int c = 0; c <= 0x7E; c++) {
        double d = fabs(oq_e4m3_value((uint8_t)c) - m);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    if (m >= 448.0)
        best = 0x7E; /* beyond the largest finite value saturates */
    return (uint8_t)((signbit(t) ? 0x80 : 0) | best);
}

void oq_e2m1_encode_array(const float *y, int64_t n, uint8_t *out, int brute)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = brute ? oq_e2m1_encode_brute(y[i]) : oq_e2m1_encode(y[i]);
}

void oq_e4m3_encode_array(const float *t, int64_t n, uint8_t *out, int brute)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = brute ? oq_e4m3_encode_brute(t[i]) : oq_e4m3_encode(t[i]);
}

/* ------------------------------------------------------------------ */
/* The block quantiser ("Quantising the KV cache", section "Code")     */
/* ------------------------------------------------------------------ */

/* Quantise one block of 16 values.  Writes 8 packed code bytes and one
 * E4M3 scale byte.  Returns 1 if the block holds a non-finite value. */
int oq_quantize_block(const float *x, uint8_t *codes, uint8_t *scale_byte)
{
    float amax = 0.0f;
    int nonfinite = 0;
    uint8_t nib[16];
    /* step 1: the block's absolute maximum (exact) */
    for (int i = 0; i < 16; i++) {
        float a = fabsf(x[i]);
        if (!isfinite(x[i]))
            nonfinite = 1;
        if (a > amax || isnan(a))
            amax = a;
    }
    /* step 2: s = RNE_e4m3(amax / 6), saturating, fp32 division */
    float t = amax / 6.0f;
    uint8_t sb = oq_e4m3_encode(t);
    /* step 3: a zero scale becomes the E4M3 minimum subnormal */
    if (oq_e4m3_value(sb) == 0.0)
        sb = 0x01;
    float s = (float)oq_e4m3_value(sb);
    /* step 4: each value divided by s (fp32), rounded to E2M1 */
    for (int i = 0; i < 16; i++) {
        float y = x[i] / s;
        nib[i] = oq_e2m1_encode(y);
    }
    /* step 5: two codes per byte, even channel in the low nibble */
    for (int j = 0; j < 8; j++)
        codes[j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    *scale_byte = sb;
    return nonfinite;
}

/* Quantise n rows of d channels (d % 16 == 0), row-major.  codes: n x d/2,
 * scales: n x d/16.  Returns the number of blocks holding a non-finite value. */
int64_t oq_quantize_rows(const float *x, int64_t n, int d, uint8_t *codes, uint8_t *scales)
{
    int64_t bad = 0;
    int nb = d / 16;
    for (int64_t r = 0; r < n; r++)
        for (int j = 0; j < nb; j++)
            bad += oq_quantize_block(x + r * d + 16 * j, codes + r * (d / 2) + 8 * j,
                                     scales + r * nb + j);
    return bad;
}

/* Dequantise n rows: value = E2M1(code) * E4M3(scale), in fp64 (exact). */
void oq_dequantize_rows(const uint8_t *codes, const uint8_t *scales, int64_t n, int d, double *out)
{
    int nb = d / 16;
    for (int64_t r = 0; r < n; r++)
        for (int c = 0; c < d; c++) {
            uint8_t byte = codes[r * (d / 2) + c / 2];
            uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            out[r * d + c] = oq_e2m1_value(nib) * oq_e4m3_value(scales[r * nb + c / 16]);
        }
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 sliding-window KV with one fp32 scale per head             */
/* ------------------------------------------------------------------ */

/* s_h = amax / 448 in fp32 over n values; 1 when amax == 0. */
float oq_fp8_head_scale(const float *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > amax || isnan(a))
            amax = a;
    }
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

/* c = RNE_e4m3(x / s) saturating, fp32 division.  Returns the number of
 * non-finite inputs. */
int64_t oq_fp8_quantize(const float *x, int64_t n, float s, uint8_t *out)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; i++) {
        float y = x[i] / s;
        if (!isfinite(x[i]))
            bad++;
        out[i] = oq_e4m3_encode(y);
    }
    return bad;
}

/* value = fp32(e4m3(c) * s), widened to fp64. */
void oq_fp8_dequantize(const uint8_t *c, int64_t n, float s, double *out)
{
    for (int64_t i = 0; i < n; i++) {
        float v = (float)oq_e4m3_value(c[i]) * s;
        out[i] = (double)v;
    }
}

/* ------------------------------------------------------------------ */
/* NVFP4: the FP4 block quantiser applied to x / S, with one fp32        */
/* second-level scale S ("KV Cache Quantisation": store the cache in FP8  */
/* or NVFP4 and handle the scales at read time).  Reading: S = amax /     */
/* (6 * 448) over a calibration tensor (1 when amax == 0), so the largest */
/* block lands on the top E4M3 scale; x / S is an fp32 division; a value  */
/* reads back as fp32(fp32(e2m1 * e4m3) * S).                             */
/* ------------------------------------------------------------------ */

float oq_nvfp4_global_scale(const float *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > amax || isnan(a))
            amax = a;
    }
    if (amax == 0.0f)
        return 1.0f;
    return amax / 2688.0f; /* 6 * 448 */
}

int64_t oq_nvfp4_quantize_rows(const float *x, int64_t n, int d, float S, uint8_t *codes, uint8_t *scales)
{
    int64_t bad = 0;
    float tmp[16];
    for (int64_t r = 0; r < n; r++)
        for (int b = 0; b < d / 16; b++) {
            for (int i = 0; i < 16; i++)
                tmp[i] = x[r * d + 16 * b + i] / S;
            bad += oq_quantize_block(tmp, codes + r * (d / 2) + 8 * b, scales + r * (d / 16) + b);
        }
    return bad;
}

void oq_nvfp4_dequantize_rows(const uint8_t *codes, const uint8_t *scales, int64_t n, int d, float S, double *out)
{
    for (int64_t r = 0; r < n; r++)
        for (int c = 0; c < d; c++) {
            uint8_t byte = codes[r * (d / 2) + c / 2];
            uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            float v = (float)(oq_e2m1_value(nib) * oq_e4m3_value(scales[r * (d / 16) + c / 16]));
            out[r * d + c] = (double)(v * S);
        }
}

/* ------------------------------------------------------------------ */
/* Bit-width sweep: symmetric INT-b with an FP16 scale per group        */
/* ("Quantising the KV cache": table rows INT8 / INT4 / INT2 per token  */
/* and "K per channel, V per token"; section "Per token or per          */
/* channel?"; section "Maths": b + s/g bits with a 16-bit scale).       */
/* ------------------------------------------------------------------ */

/* Value of an IEEE binary16 bit pattern. */
double oq_fp16_value(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double mag;
    if (e == 31)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -24); /* m/1024 * 2^-14 */
    else
        mag = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -mag : mag;
}

/* binary16 of x, round to nearest even, saturating: magnitudes that would
 * round above the largest finite value (65504) give 65504; NaN gives 0x7E00. */
uint16_t oq_fp16_encode(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double m = fabs((double)x);
    int e, k;
    if (isnan(x))
        return 0x7E00u;
    if (isinf(x)) /* saturating: above the largest finite value */
        return (uint16_t)(sign | 0x7BFFu);
    if (m == 0.0)
        return sign;
    if (m < ldexp(1.0, -14)) { /* subnormal range: multiples of 2^-24 */
        k = rne_int(ldexp(m, 24));
        return (uint16_t)(sign | (uint16_t)k); /* k == 1024 is the smallest normal */
    }
    e = (int)floor(log2(m));
    if (ldexp(1.0, e) > m) /* guard log2 rounding */
        e--;
    if (ldexp(1.0, e + 1) <= m)
        e++;
    if (e > 15)
        return (uint16_t)(sign | 0x7BFFu);
    k = rne_int(ldexp(m, 10 - e)); /* 1024 .. 2048 */
    if (k == 2048) {
        k = 1024;
        e++;
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7BFFu);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(k - 1024));
}

/* One group of n values at stride `stride`: amax over the group (exact),
 * s = fp16_RNE(amax / qmax) with qmax = 2^(bits-1) - 1 and an fp32 division,
 * a zero scale replaced by the smallest fp16 subnormal 2^-24; then each code
 * q = clamp(RNE(x / s), -qmax, qmax) with an fp32 division (NaN -> 0).
 * Writes the codes (one int8 each, at the same stride) and the scale's bit
 * pattern; returns the number of non-finite inputs. */
int64_t oq_int_quantize_group(const float *x, int64_t n, int64_t stride, int bits, int8_t *codes,
                              uint16_t *scale_bits)
{
    const int qmax = (1 << (bits - 1)) - 1;
    float amax = 0.0f;
    int64_t bad = 0;
    uint16_t sb;
    float s;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(x[i * stride]);
        if (!isfinite(x[i * stride]))
            bad++;
        if (a > amax)
            amax = a;
    }
    sb = oq_fp16_encode(amax / (float)qmax);
    if ((sb & 0x7FFFu) == 0)
        sb = 0x0001u;
    s = (float)oq_fp16_value(sb);
    for (int64_t i = 0; i < n; i++) {
        float y = x[i * stride] / s;
        int q;
        if (isnan(y))
            q = 0;
        else if (y >= (float)qmax)
            q = qmax;
        else if (y <= -(float)qmax)
            q = -qmax;
        else
            q = (y < 0.0f) ? -rne_int(-(double)y) : rne_int((double)y);
        codes[i * stride] = (int8_t)q;
    }
    *scale_bits = sb;
    return bad;
}

void oq_fp16_encode_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oq_fp16_encode(x[i]);
}

/* x: [batch][tokens][heads][d].  Per token: one group per (b, t, head), its d
 * channels; scales [batch][tokens][heads]. */
int64_t oq_int_quantize_per_token(const float *x, int64_t batch, int64_t tokens, int64_t heads, int64_t d,
                                  int bits, int8_t *codes, uint16_t *scales)
{
    int64_t bad = 0;
    for (int64_t gidx = 0; gidx < batch * tokens * heads; gidx++)
        bad += oq_int_quantize_group(x + gidx * d, d, 1, bits, codes + gidx * d, scales + gidx);
    return bad;
}

/* Per channel: one group per (b, head, channel), over the sequence's tokens;
 * scales [batch][heads][d]. */
int64_t oq_int_quantize_per_channel(const float *x, int64_t batch, int64_t tokens, int64_t heads, int64_t d,
                                    int bits, int8_t *codes, uint16_t *scales)
{
    int64_t bad = 0;
    for (int64_t b = 0; b < batch; b++)
        for (int64_t h = 0; h < heads; h++)
            for (int64_t c = 0; c < d; c++) {
                const int64_t off = (b * tokens * heads + h) * d + c;
                bad += oq_int_quantize_group(x + off, tokens, heads * d, bits, codes + off,
                                             scales + (b * heads + h) * d + c);
            }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Attention, fp64 ("an otherwise unchanged copy of the attention")    */
/* ------------------------------------------------------------------ */

/* For each of G query rows: out = sum_t softmax_t(scale * q.k_t) v_t.
 * q: G x d, k, v: T x d, out: G x d.  T == 0 gives zeros.  Also writes, per
 * query row, the max score m (in natural-log units, scale applied) and the sum
 * l = sum_t exp(score_t - m), when m_out / l_out are non-NULL. */
void oq_attend(const double *q, const double *k, const double *v, int G, int64_t T, int d,
               double scale, double *out, double *m_out, double *l_out, double *scores_tmp)
{
    for (int h = 0; h < G; h++) {
        double mx = -INFINITY, l = 0.0;
        for (int c = 0; c < d; c++)
            out[h * d + c] = 0.0;
        for (int64_t t = 0; t < T; t++) {
            double sc = 0.0;
            for (int c = 0; c < d; c++)
                sc += q[h * d + c] * k[t * d + c];
            sc *= scale;
            scores_tmp[t] = sc;
            if (sc > mx)
                mx = sc;
        }
        for (int64_t t = 0; t < T; t++) {
            double p = exp(scores_tmp[t] - mx);
            l += p;
            for (int c = 0; c < d; c++)
                out[h * d + c] += p * v[t * d + c];
        }
        if (T > 0)
            for (int c = 0; c < d; c++)
                out[h * d + c] /= l;
        if (m_out)
            m_out[h] = mx;
        if (l_out)
            l_out[h] = l;
    }
}

/* ------------------------------------------------------------------ */
/* Toy sliding-window network and its replay, fp64                     */
/* ("Week 6 -- FP4 KV Caches and Bounded Replay", Overview, Core       */
/* Concepts "Bounded replay", Lecture notes, Lab: exact replay costs   */
/* ~ L n_win; bounded replay rebuilds the SWA state from only the last */
/* n_win tokens)                                                       */
/* ------------------------------------------------------------------ */

/* The pages give no shapes; the toy is a reading: L layers, width d, one
 * attention head per layer.  Layer l maps x to x' with, for each position i,
 *   u_i  = x_i / sqrt(mean_c(x_i[c]^2) + 1e-6)         (RMS normalisation)
 *   q_i  = Wq u_i,  k_i = Wk u_i,  v_i = Wv u_i
 *   a_i  = sum_{s in win(i)} softmax_s(q_i . k_s / sqrt(d)) v_s
 *   x'_i = x_i + Wo a_i
 * with win(i) = positions max(0, i - n_win + 1) .. i of the replayed range.
 * w holds L x 4 matrices (Wq, Wk, Wv, Wo), each d x d row-major: (W u)[r] =
 * sum_c W[r*d + c] u[c].  emb: n x d, the inputs of the n replayed positions in
 * order.  Outputs: hidden (n x d), the last layer's x; states (L x 2 x n_win x
 * d), each layer's K then V rows of the last n_win positions (n >= n_win).
 * Work: x, kb, vb (n x d each), tmp (3 d + n_win). */
void oq_swa_forward(const double *w, int L, int d, const double *emb, int64_t n, int n_win, double *hidden,
                    double *states, double *x, double *kb, double *vb, double *tmp)
{
    double *u = tmp, *q = tmp + d, *a = tmp + 2 * d, *sc = tmp + 3 * d;
    const double scale = 1.0 / sqrt((double)d);
    memcpy(x, emb, (size_t)(n * d) * sizeof(double));
    for (int l = 0; l < L; l++) {
        const double *Wq = w + (size_t)(4 * l + 0) * d * d, *Wk = w + (size_t)(4 * l + 1) * d * d;
        const double *Wv = w + (size_t)(4 * l + 2) * d * d, *Wo = w + (size_t)(4 * l + 3) * d * d;
        /* keys and values of every position, from the layer's input */
        for (int64_t i = 0; i < n; i++) {
            double ms = 0.0;
            for (int c = 0; c < d; c++)
                ms += x[i * d + c] * x[i * d + c];
            const double r = 1.0 / sqrt(ms / d + 1e-6);
            for (int c = 0; c < d; c++)
                u[c] = x[i * d + c] * r;
            for (int o = 0; o < d; o++) {
                double sk = 0.0, sv = 0.0;
                for (int c = 0; c < d; c++) {
                    sk += Wk[o * d + c] * u[c];
                    sv += Wv[o * d + c] * u[c];
                }
                kb[i * d + o] = sk;
                vb[i * d + o] = sv;
            }
        }
        /* attention over each position's window, then the residual update
         * (x_i is read for q_i before it is overwritten; keys and values of
         * all positions were taken above from the layer input) */
        for (int64_t i = 0; i < n; i++) {
            double ms = 0.0;
            for (int c = 0; c < d; c++)
                ms += x[i * d + c] * x[i * d + c];
            const double r = 1.0 / sqrt(ms / d + 1e-6);
            for (int c = 0; c < d; c++)
                u[c] = x[i * d + c] * r;
            for (int o = 0; o < d; o++) {
                double s = 0.0;
                for (int c = 0; c < d; c++)
                    s += Wq[o * d + c] * u[c];
                q[o] = s;
            }
            const int64_t s0 = i - n_win + 1 > 0 ? i - n_win + 1 : 0;
            double mx = -INFINITY, den = 0.0;
            for (int64_t s = s0; s <= i; s++) {
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += q[c] * kb[s * d + c];
                sc[s - s0] = dot * scale;
                if (sc[s - s0] > mx)
                    mx = sc[s - s0];
            }
            for (int c = 0; c < d; c++)
                a[c] = 0.0;
            for (int64_t s = s0; s <= i; s++) {
                const double p = exp(sc[s - s0] - mx);
                den += p;
                for (int c = 0; c < d; c++)
                    a[c] += p * vb[s * d + c];
            }
            for (int o = 0; o < d; o++) {
                double y = 0.0;
                for (int c = 0; c < d; c++)
                    y += Wo[o * d + c] * (a[c] / den);
                x[i * d + o] += y;
            }
        }
        for (int64_t j = 0; j < n_win; j++)
            for (int c = 0; c < d; c++) {
                states[(((size_t)l * 2 + 0) * n_win + j) * d + c] = kb[(n - n_win + j) * d + c];
                states[(((size_t)l * 2 + 1) * n_win + j) * d + c] = vb[(n - n_win + j) * d + c];
            }
    }
    memcpy(hidden, x, (size_t)(n * d) * sizeof(double));
}
