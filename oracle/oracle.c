/*
 * oracle.c -- plain, slow CPU oracle for the quantized-weight matvec path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * Arithmetic is float64 unless the page being followed fixes float32
 * staging (the CQ activation preparation and dense row gather, whose
 * reference implementation stores every butterfly result in a
 * Float32Array).  Build with -O2 -ffp-contract=off and no fast-math so
 * that every float expression below is one IEEE operation, rounded to
 * nearest-even, on every host architecture.
 *
 * Citations name the page and its section:
 *   [needle-2] "Inference engine, part 2: kernels and token step"
 *              (needle.js tutorial), sections 1-3, "Row gather" and 8.
 *   [needle-1] "Inference engine, part 1: loader and tokenizer"
 *              (needle.js tutorial), sections 3-4.
 *   [ds4f-6]   "attention + tokenizer + sampling: the path to real text
 *              (milestone 6)" (ds4f-disk issue #6), work item 1, step 1
 *              and step 4.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Scalar decodes                                                            */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 -> value, [needle-1] section 3 "Decode FP16 control
 * tensors".  Written from the format's definition as a value (sign,
 * 5-bit biased exponent, 10-bit fraction): exponent 0 is subnormal
 * (fraction * 2^-24), exponent 31 is inf (fraction 0) or NaN. */
ORC_API float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return (float)(sign ? -v : v);
}

/* F8 E4M3 -> value, [ds4f-6] work item 1 and step 1 ("E4M3 LUT decode (e=0
 * subnormal, e=15 clamp to 448)").  Byte = s eeee mmm.  e=0: m * 2^-9;
 * otherwise (8+m) * 2^(e-10).  The clamp is read as saturation at 448: it
 * only changes the codes 0x7F / 0xFF (which would be 480) to +/-448. */
ORC_API float orc_e4m3_to_f32(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    if (v > 448.0)
        v = 448.0;
    return (float)(sign ? -v : v);
}

/* E8M0 block scale -> value: 2^(e-127).  The pages give the formula and no
 * exception; code 255 is read as NaN (the OCP microscaling convention for
 * this format), every other code is exact in float32 (e=0 is the
 * subnormal 2^-127). */
ORC_API float orc_e8m0_to_f32(uint8_t e)
{
    if (e == 255)
        return NAN;
    return (float)ldexp(1.0, (int)e - 127);
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard transform, [needle-2] section 1.                           */
/* Unnormalised, in place, strides 1, 2, 4, ... in increasing order; at each */
/* stride h the pair (i, i+h) with bit h clear in i becomes (a+b, a-b).      */
/* ------------------------------------------------------------------------ */

ORC_API void orc_fwht_f64(double *v, int64_t n)
{
    for (int64_t h = 1; h < n; h <<= 1)
        for (int64_t i = 0; i < n; i++)
            if ((i & h) == 0) {
                double a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
}

/* Same transform with every intermediate stored as float32, as the page's
 * implementation does (its buffer is a Float32Array). */
ORC_API void orc_fwht_f32(float *v, int64_t n)
{
    for (int64_t h = 1; h < n; h <<= 1)
        for (int64_t i = 0; i < n; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
}

/* ------------------------------------------------------------------------ */
/* CQ matrix and packed indices, [needle-1] section 4 and [needle-2] 3.      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t output, input, input_padded, group;
    int32_t bits, pad_;
    int64_t row_bytes;
    const uint8_t *packed;   /* [output, row_bytes]                      */
    const uint16_t *norms;   /* [output, input_padded / group] binary16  */
    const float *codebook;   /* [2^bits]                                 */
} orc_cq;

/* Index of column k in row r: bits [k*bits, k*bits+bits) of the row's
 * little-endian bit stream, read one bit at a time.  With 2 bits this is
 * the page's "(byte >> (crumb*2)) & 3" with the low crumb first. */
ORC_API int32_t orc_cq_index(const uint8_t *packed, int64_t row_bytes, int32_t bits,
                             int64_t r, int64_t k)
{
    const uint8_t *row = packed + r * row_bytes;
    int32_t idx = 0;
    for (int32_t i = 0; i < bits; i++) {
        int64_t t = k * bits + i;
        int bit = (row[t / 8] >> (t % 8)) & 1;
        idx |= bit << i;
    }
    return idx;
}

static double inv_sqrt_group(int64_t group)
{
    return 1.0 / sqrt((double)group);
}

/* prepare(), [needle-2] section 2: zero-pad x to input_padded, then per
 * group the unnormalised FWHT followed by multiplication by 1/sqrt(group).
 * mode 0: the page's exact float32 staging: butterflies in float32 and the
 *         scale applied as a float64 product rounded to float32.
 * mode 1: float64 throughout (used for tolerance-based checks).
 * x is [batch, input]; out32 / out64 are [batch, input_padded]. */
ORC_API int orc_cq_prepare(const float *x, int64_t batch, int64_t input,
                           int64_t input_padded, int64_t group, int mode,
                           float *out32, double *out64)
{
    double s = inv_sqrt_group(group);
    for (int64_t v = 0; v < batch; v++) {
        const float *xv = x + v * input;
        if (mode == 0) {
            float *o = out32 + v * input_padded;
            for (int64_t k = 0; k < input_padded; k++)
                o[k] = (k < input) ? xv[k] : 0.0f;
            for (int64_t g0 = 0; g0 < input_padded; g0 += group) {
                orc_fwht_f32(o + g0, group);
                for (int64_t k = 0; k < group; k++)
                    o[g0 + k] = (float)((double)o[g0 + k] * s);
            }
        } else {
            double *o = out64 + v * input_padded;
            for (int64_t k = 0; k < input_padded; k++)
                o[k] = (k < input) ? (double)xv[k] : 0.0;
            for (int64_t g0 = 0; g0 < input_padded; g0 += group) {
                orc_fwht_f64(o + g0, group);
                for (int64_t k = 0; k < group; k++)
                    o[g0 + k] *= s;
            }
        }
    }
    return 0;
}

/* cqMatvec, [needle-2] section 3:
 *   y[v,r] = sum_g norm[r,g] * sum_{k in g} codebook[index(r,k)] * p[v,k]
 * in float64 for rows [r0, r1).  mag[v,r] receives the magnitude sum
 * sum_g |norm| * sum_k |codebook * p| of exactly the terms added.
 * prepared is [batch, input_padded] float64, y and mag are [batch, output]. */
ORC_API int orc_cq_matvec(const orc_cq *m, const double *prepared, int64_t batch,
                          double *y, double *mag, int64_t r0, int64_t r1)
{
    int64_t ngroups = m->input_padded / m->group;
    for (int64_t r = r0; r < r1; r++)
        for (int64_t v = 0; v < batch; v++) {
            const double *p = prepared + v * m->input_padded;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t g = 0; g < ngroups; g++) {
                double n = orc_f16_to_f32(m->norms[r * ngroups + g]);
                double part = 0.0, abs_part = 0.0;
                for (int64_t k = g * m->group; k < (g + 1) * m->group; k++) {
                    double level = m->codebook[orc_cq_index(m->packed, m->row_bytes, m->bits, r, k)];
                    part += level * p[k];
                    abs_part += fabs(level * p[k]);
                }
                sum += n * part;
                abs_sum += fabs(n) * abs_part;
            }
            y[v * m->output + r] = sum;
            if (mag)
                mag[v * m->output + r] = abs_sum;
        }
    return 0;
}

/* dequantizeRow, [needle-2] "Row gather": per group, each level times the
 * group's norm (one float32 product), then the normalised FWHT (butterflies
 * in float32, then 1/sqrt(group) as in prepare), keeping only the first
 * `input` columns.  rows holds n row ids; out is [n, input].  A row id
 * outside [0, output) yields a row of zeros and a return value of 1. */
ORC_API int orc_cq_dequantize_row(const orc_cq *m, const int32_t *rows, int64_t n, float *out)
{
    int64_t P = m->input_padded, G = m->group, ngroups = P / G;
    double s = inv_sqrt_group(G);
    float *dense = (float *)malloc(sizeof(float) * (size_t)P);
    int bad = 0;
    if (!dense)
        return -1;
    for (int64_t i = 0; i < n; i++) {
        int64_t r = rows[i];
        float *o = out + i * m->input;
        if (r < 0 || r >= m->output) {
            bad = 1;
            for (int64_t k = 0; k < m->input; k++)
                o[k] = 0.0f;
            continue;
        }
        for (int64_t g = 0; g < ngroups; g++) {
            float n_g = orc_f16_to_f32(m->norms[r * ngroups + g]);
            for (int64_t k = g * G; k < (g + 1) * G; k++)
                dense[k] = m->codebook[orc_cq_index(m->packed, m->row_bytes, m->bits, r, k)] * n_g;
            orc_fwht_f32(dense + g * G, G);
            for (int64_t k = g * G; k < (g + 1) * G; k++)
                dense[k] = (float)((double)dense[k] * s);
        }
        memcpy(o, dense, sizeof(float) * (size_t)m->input);
    }
    free(dense);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* F8 E4M3 matvec with E8M0 block scales, [ds4f-6] step 1: weight [R, C],    */
/* scale [SR, SC]; element (r, c) uses scale[r*SR/R][c*SC/C] (integer floor).*/
/*   y[v,r] = sum_c e4m3(w[r,c]) * e8m0(scale[..][..]) * x[v,c]              */
/* in float64 for rows [r0, r1); mag = sum_c |w * s * x|.                    */
/* ------------------------------------------------------------------------ */

ORC_API int orc_f8_matvec(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                          int64_t SR, int64_t SC, const float *x, int64_t batch,
                          double *y, double *mag, int64_t r0, int64_t r1)
{
    for (int64_t r = r0; r < r1; r++) {
        int64_t rb = r * SR / R;
        for (int64_t v = 0; v < batch; v++) {
            const float *xv = x + v * C;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t c = 0; c < C; c++) {
                int64_t cb = c * SC / C;
                double term = (double)orc_e4m3_to_f32(w[r * C + c]) *
                              (double)orc_e8m0_to_f32(scale[rb * SC + cb]) * (double)xv[c];
                sum += term;
                abs_sum += fabs(term);
            }
            y[v * R + r] = sum;
            if (mag)
                mag[v * R + r] = abs_sum;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* I8 matvec with per-16 E8M0 group scales, [ds4f-6] step 4 ("I8 matvec     */
/* (int8 widen, per-16-group E8M0 scales)").  Read as: groups of 16          */
/* consecutive columns of a row share one scale; scale is [R, ceil(C/16)].  */
/*   y[v,r] = sum_c w[r,c] * e8m0(scale[r][c/16]) * x[v,c]                   */
/* in float64 for rows [r0, r1); mag = sum_c |w * s * x|.                    */
/* ------------------------------------------------------------------------ */

ORC_API int orc_i8_matvec(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                          const float *x, int64_t batch, double *y, double *mag, int64_t r0,
                          int64_t r1)
{
    int64_t ngroups = (C + 15) / 16;
    for (int64_t r = r0; r < r1; r++)
        for (int64_t v = 0; v < batch; v++) {
            const float *xv = x + v * C;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t c = 0; c < C; c++) {
                double term = (double)w[r * C + c] *
                              (double)orc_e8m0_to_f32(scale[r * ngroups + c / 16]) * (double)xv[c];
                sum += term;
                abs_sum += fabs(term);
            }
            y[v * R + r] = sum;
            if (mag)
                mag[v * R + r] = abs_sum;
        }
    (void)R;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* I8 matvec over int8 activations quantized per group of 32, Mnemonic "In  */
/* the browser", "Dot products and math": activations are quantized to int8 */
/* per group of 32 with one scale per group, the int8 x int8 dot products   */
/* are exact int32 sums, and only then become floats scaled by the          */
/* activation group's scale.  The weights are the I8 format above (int8     */
/* with per-16 E8M0 group scales, ds4f-6 step 4).                           */
/*                                                                           */
/* Quantizer (the page gives no rounding; the plainest reading): group j of  */
/* vector v covers columns [32 j, 32 j + 32) (the last may be shorter);      */
/* m = max |x| over it, d = m / 127 and q = rint(x / d) clamped to           */
/* [-127, 127], both divisions in float32 and rint to nearest-even.  d = 0   */
/* (all zeros, or m so small that m / 127 underflows) gives q = 0; a group   */
/* holding Inf or NaN gives d = NaN and q = 0, so every output it meets is   */
/* NaN.  x is [batch, C]; q is [batch, C]; d is [batch, ceil(C / 32)].       */
/* ------------------------------------------------------------------------ */

ORC_API int orc_i8_quantize_x(const float *x, int64_t C, int64_t batch, int8_t *q, float *d)
{
    int64_t ngroups = (C + 31) / 32;
    for (int64_t v = 0; v < batch; v++)
        for (int64_t g = 0; g < ngroups; g++) {
            int64_t c0 = g * 32, c1 = (g * 32 + 32 < C) ? g * 32 + 32 : C;
            const float *xv = x + v * C;
            float m = 0.0f;
            int finite = 1;
            for (int64_t c = c0; c < c1; c++) {
                if (!isfinite(xv[c]))
                    finite = 0;
                else if (fabsf(xv[c]) > m)
                    m = fabsf(xv[c]);
            }
            float dg = finite ? m / 127.0f : NAN;
            d[v * ngroups + g] = dg;
            for (int64_t c = c0; c < c1; c++) {
                int code = 0;
                if (finite && dg != 0.0f) {
                    float t = rintf(xv[c] / dg);
                    if (t > 127.0f)
                        t = 127.0f;
                    if (t < -127.0f)
                        t = -127.0f;
                    code = (int)t;
                }
                q[v * C + c] = (int8_t)code;
            }
        }
    return 0;
}

/*   y[v,r] = sum_c w[r,c] * e8m0(scale[r][c/16]) * q[v,c] * d[v][c/32]
 * in float64 for rows [r0, r1); mag = sum_c |w * s * q * d|. */
ORC_API int orc_i8_matvec_q8(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                             const int8_t *q, const float *d, int64_t batch, double *y,
                             double *mag, int64_t r0, int64_t r1)
{
    int64_t wgroups = (C + 15) / 16, xgroups = (C + 31) / 32;
    for (int64_t r = r0; r < r1; r++)
        for (int64_t v = 0; v < batch; v++) {
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t c = 0; c < C; c++) {
                double term = (double)w[r * C + c] *
                              (double)orc_e8m0_to_f32(scale[r * wgroups + c / 16]) *
                              (double)q[v * C + c] * (double)d[v * xgroups + c / 32];
                sum += term;
                abs_sum += fabs(term);
            }
            y[v * R + r] = sum;
            if (mag)
                mag[v * R + r] = abs_sum;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Hadamard MLP block, [needle-2] section 8, from the padded normalised     */
/* block input on:                                                            */
/*   z = pad(x, D); z *= d1; normalizedFwht(z); z = silu(d2 * z);             */
/*   normalizedFwht(z); z *= d3; out = (residual + z[:n]) - u                 */
/* normalizedFwht is the section-1 butterfly over the whole length D         */
/* followed by the product with 1/sqrt(D), as in prepare.  silu(v) =         */
/* v / (1 + e^-v).                                                           */
/* ------------------------------------------------------------------------ */

ORC_API double orc_silu_f64(double v)
{
    return v / (1.0 + exp(-v));
}

/* mode 0: the page's staging.  z is a Float32Array, so every stored value
 *         is rounded to float32: the diagonal products (float32 x float32,
 *         exact in float64, then rounded), each butterfly result, the
 *         1/sqrt(D) products, and silu, which takes the exact float64
 *         product d2 * z and is evaluated in float64.  The residual sum and
 *         the update difference are float32 array stores too.
 * mode 1: float64 throughout; out64 receives the result.
 * x, residual, u and out are [batch, n]; d1, d2, d3 are [D]; residual and
 * u may be NULL (the term is left out).  mag (may be NULL) receives, per
 * output, |d3| / sqrt(D) * sum_j |silu_j| + |residual| + |u|: the size of
 * the terms the last transform and the epilogue combine. */
ORC_API int orc_hadamard_mlp(const float *x, int64_t n, int64_t D, const float *d1,
                             const float *d2, const float *d3, const float *residual,
                             const float *u, int64_t batch, int mode, float *out32,
                             double *out64, double *mag)
{
    double s = inv_sqrt_group(D);
    float *z32 = (float *)malloc((size_t)D * sizeof(float));
    double *z64 = (double *)malloc((size_t)D * sizeof(double));
    if (!z32 || !z64) {
        free(z32);
        free(z64);
        return -1;
    }
    for (int64_t v = 0; v < batch; v++) {
        const float *xv = x + v * n;
        double silu_abs = 0.0;
        if (mode == 0) {
            for (int64_t i = 0; i < D; i++)
                z32[i] = (float)((double)(i < n ? xv[i] : 0.0f) * (double)d1[i]);
            orc_fwht_f32(z32, D);
            for (int64_t i = 0; i < D; i++)
                z32[i] = (float)((double)z32[i] * s);
            for (int64_t i = 0; i < D; i++) {
                z32[i] = (float)orc_silu_f64((double)d2[i] * (double)z32[i]);
                silu_abs += fabs((double)z32[i]);
            }
            orc_fwht_f32(z32, D);
            for (int64_t i = 0; i < D; i++)
                z32[i] = (float)((double)z32[i] * s);
            for (int64_t i = 0; i < n; i++) {
                float o = (float)((double)z32[i] * (double)d3[i]);
                if (residual)
                    o = (float)((double)residual[v * n + i] + (double)o);
                if (u)
                    o = (float)((double)o - (double)u[v * n + i]);
                out32[v * n + i] = o;
            }
        } else {
            for (int64_t i = 0; i < D; i++)
                z64[i] = (i < n ? (double)xv[i] : 0.0) * (double)d1[i];
            orc_fwht_f64(z64, D);
            for (int64_t i = 0; i < D; i++) {
                z64[i] = orc_silu_f64((double)d2[i] * (z64[i] * s));
                silu_abs += fabs(z64[i]);
            }
            orc_fwht_f64(z64, D);
            for (int64_t i = 0; i < n; i++) {
                double o = z64[i] * s * (double)d3[i];
                if (residual)
                    o = (double)residual[v * n + i] + o;
                if (u)
                    o = o - (double)u[v * n + i];
                out64[v * n + i] = o;
            }
        }
        if (mag)
            for (int64_t i = 0; i < n; i++)
                mag[v * n + i] = fabs((double)d3[i]) * s * silu_abs +
                                 (residual ? fabs((double)residual[v * n + i]) : 0.0) +
                                 (u ? fabs((double)u[v * n + i]) : 0.0);
    }
    free(z32);
    free(z64);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Greedy selection over one vector of head outputs (ds4f-6 work item 3 and  */
/* step 3: logits = head x state, then sampling; greedy = temperature 0).    */
/* Order: NaN above every number, larger above smaller, then the lower       */
/* index.  Returns -1 for n == 0.                                            */
/* ------------------------------------------------------------------------ */

ORC_API int64_t orc_argmax_f32(const float *y, int64_t n)
{
    int64_t best = -1;
    for (int64_t i = 0; i < n; i++) {
        if (best < 0) {
            best = i;
            continue;
        }
        int i_nan = isnan(y[i]), b_nan = isnan(y[best]);
        if (b_nan)
            continue; /* an earlier NaN is never beaten */
        if (i_nan || y[i] > y[best])
            best = i;
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* Top-k temperature sampling over one vector of head outputs (ds4f-6 work   */
/* item 3: the head's logits feed top-k / temperature sampling; step 3: the  */
/* sampler is a softmax driven by a seeded generator, so equal seeds give    */
/* equal tokens).  The pages name the steps and give no formulas; the        */
/* reading taken here, in their order:                                       */
/*   1. the k best logits in the greedy order above (NaN first, then the     */
/*      larger value, then the lower index), listed best first;              */
/*   2. weights w_i = exp((l_i - l_0) / T), l_0 the best, so w_0 = 1;        */
/*   3. probabilities p_i = w_i / S with S = w_0 + ... + w_{k-1};            */
/*   4. the token is entry i for the smallest i with w_0 + ... + w_i above   */
/*      u * S, u the caller's uniform draw (clamped into [0, 1], NaN read    */
/*      as 0); when rounding leaves no such i, the last i with w_i > 0.      */
/* Where the formula has no value the limit is taken: T = 0 is greedy        */
/* (entry 0, p = 1, 0, 0, ...); a NaN l_0 gives entry 0 and NaN            */
/* probabilities; l_0 = +inf shares the weight equally among the +inf        */
/* entries; l_0 = -inf (every entry -inf) gives equal weights.               */
/* Selection is k passes of the greedy scan with the chosen entries struck   */
/* out.  Returns 0, or -1 for k outside [1, n] or T not >= 0 (incl. NaN).    */
/* ------------------------------------------------------------------------ */

ORC_API int orc_topk_sample(const float *y, int64_t n, int64_t k, double T, double u,
                            int64_t *index, double *prob, int64_t *token)
{
    if (k < 1 || k > n || !(T >= 0))
        return -1;
    unsigned char *taken = (unsigned char *)calloc((size_t)n, 1);
    double *w = (double *)malloc((size_t)k * sizeof(double));
    if (!taken || !w) {
        free(taken);
        free(w);
        return -2;
    }
    for (int64_t j = 0; j < k; j++) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; i++) {
            if (taken[i])
                continue;
            if (best < 0) {
                best = i;
                continue;
            }
            if (isnan(y[best]))
                continue; /* an earlier NaN is never beaten */
            if (isnan(y[i]) || y[i] > y[best])
                best = i;
        }
        taken[best] = 1;
        index[j] = best;
    }
    free(taken);

    const double l0 = y[index[0]];
    if (T == 0 || isnan(l0)) {
        for (int64_t j = 0; j < k; j++)
            prob[j] = isnan(l0) ? NAN : (j == 0 ? 1.0 : 0.0);
        *token = index[0];
        free(w);
        return 0;
    }
    double S = 0;
    for (int64_t j = 0; j < k; j++) {
        const double l = y[index[j]];
        if (isinf(l0) && l0 > 0)
            w[j] = (l == l0) ? 1.0 : 0.0;
        else if (isinf(l0))
            w[j] = 1.0;
        else
            w[j] = exp((l - l0) / T);
        S += w[j];
    }
    for (int64_t j = 0; j < k; j++)
        prob[j] = w[j] / S;
    const double uu = (u > 0) ? (u < 1 ? u : 1) : 0;
    const double target = uu * S;
    double c = 0;
    int64_t pick = -1;
    for (int64_t j = 0; j < k && pick < 0; j++) {
        c += w[j];
        if (c > target)
            pick = j;
    }
    if (pick < 0)
        for (int64_t j = 0; j < k; j++)
            if (w[j] > 0)
                pick = j;
    *token = index[pick];
    free(w);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Row-range threading for timing the oracle on many host cores.  Each       */
/* thread runs the single-threaded function above on its own row range.      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int kind; /* 0 = cq, 1 = f8, 2 = i8, 3 = i8 over int8 activations */
    const orc_cq *m;
    const double *prepared;
    const uint8_t *w, *scale;
    const int8_t *xq;
    const float *xd;
    int64_t R, C, SR, SC;
    const float *x;
    int64_t batch;
    double *y, *mag;
    int64_t r0, r1;
} orc_job;

static void *orc_run_job(void *arg)
{
    orc_job *j = (orc_job *)arg;
    if (j->kind == 0)
        orc_cq_matvec(j->m, j->prepared, j->batch, j->y, j->mag, j->r0, j->r1);
    else if (j->kind == 1)
        orc_f8_matvec(j->w, j->R, j->C, j->scale, j->SR, j->SC, j->x, j->batch, j->y, j->mag,
                      j->r0, j->r1);
    else if (j->kind == 2)
        orc_i8_matvec((const int8_t *)j->w, j->R, j->C, j->scale, j->x, j->batch, j->y, j->mag,
                      j->r0, j->r1);
    else
        orc_i8_matvec_q8((const int8_t *)j->w, j->R, j->C, j->scale, j->xq, j->xd, j->batch,
                         j->y, j->mag, j->r0, j->r1);
    return NULL;
}

static int orc_run_threads(orc_job proto, int64_t r0, int64_t r1, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t tid[256];
    orc_job jobs[256];
    int64_t rows = r1 - r0;
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = proto;
        jobs[t].r0 = r0 + rows * t / nthreads;
        jobs[t].r1 = r0 + rows * (t + 1) / nthreads;
        if (t == nthreads - 1 || pthread_create(&tid[t], NULL, orc_run_job, &jobs[t]) != 0) {
            orc_run_job(&jobs[t]); /* last range (or a failed spawn) runs here */
        } else {
            started = t + 1;
        }
    }
    for (int t = 0; t < started; t++)
        pthread_join(tid[t], NULL);
    return 0;
}

ORC_API int orc_cq_matvec_mt(const orc_cq *m, const double *prepared, int64_t batch,
                             double *y, double *mag, int64_t r0, int64_t r1, int nthreads)
{
    orc_job j;
    memset(&j, 0, sizeof j);
    j.kind = 0;
    j.m = m;
    j.prepared = prepared;
    j.batch = batch;
    j.y = y;
    j.mag = mag;
    return orc_run_threads(j, r0, r1, nthreads);
}

ORC_API int orc_f8_matvec_mt(const uint8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                             int64_t SR, int64_t SC, const float *x, int64_t batch,
                             double *y, double *mag, int64_t r0, int64_t r1, int nthreads)
{
    orc_job j;
    memset(&j, 0, sizeof j);
    j.kind = 1;
    j.w = w;
    j.R = R;
    j.C = C;
    j.scale = scale;
    j.SR = SR;
    j.SC = SC;
    j.x = x;
    j.batch = batch;
    j.y = y;
    j.mag = mag;
    return orc_run_threads(j, r0, r1, nthreads);
}

ORC_API int orc_i8_matvec_mt(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                             const float *x, int64_t batch, double *y, double *mag, int64_t r0,
                             int64_t r1, int nthreads)
{
    orc_job j;
    memset(&j, 0, sizeof j);
    j.kind = 2;
    j.w = (const uint8_t *)w;
    j.R = R;
    j.C = C;
    j.scale = scale;
    j.x = x;
    j.batch = batch;
    j.y = y;
    j.mag = mag;
    return orc_run_threads(j, r0, r1, nthreads);
}

ORC_API int orc_i8_matvec_q8_mt(const int8_t *w, int64_t R, int64_t C, const uint8_t *scale,
                                const int8_t *q, const float *d, int64_t batch, double *y,
                                double *mag, int64_t r0, int64_t r1, int nthreads)
{
    orc_job j;
    memset(&j, 0, sizeof j);
    j.kind = 3;
    j.w = (const uint8_t *)w;
    j.R = R;
    j.C = C;
    j.scale = scale;
    j.xq = q;
    j.xd = d;
    j.batch = batch;
    j.y = y;
    j.mag = mag;
    return orc_run_threads(j, r0, r1, nthreads);
}
