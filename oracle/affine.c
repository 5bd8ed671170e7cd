/*
 * CPU oracle for the affine KV-cache quantizer and fp64 decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; it exists so that tests, the smoke check and the benchmark's
 * CPU baseline can check the CUDA library against an independent, slow and
 * plainly written statement of what it computes.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no SIMD intrinsics.  Every fp32
 * operation below is one separately rounded IEEE-754 binary32 operation
 * (round to nearest even); nothing is fused.
 *
 * Sources (page titles and sections):
 *  - "D-Quant: Driftable Entropy Coding for KV Cache Quantization",
 *    Sec. 3.1 Eq. (1) affine group quantization x^ = o + s*m;
 *    Sec. 4.2 Eq. (4) token-wise min-max grid s = (max-min)/(M-1), o = min,
 *    normalized Hadamard rotation per head, key channel-mean removal;
 *    App. A: scale and offset rounded to fp16 before the final assignment;
 *    App. A Eq. (7)-(9): the affine terms fold into q.k and P.V.
 *  - "WUSH-KV: KV Cache Quantization with Data-Adaptive Transforms",
 *    Methodology: a dense d x d key transform after RoPE with query
 *    compensation, and an OSCAR-style percentile-clipped affine quantizer;
 *    evaluation: the QuEST integer quantizer, per token, clipped from the
 *    group RMS (symmetric), with the near-optimality result stated for
 *    Gaussian tails.
 *  - "KVQuant-NUQ" (VeloxQuant-MLX docs), Attention Sink-Aware quantization:
 *    leading tokens kept exact in 16-bit and excluded from the fit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 conversions, written out by hand.          */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Shift m right by s (1..31) rounding to nearest, ties to even. */
static uint32_t shift_rne(uint32_t m, int s) {
    uint32_t q = m >> s;
    uint32_t r = m & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (r > half || (r == half && (q & 1u))) q++;
    return q;
}

/* binary32 -> binary16, round to nearest even; overflow -> inf; NaN kept quiet. */
uint16_t or_f32_to_f16(float f) {
    uint32_t x = f32_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u));
    int e = (int)(ax >> 23) - 127;            /* unbiased exponent */
    uint32_t mant = ax & 0x7fffffu;
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    if (e >= -14) {                           /* normal binary16 range */
        uint32_t q = shift_rne(mant, 13);     /* may carry into the exponent */
        uint32_t h = ((uint32_t)(e + 15) << 10) + q;
        if (h >= 0x7c00u) h = 0x7c00u;
        return (uint16_t)(sign | h);
    }
    /* subnormal binary16 (or zero): value = m * 2^(e-23), unit 2^-24 */
    if ((ax >> 23) == 0) return sign;         /* binary32 zero / subnormal -> 0 */
    int s = -e - 1;                           /* shift so that the unit is 2^-24 */
    if (s > 25) return sign;
    uint32_t m = mant | 0x800000u;
    return (uint16_t)(sign | shift_rne(m, s));
}

float or_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0x1fu) return bits_f32(sign | 0x7f800000u | (m << 13));
    if (e == 0) {
        /* subnormal: m * 2^-24, exact in binary32 */
        float v = (float)m * 5.9604644775390625e-08f;
        return sign ? -v : v;
    }
    return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

float or_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------------ */
/* Rotation                                                             */
/* ------------------------------------------------------------------ */

/* In-place fast Walsh-Hadamard transform (Sylvester order, unnormalized).
 * Stages h = 1, 2, 4, ..., d/2 in that order; each pair (i, i+h) with bit h
 * of i clear becomes (a+b, a-b).  H*x for the Sylvester matrix H (H*H^T = d*I). */
void or_fwht_f32(float *x, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i++)
            if (!(i & h)) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

void or_fwht_f64(double *x, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i++)
            if (!(i & h)) {
                double a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/* The binary32 normalization constant 1/sqrt(d) (0.125 for d = 64). */
float or_hadamard_scale(int d) { return (float)(1.0 / sqrt((double)d)); }

/* y = (H x) * fp32(1/sqrt(d)): the normalized Hadamard rotation of one head. */
void or_rotate_hadamard(const float *x, float *y, int d) {
    float c = or_hadamard_scale(d);
    for (int i = 0; i < d; i++) y[i] = x[i];
    or_fwht_f32(y, d);
    for (int i = 0; i < d; i++) y[i] = y[i] * c;
}

/* y_i = sum_j T[i][j] x_j, accumulated in j order from 0.0f (dense key transform). */
void or_rotate_dense(const float *T, const float *x, float *y, int d) {
    for (int i = 0; i < d; i++) {
        float acc = 0.0f;
        for (int j = 0; j < d; j++) {
            float p = T[(long)i * d + j] * x[j];
            acc = acc + p;
        }
        y[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* Affine fit and code assignment                                       */
/* ------------------------------------------------------------------ */

static float round_meta(float v, int meta_f16) {
    return meta_f16 ? or_f16_to_f32(or_f32_to_f16(v)) : v;
}

static int cmp_float(const void *a, const void *b) {
    float x = *(const float *)a, y = *(const float *)b;
    return (x > y) - (x < y);
}

/* Linear-interpolated order statistic: v[i] + f*(v[i+1]-v[i]) on sorted v. */
static float interp_sorted(const float *v, int n, int i, float f) {
    if (i + 1 >= n) return v[n - 1];
    float dlt = v[i + 1] - v[i];
    float p = f * dlt;
    return v[i] + p;
}

/* Position of the kappa quantile among n sorted values: index and fraction
 * ("linear" method, position kappa*(n-1) computed in double). */
void or_quantile_pos(double kappa, int n, int *idx, float *frac) {
    double pos = kappa * (double)(n - 1);
    double fl = floor(pos);
    *idx = (int)fl;
    *frac = (float)(pos - fl);
}

/* ------------------------------------------------------------------ */
/* QuEST INT grid: symmetric, clipped at alpha_b times the token's RMS   */
/* ------------------------------------------------------------------ */

/* Standard normal cdf and density. */
static double nrm_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }
static double nrm_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * 3.14159265358979323846); }

/* E[(X - c)^2 ; a < X < b] for X ~ N(0,1), from the closed forms
 * int phi = Phi, int x phi = -phi, int x^2 phi = Phi - x phi; a = -inf or
 * b = +inf allowed. */
static double cell_mse(double a, double b, double c) {
    double Pa = isinf(a) ? 0.0 : nrm_cdf(a), Pb = isinf(b) ? 1.0 : nrm_cdf(b);
    double pa = isinf(a) ? 0.0 : nrm_pdf(a), pb = isinf(b) ? 0.0 : nrm_pdf(b);
    double apa = isinf(a) ? 0.0 : a * pa, bpb = isinf(b) ? 0.0 : b * pb;
    double m0 = Pb - Pa;
    double m1 = -(pb - pa);
    double m2 = (Pb - Pa) - (bpb - apa);
    return m2 - 2.0 * c * m1 + c * c * m0;
}

/* Mean squared error on N(0,1) of the symmetric grid of L levels clipped at
 * +-alpha: step D = 2 alpha / L, level k at -alpha + (k + 1/2) D, decision
 * points halfway between levels, the outer cells open to +-infinity. */
double or_quest_mse(double alpha, int L) {
    double D = 2.0 * alpha / (double)L, sum = 0.0;
    for (int k = 0; k < L; k++) {
        double a = k == 0 ? -INFINITY : -alpha + (double)k * D;
        double b = k == L - 1 ? INFINITY : -alpha + (double)(k + 1) * D;
        sum += cell_mse(a, b, -alpha + ((double)k + 0.5) * D);
    }
    return sum;
}

/* The clip alpha that minimizes or_quest_mse for 2^bits levels
 * (golden-section search on [0.05, 8]; the error is unimodal in alpha). */
double or_quest_alpha_exact(int bits) {
    int L = 1 << bits;
    double lo = 0.05, hi = 8.0, g = (sqrt(5.0) - 1.0) / 2.0;
    double x1 = hi - g * (hi - lo), x2 = lo + g * (hi - lo);
    double f1 = or_quest_mse(x1, L), f2 = or_quest_mse(x2, L);
    for (int it = 0; it < 200; it++) {
        if (f1 < f2) { hi = x2; x2 = x1; f2 = f1; x1 = hi - g * (hi - lo); f1 = or_quest_mse(x1, L); }
        else { lo = x1; x1 = x2; f1 = f2; x2 = lo + g * (hi - lo); f2 = or_quest_mse(x2, L); }
    }
    return 0.5 * (lo + hi);
}

/* alpha_b as the quantizer uses it: the minimizer rounded to 4 decimals. */
double or_quest_alpha(int bits) { return floor(or_quest_alpha_exact(bits) * 1e4 + 0.5) / 1e4; }

/* The fp32 step factor c_b = fp32(2 alpha_b / 2^bits): s = c_b * rms. */
float or_quest_step_factor(int bits) { return (float)(2.0 * or_quest_alpha(bits) / (double)(1 << bits)); }

/* fp32 RMS of x[0..d) in a fixed summation order: for l = 0..31, p_l sums
 * the squares of channels l*V .. l*V+V-1 in channel order (V = d/32), then the
 * 32 partial sums combine pairwise, p_l = p_l + p_(l xor k) for
 * k = 16, 8, 4, 2, 1; rms = sqrt(p_0 / d).  Every step is one rounded fp32
 * operation. */
float or_quest_rms(const float *x, int d) {
    int V = d / 32;
    float p[32], q[32];
    for (int l = 0; l < 32; l++) {
        float a = x[l * V] * x[l * V];
        for (int j = 1; j < V; j++) {
            float t = x[l * V + j] * x[l * V + j];
            a = a + t;
        }
        p[l] = a;
    }
    for (int k = 16; k >= 1; k >>= 1) {
        for (int l = 0; l < 32; l++) q[l] = p[l] + p[l ^ k];
        memcpy(p, q, sizeof p);
    }
    float ms = p[0] / (float)d;
    return sqrtf(ms);
}

/*
 * Fit one token's grid and assign its codes.
 *   x[d]      : the (rotated, mean-removed) values
 *   clip      : 0 -> min/max grid (Eq. 4); else two-sided clip at the
 *               (1-clip) and clip quantiles of x, values clamped into it
 *   quest_c   : > 0 -> the QuEST grid instead: s = quest_c * RMS(x),
 *               o = -((L-1)/2) s (both rounded as meta_f16 says), a grid
 *               symmetric about 0 whose outer levels sit half a step inside
 *               +-alpha_b * RMS; values beyond fall to the outer codes
 *   meta_f16  : round s and o to binary16 before assigning codes (App. A)
 * Outputs codes[d] in 0..2^bits-1, and the stored scale/offset as floats.
 */
void or_affine_quantize(const float *x, int d, int bits, int meta_f16, double clip, float quest_c,
                        unsigned char *codes, float *s_out, float *o_out) {
    int L = 1 << bits;
    float lo, hi;
    if (quest_c > 0.0f) {
        float r = or_quest_rms(x, d);
        float s = round_meta(quest_c * r, meta_f16);
        float h = (float)(L - 1) * 0.5f;
        float o = round_meta(-(h * s), meta_f16);
        for (int j = 0; j < d; j++) {
            int m = 0;
            if (s != 0.0f) {
                float t = (x[j] - o) / s;
                if (t == t) {
                    float rr = nearbyintf(t);
                    if (rr < 0.0f) rr = 0.0f;
                    if (rr > (float)(L - 1)) rr = (float)(L - 1);
                    m = (int)rr;
                }
            }
            codes[j] = (unsigned char)m;
        }
        *s_out = s;
        *o_out = o;
        return;
    }
    if (clip > 0.0) {
        float *v = (float *)malloc(sizeof(float) * (size_t)d);
        memcpy(v, x, sizeof(float) * (size_t)d);
        qsort(v, (size_t)d, sizeof(float), cmp_float);
        int il, ih; float fl, fh;
        or_quantile_pos(1.0 - clip, d, &il, &fl);
        or_quantile_pos(clip, d, &ih, &fh);
        lo = interp_sorted(v, d, il, fl);
        hi = interp_sorted(v, d, ih, fh);
        free(v);
    } else {
        lo = x[0]; hi = x[0];
        for (int j = 1; j < d; j++) { if (x[j] < lo) lo = x[j]; if (x[j] > hi) hi = x[j]; }
    }
    float range = hi - lo;
    float s = range / (float)(L - 1);
    float o = lo;
    s = round_meta(s, meta_f16);
    o = round_meta(o, meta_f16);
    for (int j = 0; j < d; j++) {
        float xv = x[j];
        if (clip > 0.0) { if (xv < lo) xv = lo; if (xv > hi) xv = hi; }
        int m = 0;
        if (s != 0.0f) {
            float t = (xv - o) / s;
            if (t == t) {
                float r = nearbyintf(t);       /* default mode: nearest, ties to even */
                if (r < 0.0f) r = 0.0f;
                if (r > (float)(L - 1)) r = (float)(L - 1);
                m = (int)r;
            }
        }
        codes[j] = (unsigned char)m;
    }
    *s_out = s;
    *o_out = o;
}

/* x^ = fp32(o + fp32(s*m)), plus mu[j] when mu is given (keys). */
void or_affine_dequant(const unsigned char *codes, int d, float s, float o, const float *mu,
                       float *xhat) {
    for (int j = 0; j < d; j++) {
        float p = s * (float)codes[j];
        float v = o + p;
        if (mu) v = v + mu[j];
        xhat[j] = v;
    }
}

/* ------------------------------------------------------------------ */
/* Quantize one (batch, kv-head) unit of a cache                        */
/* ------------------------------------------------------------------ */

/*
 * x      : [n][d] raw fp32 values of tokens 0..n-1 of this unit
 * rot    : 0 none, 1 Hadamard, 2 dense (T given, [d][d])
 * mean   : 1 -> remove the channel mean of the rotated values, taken over the
 *          quantized tokens [mean_t0, mean_t1) summed in token order from 0.0f
 *          and divided by their count; mu_io receives it.  2 -> use mu_io as
 *          given (a mean frozen earlier).  0 -> no mean.
 * Tokens [q_t0, n) are quantized: codes[(t-q_t0)][d], s/o[(t-q_t0)].
 */
void or_quantize_unit(const float *x, int n, int d, int rot, const float *T, int mean,
                      int mean_t0, int mean_t1, float *mu_io, int bits, int meta_f16,
                      double clip, float quest_c, int q_t0, unsigned char *codes, float *s, float *o,
                      float *xhat) {
    float *y = (float *)malloc(sizeof(float) * (size_t)d);
    float *z = (float *)malloc(sizeof(float) * (size_t)d);
    if (mean == 1) {
        float *acc = (float *)calloc((size_t)d, sizeof(float));
        for (int t = mean_t0; t < mean_t1; t++) {
            const float *xt = x + (long)t * d;
            if (rot == 1) or_rotate_hadamard(xt, y, d);
            else if (rot == 2) or_rotate_dense(T, xt, y, d);
            else memcpy(y, xt, sizeof(float) * (size_t)d);
            for (int j = 0; j < d; j++) acc[j] = acc[j] + y[j];
        }
        int cnt = mean_t1 - mean_t0;
        for (int j = 0; j < d; j++) mu_io[j] = cnt > 0 ? acc[j] / (float)cnt : 0.0f;
        free(acc);
    }
    for (int t = q_t0; t < n; t++) {
        const float *xt = x + (long)t * d;
        if (rot == 1) or_rotate_hadamard(xt, y, d);
        else if (rot == 2) or_rotate_dense(T, xt, y, d);
        else memcpy(y, xt, sizeof(float) * (size_t)d);
        if (mean) for (int j = 0; j < d; j++) z[j] = y[j] - mu_io[j];
        else memcpy(z, y, sizeof(float) * (size_t)d);
        long r = t - q_t0;
        or_affine_quantize(z, d, bits, meta_f16, clip, quest_c, codes + r * d, s + r, o + r);
        if (xhat) or_affine_dequant(codes + r * d, d, s[r], o[r], mean ? mu_io : NULL, xhat + r * d);
    }
    free(y);
    free(z);
}

/* ------------------------------------------------------------------ */
/* fp64 dequantization back to the raw space, and fp64 attention        */
/* ------------------------------------------------------------------ */

/* out[t][j] = o_t + s_t*m_tj (+ mu_j), in fp64; then the inverse of the
 * normalized Hadamard rotation (itself) when rot == 1.  rot == 2 leaves the
 * keys in the transformed space (the query is compensated instead). */
void or_dequant_f64(const unsigned char *codes, const float *s, const float *o, const float *mu,
                    int n, int d, int rot, double *out) {
    double c = 1.0 / sqrt((double)d);
    for (int t = 0; t < n; t++) {
        double *ot = out + (long)t * d;
        for (int j = 0; j < d; j++) {
            double v = (double)o[t] + (double)s[t] * (double)codes[(long)t * d + j];
            if (mu) v += (double)mu[j];
            ot[j] = v;
        }
        if (rot == 1) {
            or_fwht_f64(ot, d);
            for (int j = 0; j < d; j++) ot[j] *= c;
        }
    }
}

/*
 * Decode attention of one kv head in fp64.
 *   q[G][d] (the G query heads that share this kv head), K[S][d], V[S][d]
 *   out[g][j] = sum_t softmax_t(sm_scale * q_g . K_t) * V[t][j]
 */
void or_attention_f64(const double *q, const double *K, const double *V, int G, int S, int d,
                      double sm_scale, double *out) {
    double *sc = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    for (int g = 0; g < G; g++) {
        const double *qg = q + (long)g * d;
        double mx = -INFINITY;
        for (int t = 0; t < S; t++) {
            double acc = 0.0;
            for (int j = 0; j < d; j++) acc += qg[j] * K[(long)t * d + j];
            sc[t] = sm_scale * acc;
            if (sc[t] > mx) mx = sc[t];
        }
        double den = 0.0;
        for (int t = 0; t < S; t++) { sc[t] = exp(sc[t] - mx); den += sc[t]; }
        double *og = out + (long)g * d;
        for (int j = 0; j < d; j++) og[j] = 0.0;
        for (int t = 0; t < S; t++) {
            double a = sc[t] / den;
            for (int j = 0; j < d; j++) og[j] += a * V[(long)t * d + j];
        }
    }
    free(sc);
}
