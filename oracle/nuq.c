/*
 * CPU oracle for the non-uniform (Lloyd-Max) KV-cache quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no SIMD intrinsics; every fp32
 * operation is one separately rounded IEEE-754 binary32 operation.
 *
 * Source: "KVQuant-NUQ" (VeloxQuant-MLX docs), How it works:
 *  - Non-uniform levels (Lloyd-Max): 2^bits levels per group, seeded at evenly
 *    spaced quantiles of the data, then assign/update sweeps (each value to its
 *    nearest level, each level to the mean of its values); distortion does not
 *    increase across sweeps.  Quantize = index of the nearest level,
 *    dequantize = table lookup.
 *  - Dense-and-Sparse outlier isolation: before the fit, the top
 *    outlier_fraction of a vector's elements by magnitude go to an fp16 side
 *    channel and are left out of the fit; selection is by rank, exactly k per
 *    vector even when magnitudes tie.
 *  - Quantization axes: keys per channel (sample axis = tokens), values per
 *    token (sample axis = channels).
 *  - Configuration reference, kvquant_group_size: the fit of a value token
 *    runs per group of g consecutive channels, each group with its own table
 *    (or_nuq_vector_grouped); the token's outliers are still chosen over the
 *    whole token.
 * Readings where the page is silent (all stated with the tests):
 *  - k = floor(f * n + 0.5); ties in |x| go to the lower index.
 *  - Quantile init: level i = sorted[floor((2i+1) * n / (2L))] of the n fit values
 *    (a -0 among them counts as +0, so equal values have one bit pattern).
 *  - Assignment ties go to the lower level; an empty level keeps its value.
 *  - A level's new value is (sum of its values) / count in fp32, the sum taken
 *    in the canonical order R32 over the vector's positions: lane l = p mod 32
 *    adds its positions in increasing order from 0.0f, then for off = 16, 8, 4,
 *    2, 1 every lane adds the lane l xor off (a butterfly; all lanes end equal).
 *  - The table is stored as fp16 (round to nearest even) and the final codes
 *    are the nearest fp16 levels.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

uint16_t or_f32_to_f16(float x);
float or_f16_to_f32(uint16_t h);

/* Rank-based top-k by magnitude: flag[i] = 1 for exactly k elements, the k
 * largest |x|, ties to the lower index.  k is clamped to [0, n]. */
void or_topk_abs(const float *x, int n, int k, uint8_t *flag) {
    memset(flag, 0, (size_t)n);
    if (k > n) k = n;
    for (int r = 0; r < k; r++) {
        int best = -1;
        float bv = 0.0f;
        for (int i = 0; i < n; i++) {
            if (flag[i]) continue;
            const float a = fabsf(x[i]);
            if (best < 0 || a > bv) {  /* strict: an equal magnitude keeps the lower index */
                best = i;
                bv = a;
            }
        }
        flag[best] = 1;
    }
}

/* Outlier count for a vector of n elements at fraction f. */
int or_outlier_count(float f, int n) {
    const int k = (int)floor((double)f * (double)n + 0.5);
    return k < 0 ? 0 : (k > n ? n : k);
}

/* R32 sum of x[p] over the positions p < n with take[p] != 0. */
static float r32_sum(const float *x, const uint8_t *take, int n) {
    float v[32];
    for (int l = 0; l < 32; l++) {
        float acc = 0.0f;
        for (int p = l; p < n; p += 32)
            if (take[p]) acc = acc + x[p];
        v[l] = acc;
    }
    for (int off = 16; off >= 1; off >>= 1) {
        float w[32];
        for (int l = 0; l < 32; l++) w[l] = v[l] + v[l ^ off];
        memcpy(v, w, sizeof v);
    }
    return v[0];
}

/* exported for the tests: R32 sum of the n values x[0..n) */
float or_r32_sum(const float *x, int n) {
    uint8_t *take = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    memset(take, 1, (size_t)(n > 0 ? n : 1));
    const float s = r32_sum(x, take, n);
    free(take);
    return s;
}

static int cmp_float(const void *a, const void *b) {
    const float x = *(const float *)a, y = *(const float *)b;
    return (x > y) - (x < y);
}

/* Nearest of the L levels lev (fp32) to x: argmin |x - lev[i]|, ties to the lower i. */
static int nearest(float x, const float *lev, int L) {
    int best = 0;
    float bd = fabsf(x - lev[0]);
    for (int i = 1; i < L; i++) {
        const float dd = fabsf(x - lev[i]);
        if (dd < bd) {
            bd = dd;
            best = i;
        }
    }
    return best;
}

/*
 * Lloyd-Max fit of L levels to the positions p < n of x with excl[p] == 0
 * (excl may be NULL).  `iters` assign/update sweeps.  lev32[L] receives the
 * fp32 levels, lut16[L] (may be NULL) their fp16 bits.  Returns the number of
 * fit values.  With no fit value at all the levels are all 0.
 */
int or_nuq_fit(const float *x, const uint8_t *excl, int n, int L, int iters, float *lev32, uint16_t *lut16) {
    float *fit = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    uint8_t *take = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    uint8_t *asg = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    int nf = 0;
    for (int p = 0; p < n; p++)
        if (!excl || !excl[p]) fit[nf++] = x[p] + 0.0f;  /* -0 -> +0: equal values sort to equal bits */
    if (nf == 0) {
        for (int i = 0; i < L; i++) lev32[i] = 0.0f;
    } else {
        qsort(fit, (size_t)nf, sizeof(float), cmp_float);
        for (int i = 0; i < L; i++) lev32[i] = fit[(long long)(2 * i + 1) * nf / (2 * L)];
        for (int it = 0; it < iters; it++) {
            for (int p = 0; p < n; p++) asg[p] = (!excl || !excl[p]) ? (uint8_t)nearest(x[p], lev32, L) : 0xff;
            for (int i = 0; i < L; i++) {
                int cnt = 0;
                for (int p = 0; p < n; p++) {
                    take[p] = asg[p] == i;
                    cnt += take[p];
                }
                if (cnt > 0) lev32[i] = r32_sum(x, take, n) / (float)cnt;
            }
        }
    }
    if (lut16)
        for (int i = 0; i < L; i++) lut16[i] = or_f32_to_f16(lev32[i]);
    free(fit);
    free(take);
    free(asg);
    return nf;
}

/* Codes of x[0..n) against an fp16 table: nearest level, ties to the lower index. */
void or_nuq_assign(const float *x, int n, const uint16_t *lut16, int L, uint8_t *codes) {
    float lev[16];
    for (int i = 0; i < L; i++) lev[i] = or_f16_to_f32(lut16[i]);
    for (int p = 0; p < n; p++) codes[p] = (uint8_t)nearest(x[p], lev, L);
}

/*
 * One vector end to end: k = outlier_count(f, n) rank outliers (flag[] out),
 * Lloyd fit of the rest, fp16 table lut16[L], codes[n] against it.  Returns k.
 */
int or_nuq_vector(const float *x, int n, int bits, int iters, float f, uint8_t *flag, uint16_t *lut16,
                  uint8_t *codes) {
    const int L = 1 << bits;
    const int k = or_outlier_count(f, n);
    or_topk_abs(x, n, k, flag);
    float lev[16];
    or_nuq_fit(x, flag, n, L, iters, lev, lut16);
    or_nuq_assign(x, n, lut16, L, codes);
    return k;
}

/*
 * A vector whose fit runs per group of g consecutive elements: the k =
 * outlier_count(f, n) rank outliers are chosen over the whole vector first
 * (Dense-and-Sparse isolation selects per channel / per token), then each
 * group's remaining values get their own Lloyd fit (positions 0 .. g-1 of the
 * group in the R32 order) and its elements are coded against the group's fp16
 * table.  lut16 receives the n / g tables of L entries in group order.  g must
 * divide n; with g == n this is or_nuq_vector.  Returns k.
 */
int or_nuq_vector_grouped(const float *x, int n, int g, int bits, int iters, float f, uint8_t *flag,
                          uint16_t *lut16, uint8_t *codes) {
    const int L = 1 << bits;
    const int k = or_outlier_count(f, n);
    or_topk_abs(x, n, k, flag);
    float lev[16];
    for (int s = 0; s + g <= n; s += g) {
        or_nuq_fit(x + s, flag + s, g, L, iters, lev, lut16 + (s / g) * L);
        or_nuq_assign(x + s, g, lut16 + (s / g) * L, L, codes + s);
    }
    return k;
}
