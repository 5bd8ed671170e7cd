/*
 * CPU oracle for the D-Quant fixed-size entropy-coded container.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no SIMD intrinsics; every fp32
 * operation is one separately rounded IEEE-754 binary32 operation.
 *
 * Source: "D-Quant: Driftable Entropy Coding for KV Cache Quantization".
 *  - Sec. 4.2 Eq. (3): a stream (the n values of one token's key or value,
 *    all KV heads) lives in a container of C bytes; the symbol costs must
 *    satisfy sum_i r(m_i) <= B = 8C - sigma.  Eq. (4): token-wise affine
 *    grid x^ = o + s m, s = (max - min)/(M - 1), o = min.  The probability
 *    table comes from Gaussian order statistics, with no calibration data.
 *  - Sec. 4.3 Eq. (5)-(6): Drift, the Lagrangian assignment
 *    argmin_m D_im + lambda r_m with lambda found by bisection.
 *  - Sec. 4.4: distribution sharpening p' ~ p^alpha.
 *  - App. A, Algorithm 1: FitMinMax, Drift, Refit (least squares), fp16
 *    s and o, Drift again, rANS encode; the bisection runs on log2(lambda)
 *    from hi = log2(8 (max D - min D)) down to hi - 40, 12 steps, and returns
 *    the assignment at hi.  Algorithm 2: the decoder (state in the first
 *    sigma/8 bytes, one table lookup per symbol, byte renormalisation
 *    below L).
 *  - Sec. 4.2: keys remove a windowed channel mean.
 * Readings where the page is silent (all stated with the tests):
 *  - Gaussian order statistics: a = E[max of n iid N(0,1)]; the M levels sit
 *    at -a + 2a m/(M-1); a level's probability is the N(0,1) mass of its bin
 *    (edges at midpoints, outer bins open).  Frequencies f_m =
 *    max(1, round(2^p p'_m)); the shortfall 2^p - sum f goes to the largest
 *    f (lowest index on ties); c_m are prefix sums.
 *  - Costs are fixed point with 16 fractional bits, rounded up:
 *    r_m = ceil(-log2(f_m / 2^p) 2^16); the budget test is on integers.
 *  - sigma = 32 (a 32-bit state), L = 2^23, bytes emitted below L.
 *  - Bisection points are multiples of 1/512; lambda = ldexp(F[k], e) for
 *    mu = e + k/512 with F[k] = fp32(2^(k/512)).  hi = ceil(log2(v)) of
 *    v = 8 fp32(max D - min D) via frexp (0 when v = 0).
 *  - Refit: S_m, S_mm exact integers, S_x and S_mx summed in R32 order in
 *    fp32; skipped when n S_mm - S_m^2 = 0.
 *  - Container: [final state, little endian][emitted bytes, last emitted
 *    first][zeros up to C].
 *  - Windowed key mean: a window is 128 consecutive quantized tokens; the
 *    mean is stored as INT8 with one fp16 scale max|mu|/127 (RNE) and the
 *    encoder subtracts the dequantized mean.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

uint16_t or_f32_to_f16(float x);
float or_f16_to_f32(uint16_t h);
float or_r32_sum(const float *x, int n);

#define RANS_L (1u << 23)

static double phi_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* E[max of n iid N(0,1)] = integral of x n phi(x) Phi(x)^(n-1), composite
 * Simpson on [-12, 12] with 240000 intervals. */
double or_dq_expected_max(int n) {
    if (n <= 1) return 0.0;
    const int N = 240000;
    const double a = -12.0, b = 12.0, h = (b - a) / N;
    double acc = 0.0;
    for (int i = 0; i <= N; i++) {
        const double x = a + h * i;
        const double pdf = exp(-0.5 * x * x) / sqrt(2.0 * 3.14159265358979323846);
        const double g = x * n * pdf * pow(phi_cdf(x), n - 1);
        const double wgt = (i == 0 || i == N) ? 1.0 : ((i & 1) ? 4.0 : 2.0);
        acc += wgt * g;
    }
    return acc * h / 3.0;
}

/*
 * Frequency table of M levels for streams of n values at precision p bits,
 * sharpened by alpha.  f[M], c[M].  Returns 0, or -1 if the adjustment would
 * leave a frequency below 1 or M is out of [2, 2^p].
 */
int or_dq_table(int n, int M, double alpha, int p, int *f, int *c, double *prob) {
    const int total = 1 << p;
    if (M < 2 || M > total) return -1;
    const double a = or_dq_expected_max(n);
    double *u = (double *)malloc(sizeof(double) * (size_t)M);
    double *pm = (double *)malloc(sizeof(double) * (size_t)M);
    for (int m = 0; m < M; m++) u[m] = -a + 2.0 * a * m / (M - 1);
    double z = 0.0;
    for (int m = 0; m < M; m++) {
        const double lo = m == 0 ? 0.0 : phi_cdf(0.5 * (u[m - 1] + u[m]));
        const double hi = m == M - 1 ? 1.0 : phi_cdf(0.5 * (u[m] + u[m + 1]));
        pm[m] = hi - lo;
        if (prob) prob[m] = pm[m];
        pm[m] = pow(pm[m], alpha);
        z += pm[m];
    }
    int sum = 0;
    for (int m = 0; m < M; m++) {
        const int v = (int)round(total * (pm[m] / z));
        f[m] = v < 1 ? 1 : v;
        sum += f[m];
    }
    int big = 0;
    for (int m = 1; m < M; m++)
        if (f[m] > f[big]) big = m;
    f[big] += total - sum;
    free(u);
    free(pm);
    if (f[big] < 1) return -1;
    int run = 0;
    for (int m = 0; m < M; m++) {
        c[m] = run;
        run += f[m];
    }
    return 0;
}

/* Fixed-point costs r_m = ceil(-log2(f_m / 2^p) * 2^16). */
void or_dq_costs(const int *f, int M, int p, long long *r) {
    for (int m = 0; m < M; m++) r[m] = (long long)ceil(((double)p - log2((double)f[m])) * 65536.0);
}

/* F[k] = fp32(2^(k/512)), k = 0..511. */
void or_dq_pow2_table(float *F) {
    for (int k = 0; k < 512; k++) F[k] = (float)exp2(k / 512.0);
}

/* Assignment at log2(lambda) = mu512 / 512; returns the integer cost. */
static long long assign_at(const float *x, int n, const float *g, int M, const long long *r, const float *F,
                           long long mu512, uint8_t *m_out) {
    const long long e = mu512 >= 0 ? mu512 / 512 : -((-mu512 + 511) / 512);  /* floor */
    const int k = (int)(mu512 - 512 * e);
    const float lam = ldexpf(F[k], (int)e);
    float lr[256];
    for (int m = 0; m < M; m++) lr[m] = lam * ((float)r[m] / 65536.0f);
    long long cost = 0;
    for (int i = 0; i < n; i++) {
        int best = 0;
        float dd = x[i] - g[0];
        float bv = dd * dd + lr[0];
        for (int m = 1; m < M; m++) {
            dd = x[i] - g[m];
            const float v = dd * dd + lr[m];
            if (v < bv) {
                bv = v;
                best = m;
            }
        }
        m_out[i] = (uint8_t)best;
        cost += r[best];
    }
    return cost;
}

/*
 * Drift: the length-constrained assignment of x[n] to the grid o + s m.
 * budget_fx = B * 2^16.  m_out[n]; *cost_out the integer cost.  Returns 1 if
 * the returned assignment satisfies the budget.
 */
int or_dq_drift(const float *x, int n, float s, float o, const long long *r, int M, long long budget_fx,
                const float *F, uint8_t *m_out, long long *cost_out) {
    float g[256];
    for (int m = 0; m < M; m++) g[m] = o + s * (float)m;
    float minD = INFINITY, maxD = -INFINITY;
    for (int i = 0; i < n; i++)
        for (int m = 0; m < M; m++) {
            const float dd = x[i] - g[m];
            const float D = dd * dd;
            if (D < minD) minD = D;
            if (D > maxD) maxD = D;
        }
    const float v = 8.0f * (maxD - minD);
    long long hi;
    if (v == 0.0f) {
        hi = 0;
    } else if (!isfinite(v)) {
        hi = 128;
    } else {
        int e;
        const float mant = frexpf(v, &e);
        hi = mant == 0.5f ? e - 1 : e;
    }
    long long hi512 = hi * 512, lo512 = hi512 - 40 * 512;
    uint8_t *tmp = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    for (int t = 0; t < 12; t++) {
        const long long mid = (lo512 + hi512) / 2;  /* always even: see the header */
        if (assign_at(x, n, g, M, r, F, mid, tmp) <= budget_fx)
            hi512 = mid;
        else
            lo512 = mid;
    }
    free(tmp);
    const long long cost = assign_at(x, n, g, M, r, F, hi512, m_out);
    if (cost_out) *cost_out = cost;
    return cost <= budget_fx;
}

/* Least-squares refit of (s, o) to the assignment; unchanged when degenerate. */
void or_dq_refit(const float *x, const uint8_t *m, int n, float *s, float *o) {
    long long Sm = 0, Smm = 0;
    float *mx = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; i++) {
        Sm += m[i];
        Smm += (long long)m[i] * m[i];
        mx[i] = (float)m[i] * x[i];
    }
    const float Sx = or_r32_sum(x, n), Smx = or_r32_sum(mx, n);
    free(mx);
    const long long den_i = (long long)n * Smm - Sm * Sm;
    if (den_i == 0) return;
    const float den = (float)den_i, nf = (float)n, smf = (float)Sm;
    const float num = nf * Smx - smf * Sx;
    const float sn = num / den;
    *s = sn;
    *o = (Sx - sn * smf) / nf;
}

/*
 * rANS encode of m[n] (last symbol first) into a container of C bytes.
 * Returns the number of emitted bytes, or -1 if 4 + emitted > C (the
 * container is then left zero-filled past what fits).
 */
int or_rans_encode(const uint8_t *m, int n, const int *f, const int *c, int p, int C, uint8_t *out) {
    uint8_t *buf = (uint8_t *)malloc((size_t)(4 * n + 8));
    uint32_t x = RANS_L;
    int pushed = 0;
    for (int i = n - 1; i >= 0; i--) {
        const uint32_t fm = (uint32_t)f[m[i]], cm = (uint32_t)c[m[i]];
        const uint32_t xmax = ((RANS_L >> p) << 8) * fm;
        while (x >= xmax) {
            buf[pushed++] = (uint8_t)(x & 255u);
            x >>= 8;
        }
        x = ((x / fm) << p) + (x % fm) + cm;
    }
    memset(out, 0, (size_t)C);
    int ok = 4 + pushed <= C;
    if (C >= 4) {
        out[0] = (uint8_t)x;
        out[1] = (uint8_t)(x >> 8);
        out[2] = (uint8_t)(x >> 16);
        out[3] = (uint8_t)(x >> 24);
    }
    for (int j = 0; j < pushed && 4 + j < C; j++) out[4 + j] = buf[pushed - 1 - j];
    free(buf);
    return ok ? pushed : -1;
}

/*
 * Decode n symbols from a container of C bytes.  m_out[n]; *x_final the
 * state after the last symbol; *consumed the bytes read after the state.
 * Returns 0, or -1 if the decoder would read past the container.
 */
int or_rans_decode(const uint8_t *pay, int C, int n, const int *f, const int *c, int M, int p, uint8_t *m_out,
                   uint32_t *x_final, int *consumed) {
    uint32_t x = (uint32_t)pay[0] | ((uint32_t)pay[1] << 8) | ((uint32_t)pay[2] << 16) | ((uint32_t)pay[3] << 24);
    int ptr = 4;
    const uint32_t mask = (1u << p) - 1u;
    for (int i = 0; i < n; i++) {
        const uint32_t z = x & mask;
        int m = 0;
        while (m + 1 < M && (uint32_t)c[m + 1] <= z) m++;
        x = (uint32_t)f[m] * (x >> p) + z - (uint32_t)c[m];
        while (x < RANS_L) {
            if (ptr >= C) return -1;
            x = (x << 8) | pay[ptr++];
        }
        m_out[i] = (uint8_t)m;
    }
    if (x_final) *x_final = x;
    if (consumed) *consumed = ptr - 4;
    return 0;
}

/*
 * One stream end to end (Algorithm 1): FitMinMax, Drift, Refit, fp16 s and
 * o, Drift, rANS encode.  Outputs the container, the fp16 bits of s and o,
 * the final symbols and the symbols of nearest rounding on the final grid
 * (m_near, may be NULL).  Returns a bit set: 1 = the final assignment is over
 * budget, 2 = the container overflowed.
 */
int or_dq_encode_stream(const float *x, int n, int M, int C, const int *f, const int *c, int p, const long long *r,
                        const float *F, uint8_t *container, uint16_t *s16, uint16_t *o16, uint8_t *m_out,
                        uint8_t *m_near) {
    float lo = x[0], hi = x[0];
    for (int i = 1; i < n; i++) {
        if (x[i] < lo) lo = x[i];
        if (x[i] > hi) hi = x[i];
    }
    float s = (hi - lo) / (float)(M - 1), o = lo;
    const long long budget_fx = (long long)(8 * C - 32) * 65536;
    or_dq_drift(x, n, s, o, r, M, budget_fx, F, m_out, NULL);
    or_dq_refit(x, m_out, n, &s, &o);
    *s16 = or_f32_to_f16(s);
    *o16 = or_f32_to_f16(o);
    const float s2 = or_f16_to_f32(*s16), o2 = or_f16_to_f32(*o16);
    const int feasible = or_dq_drift(x, n, s2, o2, r, M, budget_fx, F, m_out, NULL);
    if (m_near) {
        for (int i = 0; i < n; i++) {
            int best = 0;
            float bd = fabsf(x[i] - (o2 + s2 * 0.0f));
            for (int m = 1; m < M; m++) {
                const float dd = fabsf(x[i] - (o2 + s2 * (float)m));
                if (dd < bd) {
                    bd = dd;
                    best = m;
                }
            }
            m_near[i] = (uint8_t)best;
        }
    }
    const int pushed = or_rans_encode(m_out, n, f, c, p, C, container);
    return (feasible ? 0 : 1) | (pushed < 0 ? 2 : 0);
}

/*
 * Windowed key mean over n_tok tokens of n values (y row-major [n_tok][n]):
 * mu_j = (sum_t y_tj) / n_tok in token order, scale16 = fp16(max|mu| / 127),
 * q_j = clamp(rint(mu_j / scale), -127, 127) (0 when the scale is 0), and the
 * dequantized mean mu_hat_j = q_j * scale.
 */
void or_dq_window_mean(const float *y, int n_tok, int n, int8_t *q, uint16_t *scale16, float *mu_hat) {
    float *mu = (float *)malloc(sizeof(float) * (size_t)n);
    float amax = 0.0f;
    for (int j = 0; j < n; j++) {
        float acc = 0.0f;
        for (int t = 0; t < n_tok; t++) acc = acc + y[(size_t)t * n + j];
        mu[j] = n_tok > 0 ? acc / (float)n_tok : 0.0f;
        if (fabsf(mu[j]) > amax) amax = fabsf(mu[j]);
    }
    *scale16 = or_f32_to_f16(amax / 127.0f);
    const float sc = or_f16_to_f32(*scale16);
    for (int j = 0; j < n; j++) {
        int v = 0;
        if (sc != 0.0f) {
            const float r = rintf(mu[j] / sc);
            v = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
        }
        q[j] = (int8_t)v;
        mu_hat[j] = (float)v * sc;
    }
    free(mu);
}

/*
 * Many streams at once (independent; one thread each under OpenMP).
 * X [ns][n] fp32; containers [ns][C]; s16, o16 [ns]; m [ns][n]; flags [ns].
 */
void or_dq_encode_streams(const float *X, int ns, int n, int M, int C, const int *f, const int *c, int p,
                          const long long *r, const float *F, uint8_t *containers, uint16_t *s16, uint16_t *o16,
                          uint8_t *m, int *flags) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int i = 0; i < ns; i++)
        flags[i] = or_dq_encode_stream(X + (size_t)i * n, n, M, C, f, c, p, r, F, containers + (size_t)i * C,
                                       s16 + i, o16 + i, m + (size_t)i * n, NULL);
}

void or_rotate_hadamard(const float *x, float *y, int d);

/* The normalized Hadamard rotation of each of `rows` rows of d values. */
void or_rotate_hadamard_rows(const float *x, float *y, long rows, int d) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < rows; i++) or_rotate_hadamard(x + i * d, y + i * d, d);
}
