// D-Quant fixed-size entropy-coded KV cache, prefill (sm_103a).
//
// "D-Quant: Driftable Entropy Coding for KV Cache Quantization":
//  * Sec. 4.2: a stream is the n = Hkv * d values of one token's key (or
//    value) across all KV heads; it is stored in a container of C bytes whose
//    symbol costs satisfy sum_i r(m_i) <= B = 8C - 32 (Eq. (3), a 32-bit rANS
//    state).  Keys are Hadamard-rotated per head and have a windowed channel
//    mean removed; the grid is o + s m, m < M (Eq. (4)).  The symbol model is
//    derived from Gaussian order statistics, sharpened by alpha (Sec. 4.4).
//  * Sec. 4.3 / App. A Algorithm 1: FitMinMax, Drift (bisection of log2
//    lambda over 12 steps from hi = log2(8 (max D - min D)) to hi - 40),
//    least-squares Refit, fp16 s and o, Drift again, rANS encode.
//  * Sec. 4.5 Encoding: one warp per stream, values kept on chip, distortions
//    recomputed per bisection step, code lengths reduced with warp operations.
// The encoder here is split in two launches: the warp-per-stream Drift kernel
// writes each stream's symbols to a scratch buffer, then one thread per stream
// runs the serial rANS coder (so 32 streams advance together in a warp).
// Fixed arithmetic order (bit-exact with the oracle): fp32 steps are separate
// round-to-nearest operations; the Refit sums S_x and S_mx follow the R32
// order (lane = position mod 32 sums its positions in increasing order, then a
// xor butterfly over 16, 8, 4, 2, 1).
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

// ---- host: the symbol model (D-Quant Sec. 4.2 "Gaussian order statistics",
// Sec. 4.4 sharpening) ----------------------------------------------------------
namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// E[max of n iid N(0,1)] from its tail integrals,
//   E[X] = int_0^inf P(X > x) dx - int_0^inf P(X < -x) dx,
// with P(max > x) = 1 - Phi(x)^n and P(max < -x) = Phi(-x)^n; Simpson's rule
// on [0, 14], 140000 intervals.
double expected_max_normal(int n) {
    if (n <= 1) return 0.0;
    const int N = 140000;
    const double h = 14.0 / N;
    double acc = 0.0;
    for (int i = 0; i <= N; i++) {
        const double x = h * i;
        const double g = (1.0 - std::pow(normal_cdf(x), n)) - std::pow(normal_cdf(-x), n);
        acc += g * (i == 0 || i == N ? 1.0 : (i % 2 ? 4.0 : 2.0));
    }
    return acc * h / 3.0;
}

}  // namespace

int rans_model_probs(int n, int M, double *p) {
    if (n < 1 || M < 2 || M > RANS_MAX_LEVELS) return -1;
    const double a = expected_max_normal(n);
    for (int m = 0; m < M; m++) {
        // bin of level m: midpoints to its neighbours on the grid -a + 2a m/(M-1)
        const double um = -a + 2.0 * a * m / (M - 1);
        const double lo = m == 0 ? 0.0 : normal_cdf(um - a / (M - 1));
        const double hi = m == M - 1 ? 1.0 : normal_cdf(um + a / (M - 1));
        p[m] = hi - lo;
    }
    return 0;
}

int rans_build_table(int n, int M, double alpha, int prob_bits, int C, RansTable *t) {
    const int total = 1 << prob_bits;
    if (M < 2 || M > RANS_MAX_LEVELS || prob_bits != 8) return -1;
    double p[RANS_MAX_LEVELS], z = 0.0;
    if (rans_model_probs(n, M, p) != 0) return -1;
    for (int m = 0; m < M; m++) {
        p[m] = std::pow(p[m], alpha);
        z += p[m];
    }
    int sum = 0;
    for (int m = 0; m < M; m++) {
        const long v = std::lround(total * (p[m] / z));
        t->f[m] = v < 1 ? 1 : static_cast<int>(v);
        sum += t->f[m];
    }
    int big = 0;
    for (int m = 1; m < M; m++)
        if (t->f[m] > t->f[big]) big = m;
    t->f[big] += total - sum;
    if (t->f[big] < 1) return -1;
    t->M = M;
    t->C = C;
    int run = 0;
    long long rmin = -1;
    for (int m = 0; m < M; m++) {
        t->c[m] = run;
        run += t->f[m];
        t->r[m] = static_cast<long long>(std::ceil((prob_bits - std::log2(static_cast<double>(t->f[m]))) * 65536.0));
        t->rf[m] = static_cast<float>(t->r[m]) / 65536.0f;
        t->rcp[m] = ((1ull << 40) + static_cast<unsigned long long>(t->f[m]) - 1) / static_cast<unsigned long long>(t->f[m]);
        if (rmin < 0 || t->r[m] < rmin) rmin = t->r[m];
    }
    for (int m = M; m < RANS_MAX_LEVELS; m++) {
        t->f[m] = t->c[m] = 0;
        t->r[m] = 0;
        t->rf[m] = 0.0f;
        t->rcp[m] = 0;
    }
    for (int zz = 0; zz < total; zz++) {
        int m = 0;
        while (m + 1 < M && t->c[m + 1] <= zz) m++;
        t->dec[zz] = static_cast<uint32_t>(m) | (static_cast<uint32_t>(t->f[m]) << 4) |
                     (static_cast<uint32_t>(zz - t->c[m]) << 16);
    }
    t->budget_fx = (8LL * C - 32) * 65536;
    t->min_stream_cost = rmin * n;
    return 0;
}

void rans_pow2_table(float *F) {
    for (int k = 0; k < 512; k++) F[k] = static_cast<float>(std::pow(2.0, k / 512.0));
}

namespace {

constexpr uint32_t RANS_L = 1u << 23;

// Channels 4 lane .. 4 lane + 3 of KV head h of the token in quantized slot
// `slot` of sequence b: from this call's input when the token is one of its
// tokens, else from the 16-bit recent ring (an older token of a block flush).
__device__ __forceinline__ void load_tok4(const RansQuantArgs &a, int b, int h, long long slot, int lane,
                                          float (&r)[4]) {
    const long long t = a.n_sink + slot;
    if (t >= a.pos0) {
        const long long base = ((static_cast<long long>(b) * a.Hkv + h) * a.n_tok + (t - a.pos0)) * 128 + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; j++) r[j] = ld_in(a.x, base + j, a.in_dtype);
        return;
    }
    const long long rs = a.n_sink + t % a.n_recent, u = static_cast<long long>(b) * a.Hkv + h;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = 4 * lane + j;
        const long long off = a.is_key ? (u * a.rcap + rs) * 128 + c : ((u * (a.rcap / 2) + rs / 2) * 128 + c) * 2 + (rs & 1);
        const uint16_t bits = a.raw[off];
        r[j] = a.raw_bf16 ? __uint_as_float(static_cast<uint32_t>(bits) << 16) : __half2float(__ushort_as_half(bits));
    }
}

// ---------------------------------------------------------------------------
// Windowed key mean: one CTA per (sequence, window of 128 quantized slots),
// one warp per KV head.  Lane l holds channels 4l..4l+3 of its head; every
// rotated row is added in token order from 0.0f.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rans_mean_kernel(RansQuantArgs a) {
    __shared__ float wmax[8];
    const int b = blockIdx.x / a.n_win, w = blockIdx.x % a.n_win;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long s0 = a.slot0 + 128LL * w;
    const long long s1 = min(s0 + 128, a.slot0 + static_cast<long long>(a.n_fit));
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (long long sl = s0; sl < s1; sl++) {
        float x[4];
        load_tok4(a, b, h, sl, lane, x);
        if (a.rot) {
            fwht_warp<4>(x);
#pragma unroll
            for (int j = 0; j < 4; j++) x[j] = __fmul_rn(x[j], a.hscale);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) acc[j] = __fadd_rn(acc[j], x[j]);
    }
    const float cnt = static_cast<float>(s1 - s0);
    float mu[4], am = 0.f;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        mu[j] = s1 > s0 ? __fdiv_rn(acc[j], cnt) : 0.f;
        am = fmaxf(am, fabsf(mu[j]));
    }
    am = warp_max(am);
    if (lane == 0) wmax[h] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int i = 0; i < a.Hkv; i++) m = fmaxf(m, wmax[i]);
        wmax[0] = m;
    }
    __syncthreads();
    const __half sc16 = __float2half_rn(__fdiv_rn(wmax[0], 127.0f));
    const float sc = __half2float(sc16);
    uint8_t *rec = a.mean + (static_cast<long long>(b) * a.wcap + a.slot0 / 128 + w) * a.mean_rec;
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        int v = 0;
        if (sc != 0.f) {
            const float r = rintf(__fdiv_rn(mu[j], sc));
            v = r > 127.f ? 127 : (r < -127.f ? -127 : static_cast<int>(r));
        }
        packed |= (static_cast<uint32_t>(v) & 0xffu) << (8 * j);
    }
    reinterpret_cast<uint32_t *>(rec)[32 * h + lane] = packed;
    if (threadIdx.x == 0) *reinterpret_cast<__half *>(rec + a.n) = sc16;
}

// ---------------------------------------------------------------------------
// Drift (Algorithm 1 up to the coder): one warp per stream.  The stream sits
// in a per-warp shared row xs[n] in stream order; lane l owns positions
// 128h + 4l + j (j < 4) of every KV head h and reads them as one float4.
// ---------------------------------------------------------------------------
// Pass kinds of one assignment at a given lambda.
enum { PASS_COST = 0, PASS_REFIT = 1, PASS_STORE = 2 };

struct RefitSums {
    long long Sm, Smm;
    int changed = 0, move = 0;  // PASS_STORE: symbols off the nearest level, the largest distance
};

// One assignment argmin_m fp32(D_im + fp32(lambda r_m)) (ties to the lower m)
// at log2(lambda) = mu512 / 512; returns the stream's integer cost.
// PASS_REFIT also writes fp32(m x) to mx[] and accumulates S_m, S_mm;
// PASS_STORE writes the symbols (4 per word) to sym_out.
template <int H, int MMAX, int PASS>
__device__ __forceinline__ long long assign_at(const float *xs, const float (&g)[MMAX], const RansTable &tb,
                                               const float *F, long long mu512, int M, float *mx, RefitSums &rs,
                                               uint32_t *sym_out) {
    const int lane = threadIdx.x & 31;
    const long long e = mu512 >= 0 ? mu512 / 512 : -((-mu512 + 511) / 512);
    const int k = static_cast<int>(mu512 - 512 * e);
    const float lam = ldexpf(F[k], static_cast<int>(e));
    float lr[MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; m++) lr[m] = __fmul_rn(lam, tb.rf[m]);
    long long cost = 0;
#pragma unroll 1
    for (int h = 0; h < H; h++) {
        const float4 v4 = *reinterpret_cast<const float4 *>(xs + 128 * h + 4 * lane);
        const float xv[4] = {v4.x, v4.y, v4.z, v4.w};
        uint32_t word = 0;
        float mxv[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float dd = __fsub_rn(xv[j], g[0]);
            float bv = __fadd_rn(__fmul_rn(dd, dd), lr[0]);
            int best = 0;
#pragma unroll
            for (int m = 1; m < MMAX; m++) {
                if (m < M) {
                    dd = __fsub_rn(xv[j], g[m]);
                    const float v = __fadd_rn(__fmul_rn(dd, dd), lr[m]);
                    if (v < bv) {
                        bv = v;
                        best = m;
                    }
                }
            }
            cost += tb.r[best];
            word |= static_cast<uint32_t>(best) << (8 * j);
            if (PASS == PASS_STORE) {  // drift statistics: against the nearest level of the grid
                float bn = fabsf(__fsub_rn(xv[j], g[0]));
                int near = 0;
#pragma unroll
                for (int m = 1; m < MMAX; m++) {
                    if (m < M) {
                        const float dn = fabsf(__fsub_rn(xv[j], g[m]));
                        if (dn < bn) {
                            bn = dn;
                            near = m;
                        }
                    }
                }
                rs.changed += best != near;
                rs.move = max(rs.move, abs(best - near));
            }
            if (PASS == PASS_REFIT) {
                rs.Sm += best;
                rs.Smm += best * best;
                mxv[j] = __fmul_rn(static_cast<float>(best), xv[j]);
            }
        }
        if (PASS == PASS_REFIT)
            *reinterpret_cast<float4 *>(mx + 128 * h + 4 * lane) = make_float4(mxv[0], mxv[1], mxv[2], mxv[3]);
        if (PASS == PASS_STORE) sym_out[32 * h + lane] = word;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) cost += __shfl_xor_sync(FULL, cost, o);
    return cost;
}

// Drift at the grid o + s m: bisection of log2(lambda), then the assignment at
// the last feasible point (PASS decides what that final pass records).
template <int H, int MMAX, int PASS>
__device__ __forceinline__ bool drift(const float *xs, float s, float o, const RansTable &tb, const float *F,
                                      int M, float *mx, RefitSums &rs, uint32_t *sym_out) {
    const int lane = threadIdx.x & 31;
    float g[MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; m++) g[m] = __fadd_rn(o, __fmul_rn(s, static_cast<float>(m)));
    float mn = INFINITY, mxD = -INFINITY;
#pragma unroll 1
    for (int h = 0; h < H; h++) {
        const float4 v4 = *reinterpret_cast<const float4 *>(xs + 128 * h + 4 * lane);
        const float xv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int j = 0; j < 4; j++)
#pragma unroll
            for (int m = 0; m < MMAX; m++)
                if (m < M) {
                    const float dd = __fsub_rn(xv[j], g[m]);
                    const float D = __fmul_rn(dd, dd);
                    mn = fminf(mn, D);
                    mxD = fmaxf(mxD, D);
                }
    }
    mn = warp_min(mn);
    mxD = warp_max(mxD);
    const float v = __fmul_rn(8.0f, __fsub_rn(mxD, mn));
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
#pragma unroll 1
    for (int t = 0; t < 12; t++) {
        const long long mid = (lo512 + hi512) / 2;
        if (assign_at<H, MMAX, PASS_COST>(xs, g, tb, F, mid, M, mx, rs, sym_out) <= tb.budget_fx)
            hi512 = mid;
        else
            lo512 = mid;
    }
    return assign_at<H, MMAX, PASS>(xs, g, tb, F, hi512, M, mx, rs, sym_out) <= tb.budget_fx;
}

// R32 sum of a per-warp shared row of n floats.
__device__ __forceinline__ float r32_sum_row(const float *row, int n) {
    const int lane = threadIdx.x & 31;
    float acc = 0.0f;
    for (int p = lane; p < n; p += 32) acc = __fadd_rn(acc, row[p]);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, o));
    return acc;
}

template <int H, int MMAX>
__global__ void __launch_bounds__(128) rans_drift_kernel(RansQuantArgs a, const RansTable *tbp, const float *Fg) {
    constexpr int N = 128 * H;
    __shared__ RansTable tb;
    __shared__ float F[512];
    __shared__ __align__(16) float stage[4][2][N];
    if (threadIdx.x == 0) tb = *tbp;
    for (int i = threadIdx.x; i < 512; i += blockDim.x) F[i] = Fg[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * 4 + warp;
    if (gw >= static_cast<long long>(a.B) * a.n_fit) return;
    const int b = static_cast<int>(gw / a.n_fit);
    const long long slot = a.slot0 + gw % a.n_fit;
    const int M = tb.M;
    float *xs = stage[warp][0], *mx = stage[warp][1];
    bool finite = true;
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll 1
    for (int h = 0; h < H; h++) {
        float r[4];
        load_tok4(a, b, h, slot, lane, r);
#pragma unroll
        for (int j = 0; j < 4; j++) finite = finite && isfinite(r[j]);
        if (a.rot) {
            fwht_warp<4>(r);
#pragma unroll
            for (int j = 0; j < 4; j++) r[j] = __fmul_rn(r[j], a.hscale);
        }
        if (a.mean) {
            const uint8_t *rec = a.mean + (static_cast<long long>(b) * a.wcap + slot / 128) * a.mean_rec;
            const float sc = __half2float(*reinterpret_cast<const __half *>(rec + N));
            const uint32_t qw = reinterpret_cast<const uint32_t *>(rec)[32 * h + lane];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float mh = __fmul_rn(static_cast<float>(static_cast<int8_t>((qw >> (8 * j)) & 0xffu)), sc);
                r[j] = __fsub_rn(r[j], mh);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            lo = fminf(lo, r[j]);
            hi = fmaxf(hi, r[j]);
        }
        *reinterpret_cast<float4 *>(xs + 128 * h + 4 * lane) = make_float4(r[0], r[1], r[2], r[3]);
    }
    __syncwarp();
    if (!__all_sync(FULL, finite) && lane == 0) atomicOr(a.status, ST_NONFINITE);
    // FitMinMax
    lo = warp_min(lo);
    hi = warp_max(hi);
    float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(M - 1)), o = lo;
    RefitSums rs{0, 0};
    drift<H, MMAX, PASS_REFIT>(xs, s, o, tb, F, M, mx, rs, nullptr);
    __syncwarp();
    // Refit: integer S_m, S_mm; S_x and S_mx in R32 order over the shared rows
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) {
        rs.Sm += __shfl_xor_sync(FULL, rs.Sm, o2);
        rs.Smm += __shfl_xor_sync(FULL, rs.Smm, o2);
    }
    const float Sx = r32_sum_row(xs, N), Smx = r32_sum_row(mx, N);
    const long long den_i = static_cast<long long>(N) * rs.Smm - rs.Sm * rs.Sm;
    if (den_i != 0) {
        const float den = __ll2float_rn(den_i), nf = static_cast<float>(N), smf = static_cast<float>(rs.Sm);
        const float num = __fsub_rn(__fmul_rn(nf, Smx), __fmul_rn(smf, Sx));
        s = __fdiv_rn(num, den);
        o = __fdiv_rn(__fsub_rn(Sx, __fmul_rn(s, smf)), nf);
    }
    const __half s16 = __float2half_rn(s), o16 = __float2half_rn(o);
    uint32_t *sym = reinterpret_cast<uint32_t *>(a.sym + gw * N);
    rs.changed = rs.move = 0;
    const bool ok = drift<H, MMAX, PASS_STORE>(xs, __half2float(s16), __half2float(o16), tb, F, M, mx, rs, sym);
    if (!ok && lane == 0) atomicOr(a.status, ST_INFEASIBLE);
    if (a.drift_stats) {  // symbols drift moved off the nearest level of the final grid, and how far
        int ch = rs.changed, mv = rs.move;
#pragma unroll
        for (int o2 = 16; o2; o2 >>= 1) {
            ch += __shfl_xor_sync(FULL, ch, o2);
            mv = max(mv, __shfl_xor_sync(FULL, mv, o2));
        }
        if (lane == 0) {
            atomicAdd(a.drift_stats, static_cast<unsigned long long>(ch));
            atomicAdd(a.drift_stats + 1, static_cast<unsigned long long>(N));
            atomicMax(a.drift_stats + 2, static_cast<unsigned long long>(mv));
        }
    }
    if (lane == 0) {
        __half2 *meta = reinterpret_cast<__half2 *>(a.meta);
        meta[static_cast<long long>(b) * a.qcap + slot] = __halves2half2(s16, o16);
    }
}

// ---------------------------------------------------------------------------
// rANS encoder: one thread per stream, 32 consecutive streams of a sequence per
// CTA.  Symbols are coded last to first; emitted bytes are staged from the end
// of the thread's container in shared memory and moved behind the state.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) rans_encode_kernel(RansQuantArgs a, const RansTable *tbp) {
    extern __shared__ __align__(16) uint8_t cont[];  // [32][C]
    __shared__ RansTable tb;
    if (threadIdx.x == 0) tb = *tbp;
    __syncthreads();
    const int C = tb.C, N = a.n;
    const int b = blockIdx.y;
    const long long rel0 = 32LL * blockIdx.x, rel = rel0 + threadIdx.x;  // within the flushed range
    uint8_t *mine = cont + threadIdx.x * C;
    for (int i = 0; i < C; i++) mine[i] = 0;
    if (rel < a.n_fit) {
        const uint8_t *sym = a.sym + (static_cast<long long>(b) * a.n_fit + rel) * N;
        uint32_t x = RANS_L;
        int pushed = 0;
        bool over = false;
        for (int i0 = N - 16; i0 >= 0; i0 -= 16) {
            const uint4 w = *reinterpret_cast<const uint4 *>(sym + i0);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 15; k >= 0; k--) {
                const int m = static_cast<int>((ws[k >> 2] >> (8 * (k & 3))) & 0xffu);
                const uint32_t f = static_cast<uint32_t>(tb.f[m]);
                if (x >= (f << 23)) {
                    if (pushed < C - 4) mine[C - 1 - pushed] = static_cast<uint8_t>(x & 255u);
                    else over = true;
                    pushed++;
                    x >>= 8;
                }
                const uint32_t q = static_cast<uint32_t>((static_cast<unsigned long long>(x) * tb.rcp[m]) >> 40);
                x = (q << 8) + (x - q * f) + static_cast<uint32_t>(tb.c[m]);
            }
        }
        if (over) {
            atomicOr(a.status, ST_INFEASIBLE);
            pushed = C - 4;
        }
        for (int j = 0; j < pushed; j++) mine[4 + j] = mine[C - pushed + j];
        for (int j = 4 + pushed; j < C; j++) mine[j] = 0;
        mine[0] = static_cast<uint8_t>(x);
        mine[1] = static_cast<uint8_t>(x >> 8);
        mine[2] = static_cast<uint8_t>(x >> 16);
        mine[3] = static_cast<uint8_t>(x >> 24);
    }
    __syncthreads();
    // 32 containers are 32 * C bytes, a multiple of 16, at a 16-byte aligned offset
    uint4 *dst = reinterpret_cast<uint4 *>(a.codes + (static_cast<long long>(b) * a.qcap + a.slot0 + rel0) * C);
    const uint4 *src = reinterpret_cast<const uint4 *>(cont);
    for (int i = threadIdx.x; i < 2 * C; i += 32) dst[i] = src[i];
}

// 16-bit regions: this call's sinks (raw_ns tokens from pos0) and its tokens
// among the latest n_recent of the sequence (raw_nr tokens ending at pos0 +
// n_tok).  One warp per (unit, token) of those sets; lanes copy 4 channels each.
__global__ void __launch_bounds__(128) rans_raw_kernel(RansQuantArgs a, int n_sel) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * 4 + warp;
    const long long U = static_cast<long long>(a.B) * a.Hkv;
    if (gw >= U * n_sel) return;
    const long long u = gw / n_sel;
    const int i = static_cast<int>(gw % n_sel);
    long long t;
    int slot;
    if (i < a.raw_ns) {
        t = a.pos0 + i;
        slot = static_cast<int>(t);
    } else {
        t = a.pos0 + a.n_tok - a.raw_nr + (i - a.raw_ns);
        slot = a.n_sink + static_cast<int>(t % a.n_recent);
    }
    const long long base = (u * a.n_tok + (t - a.pos0)) * 128;
    const long long ub = u * a.rcap * 128;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = 4 * lane + j;
        const long long off = a.is_key ? static_cast<long long>(slot) * 128 + c
                                       : (static_cast<long long>(slot >> 1) * 128 + c) * 2 + (slot & 1);
        a.raw[ub + off] = raw16_of(a.x, base + c, a.in_dtype);
    }
}

template <typename F>
int rans_dispatch(int H, int M, F &&f) {
    const bool big = M > 8;
    switch (H) {
        case 1: return big ? f(std::integral_constant<int, 1>(), std::integral_constant<int, 16>())
                           : f(std::integral_constant<int, 1>(), std::integral_constant<int, 8>());
        case 2: return big ? f(std::integral_constant<int, 2>(), std::integral_constant<int, 16>())
                           : f(std::integral_constant<int, 2>(), std::integral_constant<int, 8>());
        case 4: return big ? f(std::integral_constant<int, 4>(), std::integral_constant<int, 16>())
                           : f(std::integral_constant<int, 4>(), std::integral_constant<int, 8>());
        case 8: return big ? f(std::integral_constant<int, 8>(), std::integral_constant<int, 16>())
                           : f(std::integral_constant<int, 8>(), std::integral_constant<int, 8>());
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace

int launch_rans_mean(const RansQuantArgs &a, void *stream) {
    const unsigned grid = static_cast<unsigned>(a.B * a.n_win);
    if (grid == 0) return 0;
    rans_mean_kernel<<<grid, 32 * a.Hkv, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return static_cast<int>(cudaGetLastError());
}

int launch_rans_drift(const RansQuantArgs &a, const RansTable *tb, const float *F, int M, void *stream) {
    const long long warps = static_cast<long long>(a.B) * a.n_fit;
    if (warps == 0) return 0;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    return rans_dispatch(a.Hkv, M, [&](auto h, auto mm) {
        rans_drift_kernel<decltype(h)::value, decltype(mm)::value>
            <<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, tb, F);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_rans_encode(const RansQuantArgs &a, const RansTable *tb, int C, void *stream) {
    if (a.n_fit == 0) return 0;
    const size_t smem = static_cast<size_t>(32) * C;
    cudaError_t e = cudaFuncSetAttribute(rans_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    const dim3 grid(static_cast<unsigned>((a.n_fit + 31) / 32), static_cast<unsigned>(a.B));
    rans_encode_kernel<<<grid, 32, smem, static_cast<cudaStream_t>(stream)>>>(a, tb);
    return static_cast<int>(cudaGetLastError());
}

int launch_rans_raw(const RansQuantArgs &a, void *stream) {
    const int n_sel = a.raw_ns + a.raw_nr;
    const long long warps = static_cast<long long>(a.B) * a.Hkv * n_sel;
    if (warps == 0) return 0;
    rans_raw_kernel<<<static_cast<unsigned>((warps + 3) / 4), 128, 0, static_cast<cudaStream_t>(stream)>>>(a, n_sel);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace dq
