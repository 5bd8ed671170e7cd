// Affine KV quantization kernels: key channel mean, per-token quantize + pack,
// and the dequantize export.
//
// Method ("D-Quant: Driftable Entropy Coding for KV Cache Quantization"):
//   Sec. 4.2: normalized Hadamard rotation per head, key channel-mean removal,
//   token-wise affine grid s = (max - min)/(M - 1), o = min  (Eq. (4));
//   Sec. 3.1 Eq. (1): x^ = o + s*m with m in {0 .. 2^b - 1};
//   App. A: s and o rounded to fp16 before the final code assignment.
// Percentile clip ("WUSH-KV", Methodology: clipping at a kappa-quantile, scale
// and zero point from the clipped range).  Dense key transform after RoPE
// ("WUSH-KV", Key Contributions 2).  Sink tokens kept exact ("KVQuant-NUQ",
// Attention Sink-Aware quantization) and the recent window in 16-bit
// ("D-Quant", Sec. 5.1 implementation details).
//
// Every fp32 step uses explicit round-to-nearest intrinsics so that no
// multiply-add is contracted: the codes, scale/offset and packed bytes are a
// pure function of the input bits.
#include <cuda_runtime.h>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

// ---------------------------------------------------------------------------
// Rotation of one token row held V values per lane (lane l: l*V .. l*V+V-1).
// Dense transform: y_i = sum_j T[i][j] x_j accumulated in j order from 0.
// ---------------------------------------------------------------------------
template <int V>
__device__ __forceinline__ void rotate_row(float (&x)[V], int rot, float hscale, const float *T,
                                          float *xs /* per-warp smem, d floats */) {
    constexpr int D = 32 * V;
    const int lane = threadIdx.x & 31;
    if (rot == DQ_ROT_HADAMARD) {
        fwht_warp<V>(x);
#pragma unroll
        for (int j = 0; j < V; j++) x[j] = __fmul_rn(x[j], hscale);
    } else if (rot == DQ_ROT_DENSE) {
#pragma unroll
        for (int j = 0; j < V; j++) xs[lane * V + j] = x[j];
        __syncwarp();
        float y[V];
#pragma unroll
        for (int j = 0; j < V; j++) {
            const float *Ti = T + static_cast<long long>(lane * V + j) * D;
            float acc = 0.0f;
            for (int k = 0; k < D; k++) acc = __fadd_rn(acc, __fmul_rn(__ldg(Ti + k), xs[k]));
            y[j] = acc;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < V; j++) x[j] = y[j];
    }
}

// ---------------------------------------------------------------------------
// Key channel mean over tokens [t0, t1) of each unit (prefill).  One block per
// unit, D threads; thread j accumulates channel j over the tokens in order
// (acc = acc + y_tj from 0.0f), then divides by the count.
// ---------------------------------------------------------------------------
template <int V>
__global__ void key_mean_kernel(QuantArgs a, int Hkv, long long t0, long long t1) {
    constexpr int D = 32 * V;
    constexpr int CH = 32;  // tokens per smem chunk
    __shared__ float ys[CH][D];
    __shared__ float xs[D / 32][D];
    const int u = blockIdx.x, kvh = u % Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = D / 32;
    const float *T = a.T ? a.T + static_cast<long long>(kvh) * D * D : nullptr;
    float acc = 0.0f;
    for (long long c0 = t0; c0 < t1; c0 += CH) {
        const int n = static_cast<int>(t1 - c0 < CH ? t1 - c0 : CH);
        for (int r = warp; r < n; r += nw) {
            const long long base = (static_cast<long long>(u) * a.n_tok + (c0 + r - a.pos0)) * D;
            float x[V];
#pragma unroll
            for (int j = 0; j < V; j++) x[j] = ld_in(a.x, base + lane * V + j, a.in_dtype);
            rotate_row<V>(x, a.rot, a.hscale, T, xs[warp]);
#pragma unroll
            for (int j = 0; j < V; j++) ys[r][lane * V + j] = x[j];
        }
        __syncthreads();
        for (int r = 0; r < n; r++) acc = __fadd_rn(acc, ys[r][threadIdx.x]);
        __syncthreads();
    }
    const long long cnt = t1 - t0;
    a.mean[static_cast<long long>(u) * D + threadIdx.x] = cnt > 0 ? __fdiv_rn(acc, static_cast<float>(cnt)) : 0.0f;
}

// ---------------------------------------------------------------------------
// Record packing helpers.
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// Quantize tokens [pos0, pos0 + n_tok): one warp per (unit, token).
// ---------------------------------------------------------------------------
template <int V, int BITS>
__global__ void quantize_kernel(QuantArgs a, Layout L) {
    constexpr int D = 32 * V;
    constexpr int WPB = 4;
    __shared__ float xs[WPB][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.n_tok) return;
    const int u = static_cast<int>(gw / a.n_tok);
    const long long i = gw % a.n_tok;
    const long long t = a.pos0 + i;
    const int kvh = u % L.Hkv;
    const long long base = (static_cast<long long>(u) * a.n_tok + i) * D;

    float x[V];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < V; j++) {
        x[j] = ld_in(a.x, base + lane * V + j, a.in_dtype);
        finite = finite && isfinite(x[j]);
    }
    if (!__all_sync(FULL, finite) && lane == 0) atomicOr(a.status, ST_NONFINITE);

    // 16-bit regions: sinks and the latest n_recent tokens, stored as given.
    int raw_slot = -1;
    if (t < L.n_sink) raw_slot = static_cast<int>(t);
    else if (L.n_recent > 0 && t >= a.seq_after - L.n_recent) raw_slot = L.n_sink + static_cast<int>(t % L.n_recent);
    if (raw_slot >= 0) {
        const long long ub = static_cast<long long>(u) * L.rcap * D;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int c = lane * V + j;
            const uint16_t r = raw16_of(a.x, base + c, a.in_dtype);
            long long off = a.is_key ? static_cast<long long>(raw_slot) * D + c
                                     : (static_cast<long long>(raw_slot >> 1) * D + c) * 2 + (raw_slot & 1);
            a.raw[ub + off] = r;
        }
    }
    if (t < L.n_sink) return;
    const long long slot = t - L.n_sink;

    rotate_row<V>(x, a.rot, a.hscale, a.T ? a.T + static_cast<long long>(kvh) * D * D : nullptr, xs[warp]);
    if (a.use_mean) {
        const float *mu = a.mean + static_cast<long long>(u) * D;
#pragma unroll
        for (int j = 0; j < V; j++) x[j] = __fsub_rn(x[j], mu[lane * V + j]);
    }

    // grid
    constexpr int LV = 1 << BITS;
    float lo, hi;
    if (a.clip > 0.0f) {
        // order statistics by rank (ties broken by channel index)
#pragma unroll
        for (int j = 0; j < V; j++) xs[warp][lane * V + j] = x[j];
        __syncwarp();
        float vlo0 = 0.f, vlo1 = 0.f, vhi0 = 0.f, vhi1 = 0.f;
        int have = 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int c = lane * V + j;
            const float xv = x[j];
            int rank = 0;
            for (int k = 0; k < D; k++) {
                const float y = xs[warp][k];
                rank += (y < xv) || (y == xv && k < c);
            }
            if (rank == a.clip_ilo) { vlo0 = xv; have |= 1; }
            if (rank == a.clip_ilo + 1) { vlo1 = xv; have |= 2; }
            if (rank == a.clip_ihi) { vhi0 = xv; have |= 4; }
            if (rank == a.clip_ihi + 1) { vhi1 = xv; have |= 8; }
        }
        __syncwarp();
        // gather the four order statistics (each held by exactly one lane)
        const unsigned m1 = __ballot_sync(FULL, have & 1), m2 = __ballot_sync(FULL, have & 2);
        const unsigned m4 = __ballot_sync(FULL, have & 4), m8 = __ballot_sync(FULL, have & 8);
        vlo0 = __shfl_sync(FULL, vlo0, __ffs(m1) - 1);
        vhi0 = __shfl_sync(FULL, vhi0, __ffs(m4) - 1);
        vlo1 = m2 ? __shfl_sync(FULL, vlo1, __ffs(m2) - 1) : vlo0;
        vhi1 = m8 ? __shfl_sync(FULL, vhi1, __ffs(m8) - 1) : vhi0;
        lo = (a.clip_ilo + 1 >= D) ? vlo0 : __fadd_rn(vlo0, __fmul_rn(a.clip_flo, __fsub_rn(vlo1, vlo0)));
        hi = (a.clip_ihi + 1 >= D) ? vhi0 : __fadd_rn(vhi0, __fmul_rn(a.clip_fhi, __fsub_rn(vhi1, vhi0)));
    } else {
        lo = x[0];
        hi = x[0];
#pragma unroll
        for (int j = 1; j < V; j++) { lo = fminf(lo, x[j]); hi = fmaxf(hi, x[j]); }
        lo = warp_min(lo);
        hi = warp_max(hi);
    }
    float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(LV - 1));
    float o = lo;
    if (a.meta_f16) {
        s = __half2float(__float2half_rn(s));
        o = __half2float(__float2half_rn(o));
    }

    uint32_t m[V];
#pragma unroll
    for (int j = 0; j < V; j++) {
        float xv = x[j];
        if (a.clip > 0.0f) xv = fminf(fmaxf(xv, lo), hi);
        int q = 0;
        if (s != 0.0f) {
            const float tq = __fdiv_rn(__fsub_rn(xv, o), s);
            if (tq == tq) q = min(max(__float2int_rn(tq), 0), LV - 1);
        }
        m[j] = static_cast<uint32_t>(q);
    }

    // meta
    const long long ms = static_cast<long long>(u) * L.qcap + slot;
    if (lane == 0) {
        if (a.meta_f16) {
            const uint32_t so = pack2(__half_as_ushort(__float2half_rn(s)), __half_as_ushort(__float2half_rn(o)));
            reinterpret_cast<uint32_t *>(a.meta)[ms] = so;
        } else {
            reinterpret_cast<float2 *>(a.meta)[ms] = make_float2(s, o);
        }
    }

    // pack
    constexpr int WK = Rec<D, BITS>::K_WORDS, WV = Rec<D, BITS>::V_WORDS;
    if (a.is_key) {
        uint32_t *row = reinterpret_cast<uint32_t *>(a.codes + ms * L.rowK);
        constexpr int WLO = D * 2 / 32;  // 2-bit plane words (BITS == 3)
#pragma unroll
        for (int w = 0; w < WK; w++) {
            uint32_t v = 0;
#pragma unroll
            for (int j = 0; j < V; j++) {
                const int c = lane * V + j;
                v |= contrib<D, BITS>(w, k_idx(c, D), c & 1, m[j], WLO);
            }
            v = __reduce_or_sync(FULL, v);
            if (lane == w) row[w] = v;
        }
    } else {
        const int e = static_cast<int>(slot & 1);
        uint16_t *rec = reinterpret_cast<uint16_t *>(
            a.codes + (static_cast<long long>(u) * (L.qcap / 2) + slot / 2) * L.pairV);
        constexpr int WLO = 2 * D * 2 / 32;
#pragma unroll
        for (int w = 0; w < WV; w++) {
            uint32_t v = 0;
#pragma unroll
            for (int j = 0; j < V; j++) {
                const int c = lane * V + j;
                v |= contrib<D, BITS>(w, v_idx(c, D), e, m[j], WLO);
            }
            v = __reduce_or_sync(FULL, v);
            if (lane == (w & 31)) rec[2 * w + e] = static_cast<uint16_t>(v >> (16 * e));
        }
    }
}

// ---------------------------------------------------------------------------
// Dequantize export: one warp per (unit, slot).
// ---------------------------------------------------------------------------
template <int D, int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *rec, int idx, int half, int words_lo) {
    if (BITS == 3) {
        const uint32_t lo = (rec[idx / 8] >> (16 * half + 2 * (idx % 8))) & 3u;
        const uint32_t hb = (rec[words_lo + idx / 16] >> (16 * half + idx % 16)) & 1u;
        return lo | (hb << 2);
    }
    constexpr int F = 16 / BITS;
    return (rec[idx / F] >> (16 * half + BITS * (idx % F))) & ((1u << BITS) - 1u);
}

template <int V, int BITS>
__global__ void dequant_kernel(DequantArgs a, Layout L) {
    constexpr int D = 32 * V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * 4 + warp;
    if (gw >= static_cast<long long>(L.U) * a.n) return;
    const int u = static_cast<int>(gw / a.n);
    const long long i = gw % a.n, slot = a.slot0 + i;
    const long long ms = static_cast<long long>(u) * L.qcap + slot;
    float s, o;
    if (a.meta_f16) {
        const uint32_t so = reinterpret_cast<const uint32_t *>(a.meta)[ms];
        s = __half2float(__ushort_as_half(static_cast<uint16_t>(so & 0xffffu)));
        o = __half2float(__ushort_as_half(static_cast<uint16_t>(so >> 16)));
    } else {
        const float2 so = reinterpret_cast<const float2 *>(a.meta)[ms];
        s = so.x;
        o = so.y;
    }
    const uint32_t *rec;
    int half = 0;
    if (a.is_key) {
        rec = reinterpret_cast<const uint32_t *>(a.codes + ms * L.rowK);
    } else {
        rec = reinterpret_cast<const uint32_t *>(a.codes + (static_cast<long long>(u) * (L.qcap / 2) + slot / 2) * L.pairV);
        half = static_cast<int>(slot & 1);
    }
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane * V + j;
        const uint32_t m = a.is_key ? code_at<D, BITS>(rec, k_idx(c, D), c & 1, D * 2 / 32)
                                    : code_at<D, BITS>(rec, v_idx(c, D), half, 2 * D * 2 / 32);
        float v = __fadd_rn(o, __fmul_rn(s, static_cast<float>(m)));
        if (a.mean) v = __fadd_rn(v, a.mean[static_cast<long long>(u) * D + c]);
        a.out[(static_cast<long long>(u) * a.n + i) * D + c] = v;
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
int launch_key_mean(const Layout &L, const QuantArgs &a, void *stream) {
    const long long t0 = L.n_sink;
    long long t1 = a.seq_after - L.n_recent;
    if (t1 < t0) t1 = t0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L.d == 128) key_mean_kernel<4><<<L.U, 128, 0, st>>>(a, L.Hkv, t0, t1);
    else key_mean_kernel<2><<<L.U, 64, 0, st>>>(a, L.Hkv, t0, t1);
    return static_cast<int>(cudaGetLastError());
}

template <int V>
static void launch_q_bits(const Layout &L, const QuantArgs &a, cudaStream_t st) {
    const long long warps = static_cast<long long>(L.U) * a.n_tok;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    switch (a.bits) {
        case 2: quantize_kernel<V, 2><<<grid, 128, 0, st>>>(a, L); break;
        case 3: quantize_kernel<V, 3><<<grid, 128, 0, st>>>(a, L); break;
        default: quantize_kernel<V, 4><<<grid, 128, 0, st>>>(a, L); break;
    }
}

int launch_quantize(const Layout &L, const QuantArgs &a, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L.d == 128) launch_q_bits<4>(L, a, st);
    else launch_q_bits<2>(L, a, st);
    return static_cast<int>(cudaGetLastError());
}

template <int V>
static void launch_dq_bits(const Layout &L, const DequantArgs &a, cudaStream_t st) {
    const long long warps = static_cast<long long>(L.U) * a.n;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    switch (a.bits) {
        case 2: dequant_kernel<V, 2><<<grid, 128, 0, st>>>(a, L); break;
        case 3: dequant_kernel<V, 3><<<grid, 128, 0, st>>>(a, L); break;
        default: dequant_kernel<V, 4><<<grid, 128, 0, st>>>(a, L); break;
    }
}

int launch_dequant(const Layout &L, const DequantArgs &a, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L.d == 128) launch_dq_bits<4>(L, a, st);
    else launch_dq_bits<2>(L, a, st);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace dq
