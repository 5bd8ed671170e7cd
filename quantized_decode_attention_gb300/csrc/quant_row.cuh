// One token row of the affine quantizer (keys or values), shared by the
// quantize kernel and the fused decode step.  See quant_affine.cu for the
// method and its sources.
#pragma once

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
// The global inputs of token pos0 + i of unit u, lane l holding channels
// l*V .. l*V+V-1: the values as fp32, the 16-bit bits a raw region keeps, and
// the key channel mean (zeros when the row has none).  Split from the
// arithmetic so that a caller can issue these loads early.
// ---------------------------------------------------------------------------
template <int V>
struct RowIn {
    float x[V], mu[V];
    uint16_t r[V];
};

template <int V>
__device__ __forceinline__ void load_row(const QuantArgs &a, int u, long long i, RowIn<V> &in) {
    constexpr int D = 32 * V;
    const int lane = threadIdx.x & 31;
    const long long base = (static_cast<long long>(u) * a.n_tok + i) * D;
    const long long esz = a.in_dtype == 0 ? 4 : 2;
    const bool okx = in_buf(static_cast<const char *>(a.x) + base * esz, D * esz, a.x, a.sz_x, a.status);
    const bool okm = a.use_mean && in_buf(a.mean + static_cast<long long>(u) * D, D * 4, a.mean, a.sz_mean, a.status);
#pragma unroll
    for (int j = 0; j < V; j++) {
        in.x[j] = okx ? ld_in(a.x, base + lane * V + j, a.in_dtype) : 0.f;
        in.r[j] = okx ? raw16_of(a.x, base + lane * V + j, a.in_dtype) : 0;
        in.mu[j] = okm ? a.mean[static_cast<long long>(u) * D + lane * V + j] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// Token pos0 + i of unit u from its loaded inputs: the 16-bit region copy
// (sinks and the latest n_recent tokens, stored as given), then (past the
// sinks) rotation, mean removal, the min/max or clipped grid, fp16 s and o,
// codes and the packed record.  One warp; xs is D floats of the warp's shared
// memory.
// ---------------------------------------------------------------------------
template <int V, int BITS>
__device__ __forceinline__ void quantize_loaded_row(const QuantArgs &a, const RowGeom &L, int u, long long i,
                                                    const RowIn<V> &in, float *xs) {
    constexpr int D = 32 * V;
    const int lane = threadIdx.x & 31;
    const long long t = a.pos0 + i;
    const int kvh = u % L.Hkv;

    float x[V];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < V; j++) {
        x[j] = in.x[j];
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
            long long off = a.is_key ? static_cast<long long>(raw_slot) * D + c
                                     : (static_cast<long long>(raw_slot >> 1) * D + c) * 2 + (raw_slot & 1);
            if (in_buf(a.raw + ub + off, 2, a.raw, a.sz_raw, a.status)) a.raw[ub + off] = in.r[j];
        }
    }
    if (t < L.n_sink) return;
    const long long slot = t - L.n_sink;

    rotate_row<V>(x, a.rot, a.hscale, a.T ? a.T + static_cast<long long>(kvh) * D * D : nullptr, xs);
    if (a.use_mean) {
#pragma unroll
        for (int j = 0; j < V; j++) x[j] = __fsub_rn(x[j], in.mu[j]);
    }

    // grid
    constexpr int LV = 1 << BITS;
    float lo = 0.f, hi = 0.f, s, o;
    if (a.quest_c > 0.0f) {
        // QuEST grid ("WUSH-KV", evaluation): symmetric about zero, step
        // c_b * RMS.  The sum of squares runs over the lane's channels in
        // order, then across lanes by xor butterfly (16, 8, 4, 2, 1), each
        // step one rounded fp32 operation; the RMS divides by d (a power of
        // two, exact) and takes the correctly rounded square root.
        float ss = __fmul_rn(x[0], x[0]);
#pragma unroll
        for (int j = 1; j < V; j++) ss = __fadd_rn(ss, __fmul_rn(x[j], x[j]));
#pragma unroll
        for (int k = 16; k >= 1; k >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(FULL, ss, k));
        const float rms = __fsqrt_rn(__fdiv_rn(ss, static_cast<float>(D)));
        s = __fmul_rn(a.quest_c, rms);
        if (a.meta_f16) s = __half2float(__float2half_rn(s));
        o = -__fmul_rn(static_cast<float>(LV - 1) * 0.5f, s);
        if (a.meta_f16) o = __half2float(__float2half_rn(o));
    } else if (a.clip > 0.0f) {
        // order statistics by rank (ties broken by channel index)
#pragma unroll
        for (int j = 0; j < V; j++) xs[lane * V + j] = x[j];
        __syncwarp();
        float vlo0 = 0.f, vlo1 = 0.f, vhi0 = 0.f, vhi1 = 0.f;
        int have = 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int c = lane * V + j;
            const float xv = x[j];
            int rank = 0;
            for (int k = 0; k < D; k++) {
                const float y = xs[k];
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
    if (a.quest_c <= 0.0f) {
        s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(LV - 1));
        o = lo;
        if (a.meta_f16) {
            s = __half2float(__float2half_rn(s));
            o = __half2float(__float2half_rn(o));
        }
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
            uint32_t *mp = reinterpret_cast<uint32_t *>(a.meta) + ms;
            if (in_buf(mp, 4, a.meta, a.sz_meta, a.status)) *mp = so;
        } else {
            float2 *mp = reinterpret_cast<float2 *>(a.meta) + ms;
            if (in_buf(mp, 8, a.meta, a.sz_meta, a.status)) *mp = make_float2(s, o);
        }
    }

    // pack: each code ORs its bits into its record word in the warp's scratch
    // (free again), then the record's words go out, one lane each (keys a
    // whole row, values this token's 16-bit half of its pair record)
    constexpr int WK = Rec<D, BITS>::K_WORDS, WV = Rec<D, BITS>::V_WORDS;
    uint32_t *pw = reinterpret_cast<uint32_t *>(xs);
    const int nwords = a.is_key ? WK : WV;
    const int e = static_cast<int>(slot & 1);  // values: the token's half of its pair record
    __syncwarp();
    if (lane < nwords) pw[lane] = 0u;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane * V + j;
        const int idx = a.is_key ? k_idx(c, D) : v_idx(c, D);
        const int half = a.is_key ? (c & 1) : e;
        if (BITS == 3) {
            const int wlo = (a.is_key ? 1 : 2) * D * 2 / 32;  // 2-bit plane words come first
            atomicOr(&pw[idx / 8], (m[j] & 3u) << (16 * half + 2 * (idx % 8)));
            atomicOr(&pw[wlo + idx / 16], ((m[j] >> 2) & 1u) << (16 * half + bit1_pos(idx % 16)));
        } else {
            constexpr int F = 16 / BITS;
            atomicOr(&pw[idx / F], m[j] << (16 * half + BITS * (idx % F)));
        }
    }
    __syncwarp();
    if (a.is_key) {
        uint32_t *row = reinterpret_cast<uint32_t *>(a.codes + ms * L.rowK);
        if (lane < WK && in_buf(row + lane, 4, a.codes, a.sz_codes, a.status)) row[lane] = pw[lane];
    } else {
        uint16_t *rec = reinterpret_cast<uint16_t *>(
            a.codes + (static_cast<long long>(u) * (L.qcap / 2) + slot / 2) * L.pairV);
        if (lane < WV && in_buf(rec + 2 * lane + e, 2, a.codes, a.sz_codes, a.status))
            rec[2 * lane + e] = static_cast<uint16_t>(pw[lane] >> (16 * e));
    }
    __syncwarp();  // the scratch is the caller's again
}

// Token pos0 + i of unit u: load_row, then quantize_loaded_row.
template <int V, int BITS>
__device__ __forceinline__ void quantize_row(const QuantArgs &a, const RowGeom &L, int u, long long i, float *xs) {
    RowIn<V> in;
    load_row<V>(a, u, i, in);
    quantize_loaded_row<V, BITS>(a, L, u, i, in, xs);
}

}  // namespace dq
