// Split-K GQA decode attention over the packed affine cache (sm_103a).
//
// Computes, per sequence b and query head h reading KV head h / G,
//   out_h = sum_t softmax_t(sm_scale * q_h . k^_t) v^_t
// with the affine terms applied after the contraction ("D-Quant: Driftable
// Entropy Coding for KV Cache Quantization", App. A Eq. (7)-(9)):
//   q . k^_t  = s_t * (q . m_t) + o_t * sum_j q_j + q . mu            (Eq. 8)
//   sum_t a_t v^_t = sum_t (a_t s_t) m_t + sum_t a_t o_t               (Eq. 9)
// Keys and values are rotated by the normalized Hadamard matrix Hn
// (Sec. 4.2), so q is rotated once per call and the value accumulator is
// rotated back with Hn (its own inverse) at the end.
//
// Design for GB300:
//  * One CTA = one (unit, item): a contiguous chunk of 16-token tiles of one
//    KV head, or its 16-bit sink/recent slots.  4 warps take tiles round-robin.
//  * Quantized tiles stream HBM -> shared memory with bulk asynchronous copies
//    (cp.async.bulk, completion on an mbarrier), a 4-deep ring per warp.
//  * Codes are turned into mma operands with one AND per code pair: a code m
//    placed in a binary16 bit pattern below 2048 is the exact value m*2^-24
//    (scaled by a per-field power of two, folded into q and into the output).
//  * q.K^T and P.V run on the tensor cores as mma.sync m16n8k16 with fp32
//    accumulation; the 8 mma columns hold 4 query heads x (hi, lo) halves of
//    an fp32 operand split into two binary16 numbers, so no column is wasted
//    and the operand carries ~22 significant bits.
//  * Online softmax per warp, warp partials merged per CTA, split partials
//    merged by the last CTA of each unit (atomic ticket; no spin waits).
#include <cuda_runtime.h>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

constexpr int NST = 4;          // bulk-copy ring depth per warp
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s: a healthy copy takes microseconds

struct AttnShape {
    int Hkv, G, D;
    long long qcap;
    int rcap, rowK, pairV, meta_bytes;
};

template <int D, int BK, int BV, bool M16>
struct TileCfg {
    static constexpr int ROWK = D * BK / 8;
    static constexpr int PAIRV = 2 * D * BV / 8;
    static constexpr int MB = M16 ? 2 : 4;
    static constexpr int KBYTES = 16 * ROWK;
    static constexpr int VBYTES = 8 * PAIRV;
    static constexpr int MBYTES = 16 * 2 * MB;
    static constexpr int STAGE = KBYTES + VBYTES + 2 * MBYTES;
    static constexpr int NKS = D / 16;  // k-steps of q.K^T
    static constexpr int NMT = D / 16;  // m-tiles of P.V
};

// ---- code extraction --------------------------------------------------------
// Register r of a lane's record slice: both 16-bit halves hold code fields
// at the same position; the result is the binary16 pair (m_lo, m_hi) * 2^(E-24).
template <int BITS>
__device__ __forceinline__ uint32_t extract(const uint32_t *w, int r);

template <>
__device__ __forceinline__ uint32_t extract<2>(const uint32_t *w, int r) {
    const uint32_t x = w[r >> 3];
    const int f = r & 7;
    return f <= 4 ? (x & (0x00030003u << (2 * f))) : ((x >> 10) & (0x00030003u << (2 * (f - 5))));
}
template <>
__device__ __forceinline__ uint32_t extract<4>(const uint32_t *w, int r) {
    const uint32_t x = w[r >> 2];
    const int f = r & 3;
    const uint32_t y = (f & 2) ? (x >> 8) : x;
    return y & ((f & 1) ? 0x00F000F0u : 0x000F000Fu);
}
// 3-bit: w[0..1] = 2-bit plane words, w[2] = 1-bit plane word (register r at
// bits r and 16 + r); bit 2 of the code lands two places above the 2-bit field.
template <>
__device__ __forceinline__ uint32_t extract<3>(const uint32_t *w, int r) {
    const uint32_t lo = extract<2>(w, r);
    const int f = r & 7;
    const int pos = (f <= 4 ? 2 * f : 2 * (f - 5)) + 2;
    const int sh = pos - r;
    const uint32_t hb = sh >= 0 ? (w[2] << sh) : (w[2] >> (-sh));
    return lo | (hb & (0x00010001u << pos));
}

// Words of one lane's slice: key row of one token, value pair record.
template <int D, int BITS>
struct Slice {
    static constexpr int NW = BITS == 3 ? 3 : D * BITS / 128;  // words per lane
};

template <int D, int BITS>
__device__ __forceinline__ void load_k_slice(const uint8_t *row, int tig, uint32_t *w) {
    if (BITS == 3) {
        const uint2 lo = *reinterpret_cast<const uint2 *>(row + 8 * tig);
        w[0] = lo.x;
        w[1] = lo.y;
        w[2] = *reinterpret_cast<const uint32_t *>(row + D / 4 + 4 * tig);
    } else if (Slice<D, BITS>::NW == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * tig);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if (Slice<D, BITS>::NW == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + 8 * tig);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t *>(row + 4 * tig);
    }
}
template <int D, int BITS>
__device__ __forceinline__ void load_v_slice(const uint8_t *rec, int g, uint32_t *w) {
    if (BITS == 3) {
        const uint2 lo = *reinterpret_cast<const uint2 *>(rec + 8 * g);
        w[0] = lo.x;
        w[1] = lo.y;
        w[2] = *reinterpret_cast<const uint32_t *>(rec + D / 2 + 4 * g);
    } else if (Slice<D, BITS>::NW == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rec + 16 * g);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if (Slice<D, BITS>::NW == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(rec + 8 * g);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t *>(rec + 4 * g);
    }
}

__device__ __forceinline__ float2 ld_meta(const uint8_t *p, int i, bool m16) {
    if (m16) {
        const uint32_t so = reinterpret_cast<const uint32_t *>(p)[i];
        return make_float2(__half2float(__ushort_as_half(static_cast<uint16_t>(so & 0xffffu))),
                           __half2float(__ushort_as_half(static_cast<uint16_t>(so >> 16))));
    }
    return reinterpret_cast<const float2 *>(p)[i];
}

// ---- online-softmax state of one warp ---------------------------------------
// Lane (g, tig) owns heads h0 = 2*(tig&1), h0+1 for the softmax and, in the
// P.V accumulator, the columns 2*tig, 2*tig+1 (= the same heads, hi or lo half).
template <int NMT>
struct WarpState {
    float m[2], l[2], ao[2];
    float acc[NMT][4];
};

// One 16-token tile: scores sc[4] = D[tok g][cols 2tig,2tig+1], D[tok g+8][...]
// already hi+lo-combined into (head h0, h0+1) for tokens g and g+8, as logits
// in log2 units.  p-values times `vs` (the per-token value scale) become the
// B operand of P.V; `vo` (the per-token value offset) accumulates separately.
template <int NMT, bool RAWBF16>
__device__ __forceinline__ void softmax_tile(WarpState<NMT> &st, float (&lg)[4], const float (&vs)[2],
                                             const float (&vo)[2], uint16_t *pt, uint32_t &pb0,
                                             uint32_t &pb1, bool quant) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    float mx0 = fmaxf(lg[0], lg[2]), mx1 = fmaxf(lg[1], lg[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, o));
    }
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(st.m[0] - mu0), al1 = exp2f(st.m[1] - mu1);
    st.m[0] = mn0;
    st.m[1] = mn1;
    const float p00 = exp2f(lg[0] - mu0), p01 = exp2f(lg[1] - mu1);  // token g
    const float p10 = exp2f(lg[2] - mu0), p11 = exp2f(lg[3] - mu1);  // token g+8
    st.l[0] = st.l[0] * al0 + p00 + p10;
    st.l[1] = st.l[1] * al1 + p01 + p11;
    if (quant) {
        st.ao[0] = st.ao[0] * al0 + p00 * vo[0] + p10 * vo[1];
        st.ao[1] = st.ao[1] * al1 + p01 * vo[0] + p11 * vo[1];
    }
#pragma unroll
    for (int mi = 0; mi < NMT; mi++) {
        st.acc[mi][0] *= al0;
        st.acc[mi][1] *= al1;
        st.acc[mi][2] *= al0;
        st.acc[mi][3] *= al1;
    }
    // P' (times the value scale) as hi/lo 16-bit halves; lanes tig<2 store hi,
    // tig>=2 store lo, into pt[col][tok] (col = 2*tig + {0,1}).
    const float q00 = p00 * vs[0], q01 = p01 * vs[0], q10 = p10 * vs[1], q11 = p11 * vs[1];
    const bool lo_half = tig >= 2;
    uint16_t h00, h01, h10, h11;
    if (RAWBF16 && !quant) {
        __nv_bfloat16 a, b;
        split_bf16(q00, a, b); h00 = __bfloat16_as_ushort(lo_half ? b : a);
        split_bf16(q01, a, b); h01 = __bfloat16_as_ushort(lo_half ? b : a);
        split_bf16(q10, a, b); h10 = __bfloat16_as_ushort(lo_half ? b : a);
        split_bf16(q11, a, b); h11 = __bfloat16_as_ushort(lo_half ? b : a);
    } else {
        __half a, b;
        split_f16(q00, a, b); h00 = __half_as_ushort(lo_half ? b : a);
        split_f16(q01, a, b); h01 = __half_as_ushort(lo_half ? b : a);
        split_f16(q10, a, b); h10 = __half_as_ushort(lo_half ? b : a);
        split_f16(q11, a, b); h11 = __half_as_ushort(lo_half ? b : a);
    }
    constexpr int PS = 24;  // row stride (halves) of pt: 16 tokens + pad
    pt[(2 * tig) * PS + g] = h00;
    pt[(2 * tig + 1) * PS + g] = h01;
    pt[(2 * tig) * PS + g + 8] = h10;
    pt[(2 * tig + 1) * PS + g + 8] = h11;
    __syncwarp();
    pb0 = *reinterpret_cast<const uint32_t *>(pt + g * PS + 2 * tig);
    pb1 = *reinterpret_cast<const uint32_t *>(pt + g * PS + 2 * tig + 8);
    __syncwarp();
}

// ---- the kernel ----------------------------------------------------------------
template <int D, int BK, int BV, bool M16>
__global__ void __launch_bounds__(128) attn_kernel(AttnArgs a, AttnShape sh) {
    using TC = TileCfg<D, BK, BV, M16>;
    constexpr int V = D / 32, NKS = TC::NKS, NMT = TC::NMT;
    constexpr int PS = 24;
    extern __shared__ __align__(128) uint8_t smem[];
    float *q_use = reinterpret_cast<float *>(smem);                  // [4][D]
    float *qconst = q_use + 4 * D;                                   // qsum[4], qmu[4]
    uint64_t *bars = reinterpret_cast<uint64_t *>(qconst + 8);       // [4 warps][NST]
    uint16_t *ptile = reinterpret_cast<uint16_t *>(bars + 4 * NST);  // [4 warps][8][PS]
    uint8_t *stages = reinterpret_cast<uint8_t *>(ptile + 4 * 8 * PS);
    // align stages to 128
    stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(stages) + 127) & ~uintptr_t(127));
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int u = blockIdx.x / a.items, item = blockIdx.x % a.items;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    const bool raw_item = a.has_raw && item == 0;

    // ---- query preparation: warp w handles query head w of this KV head ----
    {
        const int h = warp;
        float x[V];
        if (h < sh.G) {
            const float *qp = a.q + (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D;
#pragma unroll
            for (int j = 0; j < V; j++) x[j] = qp[lane * V + j];
            if (!raw_item) {
                if (a.rot_k == DQ_ROT_HADAMARD) {
                    fwht_warp<V>(x);
#pragma unroll
                    for (int j = 0; j < V; j++) x[j] *= a.hscale;
                } else if (a.rot_k == DQ_ROT_DENSE) {
                    // q~ = T^{-T} q with the caller's fp32 compensation matrix
                    float *xs = q_use + h * D;
#pragma unroll
                    for (int j = 0; j < V; j++) xs[lane * V + j] = x[j];
                    __syncwarp();
                    const float *Qc = a.q_comp + static_cast<long long>(kvh) * D * D;
                    float y[V];
#pragma unroll
                    for (int j = 0; j < V; j++) {
                        float acc = 0.f;
                        const float *row = Qc + static_cast<long long>(lane * V + j) * D;
                        for (int k = 0; k < D; k++) acc += row[k] * xs[k];
                        y[j] = acc;
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < V; j++) x[j] = y[j];
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < V; j++) x[j] = 0.f;
        }
        float qs = 0.f, qm = 0.f;
#pragma unroll
        for (int j = 0; j < V; j++) {
            q_use[h * D + lane * V + j] = x[j];
            qs += x[j];
            if (!raw_item && a.mean_k) qm += x[j] * a.mean_k[static_cast<long long>(u) * D + lane * V + j];
        }
        qs = warp_sum(qs);
        qm = warp_sum(qm);
        if (lane == 0) {
            qconst[h] = qs;
            qconst[4 + h] = qm;
        }
    }
    if (lane == 0) {
        for (int s = 0; s < NST; s++) mbar_init(&bars[warp * NST + s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // B operand of q.K^T: column g = head (g & 3), half (g >> 2).
    uint32_t qb[NKS][2];
    {
        const int hq = g & 3;
        const bool lo_part = (g >> 2) != 0;
#pragma unroll
        for (int i = 0; i < NKS; i++) {
#pragma unroll
            for (int sub = 0; sub < 2; sub++) {
                const int c = 16 * i + 2 * tig + 8 * sub;
                float v0 = q_use[hq * D + c], v1 = q_use[hq * D + c + 1];
                uint16_t e0, e1;
                if (!raw_item) {
                    const float sc = exp2f(static_cast<float>(-field_exp(2 * i + sub, BK)));
                    v0 *= sc;
                    v1 *= sc;
                    __half h0, l0, h1, l1;
                    split_f16(v0, h0, l0);
                    split_f16(v1, h1, l1);
                    e0 = __half_as_ushort(lo_part ? l0 : h0);
                    e1 = __half_as_ushort(lo_part ? l1 : h1);
                } else if (a.raw_bf16) {
                    __nv_bfloat16 h0, l0, h1, l1;
                    split_bf16(v0, h0, l0);
                    split_bf16(v1, h1, l1);
                    e0 = __bfloat16_as_ushort(lo_part ? l0 : h0);
                    e1 = __bfloat16_as_ushort(lo_part ? l1 : h1);
                } else {
                    __half h0, l0, h1, l1;
                    split_f16(v0, h0, l0);
                    split_f16(v1, h1, l1);
                    e0 = __half_as_ushort(lo_part ? l0 : h0);
                    e1 = __half_as_ushort(lo_part ? l1 : h1);
                }
                qb[i][sub] = pack2(e0, e1);
            }
        }
    }
    const float qsum0 = qconst[2 * (tig & 1)], qsum1 = qconst[2 * (tig & 1) + 1];
    const float qmu0 = qconst[4 + 2 * (tig & 1)], qmu1 = qconst[4 + 2 * (tig & 1) + 1];

    WarpState<NMT> st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = st.ao[0] = st.ao[1] = 0.f;
#pragma unroll
    for (int mi = 0; mi < NMT; mi++) st.acc[mi][0] = st.acc[mi][1] = st.acc[mi][2] = st.acc[mi][3] = 0.f;

    uint16_t *pt = ptile + warp * 8 * PS;
    const float two24 = 16777216.0f;

    if (!raw_item) {
        // ---------------- quantized tiles ----------------
        const int chunk = item - a.has_raw;
        const long long t_begin = a.tiles_q * chunk / a.n_split;
        const long long t_end = a.tiles_q * (chunk + 1) / a.n_split;
        const uint8_t *ck = a.codes_k + static_cast<long long>(u) * sh.qcap * TC::ROWK;
        const uint8_t *cv = a.codes_v + static_cast<long long>(u) * (sh.qcap / 2) * TC::PAIRV;
        const uint8_t *mk = static_cast<const uint8_t *>(a.meta_k) + static_cast<long long>(u) * sh.qcap * 2 * TC::MB;
        const uint8_t *mv = static_cast<const uint8_t *>(a.meta_v) + static_cast<long long>(u) * sh.qcap * 2 * TC::MB;
        uint8_t *ring = stages + warp * NST * TC::STAGE;
        uint64_t *wb = bars + warp * NST;
        // this warp's tiles: t_begin + warp, + 4, ...
        const long long my_first = t_begin + warp;
        const long long n_my = my_first < t_end ? (t_end - my_first + 3) / 4 : 0;
        auto issue = [&](long long j) {
            const long long tile = my_first + 4 * j;
            uint8_t *s = ring + (j % NST) * TC::STAGE;
            uint64_t *bar = wb + (j % NST);
            mbar_expect_tx(bar, TC::STAGE);
            bulk_g2s(s, ck + tile * 16 * TC::ROWK, TC::KBYTES, bar);
            bulk_g2s(s + TC::KBYTES, cv + tile * 8 * TC::PAIRV, TC::VBYTES, bar);
            bulk_g2s(s + TC::KBYTES + TC::VBYTES, mk + tile * 16 * 2 * TC::MB, TC::MBYTES, bar);
            bulk_g2s(s + TC::KBYTES + TC::VBYTES + TC::MBYTES, mv + tile * 16 * 2 * TC::MB, TC::MBYTES, bar);
        };
        if (lane == 0) {
            for (long long j = 0; j < n_my && j < NST; j++) issue(j);
        }
        __syncwarp();
        bool timed_out = false;
        for (long long j = 0; j < n_my; j++) {
            const long long tile = my_first + 4 * j;
            const uint8_t *s = ring + (j % NST) * TC::STAGE;
            if (!mbar_wait(wb + (j % NST), static_cast<unsigned>((j / NST) & 1), WAIT_LIMIT_NS)) timed_out = true;
            constexpr int NWK = Slice<D, BK>::NW, NWV = Slice<D, BV>::NW;
            uint32_t kw0[NWK], kw1[NWK], vw0[NWV], vw1[NWV];
            load_k_slice<D, BK>(s + g * TC::ROWK, tig, kw0);
            load_k_slice<D, BK>(s + (g + 8) * TC::ROWK, tig, kw1);
            load_v_slice<D, BV>(s + TC::KBYTES + tig * TC::PAIRV, g, vw0);
            load_v_slice<D, BV>(s + TC::KBYTES + (tig + 4) * TC::PAIRV, g, vw1);
            const uint8_t *smk = s + TC::KBYTES + TC::VBYTES;
            const float2 km0 = ld_meta(smk, g, M16), km1 = ld_meta(smk, g + 8, M16);
            const float2 vm0 = ld_meta(smk + TC::MBYTES, g, M16), vm1 = ld_meta(smk + TC::MBYTES, g + 8, M16);
            __syncwarp();
            if (lane == 0 && j + NST < n_my) {
                fence_proxy_async();
                issue(j + NST);
            }
            // q . K^T
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < NKS; i++) {
                mma_f16(sc, extract<BK>(kw0, 2 * i), extract<BK>(kw1, 2 * i), extract<BK>(kw0, 2 * i + 1),
                        extract<BK>(kw1, 2 * i + 1), qb[i][0], qb[i][1]);
            }
#pragma unroll
            for (int k = 0; k < 4; k++) sc[k] += __shfl_xor_sync(FULL, sc[k], 2);
            const long long tok0 = tile * 16 + g, tok1 = tok0 + 8;
            const bool v0 = tok0 < a.n_q, v1 = tok1 < a.n_q;
            float lg[4];
            lg[0] = v0 ? a.sm_log2 * (km0.x * two24 * sc[0] + (km0.y * qsum0 + qmu0)) : -INFINITY;
            lg[1] = v0 ? a.sm_log2 * (km0.x * two24 * sc[1] + (km0.y * qsum1 + qmu1)) : -INFINITY;
            lg[2] = v1 ? a.sm_log2 * (km1.x * two24 * sc[2] + (km1.y * qsum0 + qmu0)) : -INFINITY;
            lg[3] = v1 ? a.sm_log2 * (km1.x * two24 * sc[3] + (km1.y * qsum1 + qmu1)) : -INFINITY;
            const float vs[2] = {v0 ? vm0.x : 0.f, v1 ? vm1.x : 0.f};
            const float vo[2] = {v0 ? vm0.y : 0.f, v1 ? vm1.y : 0.f};
            uint32_t pb0, pb1;
            softmax_tile<NMT, false>(st, lg, vs, vo, pt, pb0, pb1, true);
            // P . V : A = V^T (channels x tokens), B = P'
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
                mma_f16(st.acc[mi], extract<BV>(vw0, 2 * mi), extract<BV>(vw0, 2 * mi + 1),
                        extract<BV>(vw1, 2 * mi), extract<BV>(vw1, 2 * mi + 1), pb0, pb1);
            }
        }
        if (timed_out && lane == 0) atomicOr(a.status, ST_TIMEOUT);
    } else {
        // ---------------- 16-bit sink / recent slots ----------------
        const uint16_t *rk = a.raw_k + static_cast<long long>(u) * sh.rcap * D;
        const uint16_t *rv = a.raw_v + static_cast<long long>(u) * sh.rcap * D;
        const int n_tiles = (a.n_raw_slots + 15) / 16;
        // Raw slot validity at length seq_len: sink slot s < min(seq_len, n_sink);
        // ring slot n_sink + r holds the latest token t < seq_len with
        // t mod n_recent == r, valid when that token is not itself a sink.
        auto slot_valid = [&](int slot) -> bool {
            if (slot >= a.n_raw_slots) return false;
            if (slot < a.n_sink_cfg) return slot < a.n_sink_eff;
            const long long r = slot - a.n_sink_cfg;
            const long long back = a.seq_len - 1 - r;
            if (back < 0) return false;
            const long long tr = a.seq_len - 1 - (back % a.n_recent_cfg);
            return tr >= a.n_sink_cfg;
        };
        for (int tile = warp; tile < n_tiles; tile += 4) {
            const int s0 = tile * 16;
            const bool sv[2] = {slot_valid(s0 + g), slot_valid(s0 + g + 8)};
            const bool vv[4] = {slot_valid(s0 + 2 * tig), slot_valid(s0 + 2 * tig + 1),
                                slot_valid(s0 + 2 * tig + 8), slot_valid(s0 + 2 * tig + 9)};
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint16_t *k0 = rk + static_cast<long long>(s0 + g) * D;
            const uint16_t *k1 = rk + static_cast<long long>(s0 + g + 8) * D;
#pragma unroll
            for (int i = 0; i < NKS; i++) {
                const int c = 16 * i + 2 * tig;
                const uint32_t a0 = __ldg(reinterpret_cast<const unsigned *>(k0 + c));
                const uint32_t a1 = __ldg(reinterpret_cast<const unsigned *>(k1 + c));
                const uint32_t a2 = __ldg(reinterpret_cast<const unsigned *>(k0 + c + 8));
                const uint32_t a3 = __ldg(reinterpret_cast<const unsigned *>(k1 + c + 8));
                if (a.raw_bf16) mma_bf16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
                else mma_f16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
            }
#pragma unroll
            for (int k = 0; k < 4; k++) sc[k] += __shfl_xor_sync(FULL, sc[k], 2);
            float lg[4];
            lg[0] = sv[0] ? a.sm_log2 * sc[0] : -INFINITY;
            lg[1] = sv[0] ? a.sm_log2 * sc[1] : -INFINITY;
            lg[2] = sv[1] ? a.sm_log2 * sc[2] : -INFINITY;
            lg[3] = sv[1] ? a.sm_log2 * sc[3] : -INFINITY;
            const float one[2] = {1.f, 1.f}, zero[2] = {0.f, 0.f};
            uint32_t pb0, pb1;
            if (a.raw_bf16) softmax_tile<NMT, true>(st, lg, one, zero, pt, pb0, pb1, false);
            else softmax_tile<NMT, false>(st, lg, one, zero, pt, pb0, pb1, false);
            // values: pair-interleaved, A[row ch][k slot] pairs (2tig, 2tig+1)
            const uint32_t *vp0 = reinterpret_cast<const uint32_t *>(rv) + static_cast<long long>(s0 / 2 + tig) * D;
            const uint32_t *vp1 = reinterpret_cast<const uint32_t *>(rv) + static_cast<long long>(s0 / 2 + tig + 4) * D;
            const uint32_t m0 = (vv[0] ? 0x0000ffffu : 0u) | (vv[1] ? 0xffff0000u : 0u);
            const uint32_t m1 = (vv[2] ? 0x0000ffffu : 0u) | (vv[3] ? 0xffff0000u : 0u);
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
                const int c = 16 * mi + g;
                const uint32_t a0 = __ldg(vp0 + c) & m0, a1 = __ldg(vp0 + c + 8) & m0;
                const uint32_t a2 = __ldg(vp1 + c) & m1, a3 = __ldg(vp1 + c + 8) & m1;
                if (a.raw_bf16) mma_bf16(st.acc[mi], a0, a1, a2, a3, pb0, pb1);
                else mma_f16(st.acc[mi], a0, a1, a2, a3, pb0, pb1);
            }
        }
    }

    // ---- warp partial: reduce l, ao over g; combine hi/lo columns ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        st.l[0] += __shfl_xor_sync(FULL, st.l[0], o);
        st.l[1] += __shfl_xor_sync(FULL, st.l[1], o);
        st.ao[0] += __shfl_xor_sync(FULL, st.ao[0], o);
        st.ao[1] += __shfl_xor_sync(FULL, st.ao[1], o);
    }
#pragma unroll
    for (int mi = 0; mi < NMT; mi++)
#pragma unroll
        for (int k = 0; k < 4; k++) st.acc[mi][k] += __shfl_xor_sync(FULL, st.acc[mi][k], 2);

    __syncthreads();  // stages no longer needed: reuse as the merge area
    float *mrg = reinterpret_cast<float *>(stages);  // [4 warps][4 heads][D + 2]
    constexpr int PR = D + 2;
    {
        float *wp = mrg + warp * 4 * PR;
        const int h0 = 2 * (tig & 1);
        if (tig < 2) {
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
#pragma unroll
                    for (int rr = 0; rr < 2; rr++) {
                        const int c = 16 * mi + 8 * rr + g;
                        float v = st.acc[mi][2 * rr + hh];
                        if (!raw_item) v = v * exp2f(static_cast<float>(24 - field_exp(2 * mi + rr, BV))) + st.ao[hh];
                        wp[(h0 + hh) * PR + 2 + c] = v;
                    }
                }
            }
            if (g == 0) {
                wp[h0 * PR] = st.m[0];
                wp[(h0 + 1) * PR] = st.m[1];
                wp[h0 * PR + 1] = st.l[0];
                wp[(h0 + 1) * PR + 1] = st.l[1];
            }
        }
    }
    __syncthreads();
    // CTA partial: thread t handles (head t / 32, channels ...)
    float *part = a.partials + (static_cast<long long>(u) * a.items + item) * 4 * PR;
    for (int idx = threadIdx.x; idx < 4 * PR; idx += blockDim.x) {
        const int h = idx / PR, c = idx % PR;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; w++) M = fmaxf(M, mrg[(w * 4 + h) * PR]);
        float v;
        if (c == 0) {
            v = M;
        } else {
            v = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                const float mw = mrg[(w * 4 + h) * PR];
                if (mw != -INFINITY) v += mrg[(w * 4 + h) * PR + c] * exp2f(mw - M);
            }
        }
        part[idx] = v;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int t = atomicAdd(a.counters + u, 1);
        s_last = (t == a.items - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of the unit: merge the split partials, un-rotate, write ----
    {
        const int h = warp;
        if (h < sh.G) {
            const float *pu = a.partials + static_cast<long long>(u) * a.items * 4 * PR;
            float M = -INFINITY;
            for (int it = 0; it < a.items; it++) M = fmaxf(M, __ldcg(pu + (it * 4 + h) * PR));
            float Lsum = 0.f;
            float accq[V], accr[V];
#pragma unroll
            for (int j = 0; j < V; j++) accq[j] = accr[j] = 0.f;
            for (int it = 0; it < a.items; it++) {
                const float *p = pu + (it * 4 + h) * PR;
                const float mi = __ldcg(p);
                if (mi == -INFINITY) continue;
                const float wgt = exp2f(mi - M);
                Lsum += __ldcg(p + 1) * wgt;
                const bool is_raw = a.has_raw && it == 0;
#pragma unroll
                for (int j = 0; j < V; j++) {
                    const float v = __ldcg(p + 2 + lane * V + j) * wgt;
                    if (is_raw) accr[j] += v;
                    else accq[j] += v;
                }
            }
            if (a.rot_v == DQ_ROT_HADAMARD) {
                fwht_warp<V>(accq);
#pragma unroll
                for (int j = 0; j < V; j++) accq[j] *= a.hscale;
            }
            const float inv = 1.f / Lsum;
            const long long ob = (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D;
#pragma unroll
            for (int j = 0; j < V; j++) {
                const float y = (accq[j] + accr[j]) * inv;
                const long long oi = ob + lane * V + j;
                if (a.out_dtype == DQ_F32) reinterpret_cast<float *>(a.out)[oi] = y;
                else if (a.out_dtype == DQ_F16) reinterpret_cast<__half *>(a.out)[oi] = __float2half_rn(y);
                else reinterpret_cast<__nv_bfloat16 *>(a.out)[oi] = __float2bfloat16_rn(y);
            }
        }
        if (threadIdx.x == 0) a.counters[u] = 0;
    }
}

// ---- host side -------------------------------------------------------------
template <int D, int BK, int BV, bool M16>
static size_t smem_for() {
    using TC = TileCfg<D, BK, BV, M16>;
    size_t head = 4 * D * 4 + 8 * 4 + 4 * NST * 8 + 4 * 8 * 24 * 2;
    head = (head + 127) / 128 * 128 + 128;
    size_t ring = static_cast<size_t>(4) * NST * TC::STAGE;
    size_t merge = static_cast<size_t>(4) * 4 * (D + 2) * 4;
    return head + (ring > merge ? ring : merge);
}

template <int D, int BK, int BV, bool M16>
static int launch_t(const Layout &L, const AttnArgs &a, void *stream) {
    AttnShape sh{L.Hkv, L.G, L.d, L.qcap, L.rcap, L.rowK, L.pairV, L.meta_bytes};
    const size_t smem = smem_for<D, BK, BV, M16>();
    auto kern = attn_kernel<D, BK, BV, M16>;
    // the attribute is a property of the kernel, set once (also keeps it out of
    // stream capture after the first call)
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return static_cast<int>(e);
        attr_done = true;
    }
    const unsigned grid = static_cast<unsigned>(L.U) * static_cast<unsigned>(a.items);
    kern<<<grid, 128, smem, static_cast<cudaStream_t>(stream)>>>(a, sh);
    return static_cast<int>(cudaGetLastError());
}

template <int D, bool M16>
static int launch_bits(const Layout &L, const AttnArgs &a, void *stream) {
    if (L.bits_k == 2 && L.bits_v == 2) return launch_t<D, 2, 2, M16>(L, a, stream);
    if (L.bits_k == 4 && L.bits_v == 4) return launch_t<D, 4, 4, M16>(L, a, stream);
    if (D == 128 && L.bits_k == 3 && L.bits_v == 3) return launch_t<D == 128 ? 128 : 128, 3, 3, M16>(L, a, stream);
    return static_cast<int>(cudaErrorInvalidValue);
}

int launch_attention(const Layout &L, const AttnArgs &a, int, void *stream) {
    const bool m16 = L.meta_bytes == 2;
    if (L.d == 128) return m16 ? launch_bits<128, true>(L, a, stream) : launch_bits<128, false>(L, a, stream);
    return m16 ? launch_bits<64, true>(L, a, stream) : launch_bits<64, false>(L, a, stream);
}

size_t attention_smem_bytes(const Layout &L) {
    (void)L;
    return smem_for<128, 4, 4, false>();
}

}  // namespace dq
