// Device code shared by the decode-attention kernels (sm_103a): record slices,
// code-to-operand extraction, the warp's online softmax, 16-bit tiles and the
// split-state layout.  Included by the attention translation units only.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

constexpr float RESCALE_SLACK = 8.0f;  // log2 units the running max may lag

// Unit geometry of an attention launch (unit = one sequence's KV head).
struct AttnShape {
    int U, Hkv, G, D;
    long long qcap;
    int rcap;
};

// ---- code extraction --------------------------------------------------------
// Register r of a lane's record slice: both 16-bit halves hold code fields at
// the same position; the result is the binary16 pair (m0, m1) * 2^(E-24).
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
// bits bit1_pos(r) and 16 + bit1_pos(r)); bit 2 of the code lands two places
// above the 2-bit field.  The plane's permutation gives the 16 registers of a
// slice five distinct shifts (0, -1, -10, -11, +6, +5 with 0 free), which the
// compiler computes once per slice.
template <>
__device__ __forceinline__ uint32_t extract<3>(const uint32_t *w, int r) {
    const uint32_t lo = extract<2>(w, r);
    const int f = r & 7;
    const int pos = (f <= 4 ? 2 * f : 2 * (f - 5)) + 2;
    const int sh = pos - bit1_pos(r);
    const uint32_t hb = sh >= 0 ? (w[2] << sh) : (w[2] >> (-sh));
    return lo | (hb & (0x00010001u << pos));
}

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
        const __half2 so = reinterpret_cast<const __half2 *>(p)[i];
        return __half22float2(so);
    }
    return reinterpret_cast<const float2 *>(p)[i];
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// (hi, lo) binary16 / bfloat16 halves of x, hi in the low 16 bits.
__device__ __forceinline__ uint32_t hilo_f16(float x) {
    const __half h = __float2half_rn(x);
    const __half l = __float2half_rn(x - __half2float(h));
    return pack2(__half_as_ushort(h), __half_as_ushort(l));
}
__device__ __forceinline__ uint32_t hilo_bf16(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    return pack2(__bfloat16_as_ushort(h), __bfloat16_as_ushort(l));
}

// ---- online softmax of one warp; lane (g, tig) owns query head tig --------------
// The running max m may lag the true maximum by up to RESCALE_SLACK (log2
// units): probabilities are exp2(logit - m) <= 2^RESCALE_SLACK, and the
// accumulators are rescaled only when a logit exceeds m by more than that.
template <int NMT>
struct WarpState {
    float m, l, ao;
    float acc[NMT][4];  // [m-tile]: (ch g, hi), (ch g, lo), (ch g+8, hi), (ch g+8, lo)
    __device__ __forceinline__ void init() {
        m = -INFINITY;
        l = ao = 0.f;
#pragma unroll
        for (int mi = 0; mi < NMT; mi++) acc[mi][0] = acc[mi][1] = acc[mi][2] = acc[mi][3] = 0.f;
    }
    // logits (log2 units) of NT tokens held by this lane -> probabilities
    // returns the factor the accumulators were scaled by (1 if they were not)
    template <int NT>
    __device__ __forceinline__ float update(const float (&lg)[NT], float (&p)[NT]) {
        float mx = lg[0];
#pragma unroll
        for (int k = 1; k < NT; k++) mx = fmaxf(mx, lg[k]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        const bool grow = mx > m + RESCALE_SLACK;  // also true for the first finite logit
        float al = 1.f;
        if (__any_sync(FULL, grow)) {
            const float mn = grow ? mx : m;
            al = grow ? ex2(m - mn) : 1.f;  // 0 when m was -inf
            m = mn;
            l *= al;
            ao *= al;
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
                acc[mi][0] *= al;
                acc[mi][1] *= al;
                acc[mi][2] *= al;
                acc[mi][3] *= al;
            }
        }
        const float mu = m == -INFINITY ? 0.f : m;
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NT; k++) {
            p[k] = ex2(lg[k] - mu);
            sum += p[k];
        }
        l += sum;
        return al;
    }
};
// Channel of a key record / of q that lane slot (i, tig, sub, e) stands for.
struct PermIdentity {
    __device__ __forceinline__ int operator()(int i, int tig, int sub, int e) const {
        return 16 * i + 2 * tig + 8 * sub + e;
    }
};
// 16-bit key rows are read with 16-byte vectors: lane tig takes channels
// 32j + 8tig .. +7 of each row, j = i/2; register 2(i&1)+sub of vector j holds
// channels 32j + 8tig + 4(i&1) + 2sub + {0, 1}.
struct PermRawK {
    __device__ __forceinline__ int operator()(int i, int tig, int sub, int e) const {
        return 32 * (i >> 1) + 8 * tig + 4 * (i & 1) + 2 * sub + e;
    }
};
// 16-bit value pairs are read with 16-byte vectors: lane g takes channels
// (D/8)g .. (D/8)g + D/8 - 1; P.V row 16mi + 8h + g (m-tile mi, half h) is
// the channel (D/8)g + 2mi + h.
template <int D>
__device__ __forceinline__ int raw_v_channel(int row) {
    const int g = row & 7, h = (row >> 3) & 1, mi = row >> 4;
    return (D / 8) * g + 2 * mi + h;
}

__device__ __forceinline__ uint32_t vec_word(const uint4 &v, int r) {
    return r == 0 ? v.x : (r == 1 ? v.y : (r == 2 ? v.z : v.w));
}
// One 16-bit tile (16 slots) already in shared memory -> warp state.  Rows are
// read with 16-byte vectors; the resulting channel order is folded into the q
// operand (PermRawK) and into the output rows (raw_v_channel).
template <int D, bool BF16>
__device__ __forceinline__ void process_raw(const AttnArgs &a, const uint8_t *tile, long long s0,
                                         const uint32_t (&qb)[D / 16][2], WarpState<D / 16> &st) {
    constexpr int NKS = D / 16, NMT = D / 16, NV = D / 32;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    // slot validity at length seq_len: sink slot s < min(seq_len, n_sink); ring
    // slot n_sink + r holds the latest token t < seq_len with t mod n_recent == r,
    // valid when that token is not itself a sink
    auto valid = [&](long long slot) -> bool {
        if (slot >= a.n_raw_slots) return false;
        if (a.raw_all_valid) return true;
        if (slot < a.n_sink_cfg) return slot < a.n_sink_eff;
        const long long r = slot - a.n_sink_cfg;
        const long long back = a.seq_len - 1 - r;
        if (back < 0) return false;
        const long long tr = a.seq_len - 1 - (back % a.n_recent_cfg);
        return tr >= a.n_sink_cfg;
    };
    const uint8_t *rowA = tile + g * D * 2, *rowB = tile + (g + 8) * D * 2;
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NV; j++) {
        const uint4 kA = *reinterpret_cast<const uint4 *>(rowA + 64 * j + 16 * tig);
        const uint4 kB = *reinterpret_cast<const uint4 *>(rowB + 64 * j + 16 * tig);
#pragma unroll
        for (int ii = 0; ii < 2; ii++) {
            const int i = 2 * j + ii, r = 2 * ii;
            if (i >= NKS) break;
            const uint32_t a0 = vec_word(kA, r), a1 = vec_word(kB, r);
            const uint32_t a2 = vec_word(kA, r + 1), a3 = vec_word(kB, r + 1);
            if (BF16) mma_bf16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
            else mma_f16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
        }
    }
    float lg[2];
    lg[0] = valid(s0 + g) ? a.sm_log2 * (sc[0] + sc[1]) : -INFINITY;
    lg[1] = valid(s0 + g + 8) ? a.sm_log2 * (sc[2] + sc[3]) : -INFINITY;
    float p[2];
    st.template update<2>(lg, p);
    const uint32_t b0 = movmatrix_t(BF16 ? hilo_bf16(p[0]) : hilo_f16(p[0]));
    const uint32_t b1 = movmatrix_t(BF16 ? hilo_bf16(p[1]) : hilo_f16(p[1]));
    // zero the halves of invalid slots (their bits may be anything, and
    // 0 * NaN would poison the accumulator)
    const uint32_t m0 = (valid(s0 + 2 * tig) ? 0x0000ffffu : 0u) | (valid(s0 + 2 * tig + 1) ? 0xffff0000u : 0u);
    const uint32_t m1 = (valid(s0 + 2 * tig + 8) ? 0x0000ffffu : 0u) | (valid(s0 + 2 * tig + 9) ? 0xffff0000u : 0u);
    const uint8_t *pA = tile + 32 * D + tig * D * 4 + (D / 8) * g * 4;
    const uint8_t *pB = tile + 32 * D + (tig + 4) * D * 4 + (D / 8) * g * 4;
    uint4 vA[NV], vB[NV];
#pragma unroll
    for (int j = 0; j < NV; j++) {
        vA[j] = *reinterpret_cast<const uint4 *>(pA + 16 * j);
        vB[j] = *reinterpret_cast<const uint4 *>(pB + 16 * j);
    }
#pragma unroll
    for (int mi = 0; mi < NMT; mi++) {
        const int k0 = 2 * mi, k1 = 2 * mi + 1;  // channel (D/8)g + k of this lane's vectors
        const uint32_t a0 = vec_word(vA[k0 >> 2], k0 & 3) & m0, a1 = vec_word(vA[k1 >> 2], k1 & 3) & m0;
        const uint32_t a2 = vec_word(vB[k0 >> 2], k0 & 3) & m1, a3 = vec_word(vB[k1 >> 2], k1 & 3) & m1;
        if (BF16) mma_bf16(st.acc[mi], a0, a1, a2, a3, b0, b1);
        else mma_f16(st.acc[mi], a0, a1, a2, a3, b0, b1);
    }
}

// Warp state -> [acc[D], m, l] of head tig at `dst` (stride PR per head).
// Packed tokens: undo the operand scaling and add the value offsets; 16-bit
// tokens: put each row back at its channel.
template <int D, int BV>
__device__ __forceinline__ void store_state(WarpState<D / 16> &st, bool quant, float *dst, int PR) {
    constexpr int NMT = D / 16;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        st.l += __shfl_xor_sync(FULL, st.l, o);
        st.ao += __shfl_xor_sync(FULL, st.ao, o);
    }
    float *wp = dst + tig * PR;
#pragma unroll
    for (int mi = 0; mi < NMT; mi++)
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int row = 16 * mi + 8 * rr + g;
            const float v = st.acc[mi][2 * rr] + st.acc[mi][2 * rr + 1];
            if (quant) wp[row] = v * pow2i(24 - field_exp(2 * mi + rr, BV)) + st.ao;
            else wp[raw_v_channel<D>(row)] = v;
        }
    if (g == 0) {
        wp[D] = st.m;
        wp[D + 1] = st.l;
    }
}

// owner(x): the CTA whose item range [i*N/G, (i+1)*N/G) holds global item x,
// i.e. the largest c with c N < (x + 1) G.  Estimated in fp32 and settled with
// exact 64-bit products, so no 64-bit division is needed (0 <= x < N).
__device__ __forceinline__ int owner(long long x, long long N, int G) {
    const long long t = (x + 1) * G;
    int c = static_cast<int>(__fdividef(static_cast<float>(t), static_cast<float>(N)));
    c = c < 0 ? 0 : (c > G - 1 ? G - 1 : c);
    while (c > 0 && static_cast<long long>(c) * N >= t) --c;
    while (c + 1 < G && static_cast<long long>(c + 1) * N < t) ++c;
    return c;
}

template <int V>
struct VecT;
template <>
struct VecT<4> {
    using T = float4;
};
template <>
struct VecT<2> {
    using T = float2;
};
__device__ __forceinline__ void vadd(float (&acc)[4], const float4 &v, float w) {
    acc[0] += v.x * w; acc[1] += v.y * w; acc[2] += v.z * w; acc[3] += v.w * w;
}
__device__ __forceinline__ void vadd(float (&acc)[2], const float2 &v, float w) {
    acc[0] += v.x * w; acc[1] += v.y * w;
}


}  // namespace dq
