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
//  * Work items: per KV head ("unit"), its 16-slot tiles of 16-bit sink/recent
//    tokens followed by its 64-token chunks of packed tokens.  A persistent
//    grid of one wave splits the list of all items into equal contiguous
//    ranges (stream-K); a CTA walks its range unit by unit.
//  * Packed chunks stream HBM -> shared memory with bulk asynchronous copies
//    (cp.async.bulk, completion on an mbarrier), a 2-deep ring per warp.
//  * Codes become mma operands with one AND per code pair: a code m held in a
//    binary16 bit pattern below 2048 is exactly m * 2^-24 (scaled by a
//    per-field power of two, folded into q and into the output rows).
//  * q.K^T and P.V are mma.sync m16n8k16 with fp32 accumulation.  The 8 mma
//    columns are 4 query heads x (hi, lo) binary16 halves of an fp32 operand,
//    adjacent, so each lane owns one head and adds its halves in registers.
//    P' is transposed into the B operand with movmatrix (no shared memory).
//  * Softmax bookkeeping (max, rescale) once per 64 tokens.
//  * Each CTA merges its 4 warps and writes one partial per (unit, kind);
//    the last CTA to finish a unit (atomic ticket, no waiting) merges them,
//    rotates the value accumulator back and writes the output.
#include <cuda_runtime.h>

#include <cstdlib>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

constexpr int CHUNK = 64;                           // tokens per packed work item
constexpr int RTILE = 16;                           // slots per 16-bit work item
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s; a healthy copy takes microseconds

struct AttnShape {
    int Hkv, G, D;
    long long qcap;
    int rcap;
};

template <int D, int BK, int BV, bool M16>
struct Cfg {
    static constexpr int ROWK = D * BK / 8;
    static constexpr int PAIRV = 2 * D * BV / 8;
    static constexpr int MB = M16 ? 2 : 4;
    static constexpr int KBYTES = CHUNK * ROWK;
    static constexpr int VBYTES = CHUNK / 2 * PAIRV;
    static constexpr int MBYTES = CHUNK * 2 * MB;
    static constexpr int STAGE = KBYTES + VBYTES + 2 * MBYTES;
    static constexpr int NST = 2;
    static constexpr int NKS = D / 16;
    static constexpr int NMT = D / 16;
    static constexpr int PR = D + 2;  // floats per head in a partial record
    // resident CTAs per SM the kernel is register-limited to (smem allows it)
    static constexpr int MINB = STAGE <= 5120 ? 4 : (STAGE <= 7168 ? 3 : 2);
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
    template <int NT>
    __device__ __forceinline__ void update(const float (&lg)[NT], float (&p)[NT]) {
        float mx = lg[0];
#pragma unroll
        for (int k = 1; k < NT; k++) mx = fmaxf(mx, lg[k]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        const float mn = fmaxf(m, mx);
        const float mu = mn == -INFINITY ? 0.f : mn;
        const float al = exp2f(m - mu);
        m = mn;
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NT; k++) {
            p[k] = exp2f(lg[k] - mu);
            sum += p[k];
        }
        l = l * al + sum;
        ao *= al;
        if (__any_sync(FULL, al != 1.f)) {
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
                acc[mi][0] *= al;
                acc[mi][1] *= al;
                acc[mi][2] *= al;
                acc[mi][3] *= al;
            }
        }
    }
};

// ---- shared memory -----------------------------------------------------------
template <int D, int BK, int BV, bool M16>
struct Smem {
    using C = Cfg<D, BK, BV, M16>;
    float q_raw[4][D];
    float q_rot[4][D];
    float qsum[4], qmu[4];
    float merge[4][4][C::PR];  // [warp][head][m, l, acc[D]]
    uint64_t bars[4][C::NST];
    int last;
    alignas(128) uint8_t ring[4][C::NST][C::STAGE];
};

// Bulk-copy one 64-token chunk of unit u into a stage.
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void issue_chunk(const AttnArgs &a, const AttnShape &sh, int u, long long c,
                                            uint8_t *stage, uint64_t *bar) {
    using C = Cfg<D, BK, BV, M16>;
    const long long t0 = c * CHUNK;
    const uint8_t *ck = a.codes_k + (static_cast<long long>(u) * sh.qcap + t0) * C::ROWK;
    const uint8_t *cv = a.codes_v + (static_cast<long long>(u) * (sh.qcap / 2) + t0 / 2) * C::PAIRV;
    const uint8_t *mk = static_cast<const uint8_t *>(a.meta_k) + (static_cast<long long>(u) * sh.qcap + t0) * 2 * C::MB;
    const uint8_t *mv = static_cast<const uint8_t *>(a.meta_v) + (static_cast<long long>(u) * sh.qcap + t0) * 2 * C::MB;
    mbar_expect_tx(bar, C::STAGE);
    bulk_g2s(stage, ck, C::KBYTES, bar);
    bulk_g2s(stage + C::KBYTES, cv, C::VBYTES, bar);
    bulk_g2s(stage + C::KBYTES + C::VBYTES, mk, C::MBYTES, bar);
    bulk_g2s(stage + C::KBYTES + C::VBYTES + C::MBYTES, mv, C::MBYTES, bar);
}

// B operand of q.K^T for this lane: column g = head g>>1, half g&1 of the
// (scaled) query; channels 16i + 2tig + {0,1} and +8.
template <int D, int BK, bool QUANT, bool BF16>
__device__ __forceinline__ void build_qb(const float (*q)[D], uint32_t (&qb)[D / 16][2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const int h = g >> 1, part = g & 1;
#pragma unroll
    for (int i = 0; i < D / 16; i++) {
#pragma unroll
        for (int sub = 0; sub < 2; sub++) {
            const int c = 16 * i + 2 * tig + 8 * sub;
            float v0 = q[h][c], v1 = q[h][c + 1];
            if (QUANT) {
                const float sc = exp2f(static_cast<float>(-field_exp(2 * i + sub, BK)));
                v0 *= sc;
                v1 *= sc;
            }
            const uint32_t w0 = BF16 ? hilo_bf16(v0) : hilo_f16(v0);
            const uint32_t w1 = BF16 ? hilo_bf16(v1) : hilo_f16(v1);
            const uint16_t e0 = static_cast<uint16_t>(part ? (w0 >> 16) : (w0 & 0xffffu));
            const uint16_t e1 = static_cast<uint16_t>(part ? (w1 >> 16) : (w1 & 0xffffu));
            qb[i][sub] = pack2(e0, e1);
        }
    }
}

// ---- packed chunks of one unit: this warp takes chunks c0 + warp, + 4, ... -----
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void quant_part(const AttnArgs &a, const AttnShape &sh, Smem<D, BK, BV, M16> &S, int u,
                                           long long c0, long long c1, WarpState<D / 16> &st) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int NKS = C::NKS, NMT = C::NMT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    uint32_t qb[NKS][2];
    build_qb<D, BK, true, false>(S.q_rot, qb);
    const float qs_l2 = a.sm_log2 * S.qsum[tig], qm_l2 = a.sm_log2 * S.qmu[tig];
    const float sk_l2 = a.sm_log2 * 16777216.0f;  // 2^24 undoes the operand scaling
    const long long first = c0 + warp;
    const long long n = first < c1 ? (c1 - first + 3) / 4 : 0;
    uint64_t *bars = S.bars[warp];
    if (lane == 0)
        for (long long j = 0; j < n && j < C::NST; j++)
            issue_chunk<D, BK, BV, M16>(a, sh, u, first + 4 * j, S.ring[warp][j], &bars[j]);
    __syncwarp();
    bool timed_out = false;
    for (long long j = 0; j < n; j++) {
        const long long c = first + 4 * j;
        const int s = static_cast<int>(j % C::NST);
        const uint8_t *stg = S.ring[warp][s];
        if (!mbar_wait(&bars[s], static_cast<unsigned>((j / C::NST) & 1), WAIT_LIMIT_NS)) timed_out = true;
        // q . K^T for the 4 tiles of the chunk
        float sc[4][4];
#pragma unroll
        for (int t = 0; t < 4; t++) {
            constexpr int NW = Slice<D, BK>::NW;
            uint32_t k0[NW], k1[NW];
            load_k_slice<D, BK>(stg + (16 * t + g) * C::ROWK, tig, k0);
            load_k_slice<D, BK>(stg + (16 * t + g + 8) * C::ROWK, tig, k1);
            sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
            for (int i = 0; i < NKS; i++)
                mma_f16(sc[t], extract<BK>(k0, 2 * i), extract<BK>(k1, 2 * i), extract<BK>(k0, 2 * i + 1),
                        extract<BK>(k1, 2 * i + 1), qb[i][0], qb[i][1]);
        }
        // logits of tokens 16t+g (k = 2t) and 16t+g+8 (k = 2t+1) for head tig
        const uint8_t *smk = stg + C::KBYTES + C::VBYTES;
        const uint8_t *smv = smk + C::MBYTES;
        float lg[8];
#pragma unroll
        for (int t = 0; t < 4; t++)
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {
                const float2 km = ld_meta(smk, 16 * t + g + 8 * hf, M16);
                const float dot = sc[t][2 * hf] + sc[t][2 * hf + 1];
                lg[2 * t + hf] = (km.x * sk_l2) * dot + (km.y * qs_l2 + qm_l2);
            }
        const long long tok0 = c * CHUNK;
        const bool ragged = tok0 + CHUNK > a.n_q;  // last chunk of the unit
        if (ragged) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (tok0 + 16 * (k >> 1) + g + 8 * (k & 1) >= a.n_q) lg[k] = -INFINITY;
        }
        float p[8];
        st.template update<8>(lg, p);
        // P . V per tile: A = V^T (channels x tokens), B = (P * s_v) transposed
        // by movmatrix; the offsets o_v accumulate separately (Eq. 9)
        float aos = 0.f;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            float2 vm0 = ld_meta(smv, 16 * t + g, M16), vm1 = ld_meta(smv, 16 * t + g + 8, M16);
            if (ragged) {  // masked tokens have p = 0, but their metadata may be anything
                if (tok0 + 16 * t + g >= a.n_q) vm0 = make_float2(0.f, 0.f);
                if (tok0 + 16 * t + g + 8 >= a.n_q) vm1 = make_float2(0.f, 0.f);
            }
            aos += p[2 * t] * vm0.y + p[2 * t + 1] * vm1.y;
            const uint32_t b0 = movmatrix_t(hilo_f16(p[2 * t] * vm0.x));
            const uint32_t b1 = movmatrix_t(hilo_f16(p[2 * t + 1] * vm1.x));
            constexpr int NW = Slice<D, BV>::NW;
            uint32_t v0[NW], v1[NW];
            load_v_slice<D, BV>(stg + C::KBYTES + (8 * t + tig) * C::PAIRV, g, v0);
            load_v_slice<D, BV>(stg + C::KBYTES + (8 * t + tig + 4) * C::PAIRV, g, v1);
#pragma unroll
            for (int mi = 0; mi < NMT; mi++)
                mma_f16(st.acc[mi], extract<BV>(v0, 2 * mi), extract<BV>(v0, 2 * mi + 1), extract<BV>(v1, 2 * mi),
                        extract<BV>(v1, 2 * mi + 1), b0, b1);
        }
        st.ao += aos;
        __syncwarp();
        if (lane == 0 && j + C::NST < n) {
            fence_proxy_async();
            issue_chunk<D, BK, BV, M16>(a, sh, u, first + 4 * (j + C::NST), S.ring[warp][s], &bars[s]);
        }
    }
    if (timed_out && lane == 0) atomicOr(a.status, ST_TIMEOUT);
}

// ---- 16-bit sink/recent slots of one unit: this warp takes tiles t0 + warp, + 4 --
template <int D, bool BF16>
__device__ __forceinline__ void raw_part(const AttnArgs &a, const AttnShape &sh, const float (*q_raw)[D], int u,
                                         int t0, int t1, WarpState<D / 16> &st) {
    constexpr int NKS = D / 16, NMT = D / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    uint32_t qb[NKS][2];
    build_qb<D, 2, false, BF16>(q_raw, qb);
    const uint16_t *rk = a.raw_k + static_cast<long long>(u) * sh.rcap * D;
    const uint32_t *rv = reinterpret_cast<const uint32_t *>(a.raw_v + static_cast<long long>(u) * sh.rcap * D);
    // slot validity at length seq_len: sink slot s < min(seq_len, n_sink); ring
    // slot n_sink + r holds the latest token t < seq_len with t mod n_recent == r,
    // valid when that token is not itself a sink
    auto valid = [&](int slot) -> bool {
        if (slot >= a.n_raw_slots) return false;
        if (slot < a.n_sink_cfg) return slot < a.n_sink_eff;
        const long long r = slot - a.n_sink_cfg;
        const long long back = a.seq_len - 1 - r;
        if (back < 0) return false;
        const long long tr = a.seq_len - 1 - (back % a.n_recent_cfg);
        return tr >= a.n_sink_cfg;
    };
    for (int tile = t0 + warp; tile < t1; tile += 4) {
        const int s0 = tile * RTILE;
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
            if (BF16) mma_bf16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
            else mma_f16(sc, a0, a1, a2, a3, qb[i][0], qb[i][1]);
        }
        float lg[2];
        lg[0] = valid(s0 + g) ? a.sm_log2 * (sc[0] + sc[1]) : -INFINITY;
        lg[1] = valid(s0 + g + 8) ? a.sm_log2 * (sc[2] + sc[3]) : -INFINITY;
        float p[2];
        st.template update<2>(lg, p);
        const uint32_t b0 = movmatrix_t(BF16 ? hilo_bf16(p[0]) : hilo_f16(p[0]));
        const uint32_t b1 = movmatrix_t(BF16 ? hilo_bf16(p[1]) : hilo_f16(p[1]));
        // values: pair-interleaved; zero the halves of invalid slots (their bits
        // may be anything, and 0 * NaN would poison the accumulator)
        const uint32_t m0 = (valid(s0 + 2 * tig) ? 0x0000ffffu : 0u) | (valid(s0 + 2 * tig + 1) ? 0xffff0000u : 0u);
        const uint32_t m1 =
            (valid(s0 + 2 * tig + 8) ? 0x0000ffffu : 0u) | (valid(s0 + 2 * tig + 9) ? 0xffff0000u : 0u);
        const uint32_t *vp0 = rv + static_cast<long long>(s0 / 2 + tig) * D;
        const uint32_t *vp1 = rv + static_cast<long long>(s0 / 2 + tig + 4) * D;
#pragma unroll
        for (int mi = 0; mi < NMT; mi++) {
            const int c = 16 * mi + g;
            const uint32_t a0 = __ldg(vp0 + c) & m0, a1 = __ldg(vp0 + c + 8) & m0;
            const uint32_t a2 = __ldg(vp1 + c) & m1, a3 = __ldg(vp1 + c + 8) & m1;
            if (BF16) mma_bf16(st.acc[mi], a0, a1, a2, a3, b0, b1);
            else mma_f16(st.acc[mi], a0, a1, a2, a3, b0, b1);
        }
    }
}

// Warp state -> smem merge area (head tig), then CTA merge -> global record.
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void write_record(Smem<D, BK, BV, M16> &S, WarpState<D / 16> &st, bool quant,
                                             float *rec) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int NMT = C::NMT, PR = C::PR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        st.l += __shfl_xor_sync(FULL, st.l, o);
        st.ao += __shfl_xor_sync(FULL, st.ao, o);
    }
    float *wp = &S.merge[warp][tig][0];
#pragma unroll
    for (int mi = 0; mi < NMT; mi++)
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int c = 16 * mi + 8 * rr + g;
            float v = st.acc[mi][2 * rr] + st.acc[mi][2 * rr + 1];
            if (quant) v = v * exp2f(static_cast<float>(24 - field_exp(2 * mi + rr, BV))) + st.ao;
            wp[2 + c] = v;
        }
    if (g == 0) {
        wp[0] = st.m;
        wp[1] = st.l;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 4 * PR; idx += blockDim.x) {
        const int h = idx / PR, c = idx % PR;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; w++) M = fmaxf(M, S.merge[w][h][0]);
        float v;
        if (c == 0) {
            v = M;
        } else {
            v = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                const float mw = S.merge[w][h][0];
                if (mw != -INFINITY) v += S.merge[w][h][c] * exp2f(mw - M);
            }
        }
        rec[idx] = v;
    }
    __syncthreads();
}

__device__ __forceinline__ void write_empty(float *rec, int PR) {
    if (threadIdx.x < 4) {
        rec[threadIdx.x * PR] = -INFINITY;
        rec[threadIdx.x * PR + 1] = 0.f;
    }
}

// owner(x): the CTA whose item range [i*N/G, (i+1)*N/G) holds global item x.
__device__ __forceinline__ int owner(long long x, long long N, int G) {
    return static_cast<int>(((x + 1) * G + N - 1) / N) - 1;
}

// ---- the kernel ----------------------------------------------------------------
template <int D, int BK, int BV, bool M16>
__global__ void __launch_bounds__(128, Cfg<D, BK, BV, M16>::MINB) attn_kernel(AttnArgs a, AttnShape sh) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int V = D / 32, PR = C::PR;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<D, BK, BV, M16> &S = *reinterpret_cast<Smem<D, BK, BV, M16> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, i = blockIdx.x;
    const long long N = a.total_items, ipu = a.items_per_unit;
    const long long x0 = static_cast<long long>(i) * N / G, x1 = static_cast<long long>(i + 1) * N / G;

    if (lane == 0) {
        for (int s = 0; s < C::NST; s++) mbar_init(&S.bars[warp][s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    for (long long x = x0; x < x1;) {
        const int u = static_cast<int>(x / ipu);
        const long long ub = static_cast<long long>(u) * ipu;
        const long long s0 = x - ub, s1 = (x1 < ub + ipu ? x1 : ub + ipu) - ub;
        x = ub + s1;
        const int b = u / sh.Hkv, kvh = u % sh.Hkv;

        // ---- query preparation: warp h handles query head h of this KV head ----
        __syncthreads();
        {
            const int h = warp;
            float xq[V];
            if (h < sh.G) {
                const float *qp = a.q + (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D;
#pragma unroll
                for (int j = 0; j < V; j++) xq[j] = qp[lane * V + j];
            } else {
#pragma unroll
                for (int j = 0; j < V; j++) xq[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < V; j++) S.q_raw[h][lane * V + j] = xq[j];
            if (a.rot_k == DQ_ROT_HADAMARD) {
                fwht_warp<V>(xq);
#pragma unroll
                for (int j = 0; j < V; j++) xq[j] *= a.hscale;
            } else if (a.rot_k == DQ_ROT_DENSE) {
                // q~ = T^{-T} q with the caller's fp32 compensation matrix
                __syncwarp();
                const float *Qc = a.q_comp + static_cast<long long>(kvh) * D * D;
#pragma unroll
                for (int j = 0; j < V; j++) {
                    float acc = 0.f;
                    const float *row = Qc + static_cast<long long>(lane * V + j) * D;
                    for (int k = 0; k < D; k++) acc += row[k] * S.q_raw[h][k];
                    xq[j] = acc;
                }
            }
            float qs = 0.f, qm = 0.f;
#pragma unroll
            for (int j = 0; j < V; j++) {
                S.q_rot[h][lane * V + j] = xq[j];
                qs += xq[j];
                if (a.mean_k) qm += xq[j] * a.mean_k[static_cast<long long>(u) * D + lane * V + j];
            }
            qs = warp_sum(qs);
            qm = warp_sum(qm);
            if (lane == 0) {
                S.qsum[h] = qs;
                S.qmu[h] = qm;
            }
        }
        __syncthreads();

        const int first = owner(ub, N, G), last = owner(ub + ipu - 1, N, G);
        float *recs = a.partials + (static_cast<long long>(u) * a.max_slots + (i - first)) * 2 * 4 * PR;
        // ---- 16-bit slots: items [0, n_rt) of the unit ----
        const long long r0 = s0, r1 = s1 < a.n_rt ? s1 : a.n_rt;
        if (r0 < r1) {
            WarpState<D / 16> st;
            st.init();
            if (a.raw_bf16) raw_part<D, true>(a, sh, S.q_raw, u, static_cast<int>(r0), static_cast<int>(r1), st);
            else raw_part<D, false>(a, sh, S.q_raw, u, static_cast<int>(r0), static_cast<int>(r1), st);
            write_record<D, BK, BV, M16>(S, st, false, recs);
        } else {
            write_empty(recs, PR);
        }
        // ---- packed chunks: items [n_rt, ipu) ----
        const long long q0 = (s0 > a.n_rt ? s0 : a.n_rt) - a.n_rt, q1 = s1 - a.n_rt;
        if (q0 < q1) {
            WarpState<D / 16> st;
            st.init();
            quant_part<D, BK, BV, M16>(a, sh, S, u, q0, q1, st);
            write_record<D, BK, BV, M16>(S, st, true, recs + 4 * PR);
            // the ring restarts at stage 0 for the next segment: re-arm the barriers
            if (lane == 0) {
                for (int s = 0; s < C::NST; s++) {
                    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(&S.bars[warp][s])));
                    mbar_init(&S.bars[warp][s], 1);
                }
                fence_mbar_init();
            }
            __syncwarp();
        } else {
            write_empty(recs + 4 * PR, PR);
        }

        // ---- ticket: the last CTA of the unit merges its records ----
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int t = atomicAdd(a.counters + u, 1);
            S.last = (t == last - first);
        }
        __syncthreads();
        if (!S.last) continue;
        __threadfence();
        {
            const int h = warp;
            if (h < sh.G) {
                const float *pu = a.partials + static_cast<long long>(u) * a.max_slots * 2 * 4 * PR;
                const int n_rec = 2 * (last - first + 1);
                float M = -INFINITY;
                for (int r = 0; r < n_rec; r++) M = fmaxf(M, __ldcg(pu + (r * 4 + h) * PR));
                float Lsum = 0.f;
                float accq[V], accr[V];
#pragma unroll
                for (int j = 0; j < V; j++) accq[j] = accr[j] = 0.f;
                for (int r = 0; r < n_rec; r++) {
                    const float *p = pu + (r * 4 + h) * PR;
                    const float mr = __ldcg(p);
                    if (mr == -INFINITY) continue;
                    const float wgt = exp2f(mr - M);
                    Lsum += __ldcg(p + 1) * wgt;
                    const bool is_raw = (r & 1) == 0;
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
}

// ---- host side -------------------------------------------------------------
template <int D, int BK, int BV, bool M16>
struct Launcher {
    static int occupancy;  // resident CTAs per SM, set on first use
    static size_t smem() { return sizeof(Smem<D, BK, BV, M16>); }
    static int prepare() {
        if (occupancy > 0) return 0;
        auto kern = attn_kernel<D, BK, BV, M16>;
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem()));
        if (e != cudaSuccess) return static_cast<int>(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 128, smem());
        if (e != cudaSuccess) return static_cast<int>(e);
        occupancy = occ > 0 ? occ : 1;
        return 0;
    }
    static int launch(const AttnArgs &a, const AttnShape &sh, void *stream) {
        attn_kernel<D, BK, BV, M16><<<a.grid, 128, smem(), static_cast<cudaStream_t>(stream)>>>(a, sh);
        return static_cast<int>(cudaGetLastError());
    }
};
template <int D, int BK, int BV, bool M16>
int Launcher<D, BK, BV, M16>::occupancy = 0;

template <int D, bool M16, typename F>
static int dispatch_bits(const Layout &L, F &&f) {
    if (L.bits_k == 2 && L.bits_v == 2) return f(Launcher<D, 2, 2, M16>());
    if (L.bits_k == 4 && L.bits_v == 4) return f(Launcher<D, 4, 4, M16>());
    if (L.bits_k == 3 && L.bits_v == 3) return f(Launcher<128, 3, 3, M16>());
    return static_cast<int>(cudaErrorInvalidValue);
}

template <typename F>
static int dispatch(const Layout &L, F &&f) {
    const bool m16 = L.meta_bytes == 2;
    if (L.d == 128) return m16 ? dispatch_bits<128, true>(L, f) : dispatch_bits<128, false>(L, f);
    return m16 ? dispatch_bits<64, true>(L, f) : dispatch_bits<64, false>(L, f);
}

long long attention_partial_floats(const Layout &L, const AttnArgs &a) {
    return static_cast<long long>(L.U) * a.max_slots * 2 * 4 * (L.d + 2);
}

int plan_attention(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats) {
    int occ = 0;
    const int e = dispatch(L, [&](auto l) {
        const int r = decltype(l)::prepare();
        occ = decltype(l)::occupancy;
        return r;
    });
    if (e != 0) return e;
    a.n_rt = a.has_raw ? (a.n_raw_slots + RTILE - 1) / RTILE : 0;
    a.n_qc = (a.n_q + CHUNK - 1) / CHUNK;
    a.items_per_unit = a.n_rt + a.n_qc;
    a.total_items = static_cast<long long>(L.U) * a.items_per_unit;
    long long G = static_cast<long long>(num_sms) * occ;
    if (const char *env = std::getenv("DQ_ATTN_GRID")) G = std::atoll(env);
    if (G > a.total_items) G = a.total_items;
    if (G < 1) G = 1;
    for (;;) {
        // CTAs touching one unit: at most ceil(ipu / floor(N/G)) + 1
        const long long per = a.total_items / G;
        a.max_slots = static_cast<int>((a.items_per_unit + per - 1) / per + 1);
        a.grid = static_cast<int>(G);
        if (attention_partial_floats(L, a) <= cap_floats || G == 1) break;
        G = G * 3 / 4;  // narrow the grid until the partials fit the workspace
        if (G < 1) G = 1;
    }
    return attention_partial_floats(L, a) <= cap_floats ? 0 : static_cast<int>(cudaErrorMemoryAllocation);
}

int launch_attention(const Layout &L, const AttnArgs &a, int, void *stream) {
    AttnShape sh{L.Hkv, L.G, L.d, L.qcap, L.rcap};
    return dispatch(L, [&](auto l) { return decltype(l)::launch(a, sh, stream); });
}

size_t attention_smem_bytes(const Layout &L) {
    size_t s = 0;
    dispatch(L, [&](auto l) {
        s = decltype(l)::smem();
        return 0;
    });
    return s;
}

}  // namespace dq
