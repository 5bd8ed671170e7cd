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
//  * Work items: per KV head ("unit"), its chunks of 64 packed tokens (32 at
//    4 bits); the unit's 16-slot tiles of 16-bit sink/recent tokens ride along
//    with its chunks.  A persistent grid of one wave splits the list of all
//    chunks into equal contiguous ranges (stream-K); a CTA walks its range
//    unit by unit, handing chunks to its warps one at a time.
//  * Packed chunks and 16-bit tiles stream HBM -> shared memory with bulk
//    asynchronous copies (cp.async.bulk, completion on an mbarrier), a 2-deep
//    ring per warp.
//  * Codes become mma operands with one AND per code pair: a code m held in a
//    binary16 bit pattern below 2048 is exactly m * 2^-24 (scaled by a
//    per-field power of two, folded into q and into the output rows).
//  * q.K^T and P.V are mma.sync m16n8k16 with fp32 accumulation.  The 8 mma
//    columns are 4 query heads x (hi, lo) binary16 halves of an fp32 operand,
//    adjacent, so each lane owns one head and adds its halves in registers.
//    P' is transposed into the B operand with movmatrix (no shared memory).
//  * Softmax bookkeeping once per chunk; the running max may lag by 2^8, so
//    the accumulators are rescaled only when it grows by more than that.
//  * Each CTA merges its 4 warps and writes one partial per (unit, kind);
//    the last CTA to finish a unit (atomic ticket, no waiting) merges them,
//    rotates the value accumulator back and writes the output.
#include <cuda_runtime.h>

#include <cstdlib>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

constexpr int RTILE = 16;                           // slots per 16-bit work item
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s; a healthy copy takes microseconds
constexpr float RESCALE_SLACK = 8.0f;               // log2 units the running max may lag

struct AttnShape {
    int Hkv, G, D;
    long long qcap;
    int rcap;
};

template <int D, int BK, int BV, bool M16>
struct Cfg {
    static constexpr int CK = BK == 4 ? 32 : 64;  // tokens per packed work item (chunk)
    static constexpr int SUB = 32;                // tokens per softmax step within a chunk
    static constexpr int TILES = SUB / 16;
    static constexpr int ROWK = D * BK / 8;
    static constexpr int PAIRV = 2 * D * BV / 8;
    static constexpr int MB = M16 ? 2 : 4;
    static constexpr int KBYTES = CK * ROWK;
    static constexpr int VBYTES = CK / 2 * PAIRV;
    static constexpr int MBYTES = CK * 2 * MB;
    static constexpr int STAGE = KBYTES + VBYTES + 2 * MBYTES;
    static constexpr int NST = 2;                 // bulk-copy ring depth per warp
    static constexpr int RAWBYTES = 64 * D;       // one 16-slot tile of 16-bit keys + values
    // bytes of one warp's ring: NST stages, or one 16-bit tile if that is larger
    static constexpr int RING = NST * STAGE > RAWBYTES ? NST * STAGE : RAWBYTES;
    static constexpr int NKS = D / 16;
    static constexpr int NMT = D / 16;
    static constexpr int PR = D + 4;  // floats per head in a partial record: acc[D], m, l, 0, 0
    // resident CTAs per SM the kernel is register-limited to (smem allows it)
    static constexpr int MINB = RING <= 10240 ? 4 : (RING <= 14336 ? 3 : 2);
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
    template <int NT>
    __device__ __forceinline__ void update(const float (&lg)[NT], float (&p)[NT]) {
        float mx = lg[0];
#pragma unroll
        for (int k = 1; k < NT; k++) mx = fmaxf(mx, lg[k]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        const bool grow = mx > m + RESCALE_SLACK;  // also true for the first finite logit
        if (__any_sync(FULL, grow)) {
            const float mn = grow ? mx : m;
            const float al = grow ? ex2(m - mn) : 1.f;  // 0 when m was -inf
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
    }
};

// ---- shared memory -----------------------------------------------------------
template <int D, int BK, int BV, bool M16>
struct Smem {
    using C = Cfg<D, BK, BV, M16>;
    float q_raw[2][4][D];      // prepared queries of up to two units at a time
    float q_rot[2][4][D];
    float qsum[2][4], qmu[2][4];
    float merge[4][4][C::PR];  // [warp][head][acc[D], m, l, -, -]
    uint64_t bars[4][C::NST];
    int next_chunk;            // chunks of the current segment handed out so far
    int last;
    alignas(128) uint8_t ring[4][C::RING];  // per warp: stage s at s * STAGE
};

// Global sources of one unit's packed records, and the bulk copy of chunk c
// into a stage, issued by one elected lane without branching the warp.
template <int D, int BK, int BV, bool M16>
struct ChunkSrc {
    const uint8_t *ck, *cv, *mk, *mv;
    __device__ __forceinline__ ChunkSrc(const AttnArgs &a, const AttnShape &sh, int u) {
        using C = Cfg<D, BK, BV, M16>;
        ck = a.codes_k + static_cast<long long>(u) * sh.qcap * C::ROWK;
        cv = a.codes_v + static_cast<long long>(u) * (sh.qcap / 2) * C::PAIRV;
        mk = static_cast<const uint8_t *>(a.meta_k) + static_cast<long long>(u) * sh.qcap * 2 * C::MB;
        mv = static_cast<const uint8_t *>(a.meta_v) + static_cast<long long>(u) * sh.qcap * 2 * C::MB;
    }
    __device__ __forceinline__ void issue(long long c, uint8_t *stage, uint64_t *bar) const {
        using C = Cfg<D, BK, BV, M16>;
        const uint32_t t0 = static_cast<uint32_t>(c) * C::CK;
        const uint32_t sb = smem_u32(stage), br = smem_u32(bar);
        asm volatile(
            "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
            "@p fence.proxy.async.shared::cta;\n"
            "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%11], [%12], %10, [%0];\n}\n" ::"r"(br),
            "r"(C::STAGE), "r"(sb), "l"(ck + static_cast<uint64_t>(t0) * C::ROWK), "r"(C::KBYTES),
            "r"(sb + C::KBYTES), "l"(cv + static_cast<uint64_t>(t0 / 2) * C::PAIRV), "r"(C::VBYTES),
            "r"(sb + C::KBYTES + C::VBYTES), "l"(mk + static_cast<uint64_t>(t0) * 2 * C::MB), "r"(C::MBYTES),
            "r"(sb + C::KBYTES + C::VBYTES + C::MBYTES), "l"(mv + static_cast<uint64_t>(t0) * 2 * C::MB)
            : "memory");
    }
};

// Bulk-copy 16-bit tile r (16 slots: keys then value pairs) of unit u.
template <int D>
__device__ __forceinline__ void issue_raw(const AttnArgs &a, const AttnShape &sh, int u, long long r,
                                          uint8_t *dst, uint64_t *bar) {
    const uint16_t *rk = a.raw_k + (static_cast<long long>(u) * sh.rcap + r * RTILE) * D;
    const uint16_t *rv = a.raw_v + (static_cast<long long>(u) * sh.rcap + r * RTILE) * D;
    mbar_expect_tx(bar, 64 * D);
    bulk_g2s(dst, rk, 32 * D, bar);
    bulk_g2s(dst + 32 * D, rv, 32 * D, bar);
}

// B operand of q.K^T for this lane: column g = head g>>1, half g&1 of the
// (scaled) query.  Lane slot (k-step i, sub, e) holds logical channel
// 16i + 2tig + 8sub + e; `perm` maps it to the channel of q it multiplies.
template <int D, int BK, bool QUANT, bool BF16, typename Perm>
__device__ __forceinline__ void build_qb(const float (*q)[D], uint32_t (&qb)[D / 16][2], Perm perm) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const int h = g >> 1, part = g & 1;
#pragma unroll
    for (int i = 0; i < D / 16; i++) {
#pragma unroll
        for (int sub = 0; sub < 2; sub++) {
            float v0 = q[h][perm(i, tig, sub, 0)], v1 = q[h][perm(i, tig, sub, 1)];
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

// SUB packed tokens already in shared memory -> warp state.  `stg` is the
// stage, `o` the first token of the block within the chunk, `tok0` the token
// index of the block within the unit.
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void process_block(const uint8_t *stg, int o, long long tok0, long long n_q,
                                              const uint32_t (&qb)[D / 16][2], float sk_l2, float qs_l2, float qm_l2,
                                              WarpState<D / 16> &st) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int NKS = C::NKS, NMT = C::NMT, T = C::TILES;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    // q . K^T for the tiles of the block
    float sc[T][4];
#pragma unroll
    for (int t = 0; t < T; t++) {
        constexpr int NW = Slice<D, BK>::NW;
        uint32_t k0[NW], k1[NW];
        load_k_slice<D, BK>(stg + (o + 16 * t + g) * C::ROWK, tig, k0);
        load_k_slice<D, BK>(stg + (o + 16 * t + g + 8) * C::ROWK, tig, k1);
        sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
        for (int i = 0; i < NKS; i++)
            mma_f16(sc[t], extract<BK>(k0, 2 * i), extract<BK>(k1, 2 * i), extract<BK>(k0, 2 * i + 1),
                    extract<BK>(k1, 2 * i + 1), qb[i][0], qb[i][1]);
    }
    // logits of tokens 16t+g (k = 2t) and 16t+g+8 (k = 2t+1) for head tig
    const uint8_t *smk = stg + C::KBYTES + C::VBYTES;
    const uint8_t *smv = smk + C::MBYTES;
    float lg[2 * T];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
            const float2 km = ld_meta(smk, o + 16 * t + g + 8 * hf, M16);
            const float dot = sc[t][2 * hf] + sc[t][2 * hf + 1];
            lg[2 * t + hf] = (km.x * sk_l2) * dot + (km.y * qs_l2 + qm_l2);
        }
    const bool ragged = tok0 + C::SUB > n_q;  // last block of the unit
    if (ragged) {
#pragma unroll
        for (int k = 0; k < 2 * T; k++)
            if (tok0 + 16 * (k >> 1) + g + 8 * (k & 1) >= n_q) lg[k] = -INFINITY;
    }
    float p[2 * T];
    st.template update<2 * T>(lg, p);
    // P . V per tile: A = V^T (channels x tokens), B = (P * s_v) transposed by
    // movmatrix; the offsets o_v accumulate separately (Eq. 9)
    float aos = 0.f;
#pragma unroll
    for (int t = 0; t < T; t++) {
        float2 vm0 = ld_meta(smv, o + 16 * t + g, M16), vm1 = ld_meta(smv, o + 16 * t + g + 8, M16);
        if (ragged) {  // masked tokens have p = 0, but their metadata may be anything
            if (tok0 + 16 * t + g >= n_q) vm0 = make_float2(0.f, 0.f);
            if (tok0 + 16 * t + g + 8 >= n_q) vm1 = make_float2(0.f, 0.f);
        }
        aos += p[2 * t] * vm0.y + p[2 * t + 1] * vm1.y;
        const uint32_t b0 = movmatrix_t(hilo_f16(p[2 * t] * vm0.x));
        const uint32_t b1 = movmatrix_t(hilo_f16(p[2 * t + 1] * vm1.x));
        constexpr int NW = Slice<D, BV>::NW;
        uint32_t v0[NW], v1[NW];
        load_v_slice<D, BV>(stg + C::KBYTES + (o / 2 + 8 * t + tig) * C::PAIRV, g, v0);
        load_v_slice<D, BV>(stg + C::KBYTES + (o / 2 + 8 * t + tig + 4) * C::PAIRV, g, v1);
#pragma unroll
        for (int mi = 0; mi < NMT; mi++)
            mma_f16(st.acc[mi], extract<BV>(v0, 2 * mi), extract<BV>(v0, 2 * mi + 1), extract<BV>(v1, 2 * mi),
                    extract<BV>(v1, 2 * mi + 1), b0, b1);
    }
    st.ao += aos;
}

// One 16-bit tile (16 slots) already in shared memory -> warp state.  Rows are
// read with 16-byte vectors; the resulting channel order is folded into the q
// operand (PermRawK) and into the output rows (raw_v_channel).
template <int D, bool BF16>
__device__ __noinline__ void process_raw(const AttnArgs &a, const uint8_t *tile, long long s0,
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
            if (quant) wp[row] = v * exp2f(static_cast<float>(24 - field_exp(2 * mi + rr, BV))) + st.ao;
            else wp[raw_v_channel<D>(row)] = v;
        }
    if (g == 0) {
        wp[D] = st.m;
        wp[D + 1] = st.l;
    }
}

// owner(x): the CTA whose item range [i*N/G, (i+1)*N/G) holds global item x.
__device__ __forceinline__ int owner(long long x, long long N, int G) {
    return static_cast<int>(((x + 1) * G + N - 1) / N) - 1;
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

// The last CTA of a unit: merge its split records, rotate the value
// accumulator back, normalize and write the output; reset the ticket.
// Records are read in batches of 8 whose loads are all in flight together,
// merged with a running maximum.
template <int D, int PR>
__device__ __noinline__ void combine_unit(const AttnArgs &a, const AttnShape &sh, int u, int n_ctas) {
    constexpr int V = D / 32, NB = 8;
    using VT = typename VecT<V>::T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    const int h = warp;
    if (h < sh.G) {
        const float *pu = a.partials + static_cast<long long>(u) * a.max_slots * 2 * 4 * PR + h * PR;
        const int n_rec = 2 * n_ctas;  // record r: kind r & 1 (0: 16-bit, 1: packed)
        float M = -INFINITY, Lsum = 0.f;
        float accq[V], accr[V];
#pragma unroll
        for (int j = 0; j < V; j++) accq[j] = accr[j] = 0.f;
        for (int r0 = 0; r0 < n_rec; r0 += NB) {
            float mr[NB], lr[NB];
            VT vv[NB];
#pragma unroll
            for (int k = 0; k < NB; k++) {
                const float *p = pu + (r0 + k) * 4 * PR;
                const bool in = r0 + k < n_rec;
                mr[k] = in ? __ldcg(p + D) : -INFINITY;
                lr[k] = in ? __ldcg(p + D + 1) : 0.f;
                vv[k] = in ? __ldcg(reinterpret_cast<const VT *>(p) + lane) : VT{};
            }
            float mb = M;
#pragma unroll
            for (int k = 0; k < NB; k++) mb = fmaxf(mb, mr[k]);
            if (mb == -INFINITY) continue;
            const float al = M == -INFINITY ? 0.f : exp2f(M - mb);
            M = mb;
            Lsum *= al;
#pragma unroll
            for (int j = 0; j < V; j++) {
                accq[j] *= al;
                accr[j] *= al;
            }
#pragma unroll
            for (int k = 0; k < NB; k++) {
                const float w = mr[k] == -INFINITY ? 0.f : exp2f(mr[k] - M);
                Lsum += lr[k] * w;
                if ((r0 + k) & 1) vadd(accq, vv[k], w);
                else vadd(accr, vv[k], w);
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

// Query preparation of unit u into slot qs: warp h takes query head h (raw q,
// rotated or compensated q, sum q, q . mu).
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void prep_query(const AttnArgs &a, const AttnShape &sh, Smem<D, BK, BV, M16> &S, int qs,
                                           int u) {
    constexpr int V = D / 32;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    float xq[V];
    if (h < sh.G) {
        const float *qp = a.q + (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D;
#pragma unroll
        for (int j = 0; j < V; j++) xq[j] = qp[lane * V + j];
    } else {
#pragma unroll
        for (int j = 0; j < V; j++) xq[j] = 0.f;
    }
    float mu[V];
#pragma unroll
    for (int j = 0; j < V; j++) mu[j] = a.mean_k ? a.mean_k[static_cast<long long>(u) * D + lane * V + j] : 0.f;
#pragma unroll
    for (int j = 0; j < V; j++) S.q_raw[qs][h][lane * V + j] = xq[j];
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
            for (int k = 0; k < D; k++) acc += row[k] * S.q_raw[qs][h][k];
            xq[j] = acc;
        }
    }
    float qsum = 0.f, qmu = 0.f;
#pragma unroll
    for (int j = 0; j < V; j++) {
        S.q_rot[qs][h][lane * V + j] = xq[j];
        qsum += xq[j];
        qmu += xq[j] * mu[j];
    }
    qsum = warp_sum(qsum);
    qmu = warp_sum(qmu);
    if (lane == 0) {
        S.qsum[qs][h] = qsum;
        S.qmu[qs][h] = qmu;
    }
}

// Next packed chunk (relative index) for this warp from the segment's shared
// counter, or -1 when the segment's chunks are all handed out.
__device__ __forceinline__ int grab_chunk(int *counter, int n_chunks) {
    uint32_t v = 0;
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n @p atom.shared.add.u32 %0, [%1], 1;\n}\n"
        : "+r"(v)
        : "r"(smem_u32(counter))
        : "memory");
    v = __shfl_sync(FULL, v, 0);  // lane 0 is the elected lane of a full warp
    return static_cast<int>(v) < n_chunks ? static_cast<int>(v) : -1;
}

// Items [s0, s1) of a unit -> packed chunks [q0, q1) and 16-bit tiles [r0, r1):
// a unit's items are its chunks, tile r riding with chunk floor(r * n_qc / n_rt);
// a unit without packed tokens has its tiles as items.
__device__ __forceinline__ void segment_items(const AttnArgs &a, long long s0, long long s1, long long &q0,
                                              long long &q1, long long &r0, long long &r1) {
    if (a.n_qc > 0) {
        q0 = s0;
        q1 = s1;
        r0 = (s0 * a.n_rt + a.n_qc - 1) / a.n_qc;
        r1 = (s1 * a.n_rt + a.n_qc - 1) / a.n_qc;
    } else {
        q0 = q1 = 0;
        r0 = s0;
        r1 = s1;
    }
}

// ---- the kernel ----------------------------------------------------------------
// A CTA walks its item range unit by unit.  In each unit segment, warp 0 first
// runs the segment's 16-bit tiles (if any) while warps 1-3 start on packed
// chunks; chunks are handed out one at a time from a shared counter, so the
// warps finish together.  Each warp streams its chunks through its own 2-deep
// ring of bulk copies.  Loads that later work depends on go first: warp 0's
// first 16-bit tile, then the queries of the CTA's first two units, and only
// then the packed chunks.
template <int D, int BK, int BV, bool M16>
__global__ void __launch_bounds__(128, Cfg<D, BK, BV, M16>::MINB) attn_kernel(AttnArgs a, AttnShape sh) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int PR = C::PR, NKS = C::NKS;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<D, BK, BV, M16> &S = *reinterpret_cast<Smem<D, BK, BV, M16> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3;
    const int G = gridDim.x, i = blockIdx.x;
    const long long N = a.total_items, ipu = a.items_per_unit;
    const long long x0 = static_cast<long long>(i) * N / G, x1 = static_cast<long long>(i + 1) * N / G;
    uint8_t *ring0 = S.ring[warp];
    uint64_t *bars = S.bars[warp];
    const int u_first = static_cast<int>(x0 / ipu), u_lastc = static_cast<int>((x1 - 1) / ipu);

    if (lane == 0) {
        for (int s = 0; s < C::NST; s++) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    uint32_t phase = 0;  // bit s: parity of the next completion of bars[s]
    bool timed_out = false;
    {
        // warp 0: the first segment's first 16-bit tile, before anything else
        long long q0, q1, r0, r1;
        const long long ub = static_cast<long long>(u_first) * ipu;
        segment_items(a, x0 - ub, (x1 < ub + ipu ? x1 : ub + ipu) - ub, q0, q1, r0, r1);
        if (warp == 0 && r0 < r1 && lane == 0) issue_raw<D>(a, sh, u_first, r0, ring0, &bars[0]);
        prep_query<D, BK, BV, M16>(a, sh, S, 0, u_first);
        if (u_lastc > u_first) prep_query<D, BK, BV, M16>(a, sh, S, 1, u_first + 1);
    }

    for (long long x = x0; x < x1;) {
        const int u = static_cast<int>(x / ipu);
        const long long ub = static_cast<long long>(u) * ipu;
        const bool first_seg = x == x0;
        long long q0, q1, r0, r1;
        segment_items(a, x - ub, (x1 < ub + ipu ? x1 : ub + ipu) - ub, q0, q1, r0, r1);
        x = x1 < ub + ipu ? x1 : ub + ipu;
        const int n_chunks = static_cast<int>(q1 - q0);
        const bool raw_warp = warp == 0 && r0 < r1;
        const int qs = (u - u_first) & 1;

        __syncthreads();  // the previous segment is done with the shared state
        if (threadIdx.x == 0) S.next_chunk = 0;
        if (!first_seg && raw_warp && lane == 0) issue_raw<D>(a, sh, u, r0, ring0, &bars[0]);
        if (u - u_first >= 2) prep_query<D, BK, BV, M16>(a, sh, S, qs, u);  // units past the first two
        __syncthreads();

        const ChunkSrc<D, BK, BV, M16> src(a, sh, u);
        int cq0 = -1, cq1 = -1;  // chunk (relative to q0) in flight in stage 0 / 1
        auto start_chunks = [&]() {
            cq0 = grab_chunk(&S.next_chunk, n_chunks);
            if (cq0 >= 0) src.issue(q0 + cq0, S.ring[warp], &bars[0]);
            cq1 = cq0 >= 0 ? grab_chunk(&S.next_chunk, n_chunks) : -1;
            if (cq1 >= 0) src.issue(q0 + cq1, S.ring[warp] + C::STAGE, &bars[1]);
        };
        if (!raw_warp) start_chunks();

        const int first = owner(ub, N, G), last = owner(ub + ipu - 1, N, G);
        float *recs = a.partials + (static_cast<long long>(u) * a.max_slots + (i - first)) * 2 * 4 * PR;
        WarpState<D / 16> st;

        // ---- 16-bit tiles (warp 0): record kind 0 ----
        if (raw_warp) {
            uint32_t qb[NKS][2];
            if (a.raw_bf16) build_qb<D, 2, false, true>(S.q_raw[qs], qb, PermRawK());
            else build_qb<D, 2, false, false>(S.q_raw[qs], qb, PermRawK());
            st.init();
            for (long long r = r0; r < r1; r++) {
                if (!mbar_wait(&bars[0], phase & 1u, WAIT_LIMIT_NS)) timed_out = true;
                phase ^= 1u;
                if (a.raw_bf16) process_raw<D, true>(a, ring0, r * RTILE, qb, st);
                else process_raw<D, false>(a, ring0, r * RTILE, qb, st);
                __syncwarp();
                if (lane == 0 && r + 1 < r1) {
                    fence_proxy_async();
                    issue_raw<D>(a, sh, u, r + 1, ring0, &bars[0]);
                }
            }
            store_state<D, BV>(st, false, recs, PR);
            __syncwarp();
            start_chunks();  // warp 0 joins the packed chunks
        } else if (warp == 0 && lane < 4) {
            recs[lane * PR + D] = -INFINITY;  // no 16-bit tiles in this segment
            recs[lane * PR + D + 1] = 0.f;
        }

        // ---- packed chunks: all warps, handed out one at a time ----
        st.init();
        if (cq0 >= 0) {
            uint32_t qb[NKS][2];
            build_qb<D, BK, true, false>(S.q_rot[qs], qb, PermIdentity());
            const float qs_l2 = a.sm_log2 * S.qsum[qs][tig], qm_l2 = a.sm_log2 * S.qmu[qs][tig];
            const float sk_l2 = a.sm_log2 * 16777216.0f;  // 2^24 undoes the operand scaling
            const long long n_q = a.n_q;
            int s = 0;
            for (;;) {
                const int cur = s ? cq1 : cq0;
                if (cur < 0) break;
                if (!mbar_wait(&bars[s], (phase >> s) & 1u, WAIT_LIMIT_NS)) timed_out = true;
                phase ^= 1u << s;
                const uint8_t *stg = S.ring[warp] + s * C::STAGE;
                const long long tok0 = (q0 + cur) * C::CK;
#pragma unroll 1
                for (int o = 0; o < C::CK; o += C::SUB)
                    process_block<D, BK, BV, M16>(stg, o, tok0 + o, n_q, qb, sk_l2, qs_l2, qm_l2, st);
                __syncwarp();
                const int nxt = grab_chunk(&S.next_chunk, n_chunks);
                if (nxt >= 0) src.issue(q0 + nxt, S.ring[warp] + s * C::STAGE, &bars[s]);
                if (s) cq1 = nxt;
                else cq0 = nxt;
                s ^= 1;
            }
        }
        store_state<D, BV>(st, true, &S.merge[warp][0][0], PR);
        __syncthreads();
        // CTA merge of the 4 warps -> record kind 1
        for (int idx = threadIdx.x; idx < 4 * PR; idx += blockDim.x) {
            const int h = idx / PR, c = idx % PR;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; w++) M = fmaxf(M, S.merge[w][h][D]);
            float v = 0.f;
            if (c == D) {
                v = M;
            } else if (c < D + 2) {
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    const float mw = S.merge[w][h][D];
                    if (mw != -INFINITY) v += S.merge[w][h][c] * exp2f(mw - M);
                }
            }
            recs[4 * PR + idx] = v;
        }

        // ---- ticket: the last CTA of the unit merges the records ----
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int t = atomicAdd(a.counters + u, 1);
            S.last = (t == last - first);
        }
        __syncthreads();
        if (!S.last) continue;
        __threadfence();
        combine_unit<D, PR>(a, sh, u, last - first + 1);
    }
    if (timed_out && lane == 0) atomicOr(a.status, ST_TIMEOUT);
}

// ---- host side -------------------------------------------------------------
template <int D, int BK, int BV, bool M16>
struct Launcher {
    static constexpr int CK = Cfg<D, BK, BV, M16>::CK;
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
    return static_cast<long long>(L.U) * a.max_slots * 2 * 4 * (L.d + 4);
}

int plan_attention(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats) {
    int occ = 0, ck = 0;
    const int e = dispatch(L, [&](auto l) {
        const int r = decltype(l)::prepare();
        occ = decltype(l)::occupancy;
        ck = decltype(l)::CK;
        return r;
    });
    if (e != 0) return e;
    a.n_rt = a.has_raw ? (a.n_raw_slots + RTILE - 1) / RTILE : 0;
    a.raw_all_valid = a.seq_len >= static_cast<long long>(a.n_sink_cfg) + a.n_recent_cfg;
    a.n_qc = (a.n_q + ck - 1) / ck;
    // a unit's items are its packed chunks (its 16-bit tiles ride along with
    // them), or its 16-bit tiles when it has no packed tokens
    a.items_per_unit = a.n_qc > 0 ? a.n_qc : a.n_rt;
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
