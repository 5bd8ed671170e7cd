// Split-K GQA decode attention over the packed affine cache with 2-, 3- or
// 4-bit codes (sm_103a).
//
// Per sequence b and query head h reading KV head h / G it computes
//   out_h = sum_t softmax_t(sm_scale * q_h . k^_t) v^_t,
// with the affine terms applied after the contractions ("D-Quant: Driftable
// Entropy Coding for KV Cache Quantization", App. A Eq. (7)-(9)):
//   q . k^_t = s_t (q . m_t) + o_t sum_j q_j + q . mu                   (Eq. 8)
//   sum_t a_t v^_t = sum_t (a_t s_t) m_t + sum_t a_t o_t                 (Eq. 9)
// Keys and values carry the normalized Hadamard rotation (Sec. 4.2), so q is
// rotated once and the value accumulator is rotated back at the end; the
// n_sink first and n_recent latest tokens are exact 16-bit slots.
//
// Design for GB300:
//  * One CTA of 16 warps per SM.  The packed chunks (up to TPC 16-token tiles
//    of one unit) of all (sequence, KV head) units form one list; the grid
//    splits it into equal contiguous ranges and a CTA's packed warps take its
//    chunks one at a time from a shared counter.  The CTA prepares the query
//    operands of its (at most four) units once, shared by all its warps; a warp
//    that moves on to the next unit folds its state into that unit's shared
//    accumulator.
//  * Every packed warp streams its range through its own ring of shared-memory
//    slots: one elected lane issues the bulk copies (cp.async.bulk, completion
//    on the slot's mbarrier) of a chunk of up to TPC tiles -- key records,
//    value pair records, key and value metadata -- and refills the slot as
//    soon as the warp is done with it.  No warp waits on another.
//  * q . K^T and P . V run on binary16 tensor-core operands (mma.sync
//    m16n8k16, fp32 accumulation): a code m held below bit 10 of a 16-bit half
//    is exactly m * 2^-24 (binary16 subnormals and the first binade share one
//    spacing), times a per-field power of two folded into q and into the output
//    rows, so one AND turns two codes into an operand register.  q and P' = p s_v
//    enter as (hi, lo) binary16 halves (about 22 significant bits) in the 8 mma
//    columns = 4 heads x (hi, lo); P' is transposed into the B operand by
//    movmatrix.  (8-bit tensor operands of mma.sync are not native on sm_103a:
//    they are widened to binary16 in registers, which costs more than the codes
//    they would save.)
//  * The sink and recent 16-bit tiles go to the CTA's last warp, which has a
//    ring of its own.
//  * Online softmax with a lagging maximum: accumulators are rescaled only when
//    a logit exceeds the running maximum by more than 2^8, and the cross-lane
//    reduction runs only then.
//  * Each CTA merges its warps' states per unit and publishes one record per
//    (unit, CTA); whoever publishes a unit's last record (a CTA or a 16-bit-tile
//    warp, counted with an atomic ticket) merges the unit's records, rotates
//    the value accumulator back, normalizes and casts.  No block waits for
//    another.
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "dq_internal.h"
#include "quant_row.cuh"

namespace dq {
namespace {

static_assert(ST_OOB == 32u, "in_buf latches ST_OOB");

constexpr int AF_WPB = 16;                       // warps per CTA
constexpr int AF_NUS = 4;                        // units a CTA's packed range may touch
constexpr int AF_NSR = 2;                        // ring slots of the 16-bit-tile warp
constexpr int AF_NUR = 3;                        // units the 16-bit-tile warp's range may touch
constexpr int AF_RTILE = 16;                     // slots per 16-bit tile
constexpr uint64_t AF_WAIT_NS = 2000000000ull;   // 2 s; a healthy copy lands in microseconds

template <int D, int BITS, bool M16>
struct ACfg {
    static constexpr int TPC = BITS == 2 ? 4 : (BITS == 3 ? 3 : 2);  // 16-token tiles per chunk (what fits)
    static constexpr int NS = 2;                    // ring slots per packed warp
    static constexpr int ROWK = D * BITS / 8;       // bytes per key record
    static constexpr int PAIRV = 2 * D * BITS / 8;  // bytes per value pair record
    static constexpr int MB = M16 ? 2 : 4;          // bytes per metadata value
    static constexpr int CT = 16 * TPC;             // tokens per chunk
    static constexpr int VOFF = CT * ROWK;
    static constexpr int MKOFF = VOFF + CT / 2 * PAIRV;
    static constexpr int MVOFF = MKOFF + CT * 2 * MB;
    static constexpr int SLOT = (MVOFF + CT * 2 * MB + 127) / 128 * 128;
    static constexpr int RSLOT = 64 * D;            // a 16-slot tile of 16-bit keys and values
    static constexpr int NMT = D / 16;              // m-tiles of P . V
    static constexpr int PR = D + 4;                // floats per head in a state record
    static constexpr int RING_P = AF_WPB * NS * SLOT;
    static constexpr int RING_R = (AF_WPB - 1) * NS * SLOT + AF_NSR * RSLOT;
    static constexpr int RING = RING_P > RING_R ? RING_P : RING_R;
    static_assert(AF_WPB * 4 * PR * 4 <= RING, "the warps' final states overlay the rings");
};

template <int D, int BITS, bool M16>
struct ASmem {
    using C = ACfg<D, BITS, M16>;
    uint16_t qh[AF_NUS][2][4][D + 8];  // packed keys: (hi, lo) halves of the prepared q, rows padded by 8
    float qsc[AF_NUS][4][4];           // per head: sum q and q . mu (log2 units)
    uint16_t rqh[AF_NUR][2][4][D + 8]; // 16-bit-tile warp: (hi, lo) halves of its units' raw q
    float uacc[AF_NUS][4][C::PR];      // per unit: states folded in by warps on their second move
    float save[AF_WPB][4][C::PR];      // a warp's first finished unit segment
    int ulock[AF_NUS];
    int fin_u[AF_WPB];                 // unit of a warp's final state (-1: none)
    int save_u[AF_WPB];                // unit of a warp's saved state (-1: none)
    int done_u[AF_NUS + AF_NUR];       // units whose last record this CTA published (-1: none)
    int next;                          // next chunk of the CTA's range
    uint64_t full[AF_WPB][C::NS];
    uint64_t rfull[AF_NSR];
    alignas(128) uint8_t ring[C::RING];
};

// The query of unit u, head h, as this lane's V channels (lane l: channels
// lV .. lV+V-1) and the key channel mean; loaded before any cache copy is
// issued so that these loads do not queue behind the copies.
template <int D>
struct QLoad {
    float x[D / 32], mu[D / 32];
};
template <int D>
__device__ __forceinline__ void load_unit_query(const AttnArgs &a, const AttnShape &sh, int u, int h, QLoad<D> &in) {
    constexpr int V = D / 32;
    const int lane = threadIdx.x & 31;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    const long long qo = (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D + lane * V;
    const bool okq = h < sh.G && in_buf(a.q + qo - lane * V, D * 4, a.q, a.sz_q, a.status);
    const bool okm = a.mean_k && in_buf(a.mean_k + static_cast<long long>(u) * D, D * 4, a.mean_k, a.sz_mean_k,
                                        a.status);
#pragma unroll
    for (int j = 0; j < V; j++) {
        in.x[j] = okq ? __ldg(a.q + qo + j) : 0.f;
        in.mu[j] = okm ? __ldg(a.mean_k + static_cast<long long>(u) * D + lane * V + j) : 0.f;
        if (a.rot_k == DQ_ROT_DENSE && a.q_tilde) in.x[j] = okq ? __ldg(a.q_tilde + qo + j) : 0.f;
    }
}

// Query operands of unit u for head h into unit slot i (one warp per head):
// q rotated (Hadamard), compensated (dense key transform) or as is, scaled by
// 2^-E for the code field E that channel c meets in the key operand, as (hi,
// lo) binary16 halves; sum q and q . mu for the fold of the affine code (Eq. 8).
template <int D, int BITS, bool M16>
__device__ void prep_unit(const AttnArgs &a, const AttnShape &sh, ASmem<D, BITS, M16> &S, int i, int u, int h,
                          QLoad<D> &in) {
    constexpr int V = D / 32;
    const int lane = threadIdx.x & 31;
    float *x = in.x;
    if (a.rot_k == DQ_ROT_HADAMARD) {
        fwht_warp<V>(in.x);
#pragma unroll
        for (int j = 0; j < V; j++) x[j] *= a.hscale;
    } else if (a.rot_k == DQ_ROT_DENSE && !a.q_tilde) {
        // q~ = T^{-T} q with the caller's fp32 compensation matrix, summed over k
        // in order (as the compensation kernel does); the rows of this warp's
        // head go through its unit slot's accumulator rows as scratch
        float *scr = &S.uacc[i][h][0];
        __syncwarp();
#pragma unroll
        for (int j = 0; j < V; j++) scr[lane * V + j] = x[j];
        __syncwarp();
        const float *Qc = a.q_comp + static_cast<long long>(u % sh.Hkv) * D * D;
        const bool okc = in_buf(Qc, static_cast<long long>(D) * D * 4, a.q_comp, a.sz_q_comp, a.status);
#pragma unroll
        for (int j = 0; j < V; j++) {
            const float *row = Qc + static_cast<long long>(lane * V + j) * D;
            float acc = 0.f;
            if (okc)
                for (int k = 0; k < D; k++) acc += __ldg(row + k) * scr[k];
            x[j] = h < sh.G ? acc : 0.f;
        }
        __syncwarp();
    }
    float qsum = 0.f, qmu = 0.f;
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane * V + j;
        qsum += x[j];
        qmu += x[j] * in.mu[j];
        const uint32_t w = hilo_f16(x[j] * __int_as_float((127 - field_exp(c >> 3, BITS)) << 23));
        S.qh[i][0][h][c] = static_cast<uint16_t>(w & 0xffffu);
        S.qh[i][1][h][c] = static_cast<uint16_t>(w >> 16);
    }
    qsum = warp_sum(qsum);
    qmu = warp_sum(qmu);
    __syncwarp();
    // the unit's accumulator starts empty (rows were scratch above)
    for (int c = lane; c < D + 4; c += 32) S.uacc[i][h][c] = c == D ? -INFINITY : 0.f;
    if (lane == 0) {
        S.qsc[i][h][0] = a.sm_log2 * qsum;
        S.qsc[i][h][1] = a.sm_log2 * qmu;
    }
}

// Copies of packed tiles [tin, tin + T) of unit u into a slot: key records,
// value pair records, key metadata, value metadata at their fixed offsets.
template <int D, int BITS, bool M16>
__device__ __forceinline__ void issue_chunk(const AttnArgs &a, long long qcap, int u, long long tin, int T,
                                            uint8_t *slot, uint64_t *bar) {
    using C = ACfg<D, BITS, M16>;
    const long long g0 = static_cast<long long>(u) * qcap + tin * 16;
    const uint32_t nt = 16u * static_cast<uint32_t>(T);
    const uint8_t *ck = a.codes_k + g0 * C::ROWK;
    const uint8_t *cv = a.codes_v + g0 / 2 * C::PAIRV;
    const uint8_t *mk = static_cast<const uint8_t *>(a.meta_k) + g0 * 2 * C::MB;
    const uint8_t *mv = static_cast<const uint8_t *>(a.meta_v) + g0 * 2 * C::MB;
    const uint32_t kb = nt * C::ROWK, vb = nt / 2 * C::PAIRV, mb = nt * 2 * C::MB;
    const uint32_t sb = smem_u32(slot), br = smem_u32(bar);
    if (!(in_buf(ck, kb, a.codes_k, a.sz_codes_k, a.status) && in_buf(cv, vb, a.codes_v, a.sz_codes_v, a.status) &&
          in_buf(mk, mb, a.meta_k, a.sz_meta_k, a.status) && in_buf(mv, mb, a.meta_v, a.sz_meta_v, a.status))) {
        // checked build: the copies are skipped and the slot's phase completes empty
        asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
                     "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(br) : "memory");
        return;
    }
    if (T == C::TPC) {  // a full chunk: the sizes are constants
        constexpr uint32_t KB = 16 * C::TPC * C::ROWK, VB = 8 * C::TPC * C::PAIRV, MB2 = 32 * C::TPC * C::MB;
        asm volatile(
            "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
            "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%11], [%12], %10, [%0];\n}\n" ::"r"(br),
            "n"(KB + VB + 2 * MB2), "r"(sb), "l"(ck), "n"(KB), "r"(sb + C::VOFF), "l"(cv), "n"(VB),
            "r"(sb + C::MKOFF), "l"(mk), "n"(MB2), "r"(sb + C::MVOFF), "l"(mv)
            : "memory");
        return;
    }
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%11], [%12], %10, [%0];\n}\n" ::"r"(br),
        "r"(kb + vb + 2 * mb), "r"(sb), "l"(ck), "r"(kb), "r"(sb + C::VOFF), "l"(cv), "r"(vb), "r"(sb + C::MKOFF),
        "l"(mk), "r"(mb), "r"(sb + C::MVOFF), "l"(mv)
        : "memory");
}

// 16-slot tile e of unit u's 16-bit slots into a slot (keys, then value pairs).
template <int D>
__device__ __forceinline__ void issue_raw(const AttnArgs &a, int rcap, int u, int e, uint8_t *slot, uint64_t *bar) {
    const long long r0 = static_cast<long long>(u) * rcap + static_cast<long long>(e) * AF_RTILE;
    const uint16_t *rk = a.raw_k + r0 * D, *rv = a.raw_v + r0 * D;
    if (!(in_buf(rk, 32 * D, a.raw_k, a.sz_raw_k, a.status) && in_buf(rv, 32 * D, a.raw_v, a.sz_raw_v, a.status))) {
        // checked build: the copies are skipped and the slot's phase completes empty
        asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
                     "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(smem_u32(bar)) : "memory");
        return;
    }
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %4, [%0];\n}\n" ::"r"(
            smem_u32(bar)),
        "n"(64 * D), "r"(smem_u32(slot)), "l"(rk), "n"(32 * D), "r"(smem_u32(slot) + 32 * D), "l"(rv)
        : "memory");
}

// Online-softmax step over NT logits of this lane (head tig); the running
// maximum is shared by the 8 lanes of a head and may lag by RESCALE_SLACK.
// The cross-lane maximum is taken only when some lane's logit exceeds the
// running maximum by more than the slack.
template <int NT, int NMT>
__device__ __forceinline__ void softmax_step(WarpState<NMT> &st, const float (&lg)[NT], float (&p)[NT]) {
    float mx = lg[0];
#pragma unroll
    for (int k = 1; k < NT; k++) mx = fmaxf(mx, lg[k]);
    if (__any_sync(FULL, mx > st.m + RESCALE_SLACK)) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        if (mx > st.m + RESCALE_SLACK) {  // uniform over a head's lanes
            const float al = ex2(st.m - mx);  // 0 when the maximum was -inf
            st.m = mx;
            st.l *= al;
            st.ao *= al;
#pragma unroll
            for (int mi = 0; mi < NMT; mi++) {
                st.acc[mi][0] *= al;
                st.acc[mi][1] *= al;
                st.acc[mi][2] *= al;
                st.acc[mi][3] *= al;
            }
        }
    }
    const float mu = st.m == -INFINITY ? 0.f : st.m;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < NT; k++) {
        p[k] = ex2(lg[k] - mu);
        sum += p[k];
    }
    st.l += sum;
}

// One chunk of T tiles (T <= TPC) in a slot -> this warp's state.  Tokens at
// or past nv in the chunk's last tile, and tiles at or past T, are masked
// (their bytes are whatever the slot held).
template <int D, int BITS, bool M16, bool FULLC>
__device__ __forceinline__ void process_chunk(const uint8_t *slot, int T, int nv, const uint32_t (&qb)[D / 16][2],
                                              float qs, float qm, float sk, WarpState<D / 16> &st) {
    using C = ACfg<D, BITS, M16>;
    constexpr int TPC = C::TPC, NMT = C::NMT, NWK = Slice<D, BITS>::NW;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const uint8_t *kp = slot, *vp = slot + C::VOFF, *mkp = slot + C::MKOFF, *mvp = slot + C::MVOFF;
    if (FULLC) {  // a full chunk: no tile or token checks
        T = TPC;
        nv = 16;
    }
    const int nvc = 16 * (T - 1) + nv;               // valid tokens of the chunk
    const bool ragged = !FULLC && nvc < 16 * TPC;  // warp-uniform
    float lg[2 * TPC];
#pragma unroll
    for (int t = 0; t < TPC; t++) {
        if (t < T) {
            uint32_t k0[NWK], k1[NWK];
            load_k_slice<D, BITS>(kp + (16 * t + g) * C::ROWK, tig, k0);
            load_k_slice<D, BITS>(kp + (16 * t + g + 8) * C::ROWK, tig, k1);
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < D / 16; i++)
                mma_f16(sc, extract<BITS>(k0, 2 * i), extract<BITS>(k1, 2 * i), extract<BITS>(k0, 2 * i + 1),
                        extract<BITS>(k1, 2 * i + 1), qb[i][0], qb[i][1]);
            const float2 ma = ld_meta(mkp, 16 * t + g, M16), mb = ld_meta(mkp, 16 * t + g + 8, M16);
            lg[2 * t] = (ma.x * sk) * (sc[0] + sc[1]) + fmaf(ma.y, qs, qm);
            lg[2 * t + 1] = (mb.x * sk) * (sc[2] + sc[3]) + fmaf(mb.y, qs, qm);
        }
    }
    if (ragged) {  // tokens past the chunk's valid ones (including whole tiles t >= T)
#pragma unroll
        for (int t = 0; t < TPC; t++) {
            if (16 * t + g >= nvc) lg[2 * t] = -INFINITY;
            if (16 * t + g + 8 >= nvc) lg[2 * t + 1] = -INFINITY;
        }
    }
    float p[2 * TPC];
    softmax_step<2 * TPC, NMT>(st, lg, p);
    float aos = 0.f;
#pragma unroll
    for (int t = 0; t < TPC; t++) {
        if (t < T) {
            float2 va = ld_meta(mvp, 16 * t + g, M16), vb = ld_meta(mvp, 16 * t + g + 8, M16);
            if (ragged) {  // masked tokens have p = 0, but their metadata may be anything
                if (16 * t + g >= nvc) va = make_float2(0.f, 0.f);
                if (16 * t + g + 8 >= nvc) vb = make_float2(0.f, 0.f);
            }
            aos += p[2 * t] * va.y + p[2 * t + 1] * vb.y;
            const uint32_t b0 = movmatrix_t(hilo_f16(p[2 * t] * va.x));
            const uint32_t b1 = movmatrix_t(hilo_f16(p[2 * t + 1] * vb.x));
            uint32_t v0[NWK], v1[NWK];
            load_v_slice<D, BITS>(vp + (8 * t + tig) * C::PAIRV, g, v0);
            load_v_slice<D, BITS>(vp + (8 * t + tig + 4) * C::PAIRV, g, v1);
#pragma unroll
            for (int mi = 0; mi < NMT; mi++)
                mma_f16(st.acc[mi], extract<BITS>(v0, 2 * mi), extract<BITS>(v0, 2 * mi + 1),
                        extract<BITS>(v1, 2 * mi), extract<BITS>(v1, 2 * mi + 1), b0, b1);
        }
    }
    st.ao += aos;
}

// Fold this warp's state into unit slot i's shared accumulator (one warp at a
// time: a lock per slot).  Each lane owns rows 16 mi + 8 rr + g of head tig.
template <int D, int BITS, bool M16>
__device__ __forceinline__ void fold_into_unit(ASmem<D, BITS, M16> &S, int i, WarpState<D / 16> &st, unsigned *status) {
    constexpr int NMT = D / 16;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        st.l += __shfl_xor_sync(FULL, st.l, o);
        st.ao += __shfl_xor_sync(FULL, st.ao, o);
    }
    if (lane == 0) {
        const uint64_t t0 = global_ns();
        while (atomicCAS(&S.ulock[i], 0, 1) != 0) {
            if (global_ns() - t0 > AF_WAIT_NS) {
                atomicOr(status, ST_TIMEOUT);
                break;
            }
        }
    }
    __syncwarp();
    __threadfence_block();
    float *ua = S.uacc[i][tig];
    const float Ms = ua[D], Ls = ua[D + 1];
    __syncwarp();
    const float Mn = fmaxf(Ms, st.m);
    const float as = Ms == -INFINITY ? 0.f : ex2(Ms - Mn);
    const float aw = st.m == -INFINITY ? 0.f : ex2(st.m - Mn);
#pragma unroll
    for (int mi = 0; mi < NMT; mi++)
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int row = 16 * mi + 8 * rr + g;
            const float v = (st.acc[mi][2 * rr] + st.acc[mi][2 * rr + 1]) *
                                pow2i(24 - field_exp(2 * mi + rr, BITS)) +
                            st.ao;
            ua[row] = ua[row] * as + v * aw;
        }
    if (g == 0) {
        ua[D] = Mn;
        ua[D + 1] = Ls * as + st.l * aw;
    }
    __threadfence_block();
    __syncwarp();
    if (lane == 0) atomicExch(&S.ulock[i], 0);
}

// Record counts of unit u: np packed CTAs (slots [0, np)) and nr 16-bit-tile
// warps (slots [mps, mps + nr)).
__device__ __forceinline__ void unit_records(const AttnArgs &a, int u, int G, int &np, int &nr) {
    np = nr = 0;
    if (a.np_total > 0) {
        const int fp = owner(static_cast<long long>(u) * a.cpu, a.np_total, G);
        np = owner(static_cast<long long>(u) * a.cpu + a.cpu - 1, a.np_total, G) - fp + 1;
    }
    if (a.nr_total > 0) {
        const int fr = owner(static_cast<long long>(u) * a.n_rt, a.nr_total, G);
        nr = owner(static_cast<long long>(u) * a.n_rt + a.n_rt - 1, a.nr_total, G) - fr + 1;
    }
}

// One warp: merge the records of unit u for query head h (packed value
// accumulators in the rotated basis, 16-bit ones in the original basis),
// rotate back, normalize and write the output row.  The caller has seen every
// record of the unit published (its count reached np + nr) and fenced.
template <int D>
__device__ void finish_head(const AttnArgs &a, const AttnShape &sh, int u, int h, int np, int nr) {
    constexpr int V = D / 32, PR = D + 4, NB = 8;
    using VT = typename VecT<V>::T;
    const int lane = threadIdx.x & 31;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    const float *pu = a.partials + static_cast<long long>(u) * a.max_slots * 4 * PR + h * PR;
    const int n_rec = np + nr;
    float M = -INFINITY, Lsum = 0.f;
    float accq[V], accr[V];
#pragma unroll
    for (int j = 0; j < V; j++) accq[j] = accr[j] = 0.f;
    for (int r0 = 0; r0 < n_rec; r0 += NB) {
        float mr[NB], lr[NB];
        VT vv[NB];
#pragma unroll
        for (int k = 0; k < NB; k++) {
            const int r = r0 + k;
            const bool in = r < n_rec;
            const int slot = r < np ? r : a.mps + (r - np);
            const float *p = pu + static_cast<long long>(in ? slot : 0) * 4 * PR;
            const bool ok = in && in_buf(p, PR * 4, a.partials, a.sz_partials, a.status);
            mr[k] = ok ? __ldcg(p + D) : -INFINITY;
            lr[k] = ok ? __ldcg(p + D + 1) : 0.f;
            vv[k] = ok ? __ldcg(reinterpret_cast<const VT *>(p) + lane) : VT{};
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
            if (mr[k] == -INFINITY) continue;  // empty record: its value row was never written
            const float w = exp2f(mr[k] - M);
            Lsum += lr[k] * w;
            if (r0 + k < np) vadd(accq, vv[k], w);
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
    const int osz = a.out_dtype == DQ_F32 ? 4 : 2;
    if (!in_buf(static_cast<char *>(a.out) + ob * osz, D * osz, a.out, a.sz_out, a.status)) return;
#pragma unroll
    for (int j = 0; j < V; j++) {
        const float y = (accq[j] + accr[j]) * inv;
        const long long oi = ob + lane * V + j;
        if (a.out_dtype == DQ_F32) reinterpret_cast<float *>(a.out)[oi] = y;
        else if (a.out_dtype == DQ_F16) reinterpret_cast<__half *>(a.out)[oi] = __float2half_rn(y);
        else reinterpret_cast<__nv_bfloat16 *>(a.out)[oi] = __float2bfloat16_rn(y);
    }
}

// The fused step's append of one unit's new token (its keys or its values)
// from inputs loaded earlier, kept out of line: the attention's own loops keep
// the code layout they have without it.
template <int V, int BITS>
__device__ __noinline__ void append_row(const QuantArgs &qa, const RowGeom &rg, int u, const RowIn<V> &in,
                                        float *xs) {
    quantize_loaded_row<V, BITS>(qa, rg, u, 0, in, xs);
}

// ---- the kernel ---------------------------------------------------------------
// Chunks: chunk j of unit u holds its packed tiles [j TPC, min((j + 1) TPC,
// n_pt)).  CTA c owns chunks [c N / G, (c + 1) N / G) of the list of all units'
// chunks; its packed warps take them one at a time from a shared counter (in
// increasing order, so a warp meets its units in order), each warp's first
// chunk being fixed so that its copy goes out at once.
template <int D, int BITS, bool M16>
__global__ void __launch_bounds__(AF_WPB * 32, 1) attn_affine_kernel(AttnArgs a, AttnShape sh) {
    using C = ACfg<D, BITS, M16>;
    constexpr int NS = C::NS, TPC = C::TPC, PR = C::PR;
    static_assert(NS == 2 || NS == 3, "the ring holds two or three slots");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ASmem<D, BITS, M16> &S = *reinterpret_cast<ASmem<D, BITS, M16> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3, g = lane >> 2;
    const int cta = blockIdx.x, G = gridDim.x;
    const long long cpu = a.cpu, NP = a.np_total, NR = a.nr_total;
    const int WP = a.wp;
    const bool raw_warp = warp >= WP;
    const long long x0 = static_cast<long long>(cta) * NP / G, x1 = static_cast<long long>(cta + 1) * NP / G;
    const int u_first = x1 > x0 ? static_cast<int>(x0 / cpu) : 0;
    const int n_units = x1 > x0 ? static_cast<int>((x1 - 1) / cpu) - u_first + 1 : 0;
    const bool preps = (warp >> 2) < n_units;
    bool timed_out = false;

    // the query loads go out first, with the new token's rows in a fused step
    // (loaded before any cache copy is issued, they do not queue behind them,
    // and parked in shared memory until the append at the end)
    QLoad<D> qin;
    if (preps) load_unit_query<D>(a, sh, u_first + (warp >> 2), warp & 3, qin);
    const bool appends = a.append && !raw_warp && warp >= WP - 2;
    const int which = warp == WP - 1 ? 0 : 1;  // keys, values
    // parking place: the save slot of the 16-bit-tile warp (a fused step has
    // 16-bit slots, so that warp exists and never saves a state): keys and
    // values as fp32 at [0, 2D), the key mean at [2D, 3D), the 16-bit bits
    // from float 3D on
    float *park = &S.save[AF_WPB - 1][0][0];
    static_assert(4 * D <= 4 * PR, "the new token's rows fit a save slot");
    if (appends && cta < sh.U) {
        RowIn<D / 32> ain;
        load_row<D / 32>(a.qa[which], cta, 0, ain);
#pragma unroll
        for (int j = 0; j < D / 32; j++) {
            const int c = lane * (D / 32) + j;
            park[which * D + c] = ain.x[j];
            if (which == 0) park[2 * D + c] = ain.mu[j];
            reinterpret_cast<uint16_t *>(park + 3 * D)[which * D + c] = ain.r[j];
        }
    }
    if (lane == 0) {
        if (!raw_warp) {
            for (int s = 0; s < NS; s++) mbar_init(&S.full[warp][s], 1);
        } else {
            for (int s = 0; s < AF_NSR; s++) mbar_init(&S.rfull[s], 1);
        }
        fence_mbar_init();
        S.save_u[warp] = -1;
        if (warp < AF_NUS + AF_NUR) S.done_u[warp] = -1;
        if (warp < AF_NUS) S.ulock[warp] = 0;
        if (warp == 0) S.next = static_cast<int>(x0 + WP);
    }
    __syncwarp();

    uint8_t *myring = S.ring + static_cast<size_t>(warp) * NS * C::SLOT;
    // chunk indices fit 32 bits (the planner checks it); a warp meets its chunks
    // in increasing order, so units are tracked by comparison, not division
    const int cpu32 = static_cast<int>(cpu), npt = static_cast<int>(a.n_pt);
    int iu = -1, iend = 0;  // issue side: unit of the last issued chunk and its end
    auto issue = [&](int c, int s) {
        while (c >= iend) {
            iu = iu < 0 ? c / cpu32 : iu + 1;
            iend = (iu + 1) * cpu32;
        }
        const int tin = (c - (iend - cpu32)) * TPC;
        const int T = npt - tin < TPC ? npt - tin : TPC;
        issue_chunk<D, BITS, M16>(a, sh.qcap, iu, tin, T, myring + s * C::SLOT, &S.full[warp][s]);
    };
    const int x1i = static_cast<int>(x1);
    // each packed warp's first chunk, before the query preparation
    // the 16-bit tiles of this CTA's share of all units: the first AF_NSR
    // copies go out now, with the packed warps' first chunks
    const long long r0 = static_cast<long long>(cta) * NR / G, r1 = static_cast<long long>(cta + 1) * NR / G;
    uint8_t *rring = S.ring + static_cast<size_t>(WP) * NS * C::SLOT;
    auto issue_raw_tile = [&](long long x, int s) {
        const int u = static_cast<int>(x / a.n_rt);
        issue_raw<D>(a, sh.rcap, u, static_cast<int>(x - static_cast<long long>(u) * a.n_rt), rring + s * C::RSLOT,
                     &S.rfull[s]);
    };
    const int ru0 = r0 < r1 ? static_cast<int>(r0 / a.n_rt) : 0;
    const int n_runits = r0 < r1 ? static_cast<int>((r1 - 1) / a.n_rt) - ru0 + 1 : 0;  // <= AF_NUR (planner)
    if (raw_warp && r0 < r1) {
        for (int s = 0; s < AF_NSR && r0 + s < r1; s++) issue_raw_tile(r0 + s, s);
        // (hi, lo) 16-bit halves of the raw queries of the warp's units, loaded
        // now so that no load waits behind the cache stream later
        constexpr int V = D / 32;
        for (int j = 0; j < n_runits; j++) {
            const int u = ru0 + j, b = u / sh.Hkv, kvh = u % sh.Hkv;
#pragma unroll
            for (int h = 0; h < 4; h++) {
                const long long qo = (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D;
                const bool okq = h < sh.G && in_buf(a.q + qo, D * 4, a.q, a.sz_q, a.status);
#pragma unroll
                for (int jj = 0; jj < V; jj++) {
                    const int c = lane * V + jj;
                    const float xq = okq ? __ldg(a.q + qo + c) : 0.f;
                    const uint32_t w = a.raw_bf16 ? hilo_bf16(xq) : hilo_f16(xq);
                    S.rqh[j][0][h][c] = static_cast<uint16_t>(w & 0xffffu);
                    S.rqh[j][1][h][c] = static_cast<uint16_t>(w >> 16);
                }
            }
        }
    }
    // fused decode step: the new token's 16-bit slot of unit u sits in tile
    // e_new, and the warp holding that tile reads the token's 16-bit row from
    // the input instead of the cache.  The append itself is made by the
    // packed warps below; nothing in this call reads what it writes (the
    // token's packed slot lies in the recent window, its 16-bit row comes from
    // the input).
    int rs_new = -1, e_new = -1;
    if (a.append) {
        const long long tn = a.qa[0].pos0;
        rs_new = tn < a.rg.n_sink ? static_cast<int>(tn) : a.rg.n_sink + static_cast<int>(tn % a.rg.n_recent);
        e_new = rs_new / AF_RTILE;
    }
    // chunks in flight, oldest first: q0 in slot s, q1 in the next slot, ...
    int q0 = -1, q1 = -1, q2 = -1;
    if (!raw_warp && x0 + warp < x1) {
        q0 = static_cast<int>(x0) + warp;
        issue(q0, 0);
    }
    if (preps) prep_unit<D, BITS, M16>(a, sh, S, warp >> 2, u_first + (warp >> 2), warp & 3, qin);
    __syncthreads();

    WarpState<D / 16> st;
    st.init();
    int cu = -1;  // packed: unit of the segment in progress
    if (!raw_warp) {
        auto grab = [&]() {
            int c = 0;
            if (lane == 0) c = atomicAdd(&S.next, 1);
            c = __shfl_sync(FULL, c, 0);
            return c < x1i ? c : -1;
        };
        if (q0 >= 0) {
            q1 = grab();
            if (q1 >= 0) issue(q1, 1);
            if (NS == 3 && q1 >= 0) {
                q2 = grab();
                if (q2 >= 0) issue(q2, 2);
            }
        }
        uint32_t qb[D / 16][2];
        float qs = 0.f, qm = 0.f;
        const float sk = a.sm_log2 * 16777216.0f;  // 2^24 undoes the operand scaling
        unsigned ph = 0;                           // bit s: phase of slot s
        int uend = 0;                              // end of unit cu's chunks
        for (int s = 0;; s = s + 1 == NS ? 0 : s + 1) {
            const int c = q0;
            if (c < 0) break;
            // the next chunk's number is taken now; its latency hides behind this chunk
            int nx = 0;
            if (lane == 0) nx = atomicAdd(&S.next, 1);
            if (!mbar_wait(&S.full[warp][s], (ph >> s) & 1u, AF_WAIT_NS)) timed_out = true;
            ph ^= 1u << s;
            if (c >= uend) {
                if (cu >= 0) {
                    // the first finished segment goes to the warp's own slot; a
                    // later one (a CTA range over three or more units) is folded
                    // into the unit's shared accumulator under its lock
                    if (S.save_u[warp] < 0) {
                        store_state<D, BITS>(st, true, &S.save[warp][0][0], PR);
                        __syncwarp();
                        if (lane == 0) S.save_u[warp] = cu;
                        __syncwarp();
                    } else {
                        fold_into_unit<D, BITS, M16>(S, cu - u_first, st, a.status);
                    }
                }
                do {
                    cu = cu < 0 ? c / cpu32 : cu + 1;
                    uend = (cu + 1) * cpu32;
                } while (c >= uend);
                const int i = cu - u_first;
                const uint16_t *row = S.qh[i][g & 1][g >> 1];
#pragma unroll
                for (int k = 0; k < D / 16; k++)
#pragma unroll
                    for (int sub = 0; sub < 2; sub++)
                        qb[k][sub] = *reinterpret_cast<const uint32_t *>(row + PermIdentity()(k, tig, sub, 0));
                qs = S.qsc[i][tig][0];
                qm = S.qsc[i][tig][1];
                st.init();
            }
            const int tin = (c - (uend - cpu32)) * TPC;
            const int T = npt - tin < TPC ? npt - tin : TPC;
            const long long left = a.n_q - static_cast<long long>(tin + T - 1) * 16;
            const int nv = left < 16 ? static_cast<int>(left) : 16;
            uint8_t *slot = myring + s * C::SLOT;
            if (T == TPC && nv == 16) process_chunk<D, BITS, M16, true>(slot, T, nv, qb, qs, qm, sk, st);
            else process_chunk<D, BITS, M16, false>(slot, T, nv, qb, qs, qm, sk, st);
            __syncwarp();
            nx = __shfl_sync(FULL, nx, 0);
            if (nx >= x1i) nx = -1;
            if (nx >= 0) issue(nx, s);
            q0 = q1;
            if (NS == 3) {
                q1 = q2;
                q2 = nx;
            } else {
                q1 = nx;
            }
        }
    } else {
        // ---- the 16-bit tiles (their first copies went out above); a unit's
        // record is written here and published with the CTA's at the end
        if (r0 < r1) {
            const int n_rt = a.n_rt;
            uint32_t qb[D / 16][2];
            int ru = -1;
            auto flush = [&]() {
                const int first = owner(static_cast<long long>(ru) * n_rt, NR, G);
                float *rec = a.partials +
                             (static_cast<long long>(ru) * a.max_slots + a.mps + (cta - first)) * 4 * PR;
                if (in_buf(rec, 4 * PR * 4, a.partials, a.sz_partials, a.status)) store_state<D, BITS>(st, false, rec, PR);
            };
            for (long long x = r0; x < r1; x++) {
                const int k = static_cast<int>(x - r0), s = k % AF_NSR;
                const int u = static_cast<int>(x / n_rt), e = static_cast<int>(x - static_cast<long long>(u) * n_rt);
                if (u != ru) {
                    if (ru >= 0) flush();
                    ru = u;
                    const uint16_t *row = S.rqh[u - ru0][g & 1][g >> 1];
#pragma unroll
                    for (int i = 0; i < D / 16; i++)
#pragma unroll
                        for (int sub = 0; sub < 2; sub++)
                            qb[i][sub] = *reinterpret_cast<const uint32_t *>(row + PermRawK()(i, tig, sub, 0));
                    st.init();
                }
                if (!mbar_wait(&S.rfull[s], (k / AF_NSR) & 1, AF_WAIT_NS)) timed_out = true;
                uint8_t *tile = rring + s * C::RSLOT;
                if (e == e_new) {  // the new token's 16-bit row, from the input
                    const int sl = rs_new - e * AF_RTILE;
                    uint16_t *kr = reinterpret_cast<uint16_t *>(tile) + sl * D;
                    uint16_t *vr = reinterpret_cast<uint16_t *>(tile + 32 * D) + (sl >> 1) * 2 * D + (sl & 1);
                    constexpr int V = D / 32;
                    const long long base = static_cast<long long>(u) * D;
                    const long long esz = a.qa[0].in_dtype == 0 ? 4 : 2;
                    const bool okk = in_buf(static_cast<const char *>(a.qa[0].x) + base * esz, D * esz, a.qa[0].x,
                                            a.qa[0].sz_x, a.status);
                    const bool okv = in_buf(static_cast<const char *>(a.qa[1].x) + base * esz, D * esz, a.qa[1].x,
                                            a.qa[1].sz_x, a.status);
#pragma unroll
                    for (int j = 0; j < V; j++) {
                        const int c = lane * V + j;
                        kr[c] = okk ? raw16_of(a.qa[0].x, base + c, a.qa[0].in_dtype) : 0;
                        vr[2 * c] = okv ? raw16_of(a.qa[1].x, base + c, a.qa[1].in_dtype) : 0;
                    }
                    __syncwarp();
                }
                if (a.raw_bf16) process_raw<D, true>(a, tile, static_cast<long long>(e) * AF_RTILE, qb, st);
                else process_raw<D, false>(a, tile, static_cast<long long>(e) * AF_RTILE, qb, st);
                __syncwarp();
                if (x + AF_NSR < r1) issue_raw_tile(x + AF_NSR, s);
            }
            flush();
        }
    }
    if (timed_out && lane == 0) atomicOr(a.status, ST_TIMEOUT);

    // ---- merge per unit: each warp's final state (stored over the now idle
    // rings), the warps' saved states and the unit's shared accumulator are
    // summed, scaled to the unit's maximum, by one warp per (unit, head)
    __syncthreads();
    float *fin = reinterpret_cast<float *>(S.ring);  // [AF_WPB][4][PR]
    if (cu >= 0) store_state<D, BITS>(st, true, fin + warp * 4 * PR, PR);
    if (lane == 0) S.fin_u[warp] = cu;
    __syncthreads();
    constexpr int NSRC = 2 * AF_WPB + 1;  // warp z's final state, its saved state, the shared accumulator
    static_assert(NSRC <= 64, "two sources per lane");
    const float *sbase = reinterpret_cast<const float *>(smem_raw);
    // per warp, the live sources of the pair it merges (the query operands'
    // space: they are dead once the chunks are done)
    int2 *lists = reinterpret_cast<int2 *>(&S.qh[0][0][0][0]);
    static_assert(sizeof(S.qh) >= AF_WPB * (NSRC + 1) * sizeof(int2), "merge lists fit the query operands' space");
    for (int ih = warp; ih < 4 * n_units; ih += AF_WPB) {
        const int i = ih >> 2, h = ih & 3, u = u_first + i;
        // source z as a float offset into shared memory (-1: no state of unit u)
        auto src = [&](int z) -> int {
            const float *p = nullptr;
            if (z < AF_WPB) p = S.fin_u[z] == u ? fin + (z * 4 + h) * PR : nullptr;
            else if (z < 2 * AF_WPB) p = S.save_u[z - AF_WPB] == u ? &S.save[z - AF_WPB][h][0] : nullptr;
            else if (z == 2 * AF_WPB) p = &S.uacc[i][h][0];
            return p ? static_cast<int>(p - sbase) : -1;
        };
        // lane l holds sources l and l + 32: their maxima, then their weights
        const int o0 = src(lane), o1 = src(lane + 32);
        const float m0 = o0 >= 0 ? sbase[o0 + D] : -INFINITY, m1 = o1 >= 0 ? sbase[o1 + D] : -INFINITY;
        const float M = warp_max(fmaxf(m0, m1));
        const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - M), w1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
        const float L = warp_sum((o0 >= 0 ? w0 * sbase[o0 + D + 1] : 0.f) + (o1 >= 0 ? w1 * sbase[o1 + D + 1] : 0.f));
        constexpr int CPL = (D + 31) / 32;  // columns per lane
        float acc[CPL];
#pragma unroll
        for (int j = 0; j < CPL; j++) acc[j] = 0.f;
        // the live sources, compacted into this warp's list as (offset, weight
        // bits), then summed four at a time: every load address comes from a
        // broadcast read, not from a chain of shuffles
        int2 *lst = lists + warp * (NSRC + 1);
        const unsigned b0 = __ballot_sync(FULL, w0 != 0.f), b1 = __ballot_sync(FULL, w1 != 0.f);
        const unsigned below = (1u << lane) - 1u;
        if (w0 != 0.f) lst[__popc(b0 & below)] = make_int2(o0, __float_as_int(w0));
        if (w1 != 0.f) lst[__popc(b0) + __popc(b1 & below)] = make_int2(o1, __float_as_int(w1));
        __syncwarp();
        const int nlive = __popc(b0) + __popc(b1);
        for (int k0 = 0; k0 < nlive; k0 += 4) {
            int2 e[4];
            float v[4][CPL];
#pragma unroll
            for (int k = 0; k < 4; k++) e[k] = k0 + k < nlive ? lst[k0 + k] : make_int2(0, 0);
#pragma unroll
            for (int k = 0; k < 4; k++)
#pragma unroll
                for (int j = 0; j < CPL; j++) v[k][j] = e[k].y != 0 ? sbase[e[k].x + lane + 32 * j] : 0.f;
#pragma unroll
            for (int k = 0; k < 4; k++)
#pragma unroll
                for (int j = 0; j < CPL; j++) acc[j] = fmaf(__int_as_float(e[k].y), v[k][j], acc[j]);
        }
        __syncwarp();  // the list is rewritten for this warp's next pair
        const int first = owner(static_cast<long long>(u) * cpu, NP, G);
        float *rec = a.partials + (static_cast<long long>(u) * a.max_slots + (cta - first)) * 4 * PR + h * PR;
        if (in_buf(rec, PR * 4, a.partials, a.sz_partials, a.status)) {
#pragma unroll
            for (int j = 0; j < CPL; j++) rec[lane + 32 * j] = acc[j];
            if (lane == 0) {
                rec[D] = M;
                rec[D + 1] = L;
            }
        }
    }
    // publish: the records are visible GPU-wide before the units' counts move
    // (the barrier orders every thread's record stores before the releasing
    // add of the threads that take the tickets); the CTA whose record
    // completes a unit merges that unit's records (the add also acquires: the
    // unit's other records are visible to it, and to the CTA after the barrier)
    __syncthreads();
    if (threadIdx.x < n_units + n_runits) {  // one ticket per record: packed units, then 16-bit ones
        const int t = threadIdx.x;
        const int u = t < n_units ? u_first + t : ru0 + (t - n_units);
        int np, nr;
        unit_records(a, u, G, np, nr);
        const bool last = in_buf(a.counters + u, 4, a.counters, a.sz_counters, a.status) &&
                          atomic_add_acq_rel_gpu(a.counters + u, 1) + 1 == np + nr;
        S.done_u[t] = last ? u : -1;
    }
    __syncthreads();
    // the completed units, four warps (one per query head) per unit at a time
    int k = 0;
    for (int i = 0; i < n_units + n_runits; i++) {
        const int u = S.done_u[i];
        if (u < 0) continue;
        if ((warp >> 2) == (k & 3) && (warp & 3) < sh.G) {
            int np, nr;
            unit_records(a, u, G, np, nr);
            finish_head<D>(a, sh, u, warp & 3, np, nr);
            if (lane == 0 && (warp & 3) == 0 && in_buf(a.counters + u, 4, a.counters, a.sz_counters, a.status))
                a.counters[u] = 0;  // every record of this call has arrived
        }
        ++k;
    }
    // fused decode step: CTA c appends the new token of units c, c + G, ...;
    // its last two packed warps quantize the keys and the values here, at the
    // end, where they overlap the warps finishing units instead of taking
    // issue slots from the chunk loop
    if (appends) {
        for (int u = cta; u < sh.U; u += G) {
            RowIn<D / 32> ain;
            if (u == cta) {
#pragma unroll
                for (int j = 0; j < D / 32; j++) {
                    const int c = lane * (D / 32) + j;
                    ain.x[j] = park[which * D + c];
                    ain.mu[j] = which == 0 ? park[2 * D + c] : 0.f;
                    ain.r[j] = reinterpret_cast<const uint16_t *>(park + 3 * D)[which * D + c];
                }
            } else {
                load_row<D / 32>(a.qa[which], u, 0, ain);
            }
            append_row<D / 32, BITS>(a.qa[which], a.rg, u, ain, &S.save[warp][0][0]);
        }
    }
}

template <int D, int BITS, bool M16>
struct AffineLauncher {
    using C = ACfg<D, BITS, M16>;
    static constexpr int TPC = C::TPC;
    static size_t smem() { return sizeof(ASmem<D, BITS, M16>); }
    // a CTA's shared memory must fit the 227 KB an sm_103a block may use (2-bit
    // head_dim 128 records with fp32 metadata do not: the older kernel serves them)
    static constexpr bool FITS = sizeof(ASmem<D, BITS, M16>) <= 227 * 1024;

    static int prepare() {
        static bool done = false;
        if (done) return 0;
        const cudaError_t e = cudaFuncSetAttribute(attn_affine_kernel<D, BITS, M16>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem()));
        if (e != cudaSuccess) return static_cast<int>(e);
        done = true;
        return 0;
    }
    static int launch(const AttnArgs &a, const AttnShape &sh, void *stream) {
        attn_affine_kernel<D, BITS, M16><<<a.grid, AF_WPB * 32, smem(), static_cast<cudaStream_t>(stream)>>>(a, sh);
        return static_cast<int>(cudaGetLastError());
    }
};

template <typename F>
int dispatch_affine(const Layout &L, F &&f) {
    const bool m16 = L.meta_bytes == 2;
    if (L.d == 128) {
        if (L.bits_k == 2) return m16 ? f(AffineLauncher<128, 2, true>()) : f(AffineLauncher<128, 2, false>());
        if (L.bits_k == 3) return m16 ? f(AffineLauncher<128, 3, true>()) : f(AffineLauncher<128, 3, false>());
        return m16 ? f(AffineLauncher<128, 4, true>()) : f(AffineLauncher<128, 4, false>());
    }
    if (L.bits_k == 2) return m16 ? f(AffineLauncher<64, 2, true>()) : f(AffineLauncher<64, 2, false>());
    return m16 ? f(AffineLauncher<64, 4, true>()) : f(AffineLauncher<64, 4, false>());
}

long long ceil_div(long long x, long long y) { return (x + y - 1) / y; }

}  // namespace

bool affine_kernel_applies(const Layout &L, const AttnArgs &a) {
    if (!(L.scheme == DQ_AFFINE && L.bits_k == L.bits_v && L.G <= 4 &&
          ((L.d == 128 && L.bits_k >= 2 && L.bits_k <= 4) || (L.d == 64 && (L.bits_k == 2 || L.bits_k == 4)))))
        return false;
    if (!dispatch_affine(L, [](auto l) { return decltype(l)::FITS ? 1 : 0; })) return false;
    // a cache read mostly as 16-bit slots streams better through the CTA-wide
    // ring of attn_kernel, whose every warp takes 16-bit tiles
    const long long packed = a.n_q * (L.rowK + L.pairV / 2 + 4LL * L.meta_bytes);
    const long long raw = (a.has_raw ? static_cast<long long>(a.n_raw_slots) : 0) * L.d * 4;
    return packed >= raw;
}

int plan_affine(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats) {
    int tpc = 0;
    const int e = dispatch_affine(L, [&](auto l) {
        tpc = decltype(l)::TPC;
        return decltype(l)::prepare();
    });
    if (e != 0) return e;
    a.affine = 1;
    a.n_rt = a.has_raw ? (a.n_raw_slots + AF_RTILE - 1) / AF_RTILE : 0;
    a.raw_all_valid = a.seq_len >= static_cast<long long>(a.n_sink_cfg) + a.n_recent_cfg;
    a.n_pt = (a.n_q + 15) / 16;
    a.cpu = ceil_div(a.n_pt, tpc);
    a.np_total = static_cast<long long>(L.U) * a.cpu;
    a.nr_total = static_cast<long long>(L.U) * a.n_rt;
    a.wp = a.n_rt > 0 ? AF_WPB - 1 : AF_WPB;
    const long long NP = a.np_total, NR = a.nr_total;
    if (NP >= (1LL << 31)) return static_cast<int>(cudaErrorInvalidValue);  // chunks are counted in 32 bits
    long long G;
    if (NP > 0) {
        G = ceil_div(NP, 2LL * a.wp);  // at least two chunks per warp on average
        if (G > num_sms) G = num_sms;
        if (G < 1) G = 1;
    } else {
        G = NR < num_sms ? NR : num_sms;
        if (G < 1) G = 1;
    }
    // a CTA's packed range touches at most AF_NUS units, its 16-bit tiles at most
    // AF_NUR (one query-operand slot each)
    for (;;) {
        const bool p_ok = NP == 0 || ceil_div(ceil_div(NP, G) - 1, a.cpu) + 1 <= AF_NUS;
        const bool r_ok = NR == 0 || ceil_div(ceil_div(NR, G) - 1, a.n_rt) + 1 <= AF_NUR;
        if (p_ok && r_ok) break;
        G += ceil_div(G, 8);
    }
    if (G >= (1LL << 31)) return static_cast<int>(cudaErrorInvalidValue);
    a.grid = static_cast<int>(G);
    // record slots per unit: packed CTAs touching it, then 16-bit-tile warps
    long long mps = 0, mrs = 0;
    if (NP > 0) {
        const long long per = NP / G;
        mps = per > 0 ? ceil_div(a.cpu, per) + 1 : a.cpu;
        if (mps > a.cpu) mps = a.cpu;
    }
    if (NR > 0) {
        const long long per = NR / G;
        mrs = per > 0 ? ceil_div(a.n_rt, per) + 1 : a.n_rt;
        if (mrs > a.n_rt) mrs = a.n_rt;
    }
    a.mps = static_cast<int>(mps);
    a.max_slots = static_cast<int>(mps + mrs);
    a.items_per_unit = a.cpu;
    a.total_items = NP;
    return affine_partial_floats(L, a) <= cap_floats ? 0 : static_cast<int>(cudaErrorMemoryAllocation);
}

long long affine_partial_floats(const Layout &L, const AttnArgs &a) {
    return static_cast<long long>(L.U) * a.max_slots * 4 * (L.d + 4);
}

int launch_affine(const Layout &L, const AttnArgs &a, void *stream) {
    AttnShape sh{L.U, L.Hkv, L.G, L.d, L.qcap, L.rcap};
    return dispatch_affine(L, [&](auto l) { return decltype(l)::launch(a, sh, stream); });
}

size_t affine_smem_bytes(const Layout &L) {
    size_t s = 0;
    dispatch_affine(L, [&](auto l) {
        s = decltype(l)::smem();
        return 0;
    });
    return s;
}

}  // namespace dq
