// Split-K GQA decode attention, the CTA-ring kernel (sm_103a): caches read
// mostly as 16-bit slots, non-uniform (table) caches, and the affine shapes
// the warp-ring kernel in attn_affine.cu does not take.  Also the planner that
// routes each call, the query compensation kernel and test-support kernels.
//
// Computes, per sequence b and query head h reading KV head h / G,
//   out_h = sum_t softmax_t(sm_scale * q_h . k^_t) v^_t
// with the affine terms applied after the contraction ("D-Quant: Driftable
// Entropy Coding for KV Cache Quantization", App. A Eq. (7)-(9)):
//   q . k^_t  = s_t * (q . m_t) + o_t * sum_j q_j + q . mu            (Eq. 8)
//   sum_t a_t v^_t = sum_t (a_t s_t) m_t + sum_t a_t o_t               (Eq. 9)
// Keys and values are rotated by the normalized Hadamard matrix Hn
// (Sec. 4.2), so q is rotated once per call and the value accumulator is
// rotated back with Hn (its own inverse) at the end.  Non-uniform caches
// ("KVQuant-NUQ", How it works) take table values as operands instead and add
// their outliers' corrections.
//
// Design for GB300:
//  * Work items: per KV head ("unit"), its 16-slot tiles of 16-bit sink and
//    recent tokens, then its packed entries of 128 tokens (the last ragged).
//    A persistent grid of 3-4 CTAs per SM splits the list of all units'
//    entries into equal contiguous ranges (stream-K).
//  * Each CTA streams its range through one ring of 3-4 slots, one entry per
//    slot (bulk asynchronous copies, completion on the slot's mbarrier); every
//    warp takes 32 tokens of every entry, and the last warp to release a slot
//    issues the copies of the entry the ring's depth later.
//  * Codes become mma operands with one AND per code pair: a code m held in a
//    binary16 bit pattern below 2048 is exactly m * 2^-24 (scaled by a
//    per-field power of two, folded into q and into the output rows).
//  * q.K^T and P.V are mma.sync m16n8k16 with fp32 accumulation.  The 8 mma
//    columns are 4 query heads x (hi, lo) binary16 halves of an fp32 operand,
//    adjacent, so each lane owns one head and adds its halves in registers.
//    P' is transposed into the B operand with movmatrix (no shared memory).
//  * The running max may lag by 2^8, so the accumulators are rescaled only
//    when it grows by more than that.
//  * Each CTA merges its 4 warps and writes one partial per (unit, kind); a
//    second grid (combine_kernel), launched as a programmatic dependent of the
//    first, waits for each unit's partials, merges them, rotates the value
//    accumulator back and writes the output.
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "dq_internal.h"

namespace dq {

constexpr int RTILE = 16;                           // slots per 16-bit work item
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s; a healthy copy takes microseconds


// NUQ: 1 = the non-uniform scheme (per-channel key tables, per-token value
// tables, fp16 outlier side channel) instead of the affine one; 2 = the same
// with value tables per 32-channel group and/or key tables per refit block
// (copied with each entry), head_dim 128.
template <int D, int BK, int BV, bool M16, int NUQ = 0>
struct Cfg {
    static constexpr int ST = 128;                // packed tokens per pipeline entry
    static constexpr int SUB = 32;                // tokens of an entry per warp (one softmax step)
    static constexpr int TILES = SUB / 16;
    static constexpr int ROWK = D * BK / 8;
    static constexpr int PAIRV = 2 * D * BV / 8;
    static constexpr int MB = M16 ? 2 : 4;
    static constexpr int LV = 1 << BV;            // table entries (non-uniform scheme)
    // stage layout: keys, value pairs, then (affine) key meta, value meta or
    // (non-uniform) the tokens' value tables
    static constexpr int KBYTES = ST * ROWK;
    static constexpr int VBYTES = ST / 2 * PAIRV;
    static constexpr int MBYTES = NUQ ? 0 : ST * 2 * MB;
    static constexpr int GVMAX = NUQ == 2 ? D / 32 : 1;  // value tables per token, at most
    static constexpr int LUTV = NUQ ? ST * GVMAX * LV * 2 : 0;
    static constexpr int LUTK = NUQ == 2 ? D * (1 << BK) * 2 : 0;  // the entry's key tables (refit blocks)
    static constexpr int ENTRY = KBYTES + VBYTES + 2 * MBYTES + LUTV + LUTK;
    static constexpr int RAWBYTES = 64 * D;       // one 16-slot tile of 16-bit keys + values
    static constexpr int SLOT = ((ENTRY > RAWBYTES ? ENTRY : RAWBYTES) + 127) / 128 * 128;
    // ring depth: four slots where four CTAs per SM still fit, else as many as
    // fit three CTAs per SM (the 3-bit kernel is register-limited to three)
    static constexpr int NST = NUQ ? (SLOT <= 10240 ? 3 : 2) : (SLOT <= 13312 ? 4 : 3);
    static constexpr int NKS = D / 16;
    static constexpr int NMT = D / 16;
    static constexpr int PR = D + 4;  // floats per head in a partial record: acc[D], m, l, 0, 0
    static constexpr int MINB = (NUQ || BK == 3 || SLOT > 9216) ? 3 : 4;  // resident CTAs per SM
};


// ---- shared memory -----------------------------------------------------------
template <int D, int BK, int BV, bool M16, int NUQ = 0>
struct Smem {
    using C = Cfg<D, BK, BV, M16, NUQ>;
    // query operands of up to two units at a time: [unit slot][kind: 0 16-bit
    // tiles, 1 packed][half: 0 hi, 1 lo][head][channel] 16-bit values, rows
    // padded by 8 so that the 8 (half, head) rows of a warp's load hit
    // different banks
    uint16_t qh[2][2][2][4][D + 8];
    float qsum[2][4], qmu[2][4];
    float msc[4][4], mM[4], mL[4];  // CTA merge: per-warp scale, max and sum per head
    union {
        float merge[4][4][C::PR];  // [warp][head][acc[D], m, l, -, -]
        float qscr[4][D];          // query preparation (dense rotation): raw q per head
    };
    uint64_t full[C::NST];         // slot filled (transaction count of its copies)
    unsigned rel[C::NST];          // releases of a slot so far (4 per entry)
    // non-uniform scheme only (one element otherwise): key tables [unit slot]
    // [channel][level], this block's probabilities per warp, and the value
    // side channel's corrections per warp [warp][head][channel]
    uint16_t lutk[NUQ ? 2 : 1][NUQ ? D * C::LV : 1];
    float pb[NUQ ? 4 : 1][4][NUQ ? C::SUB : 1];
    float corr[NUQ ? 4 : 1][4][NUQ ? D : 1];
    alignas(128) uint8_t ring[C::NST][C::SLOT];
};

// Shared-memory counter increment with acquire-release ordering at CTA scope;
// returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p) {
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;\n" : "=r"(old) : "r"(smem_u32(p)) : "memory");
    return old;
}

// Arrive on an mbarrier from one elected lane of the warp.
__device__ __forceinline__ void mbar_arrive_elect(uint64_t *bar) {
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(smem_u32(bar))
        : "memory");
}

// Pipeline entry e of unit u into a ring slot, issued by one elected lane of
// the calling warp (all lanes call it with the same arguments).  Entries
// [0, n_rt) are 16-slot tiles of 16-bit keys and values; entry n_rt + p holds
// packed tokens [p*ST, p*ST + ST): keys, value pairs, key meta, value meta,
// each at its fixed offset in the slot.  A last entry that would run past the
// unit's capacity copies the 64 tokens that exist (capacity is a multiple of 64).
template <int D, int BK, int BV, bool M16, int NUQ = 0>
__device__ __forceinline__ void issue_entry(const AttnArgs &a, const AttnShape &sh, int u, int e, uint8_t *slot,
                                            uint64_t *bar) {
    using C = Cfg<D, BK, BV, M16, NUQ>;
    const uint32_t sb = smem_u32(slot), br = smem_u32(bar);
    if (e < a.n_rt) {
        const long long r0 = static_cast<long long>(u) * sh.rcap + static_cast<long long>(e) * RTILE;
        const uint16_t *rk = a.raw_k + r0 * D, *rv = a.raw_v + r0 * D;
        asm volatile(
            "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
            "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %4, [%0];\n}\n" ::"r"(br),
            "n"(64 * D), "r"(sb), "l"(rk), "n"(32 * D), "r"(sb + 32 * D), "l"(rv)
            : "memory");
        return;
    }
    const long long t0 = static_cast<long long>(e - a.n_rt) * C::ST;
    const uint32_t nt = sh.qcap - t0 >= C::ST ? C::ST : static_cast<uint32_t>(sh.qcap - t0);
    const long long g0 = static_cast<long long>(u) * sh.qcap + t0;
    const uint8_t *ck = a.codes_k + g0 * C::ROWK;
    const uint8_t *cv = a.codes_v + g0 / 2 * C::PAIRV;
    if constexpr (NUQ) {
        const int gv = NUQ == 2 ? a.gv : 1;
        const uint8_t *lv = reinterpret_cast<const uint8_t *>(a.lut_v) + g0 * gv * C::LV * 2;
        const uint32_t kb = nt * C::ROWK, vb = nt / 2 * C::PAIRV, lb = nt * gv * C::LV * 2;
        if constexpr (NUQ == 2) if (a.refit) {  // plus the key tables of the entry's block
            const uint8_t *lk = reinterpret_cast<const uint8_t *>(a.lut_k) +
                                (static_cast<long long>(u) * a.nbk + t0 / a.refit) * C::LUTK;
            asm volatile(
                "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
                "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
                "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
                "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n"
                "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%11], [%12], %13, [%0];\n}\n" ::"r"(br),
                "r"(kb + vb + lb + static_cast<uint32_t>(C::LUTK)), "r"(sb), "l"(ck), "r"(kb), "r"(sb + C::KBYTES), "l"(cv),
                "r"(vb), "r"(sb + C::KBYTES + C::VBYTES), "l"(lv), "r"(lb), "r"(sb + C::KBYTES + C::VBYTES + C::LUTV),
                "l"(lk), "n"(C::LUTK)
                : "memory");
            return;
        }
        asm volatile(
            "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
            "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
            "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n}\n" ::"r"(br),
            "r"(kb + vb + lb), "r"(sb), "l"(ck), "r"(kb), "r"(sb + C::KBYTES), "l"(cv), "r"(vb),
            "r"(sb + C::KBYTES + C::VBYTES), "l"(lv), "r"(lb)
            : "memory");
        return;
    }
    const uint8_t *mk = static_cast<const uint8_t *>(a.meta_k) + g0 * 2 * C::MB;
    const uint8_t *mv = static_cast<const uint8_t *>(a.meta_v) + g0 * 2 * C::MB;
    const uint32_t kb = nt * C::ROWK, vb = nt / 2 * C::PAIRV, mb = nt * 2 * C::MB;
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%2], [%3], %4, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%5], [%6], %7, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%0];\n"
        "@p cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%11], [%12], %10, [%0];\n}\n" ::"r"(br),
        "r"(kb + vb + 2 * mb), "r"(sb), "l"(ck), "r"(kb), "r"(sb + C::KBYTES), "l"(cv), "r"(vb),
        "r"(sb + C::KBYTES + C::VBYTES), "l"(mk), "r"(mb), "r"(sb + C::KBYTES + C::VBYTES + C::MBYTES), "l"(mv)
        : "memory");
}


// ---- non-uniform scheme ---------------------------------------------------------
// Integer codes (half 0, half 1) of field r of a lane's record slice; the same
// fields extract<BITS> turns into mma operands in the affine scheme.
template <int BITS>
__device__ __forceinline__ void field_codes(const uint32_t *w, int r, uint32_t &m0, uint32_t &m1) {
    if (BITS == 4) {
        const uint32_t x = w[r >> 2], sh = 4 * (r & 3);
        m0 = (x >> sh) & 15u;
        m1 = (x >> (16 + sh)) & 15u;
        return;
    }
    const uint32_t x = w[r >> 3], sh = 2 * (r & 7);
    m0 = (x >> sh) & 3u;
    m1 = (x >> (16 + sh)) & 3u;
    if (BITS == 3) {  // the 1-bit plane word holds register r at bits bit1_pos(r) and 16 + bit1_pos(r)
        m0 |= ((w[2] >> bit1_pos(r)) & 1u) << 2;
        m1 |= ((w[2] >> (16 + bit1_pos(r))) & 1u) << 2;
    }
}

// Code of field idx, half `half` of a whole record (words_lo: 2-bit plane
// words of a 3-bit record).
template <int BITS>
__device__ __forceinline__ uint32_t code_in_rec(const uint8_t *rec, int idx, int half, int words_lo) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(rec);
    if (BITS == 3) {
        const uint32_t lo = (w[idx >> 3] >> (16 * half + 2 * (idx & 7))) & 3u;
        const uint32_t hi = (w[words_lo + (idx >> 4)] >> (16 * half + bit1_pos(idx & 15))) & 1u;
        return lo | (hi << 2);
    }
    constexpr int F = 16 / BITS;
    return (w[idx / F] >> (16 * half + BITS * (idx % F))) & ((1u << BITS) - 1u);
}

__device__ __forceinline__ float f16v(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// This warp's SUB tokens of a non-uniform entry -> warp state.  Operands are
// table values: K^[r][c] = lut_k[c][code] from the unit's key tables in
// shared memory, V^[t][c] = lut_v[t][code] from the tokens' tables in the
// slot ("KVQuant-NUQ" page: dequantize = table lookup).  Outliers keep their
// fp16 value: a key outlier adds q_c (x - table value) to its logit, a value
// outlier adds p_t (x - table value) to corr[head][c] (kept in the warp
// state's scale).  Both side channels are read a whole warp at a time, their
// loads issued before the key contraction; contributions meet in shared
// memory (pb holds the logit corrections, then the probabilities).
template <int D, int BK, int BV>
__device__ __forceinline__ void process_block_nuq(const uint8_t *kp, const uint8_t *vp, const uint16_t *lvp, int gv,
                                                  int valid, const uint32_t (&qb)[D / 16][2], const uint16_t *lutk,
                                                  const uint16_t (*qhl)[4][D + 8], float sm_l2, WarpState<D / 16> &st,
                                                  float (*corr)[D], float (*pb)[32], const AttnArgs &a,
                                                  const AttnShape &sh, int u, long long s0) {
    constexpr int NKS = D / 16, NMT = D / 16, T = 2, LV = 1 << BV, ROWK = D * BK / 8, PAIRV = 2 * D * BV / 8;
    constexpr int NWK = Slice<D, BK>::NW, NWV = Slice<D, BV>::NW;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    // side-channel loads first: key row starts of this warp's tokens, value outliers of this lane's token
    const int *rp = a.ol_rowptr_k ? a.ol_rowptr_k + static_cast<long long>(u) * a.rp_stride + s0 : nullptr;
    int rpv = 0, e_end = 0;
    if (rp) {  // valid counts every token to the end of the cache; this warp's rows are the first 32
        const int vr = valid < 32 ? valid : 32;
        rpv = rp[lane < vr ? lane : vr];
        e_end = rp[vr];
    }
    const int kv = a.k_out_v;
    const long long tv = static_cast<long long>(u) * sh.qcap + s0 + lane;
    uint32_t cv0 = 0xffffu, xv0 = 0u;
    if (kv > 0 && lane < valid) {
        cv0 = a.ol_col_v[tv * kv];
        xv0 = a.ol_val_v[tv * kv];
    }
    const uint16_t *lk = lutk + 2 * tig * LV;  // table rows of this lane's channels 16i + 2tig + 8sub + e
    // the two key tiles run through one copy of the (large, table-lookup) code
    float lg[2 * T];
#pragma unroll 1
    for (int t = 0; t < T; t++) {
        uint32_t k0[NWK], k1[NWK];
        load_k_slice<D, BK>(kp + (16 * t + g) * ROWK, tig, k0);
        load_k_slice<D, BK>(kp + (16 * t + g + 8) * ROWK, tig, k1);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < NKS; i++) {
            uint32_t m0, m1, r[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int f = 2 * i + (q >> 1);
                field_codes<BK>((q & 1) ? k1 : k0, f, m0, m1);
                const uint16_t *l0 = lk + (16 * i + 8 * (q >> 1)) * LV;
                r[q] = pack2(l0[m0], l0[LV + m1]);
            }
            mma_f16(s4, r[0], r[1], r[2], r[3], qb[i][0], qb[i][1]);
        }
        const float l0 = sm_l2 * (s4[0] + s4[1]), l1 = sm_l2 * (s4[2] + s4[3]);
        if (t == 0) {
            lg[0] = l0;
            lg[1] = l1;
        } else {
            lg[2] = l0;
            lg[3] = l1;
        }
    }
    if (rp) {  // key side channel: one lane per entry of [row start of token 0, end of the last token)
        pb[0][lane] = pb[1][lane] = pb[2][lane] = pb[3][lane] = 0.f;
        __syncwarp();
        const int e_beg = __shfl_sync(FULL, rpv, 0);
        for (int eb = e_beg; eb < e_end; eb += 32) {
            const int e = eb + lane;
            int r = 0;  // the token of entry e: the last row starting at or before it
#pragma unroll
            for (int stp = 16; stp; stp >>= 1) {
                const int s = __shfl_sync(FULL, rpv, r + stp);
                if (r + stp < 32 && s <= e) r += stp;
            }
            if (e < e_end) {
                const long long ei = static_cast<long long>(u) * a.nnzk_cap + e;
                const int c = a.ol_col_k[ei];
                const float x = f16v(a.ol_val_k[ei]);
                const uint32_t m = code_in_rec<BK>(kp + r * ROWK, k_idx(c, D), c & 1, D / 16);
                const float dlt = x - f16v(lutk[c * LV + m]);
#pragma unroll
                for (int h = 0; h < 4; h++)  // q = its fp16 hi + lo halves (about 22 significant bits)
                    atomicAdd(&pb[h][r], (f16v(qhl[0][h][c]) + f16v(qhl[1][h][c])) * dlt);
            }
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2 * T; k++) lg[k] += sm_l2 * pb[tig][16 * (k >> 1) + g + 8 * (k & 1)];
        __syncwarp();
    }
    const bool ragged = valid < 32;
    if (ragged) {
#pragma unroll
        for (int k = 0; k < 2 * T; k++)
            if (16 * (k >> 1) + g + 8 * (k & 1) >= valid) lg[k] = -INFINITY;
    }
    float p[2 * T];
    const float al = st.template update<2 * T>(lg, p);
    if (kv > 0) {
        if (al != 1.f) {
#pragma unroll
            for (int j = 0; j < D / 8; j++) corr[tig][8 * j + g] *= al;
        }
#pragma unroll
        for (int k = 0; k < 2 * T; k++) pb[tig][16 * (k >> 1) + g + 8 * (k & 1)] = p[k];
        __syncwarp();
    }
    // P . V per tile: A = V^T (channels x tokens) from the tokens' tables
#pragma unroll 1
    for (int t = 0; t < T; t++) {
        const uint32_t b0 = movmatrix_t(hilo_f16(t == 0 ? p[0] : p[2]));
        const uint32_t b1 = movmatrix_t(hilo_f16(t == 0 ? p[1] : p[3]));
        uint32_t v0[NWV], v1[NWV];
        load_v_slice<D, BV>(vp + (8 * t + tig) * PAIRV, g, v0);
        load_v_slice<D, BV>(vp + (8 * t + tig + 4) * PAIRV, g, v1);
        // token 16t + 2tig (+1, +8, +9)'s tables; channels 16mi .. 16mi + 15 share one group's
        const int TV = gv * LV;  // table entries per token
        const uint16_t *la0 = lvp + (16 * t + 2 * tig) * TV, *lb0 = la0 + 8 * TV;
#pragma unroll
        for (int mi = 0; mi < NMT; mi++) {
            const int go = (16 * mi * gv) / D * LV;
            const uint16_t *la = la0 + go, *lb = lb0 + go;
            uint32_t m0, m1, r[4];
            field_codes<BV>(v0, 2 * mi, m0, m1);
            r[0] = pack2(la[m0], la[TV + m1]);
            field_codes<BV>(v0, 2 * mi + 1, m0, m1);
            r[1] = pack2(la[m0], la[TV + m1]);
            field_codes<BV>(v1, 2 * mi, m0, m1);
            r[2] = pack2(lb[m0], lb[TV + m1]);
            field_codes<BV>(v1, 2 * mi + 1, m0, m1);
            r[3] = pack2(lb[m0], lb[TV + m1]);
            mma_f16(st.acc[mi], r[0], r[1], r[2], r[3], b0, b1);
        }
    }
    if (kv > 0) {  // value side channel: lane t adds p_t (x - table value) at its outlier channels
        for (int j = 0; j < kv; j++) {
            uint32_t c = cv0, xb = xv0;
            if (j > 0 && lane < valid) {
                c = a.ol_col_v[tv * kv + j];
                xb = a.ol_val_v[tv * kv + j];
            }
            if (lane < valid && c != 0xffffu) {
                const uint32_t m = code_in_rec<BV>(vp + (lane >> 1) * PAIRV, v_idx(static_cast<int>(c), D), lane & 1, D / 8);
                const float dlt = f16v(static_cast<uint16_t>(xb)) - f16v(lvp[(lane * gv + static_cast<int>(c) * gv / D) * LV + m]);
#pragma unroll
                for (int h = 0; h < 4; h++) atomicAdd(&corr[h][c], pb[h][lane] * dlt);
            }
        }
        __syncwarp();
    }
}

// Warp state of a non-uniform segment -> [acc[D], m, l] of head tig at dst:
// rows are channels, plus the value side channel's corrections.
template <int D>
__device__ __forceinline__ void store_state_nuq(WarpState<D / 16> &st, const float (*corr)[D], float *dst, int PR) {
    constexpr int NMT = D / 16;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l += __shfl_xor_sync(FULL, st.l, o);
    float *wp = dst + tig * PR;
#pragma unroll
    for (int mi = 0; mi < NMT; mi++)
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int row = 16 * mi + 8 * rr + g;
            wp[row] = st.acc[mi][2 * rr] + st.acc[mi][2 * rr + 1] + corr[tig][row];
        }
    if (g == 0) {
        wp[D] = st.m;
        wp[D + 1] = st.l;
    }
}

// This warp's SUB packed tokens of an entry -> warp state.  `kp`, `vp`, `mkp`,
// `mvp` point at the warp's first key record, value pair record, key meta and
// value meta in the slot; tokens at or past `valid` (0 < valid) are masked.
template <int D, int BK, int BV, bool M16>
__device__ __forceinline__ void process_block(const uint8_t *kp, const uint8_t *vp, const uint8_t *mkp,
                                              const uint8_t *mvp, int valid, const uint32_t (&qb)[D / 16][2],
                                              float sk_l2, float qs_l2, float qm_l2, WarpState<D / 16> &st) {
    using C = Cfg<D, BK, BV, M16>;
    constexpr int NKS = C::NKS, NMT = C::NMT, T = C::TILES;
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    // q . K^T for the tiles of the block
    float sc[T][4];
#pragma unroll
    for (int t = 0; t < T; t++) {
        constexpr int NW = Slice<D, BK>::NW;
        uint32_t k0[NW], k1[NW];
        load_k_slice<D, BK>(kp + (16 * t + g) * C::ROWK, tig, k0);
        load_k_slice<D, BK>(kp + (16 * t + g + 8) * C::ROWK, tig, k1);
        sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
        for (int i = 0; i < NKS; i++)
            mma_f16(sc[t], extract<BK>(k0, 2 * i), extract<BK>(k1, 2 * i), extract<BK>(k0, 2 * i + 1),
                    extract<BK>(k1, 2 * i + 1), qb[i][0], qb[i][1]);
    }
    // logits of tokens 16t+g (k = 2t) and 16t+g+8 (k = 2t+1) for head tig
    float lg[2 * T];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
            const float2 km = ld_meta(mkp, 16 * t + g + 8 * hf, M16);
            const float dot = sc[t][2 * hf] + sc[t][2 * hf + 1];
            lg[2 * t + hf] = (km.x * sk_l2) * dot + (km.y * qs_l2 + qm_l2);
        }
    const bool ragged = valid < C::SUB;  // warp-uniform: the unit's last entry
    if (ragged) {
#pragma unroll
        for (int k = 0; k < 2 * T; k++)
            if (16 * (k >> 1) + g + 8 * (k & 1) >= valid) lg[k] = -INFINITY;
    }
    float p[2 * T];
    st.template update<2 * T>(lg, p);
    // P . V per tile: A = V^T (channels x tokens), B = (P * s_v) transposed by
    // movmatrix; the offsets o_v accumulate separately (Eq. 9)
    float aos = 0.f;
#pragma unroll
    for (int t = 0; t < T; t++) {
        float2 vm0 = ld_meta(mvp, 16 * t + g, M16), vm1 = ld_meta(mvp, 16 * t + g + 8, M16);
        if (ragged) {  // masked tokens have p = 0, but their metadata may be anything
            if (16 * t + g >= valid) vm0 = make_float2(0.f, 0.f);
            if (16 * t + g + 8 >= valid) vm1 = make_float2(0.f, 0.f);
        }
        aos += p[2 * t] * vm0.y + p[2 * t + 1] * vm1.y;
        const uint32_t b0 = movmatrix_t(hilo_f16(p[2 * t] * vm0.x));
        const uint32_t b1 = movmatrix_t(hilo_f16(p[2 * t + 1] * vm1.x));
        constexpr int NW = Slice<D, BV>::NW;
        uint32_t v0[NW], v1[NW];
        load_v_slice<D, BV>(vp + (8 * t + tig) * C::PAIRV, g, v0);
        load_v_slice<D, BV>(vp + (8 * t + tig + 4) * C::PAIRV, g, v1);
#pragma unroll
        for (int mi = 0; mi < NMT; mi++)
            mma_f16(st.acc[mi], extract<BV>(v0, 2 * mi), extract<BV>(v0, 2 * mi + 1), extract<BV>(v1, 2 * mi),
                    extract<BV>(v1, 2 * mi + 1), b0, b1);
    }
    st.ao += aos;
}

// Merge the split records of unit u, rotate the value accumulator back,
// normalize and write the output.
// Records are read in batches of 16 whose loads are all in flight together
// (one batch for up to 8 CTAs per unit), merged with a running maximum.
template <int D, int PR>
__device__ __forceinline__ void combine_unit(const AttnArgs &a, const AttnShape &sh, int u, int n_ctas) {
    constexpr int V = D / 32, NB = 16;
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
                if (mr[k] == -INFINITY) continue;  // empty record: its value row was never written
                const float w = exp2f(mr[k] - M);
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
}

// One lane's share of a unit's query head (warp h takes head h; lane l holds
// channels l*V .. l*V+V-1) and of the key channel mean.  Loaded first thing, so
// that the loads are in flight before the cache copies.
template <int V>
struct QIn {
    float xq[V], mu[V], xt[V];  // xt: the compensated query when it was computed beforehand
};
template <int D>
__device__ __forceinline__ void load_query(const AttnArgs &a, const AttnShape &sh, int u, QIn<D / 32> &in) {
    constexpr int V = D / 32;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = u / sh.Hkv, kvh = u % sh.Hkv;
    const long long qo = (static_cast<long long>(b) * sh.Hkv * sh.G + kvh * sh.G + h) * D + lane * V;
    const long long mo = static_cast<long long>(u) * D + lane * V;
#pragma unroll
    for (int j = 0; j < V; j++) {
        in.xq[j] = h < sh.G ? __ldg(a.q + qo + j) : 0.f;
        in.mu[j] = a.mean_k ? __ldg(a.mean_k + mo + j) : 0.f;
        in.xt[j] = a.q_tilde && h < sh.G ? __ldg(a.q_tilde + qo + j) : 0.f;
    }
}

// The (hi, lo) 16-bit halves of v into S.qh[qs][kind][0 / 1][h][c].
template <int D, int BK, int BV, bool M16, int NUQ>
__device__ __forceinline__ void put_hilo(Smem<D, BK, BV, M16, NUQ> &S, int qs, int kind, int h, int c, float v,
                                         bool bf16) {
    const uint32_t w = bf16 ? hilo_bf16(v) : hilo_f16(v);
    S.qh[qs][kind][0][h][c] = static_cast<uint16_t>(w & 0xffffu);
    S.qh[qs][kind][1][h][c] = static_cast<uint16_t>(w >> 16);
}

// Query preparation of unit u into slot qs (warp h: head h).  Kind 0 (16-bit
// keys): raw q in the raw region's 16-bit type.  Kind 1 (packed keys): q
// rotated (or compensated) and scaled by 2^-E for the code field E that
// channel c meets in the key operand (register c>>3 of a lane's slice); also
// sum q and q . mu for the fold of the affine code (Eq. 8).
template <int D, int BK, int BV, bool M16, int NUQ>
__device__ __forceinline__ void prep_query(const AttnArgs &a, const AttnShape &sh, Smem<D, BK, BV, M16, NUQ> &S,
                                           int qs, int u, const QIn<D / 32> &in) {
    constexpr int V = D / 32;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float xq[V];
#pragma unroll
    for (int j = 0; j < V; j++) {
        xq[j] = in.xq[j];
        put_hilo(S, qs, 0, h, lane * V + j, xq[j], a.raw_bf16 != 0);
    }
    if (a.rot_k == DQ_ROT_HADAMARD) {
        fwht_warp<V>(xq);
#pragma unroll
        for (int j = 0; j < V; j++) xq[j] *= a.hscale;
    } else if (a.rot_k == DQ_ROT_DENSE && a.q_tilde) {
        // q~ = T^{-T} q, computed once per call by qcomp_kernel
#pragma unroll
        for (int j = 0; j < V; j++) xq[j] = in.xt[j];
    } else if (a.rot_k == DQ_ROT_DENSE) {
        // q~ = T^{-T} q with the caller's fp32 compensation matrix (no workspace for it)
        __syncwarp();
#pragma unroll
        for (int j = 0; j < V; j++) S.qscr[h][lane * V + j] = xq[j];
        __syncwarp();
        const float *Qc = a.q_comp + static_cast<long long>(u % sh.Hkv) * D * D;
#pragma unroll
        for (int j = 0; j < V; j++) {
            float acc = 0.f;
            const float *row = Qc + static_cast<long long>(lane * V + j) * D;
            for (int k = 0; k < D; k++) acc += row[k] * S.qscr[h][k];
            xq[j] = acc;
        }
        __syncwarp();
    }
    float qsum = 0.f, qmu = 0.f;
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane * V + j;
        qsum += xq[j];
        qmu += xq[j] * in.mu[j];
        // packed keys: 2^-E of the code field (affine), or 1 (table values)
        const float sc = NUQ ? 1.f : __int_as_float((127 - field_exp(c >> 3, BK)) << 23);
        put_hilo(S, qs, 1, h, c, xq[j] * sc, false);
    }
    qsum = warp_sum(qsum);
    qmu = warp_sum(qmu);
    if (lane == 0) {
        S.qsum[qs][h] = qsum;
        S.qmu[qs][h] = qmu;
    }
    if constexpr (NUQ) {  // the unit's key tables
        constexpr int LV = Cfg<D, BK, BV, M16, NUQ>::LV;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.lut_k + static_cast<long long>(u) * a.nbk * D * LV);
        uint32_t *dst = reinterpret_cast<uint32_t *>(S.lutk[qs]);
        for (int i = threadIdx.x; i < D * LV / 2; i += blockDim.x) dst[i] = src[i];
    }
}

// This lane's mma B operand of q.K^T from the prepared halves: column g of the
// operand is head g>>1, half g&1; lane slot (k-step i, sub, e) holds channel
// perm(i, tig, sub, e), and e = 0, 1 are adjacent channels (one 32-bit load).
template <int D, int BK, int BV, bool M16, int NUQ, typename Perm>
__device__ __forceinline__ void load_qb(const Smem<D, BK, BV, M16, NUQ> &S, int qs, int kind, Perm perm,
                                        uint32_t (&qb)[D / 16][2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const uint16_t *row = S.qh[qs][kind][g & 1][g >> 1];
#pragma unroll
    for (int i = 0; i < D / 16; i++)
#pragma unroll
        for (int sub = 0; sub < 2; sub++) qb[i][sub] = *reinterpret_cast<const uint32_t *>(row + perm(i, tig, sub, 0));
}

// ---- the kernel ----------------------------------------------------------------
// A CTA walks its range [x0, x1) of pipeline entries unit by unit; a unit's
// entries are its 16-slot tiles of 16-bit tokens, then its packed entries of
// ST tokens.  NST entries are in flight in a CTA-wide ring of bulk copies
// (completion on full[s]); the last of the four warps to be done with a slot
// refills it.  Every warp takes SUB tokens of each packed entry; a 16-bit tile
// goes to warp (tile index mod 4).  The query loads go out first, then the
// first NST copies, then the queries are prepared.  Every warp waits on full[]
// for every entry (also the 16-bit tiles it leaves to another warp): a warp is
// then never more than one phase ahead of a slot, which the parity test of the
// wait requires.
template <int D, int BK, int BV, bool M16, int NUQ = 0>
__global__ void __launch_bounds__(128, Cfg<D, BK, BV, M16, NUQ>::MINB) attn_kernel(AttnArgs a, AttnShape sh) {
    using C = Cfg<D, BK, BV, M16, NUQ>;
    constexpr int PR = C::PR, NKS = C::NKS, NST = C::NST;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<D, BK, BV, M16, NUQ> &S = *reinterpret_cast<Smem<D, BK, BV, M16, NUQ> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3;
    const int G = gridDim.x, i = blockIdx.x;
    const long long N = a.total_items;
    const int ipu = static_cast<int>(a.items_per_unit), n_rt = a.n_rt;
    const long long x0 = static_cast<long long>(i) * N / G, x1 = static_cast<long long>(i + 1) * N / G;
    const int n_ent = static_cast<int>(x1 - x0);
    // the combine grid may be scheduled now; it waits for this whole grid
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    if (n_ent <= 0 || ipu <= 0) return;
    const int u_first = static_cast<int>(x0 / ipu), u_lastc = static_cast<int>((x1 - 1) / ipu);
    bool timed_out = false;

    // the queries of the CTA's first two units: their loads go out before the copies
    QIn<D / 32> qin0, qin1;
    load_query<D>(a, sh, u_first, qin0);
    if (u_lastc > u_first) load_query<D>(a, sh, u_first + 1, qin1);

    // the CTA's entry k -> (unit, entry of the unit), copied into slot k % NST
    // (all lanes of a warp call it; one elected lane issues)
    auto issue_k = [&](int k) {
        const unsigned x = static_cast<unsigned>(x0) + static_cast<unsigned>(k);
        const unsigned u = x / static_cast<unsigned>(ipu);
        issue_entry<D, BK, BV, M16, NUQ>(a, sh, static_cast<int>(u), static_cast<int>(x - u * ipu), S.ring[k % NST],
                                    &S.full[k % NST]);
    };
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < NST; s++) {
                mbar_init(&S.full[s], 1);
                S.rel[s] = 0;
            }
            fence_mbar_init();
        }
        __syncwarp();
        for (int k = 0; k < NST && k < n_ent; k++) issue_k(k);
    }
    prep_query<D, BK, BV, M16, NUQ>(a, sh, S, 0, u_first, qin0);
    if (u_lastc > u_first) prep_query<D, BK, BV, M16, NUQ>(a, sh, S, 1, u_first + 1, qin1);

    int j = 0;  // the CTA's entry being consumed
    auto acquire = [&]() -> const uint8_t * {
        if (!mbar_wait(&S.full[j % NST], (j / NST) & 1, WAIT_LIMIT_NS)) timed_out = true;
        return S.ring[j % NST];
    };
    // done with slot j % NST: the last of the four warps to release it (an
    // acquire-release count of releases) loads entry j + NST into it
    auto release = [&]() {
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atom_add_acq_rel(&S.rel[j % NST]);
        old = __shfl_sync(FULL, old, 0);
        if ((old & 3u) == 3u && j + NST < n_ent) issue_k(j + NST);
        ++j;
    };
    // CTA merge of the 4 warps' states in S.merge -> one record of 4 heads at
    // dst (called after a __syncthreads that follows the warps' stores)
    auto cta_merge = [&](float *dst) {
        if (threadIdx.x < 4) {
            const int h = threadIdx.x;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; w++) M = fmaxf(M, S.merge[w][h][D]);
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                const float mw = S.merge[w][h][D];
                const float sw = mw == -INFINITY ? 0.f : exp2f(mw - M);
                S.msc[w][h] = sw;
                L += sw * S.merge[w][h][D + 1];
            }
            S.mM[h] = M;
            S.mL[h] = L;
        }
        __syncthreads();
        constexpr int P4 = PR / 4;
        for (int idx = threadIdx.x; idx < 4 * P4; idx += blockDim.x) {
            const int h = idx / P4, c4 = idx - h * P4;
            float4 r;
            if (c4 < D / 4) {
                r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    const float sw = S.msc[w][h];
                    const float4 v = reinterpret_cast<const float4 *>(S.merge[w][h])[c4];
                    r.x += sw * v.x;
                    r.y += sw * v.y;
                    r.z += sw * v.z;
                    r.w += sw * v.w;
                }
            } else {
                r = make_float4(S.mM[h], S.mL[h], 0.f, 0.f);
            }
            reinterpret_cast<float4 *>(dst)[idx] = r;
        }
    };

    for (long long x = x0; x < x1;) {
        const int u = static_cast<int>(x / ipu);
        const long long ub = static_cast<long long>(u) * ipu;
        const long long xe = x1 < ub + ipu ? x1 : ub + ipu;
        const int e0 = static_cast<int>(x - ub), e1 = static_cast<int>(xe - ub);
        x = xe;
        const int qs = (u - u_first) & 1;
        __syncthreads();  // barriers and queries published; the last segment is done with S
        if (u - u_first >= 2) {
            QIn<D / 32> qin;
            load_query<D>(a, sh, u, qin);
            prep_query<D, BK, BV, M16, NUQ>(a, sh, S, qs, u, qin);
            __syncthreads();
        }
        const int first = owner(ub, N, G);
        float *recs = a.partials + (static_cast<long long>(u) * a.max_slots + (i - first)) * 2 * 4 * PR;
        WarpState<D / 16> st;

        // ---- 16-bit tiles: record kind 0 ----
        const int r1 = e1 < n_rt ? e1 : n_rt;
        if (e0 < r1) {
            uint32_t qb[NKS][2];
            load_qb(S, qs, 0, PermRawK(), qb);
            st.init();
            for (int e = e0; e < r1; e++) {
                // every warp waits for every entry, so that no warp runs a full
                // ring ahead and tests a slot's barrier two phases early
                const uint8_t *slot = acquire();
                if ((e & 3) == warp) {
                    if (a.raw_bf16) process_raw<D, true>(a, slot, static_cast<long long>(e) * RTILE, qb, st);
                    else process_raw<D, false>(a, slot, static_cast<long long>(e) * RTILE, qb, st);
                }
                release();
            }
            store_state<D, BV>(st, false, &S.merge[warp][0][0], PR);
            __syncthreads();
            cta_merge(recs);
            __syncthreads();  // S.merge is free again
        } else if (warp == 0 && lane < 4) {
            recs[lane * PR + D] = -INFINITY;  // no 16-bit tiles in this segment
            recs[lane * PR + D + 1] = 0.f;
        }

        // ---- packed entries: SUB tokens per warp; record kind 1 ----
        st.init();
        const int p0 = (e0 > n_rt ? e0 : n_rt) - n_rt, p1 = e1 - n_rt;
        if constexpr (NUQ) {
#pragma unroll
            for (int j = 0; j < D / 8; j++) S.corr[warp][tig][8 * j + (lane >> 2)] = 0.f;  // this lane's channels
            __syncwarp();
            if (p0 < p1) {
                uint32_t qb[NKS][2];
                load_qb(S, qs, 1, PermIdentity(), qb);
                const int wv = static_cast<int>(a.n_q) - warp * C::SUB;
                const int ok = warp * C::SUB * C::ROWK;
                const int ov = C::KBYTES + warp * (C::SUB / 2) * C::PAIRV;
                const int gv = NUQ == 2 ? a.gv : 1;
                const int ol = C::KBYTES + C::VBYTES + warp * C::SUB * gv * C::LV * 2;
                const bool blk_tables = NUQ == 2 && a.refit;  // key tables of the entry's refit block
#pragma unroll 1
                for (int q = p0; q < p1; q++) {
                    const uint8_t *slot = acquire();
                    const int valid = wv - q * C::ST;
                    const uint16_t *lutk = blk_tables ? reinterpret_cast<const uint16_t *>(slot + C::KBYTES + C::VBYTES + C::LUTV)
                                                      : S.lutk[qs];
                    if (valid > 0)
                        process_block_nuq<D, BK, BV>(slot + ok, slot + ov, reinterpret_cast<const uint16_t *>(slot + ol),
                                                     gv, valid, qb, lutk, S.qh[qs][1], a.sm_log2, st, S.corr[warp],
                                                     S.pb[warp], a, sh, u,
                                                     static_cast<long long>(q) * C::ST + warp * C::SUB);
                    release();
                }
            }
            store_state_nuq<D>(st, S.corr[warp], &S.merge[warp][0][0], PR);
        } else {
        if (p0 < p1) {
            uint32_t qb[NKS][2];
            load_qb(S, qs, 1, PermIdentity(), qb);
            const float qs_l2 = a.sm_log2 * S.qsum[qs][tig], qm_l2 = a.sm_log2 * S.qmu[qs][tig];
            const float sk_l2 = a.sm_log2 * 16777216.0f;  // 2^24 undoes the operand scaling
            const int wv = static_cast<int>(a.n_q) - warp * C::SUB;  // valid tokens of entry 0 for this warp
            // this warp's records in a slot: keys, value pairs, key meta, value meta
            const int ok = warp * C::SUB * C::ROWK;
            const int ov = C::KBYTES + warp * (C::SUB / 2) * C::PAIRV;
            const int omk = C::KBYTES + C::VBYTES + warp * C::SUB * 2 * C::MB;
            const int omv = omk + C::MBYTES;
#pragma unroll 1
            for (int q = p0; q < p1; q++) {
                const uint8_t *slot = acquire();
                const int valid = wv - q * C::ST;
                if (valid > 0)
                    process_block<D, BK, BV, M16>(slot + ok, slot + ov, slot + omk, slot + omv, valid, qb, sk_l2,
                                                  qs_l2, qm_l2, st);
                release();
            }
        }
        store_state<D, BV>(st, true, &S.merge[warp][0][0], PR);
        }
        __syncthreads();
        cta_merge(recs + 4 * PR);
        // publish: the records are visible GPU-wide before the unit's count moves
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) atomicAdd(a.counters + u, 1);
    }
    if (timed_out && lane == 0) atomicOr(a.status, ST_TIMEOUT);
}

// The split records of unit u -> output.  This grid is a programmatic
// dependent of the attention grid, so its CTAs can start as SMs free up; CTA u
// waits (bounded) until all CTAs that touch unit u have published their
// records, merges them and clears the unit's count for the next call.  The
// attention grid never waits on this one, so the wait always ends.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(AttnArgs a, AttnShape sh) {
    __shared__ int ok;
    const int u = blockIdx.x;
    const long long N = a.total_items, ipu = a.items_per_unit;
    const int first = owner(static_cast<long long>(u) * ipu, N, a.grid);
    const int last = owner(static_cast<long long>(u) * ipu + ipu - 1, N, a.grid);
    if (threadIdx.x == 0) {
        const int need = last - first + 1;
        const uint64_t t0 = global_ns();
        int got;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(got) : "l"(a.counters + u) : "memory");
            if (got >= need || global_ns() - t0 > WAIT_LIMIT_NS) break;
            __nanosleep(256);
        }
        ok = got >= need;
        if (!ok) atomicOr(a.status, ST_TIMEOUT);
    }
    __syncthreads();
    if (!ok) return;
    combine_unit<D, D + 4>(a, sh, u, last - first + 1);
    __syncthreads();
    if (threadIdx.x == 0) a.counters[u] = 0;
}

// ---- host side -------------------------------------------------------------
template <int D, int BK, int BV, bool M16, int NUQ = 0>
struct Launcher {
    static constexpr int ST = Cfg<D, BK, BV, M16, NUQ>::ST;
    static int occupancy;  // resident CTAs per SM, set on first use
    static size_t smem() { return sizeof(Smem<D, BK, BV, M16, NUQ>); }
    static int prepare() {
        if (occupancy > 0) return 0;
        auto kern = attn_kernel<D, BK, BV, M16, NUQ>;
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
        const cudaStream_t st = static_cast<cudaStream_t>(stream);
        attn_kernel<D, BK, BV, M16, NUQ><<<a.grid, 128, smem(), st>>>(a, sh);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return static_cast<int>(e);
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>(sh.U));
        lc.blockDim = dim3(128);
        lc.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        return static_cast<int>(cudaLaunchKernelEx(&lc, combine_kernel<D>, a, sh));
    }
};
template <int D, int BK, int BV, bool M16, int NUQ>
int Launcher<D, BK, BV, M16, NUQ>::occupancy = 0;

template <int D, bool M16, typename F>
static int dispatch_bits(const Layout &L, F &&f) {
    if (L.bits_k == 2 && L.bits_v == 2) return f(Launcher<D, 2, 2, M16>());
    if (L.bits_k == 4 && L.bits_v == 4) return f(Launcher<D, 4, 4, M16>());
    if (L.bits_k == 3 && L.bits_v == 3) return f(Launcher<128, 3, 3, M16>());
    return static_cast<int>(cudaErrorInvalidValue);
}

template <typename F>
static int dispatch(const Layout &L, F &&f) {
    if (L.scheme == DQ_NUQ) {  // no meta: one instantiation per (d, bits, table kind)
        if (L.d == 128 && (L.gv > 1 || L.refit > 0)) {
            if (L.bits_k == 2) return f(Launcher<128, 2, 2, true, 2>());
            if (L.bits_k == 3) return f(Launcher<128, 3, 3, true, 2>());
            return f(Launcher<128, 4, 4, true, 2>());
        }
        if (L.d == 128) {
            if (L.bits_k == 2) return f(Launcher<128, 2, 2, true, 1>());
            if (L.bits_k == 3) return f(Launcher<128, 3, 3, true, 1>());
            return f(Launcher<128, 4, 4, true, 1>());
        }
        if (L.bits_k == 2) return f(Launcher<64, 2, 2, true, 1>());
        return f(Launcher<64, 4, 4, true, 1>());
    }
    const bool m16 = L.meta_bytes == 2;
    if (L.d == 128) return m16 ? dispatch_bits<128, true>(L, f) : dispatch_bits<128, false>(L, f);
    return m16 ? dispatch_bits<64, true>(L, f) : dispatch_bits<64, false>(L, f);
}

long long attention_partial_floats(const Layout &L, const AttnArgs &a) {
    if (a.affine) return affine_partial_floats(L, a);
    return static_cast<long long>(L.U) * a.max_slots * 2 * 4 * (L.d + 4);
}

int plan_attention(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats) {
    a.affine = 0;
    if (affine_kernel_applies(L, a)) return plan_affine(L, a, num_sms, cap_floats);
    int occ = 0, st = 0;
    const int e = dispatch(L, [&](auto l) {
        const int r = decltype(l)::prepare();
        occ = decltype(l)::occupancy;
        st = decltype(l)::ST;
        return r;
    });
    if (e != 0) return e;
    a.n_rt = a.has_raw ? (a.n_raw_slots + RTILE - 1) / RTILE : 0;
    a.raw_all_valid = a.seq_len >= static_cast<long long>(a.n_sink_cfg) + a.n_recent_cfg;
    a.n_qc = (a.n_q + st - 1) / st;
    // a unit's pipeline entries: its 16-slot tiles of 16-bit tokens, then its
    // packed entries of st tokens
    a.items_per_unit = a.n_rt + a.n_qc;
    a.total_items = static_cast<long long>(L.U) * a.items_per_unit;
    if (a.total_items >= (1LL << 31)) return static_cast<int>(cudaErrorInvalidValue);  // entries are indexed in 32 bits
    long long G = static_cast<long long>(num_sms) * occ;
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

// q~ = T^{-T} q for every query head (WUSH-KV, Methodology: queries are
// compensated with the inverse transform).  One warp per (sequence, KV head,
// 32 output channels); lane i computes output channel 32 blk + i of the G
// query heads from its row of the fp32 compensation matrix (loads unrolled,
// so a lane has its whole row in flight at once).
template <int D>
__global__ void __launch_bounds__(32) qcomp_kernel(const float *q, const float *qc, float *qt, int Hkv, int G) {
    __shared__ float qs[4][D];
    constexpr int NB = D / 32;
    const int blk = blockIdx.x % NB, bk = blockIdx.x / NB;
    const int b = bk / Hkv, kvh = bk % Hkv, lane = threadIdx.x, i = 32 * blk + lane;
    const long long q0 = (static_cast<long long>(b) * Hkv + kvh) * G * D;
    for (int g = 0; g < G; g++)
        for (int c = lane; c < D; c += 32) qs[g][c] = q[q0 + static_cast<long long>(g) * D + c];
    __syncwarp();
    const float4 *row = reinterpret_cast<const float4 *>(qc + (static_cast<long long>(kvh) * D + i) * D);
    float4 r[D / 4];
#pragma unroll
    for (int k4 = 0; k4 < D / 4; k4++) r[k4] = __ldg(row + k4);
    for (int g = 0; g < G; g++) {
        float acc = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < D / 4; k4++)
            acc += r[k4].x * qs[g][4 * k4] + r[k4].y * qs[g][4 * k4 + 1] + r[k4].z * qs[g][4 * k4 + 2] +
                   r[k4].w * qs[g][4 * k4 + 3];
        qt[q0 + static_cast<long long>(g) * D + i] = acc;
    }
}

int launch_qcomp(const Layout &L, const float *q, const float *qc, float *qt, void *stream) {
    const unsigned grid = static_cast<unsigned>(L.U) * static_cast<unsigned>(L.d / 32);
    if (L.d == 128) qcomp_kernel<128><<<grid, 32, 0, static_cast<cudaStream_t>(stream)>>>(q, qc, qt, L.Hkv, L.G);
    else qcomp_kernel<64><<<grid, 32, 0, static_cast<cudaStream_t>(stream)>>>(q, qc, qt, L.Hkv, L.G);
    return static_cast<int>(cudaGetLastError());
}

int launch_attention(const Layout &L, const AttnArgs &a, int, void *stream) {
    if (a.affine) return launch_affine(L, a, stream);
    AttnShape sh{L.U, L.Hkv, L.G, L.d, L.qcap, L.rcap};
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

namespace dq {
namespace {

// One warp; lane 0 initialises an mbarrier that nothing arrives at and waits
// on it with the bounded wait every pipeline here uses.  When the wait gives
// up it latches ST_TIMEOUT and bumps unit 0's record count, as an attention
// CTA that stopped waiting midway can, then completes the phase itself so the
// barrier is quiet before it is invalidated.
__global__ void __launch_bounds__(32) expire_wait_kernel(unsigned *status, int *counters, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(b) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    if (!mbar_wait(&bar, 0, limit_ns)) {
        atomicOr(status, ST_TIMEOUT);
        atomicAdd(counters, 1);
    }
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(b) : "memory");
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(b) : "memory");
}

// One lane tests a byte range that ends one byte past a 4-byte buffer (the
// status word itself): the checked build latches ST_OOB; nothing is accessed.
__global__ void __launch_bounds__(32) checked_probe_kernel(unsigned *status) {
    if (threadIdx.x == 0) (void)in_buf(reinterpret_cast<const char *>(status) + 1, 4, status, 4, status);
}

}  // namespace

int launch_checked_probe(unsigned *status, void *stream) {
    checked_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return static_cast<int>(cudaGetLastError());
}

int launch_expire_wait(unsigned *status, int *counters, unsigned long long limit_ns, void *stream) {
    expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, counters, limit_ns);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace dq
