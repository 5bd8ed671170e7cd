// Decode attention over D-Quant entropy-coded containers (sm_103a).
//
// "D-Quant: Driftable Entropy Coding for KV Cache Quantization", Sec. 4.5
// Decoding and App. A:
//  * a stream spans all KV heads of a token, so decoding is organised around
//    tokens: every stream is decoded once, one lane per token, head after
//    head (the stream's order), and the decoded levels feed that head's
//    query heads directly;
//  * Algorithm 2: state from the first 4 bytes, z = x mod 2^8 selects the
//    table entry (level, f, c), x <- f floor(x / 2^8) + z - c, one byte shifted
//    in while x < 2^23; one lookup serves decoding and reconstruction;
//  * Eq. (8): q . k^_t = s_t sum_j q_j m_tj + o_t sum_j q_j + sum_j q_j mu_j, so
//    keys contract decoded levels and apply the affine terms afterwards;
//  * Eq. (9): sum_t a_t v^_tj = sum_t (a_t s_t) m_tj + sum_t a_t o_t, so the
//    value scale folds into the attention weight and the offset is summed
//    apart.
// Work: an item is 512 quantized tokens of one sequence (4 warps x 4 chunks of
// 32 tokens) or the 16-bit tokens (sinks + recent window) of one sequence.
// Per KV head h a warp, for each of its chunks, decodes 128 key and 128 value
// symbols per lane, takes the key dot products with the rotated query rows
// (scalar FMAs, the rows of head h's query heads prepared in shared memory at
// the start of the head and broadcast from there), updates the online
// softmax of the G query heads, stages the value levels in shared memory and
// runs P.V on the tensor cores (mma m16n8k16, 8 columns = 4 query heads x hi/lo
// halves of P' = p s).  The decoder states of a lane's 4 tokens stay in
// registers between heads.  The 4 warps merge their states per head and write
// one record per query head; a second grid merges the items of a sequence,
// rotates the value space back and normalises.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {
namespace {

constexpr int RW = 4;                  // warps per CTA
constexpr int RCH = 4;                 // 32-token chunks per warp
constexpr int ITEM = 32 * RW * RCH;    // quantized tokens per item
constexpr int REC = 132;               // floats per record: acc[128], m, l, 2 pad
constexpr uint32_t RANS_L = 1u << 23;
constexpr int VST = 40;                // u16 per staged value row (32 tokens + pad)

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Predicated 32-bit read-only load into v: v = base[i] when pred, else v is
// kept.  Nothing reads v here, so the load's latency is only paid where v is
// next used.
__device__ __forceinline__ void ldg_into_if(uint32_t &v, const uint32_t *base, uint32_t i, bool pred) {
    asm("{\n .reg .pred q;\n .reg .u64 a;\n setp.ne.b32 q, %3, 0;\n mad.wide.u32 a, %2, 4, %1;\n"
        " @q ld.global.nc.u32 %0, [a];\n}\n"
        : "+r"(v)
        : "l"(base), "r"(i), "r"(static_cast<int>(pred)));
}

// One rANS stream being decoded by a lane.  The container bytes after the
// state sit in two words, lo then hi, the next byte being byte k of the pair
// (one byte permute picks it); every 4 symbols refill() moves hi and the word
// prefetched at the previous refill in and fetches the next one (a predicated
// load, so there is no branch and no wait), which keeps at least 4 unread bytes
// in the pair - enough for 4 symbols, each taking at most one byte.  Loads stay
// inside the aligned words that overlap the container; an idle lane loads
// nothing.  A well-formed stream ends in the state the encoder started from
// (2^23), which the caller checks.  Six registers: kw holds k (bits 0-3) and
// the words overlapping the container not yet loaded (bits 8 up); wi is the
// next word's index from the tensor's base.
struct Dec {
    uint32_t x, lo, hi, nxt, kw, wi;
    __device__ __forceinline__ void open(const uint8_t *codes, long long off0, int C, bool valid) {
        if (!valid) {  // an idle lane: decodes zeros, reads nothing
            x = RANS_L;
            lo = hi = nxt = kw = wi = 0;
            return;
        }
        const uint8_t *base = codes + off0;
        x = static_cast<uint32_t>(base[0]) | (static_cast<uint32_t>(base[1]) << 8) |
            (static_cast<uint32_t>(base[2]) << 16) | (static_cast<uint32_t>(base[3]) << 24);
        const long long p0 = off0 + 4, pe = off0 + C - 1;  // C >= 8: pe >= p0; codes is 16-byte aligned
        const int off = static_cast<int>(p0 & 3);
        const long long w0 = (p0 - off) / 4;
        const int words = static_cast<int>((pe & ~3LL) / 4 - w0) + 1;
        const uint32_t *cw = reinterpret_cast<const uint32_t *>(codes);
        lo = __ldg(cw + w0);
        hi = words > 1 ? __ldg(cw + w0 + 1) : 0u;
        nxt = words > 2 ? __ldg(cw + w0 + 2) : 0u;
        kw = static_cast<uint32_t>(off) | (static_cast<uint32_t>(words - 3 > 0 ? words - 3 : 0) << 8);
        wi = static_cast<uint32_t>(w0 + 3);
    }
    // Past the container's last word nxt keeps a stale word: a well-formed
    // stream never consumes those bytes (the final-state check catches one that does).
    __device__ __forceinline__ void refill(const uint32_t *cw) {
        const bool r = (kw & 0xffu) >= 4u;
        lo = r ? hi : lo;
        hi = r ? nxt : hi;
        ldg_into_if(nxt, cw, wi, r && kw >= 256u);
        wi += (r && kw >= 256u) ? 1u : 0u;
        kw -= r ? (kw >= 256u ? 260u : 4u) : 0u;
    }
};

// One symbol of each of N streams, written phase by phase across the streams
// (table lookups, state updates, byte merges) so their dependent chains
// interleave.  e[ch] receives stream ch's table entry.
template <int N>
__device__ __forceinline__ void step_all(Dec (&d)[N], const uint2 *dec, uint2 (&e)[N]) {
#pragma unroll
    for (int ch = 0; ch < N; ch++) e[ch] = dec[d[ch].x & 255u];
#pragma unroll
    for (int ch = 0; ch < N; ch++) d[ch].x = (e[ch].x & 0x1ffu) * (d[ch].x >> 8) + (e[ch].x >> 16);
#pragma unroll
    for (int ch = 0; ch < N; ch++) {
        const bool need = d[ch].x < RANS_L;
        const uint32_t byte = __byte_perm(d[ch].lo, d[ch].hi, d[ch].kw);  // byte k of (hi, lo) in byte 0
        d[ch].x = need ? __byte_perm(byte, d[ch].x, 0x6540) : d[ch].x;    // (x << 8) | byte
        d[ch].kw += need ? 1u : 0u;
    }
}

struct RecMerge {
    float m[RW][4], l[RW][4];
    float acc[RW][4][128];
};

template <int H>
struct RansSmem {
    uint2 dec_k[256], dec_v[256];   // (f | (z - c) << 16, level as fp32 bits / fp16 bits)
    float4 qk[128];                  // rotated query rows of the current head's 4 query heads, by channel
    float qsum[4];                   // sum_c q_rot[qh][c] of those heads
    float qmu[4][4];                 // sum_c q_rot[qh][c] mu^_w[c] for the item's 4 windows
    uint16_t pst[RW][RCH][8][VST];   // staged P' (fp16 hi/lo), [chunk][column][token]
    union {                          // the merge follows the head's value pass
        uint16_t vst[RW][RCH][16][VST];  // staged value levels (fp16) of 16 channels, [chunk][channel][token]
        RecMerge mg;
    };
};

// ---------------------------------------------------------------------------
// Quantized item: 512 tokens of one sequence.
// ---------------------------------------------------------------------------
template <int H>
__device__ void rans_quant_item(RansSmem<H> &S, const RansAttnArgs &a, int b, long long s0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    constexpr int N = 128 * H, HQ = 4 * H;
    // rotated query rows of KV head h's query heads (warp gq takes head 4h +
    // gq), their sums and their dot products with the item's window means
    auto prep_queries = [&](int h) {
        const int gq = warp, qh = 4 * h + gq;
        float q4[4];
        const float *qp = a.q + (static_cast<long long>(b) * HQ + qh) * 128 + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; j++) q4[j] = qp[j];
        if (a.rot_k) {
            fwht_warp<4>(q4);
#pragma unroll
            for (int j = 0; j < 4; j++) q4[j] = __fmul_rn(q4[j], a.hscale);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) reinterpret_cast<float *>(&S.qk[4 * lane + j])[gq] = q4[j];
        const float sum = warp_sum(q4[0] + q4[1] + q4[2] + q4[3]);
        if (lane == 0) S.qsum[gq] = sum;
        // window means: INT8 q times the fp16 scale
        for (int w = 0; w < 4; w++) {
            const long long win = s0 / 128 + w;
            float dmu = 0.f;
            if (a.mean && win < a.wcap) {
                const uint8_t *rec = a.mean + (static_cast<long long>(b) * a.wcap + win) * a.mean_rec;
                const float sc = __half2float(*reinterpret_cast<const __half *>(rec + N));
                const uint32_t qw = reinterpret_cast<const uint32_t *>(rec)[32 * h + lane];
#pragma unroll
                for (int j = 0; j < 4; j++)
                    dmu += q4[j] * (static_cast<float>(static_cast<int8_t>((qw >> (8 * j)) & 0xffu)) * sc);
            }
            dmu = warp_sum(dmu);
            if (lane == 0) S.qmu[w][gq] = dmu;
        }
    };
    // this lane's 4 tokens (one per chunk), their decoders and metadata
    Dec dk[RCH], dv[RCH];
    bool bad = false, valid[RCH];
    float sk[RCH], ok[RCH], sv[RCH], ov[RCH];
    // the token's 128-slot mean window within the item: slot - s0 = 128 warp +
    // 32 ch + lane, so it is window `warp` for every chunk of the lane
#pragma unroll
    for (int ch = 0; ch < RCH; ch++) {
        const long long slot = s0 + 32 * (RCH * warp + ch) + lane;
        valid[ch] = slot < a.n_q;
        const long long rs = static_cast<long long>(b) * a.qcap + (valid[ch] ? slot : 0);
        dk[ch].open(a.codes_k, rs * a.ck, a.ck, valid[ch]);
        dv[ch].open(a.codes_v, rs * a.cv, a.cv, valid[ch]);
        sk[ch] = ok[ch] = sv[ch] = ov[ch] = 0.f;
        if (valid[ch]) {
            const __half2 mk = reinterpret_cast<const __half2 *>(a.meta_k)[rs];
            const __half2 mv = reinterpret_cast<const __half2 *>(a.meta_v)[rs];
            sk[ch] = __low2float(mk);
            ok[ch] = __high2float(mk);
            sv[ch] = __low2float(mv);
            ov[ch] = __high2float(mv);
        }
    }
    uint16_t(*vst)[16][VST] = S.vst[warp];
    uint16_t(*pst)[8][VST] = S.pst[warp];
    const uint32_t *ckw = reinterpret_cast<const uint32_t *>(a.codes_k);
    const uint32_t *cvw = reinterpret_cast<const uint32_t *>(a.codes_v);
#pragma unroll 1
    for (int h = 0; h < H; h++) {
        prep_queries(h);
        __syncthreads();
        // keys of head h: 128 symbols of each of the 4 streams, interleaved
        float dot[RCH][4];
#pragma unroll
        for (int ch = 0; ch < RCH; ch++) dot[ch][0] = dot[ch][1] = dot[ch][2] = dot[ch][3] = 0.f;
#pragma unroll 4
        for (int c = 0; c < 128; c++) {
            if ((c & 3) == 0) {
#pragma unroll
                for (int ch = 0; ch < RCH; ch++) dk[ch].refill(ckw);
            }
            const float4 q4 = S.qk[c];
            uint2 ek[RCH];
            step_all<RCH>(dk, S.dec_k, ek);
#pragma unroll
            for (int ch = 0; ch < RCH; ch++) {
                const float lev = __uint_as_float(ek[ch].y);
                dot[ch][0] = fmaf(q4.x, lev, dot[ch][0]);
                dot[ch][1] = fmaf(q4.y, lev, dot[ch][1]);
                dot[ch][2] = fmaf(q4.z, lev, dot[ch][2]);
                dot[ch][3] = fmaf(q4.w, lev, dot[ch][3]);
            }
        }
        // Eq. (8) affine terms (log2 units) and one softmax step over the warp's 128 tokens
        float mrun[4], lsum[4], osum[4];
#pragma unroll
        for (int gq = 0; gq < 4; gq++) {
            float lg[RCH], mx = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < RCH; ch++) {
                lg[ch] = valid[ch] ? a.sm_log2 * (sk[ch] * dot[ch][gq] + ok[ch] * S.qsum[gq] + S.qmu[warp][gq])
                                   : -INFINITY;
                mx = fmaxf(mx, lg[ch]);
            }
            mx = warp_max(mx);
            mrun[gq] = mx;
            float ls = 0.f, os = 0.f;
#pragma unroll
            for (int ch = 0; ch < RCH; ch++) {
                const float p = valid[ch] ? ex2(lg[ch] - mx) : 0.f;
                ls += p;
                os = fmaf(p, ov[ch], os);
                const __half hi = __float2half_rn(p * sv[ch]);
                const __half lo = __float2half_rn(p * sv[ch] - __half2float(hi));
                pst[ch][2 * gq][lane] = __half_as_ushort(hi);
                pst[ch][2 * gq + 1][lane] = __half_as_ushort(lo);
            }
            lsum[gq] = warp_sum(ls);
            osum[gq] = warp_sum(os);
        }
        __syncwarp();
        uint32_t bf[RCH][2][2];
#pragma unroll
        for (int ch = 0; ch < RCH; ch++)
#pragma unroll
            for (int kt = 0; kt < 2; kt++) {
                bf[ch][kt][0] = *reinterpret_cast<const uint32_t *>(&pst[ch][g][16 * kt + 2 * tig]);
                bf[ch][kt][1] = *reinterpret_cast<const uint32_t *>(&pst[ch][g][16 * kt + 2 * tig + 8]);
            }
        // values of head h, 16 channels at a time: stage the levels, then P . V
        // (A = V^T: 16 channels x 16 tokens, B = P': 16 tokens x 8 columns)
        float acc[8][4];
#pragma unroll
        for (int mi = 0; mi < 8; mi++) {
            acc[mi][0] = acc[mi][1] = acc[mi][2] = acc[mi][3] = 0.f;
#pragma unroll 4
            for (int cc = 0; cc < 16; cc++) {
                if ((cc & 3) == 0) {
#pragma unroll
                    for (int ch = 0; ch < RCH; ch++) dv[ch].refill(cvw);
                }
                uint2 ev[RCH];
                step_all<RCH>(dv, S.dec_v, ev);
#pragma unroll
                for (int ch = 0; ch < RCH; ch++) vst[ch][cc][lane] = static_cast<uint16_t>(ev[ch].y);
            }
            __syncwarp();
#pragma unroll
            for (int ch = 0; ch < RCH; ch++)
#pragma unroll
                for (int kt = 0; kt < 2; kt++) {
                    const uint32_t a0 = *reinterpret_cast<const uint32_t *>(&vst[ch][g][16 * kt + 2 * tig]);
                    const uint32_t a1 = *reinterpret_cast<const uint32_t *>(&vst[ch][g + 8][16 * kt + 2 * tig]);
                    const uint32_t a2 = *reinterpret_cast<const uint32_t *>(&vst[ch][g][16 * kt + 2 * tig + 8]);
                    const uint32_t a3 = *reinterpret_cast<const uint32_t *>(&vst[ch][g + 8][16 * kt + 2 * tig + 8]);
                    mma16816(acc[mi], a0, a1, a2, a3, bf[ch][kt][0], bf[ch][kt][1]);
                }
            __syncwarp();
        }
        // this warp's record per query head into the merge area (which overlays
        // the staging tiles: every warp must be done with its value pass)
        __syncthreads();
        const float my_o = tig == 0 ? osum[0] : (tig == 1 ? osum[1] : (tig == 2 ? osum[2] : osum[3]));
#pragma unroll
        for (int mi = 0; mi < 8; mi++) {
            S.mg.acc[warp][tig][16 * mi + g] = acc[mi][0] + acc[mi][1] + my_o;
            S.mg.acc[warp][tig][16 * mi + g + 8] = acc[mi][2] + acc[mi][3] + my_o;
        }
        if (lane < 4) {
            S.mg.m[warp][lane] = lane == 0 ? mrun[0] : (lane == 1 ? mrun[1] : (lane == 2 ? mrun[2] : mrun[3]));
            S.mg.l[warp][lane] = lane == 0 ? lsum[0] : (lane == 1 ? lsum[1] : (lane == 2 ? lsum[2] : lsum[3]));
        }
        __syncthreads();
        // merge the 4 warps: warp gq writes the record of query head 4h + gq
        {
            const int gq = warp;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < RW; w++) M = fmaxf(M, S.mg.m[w][gq]);
            float sc[RW], L = 0.f;
#pragma unroll
            for (int w = 0; w < RW; w++) {
                sc[w] = S.mg.m[w][gq] == -INFINITY ? 0.f : ex2(S.mg.m[w][gq] - M);
                L += S.mg.l[w][gq] * sc[w];
            }
            float *rec = a.partials + ((static_cast<long long>(b) * a.items_per_b + s0 / ITEM) * HQ + 4 * h + gq) * REC;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int c = lane + 32 * j;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < RW; w++) v += S.mg.acc[w][gq][c] * sc[w];
                rec[c] = v;
            }
            if (lane == 0) {
                rec[128] = M;
                rec[129] = L;
            }
        }
        __syncthreads();
    }
    // a well-formed container decodes back to the encoder's initial state
#pragma unroll
    for (int ch = 0; ch < RCH; ch++) bad = bad || (valid[ch] && (dk[ch].x != RANS_L || dv[ch].x != RANS_L));
    if (bad) atomicOr(a.status, ST_BOUNDS);
}

// ---------------------------------------------------------------------------
// 16-bit item: the sinks and the recent window of one sequence, every head.
// Warp gq handles query head 4h + gq of KV head h; lanes own 4 channels.
// ---------------------------------------------------------------------------
template <int H>
__device__ void rans_raw_item(RansSmem<H> &S, const RansAttnArgs &a, int b) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int HQ = 4 * H;
    for (int h = 0; h < H; h++) {
        const int qh = 4 * h + warp;
        const long long u = static_cast<long long>(b) * H + h;
        float q4[4];
        const float *qp = a.q + (static_cast<long long>(b) * HQ + qh) * 128 + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; j++) q4[j] = qp[j];
        float M = -INFINITY, L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < a.n_raw; i++) {
            const int slot = i < a.n_sink_eff ? i : a.n_sink_cfg + static_cast<int>((a.recent_t0 + (i - a.n_sink_eff)) % a.n_recent_cfg);
            const uint16_t *kr = a.raw_k + (u * a.rcap + slot) * 128 + 4 * lane;
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint16_t bits = kr[j];
                const float kv = a.raw_bf16 ? __uint_as_float(static_cast<uint32_t>(bits) << 16)
                                            : __half2float(__ushort_as_half(bits));
                s = fmaf(q4[j], kv, s);
            }
            const float lg = a.sm_log2 * warp_sum(s);
            const float Mn = fmaxf(M, lg);
            const float al = M == -INFINITY ? 0.f : ex2(M - Mn);
            const float p = ex2(lg - Mn);
            L = L * al + p;
            const uint16_t *vr = a.raw_v + ((u * (a.rcap / 2) + slot / 2) * 128 + 4 * lane) * 2 + (slot & 1);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint16_t bits = vr[2 * j];
                const float vv = a.raw_bf16 ? __uint_as_float(static_cast<uint32_t>(bits) << 16)
                                            : __half2float(__ushort_as_half(bits));
                acc[j] = fmaf(p, vv, acc[j] * al);
            }
            M = Mn;
        }
        float *rec = a.partials + ((static_cast<long long>(b) * a.items_per_b + a.items_per_b - 1) * HQ + qh) * REC;
#pragma unroll
        for (int j = 0; j < 4; j++) rec[4 * lane + j] = acc[j];
        if (lane == 0) {
            rec[128] = M;
            rec[129] = L;
        }
    }
}

template <int H>
__global__ void __launch_bounds__(128, 4) attn_rans_kernel(RansAttnArgs a, const RansDevTables *tabs) {
    extern __shared__ __align__(16) unsigned char smraw[];
    RansSmem<H> &S = *reinterpret_cast<RansSmem<H> *>(smraw);
    const int b = blockIdx.x / a.items_per_b, it = blockIdx.x % a.items_per_b;
    if (it == a.items_per_b - 1) {
        rans_raw_item<H>(S, a, b);
        return;
    }
    // decoder tables: entry = (f | (z - c) << 16, level as fp32 bits) for keys,
    // (f | (z - c) << 16, level as fp16 bits) for values
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        const uint32_t ek = tabs->k.dec[i], ev = tabs->v.dec[i];
        S.dec_k[i] = make_uint2(((ek >> 4) & 0x1ffu) | ((ek >> 16) << 16), __float_as_uint(static_cast<float>(ek & 15u)));
        S.dec_v[i] = make_uint2(((ev >> 4) & 0x1ffu) | ((ev >> 16) << 16),
                                static_cast<uint32_t>(__half_as_ushort(__uint2half_rn(ev & 15u))));
    }
    __syncthreads();
    rans_quant_item<H>(S, a, b, static_cast<long long>(it) * ITEM);
}

// ---------------------------------------------------------------------------
// Merge the records of a sequence: one CTA per (sequence, KV head), warp gq
// for query head 4h + gq.  Quantized records live in the value space the
// encoder saw (rotated back here when values were rotated); the 16-bit record
// is in the original space.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) rans_combine_kernel(RansAttnArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / a.Hkv, h = blockIdx.x % a.Hkv;
    const int HQ = 4 * a.Hkv, qh = 4 * h + warp;
    const int nqi = a.items_per_b - 1;
    float M = -INFINITY;  // lanes read the records' maxima in parallel
    for (int i = lane; i < a.items_per_b; i += 32) {
        const float *rec = a.partials + ((static_cast<long long>(b) * a.items_per_b + i) * HQ + qh) * REC;
        if (i < nqi ? i < a.n_qitems : a.n_raw > 0) M = fmaxf(M, rec[128]);
    }
    M = warp_max(M);
    float L = 0.f, aq[4] = {0.f, 0.f, 0.f, 0.f}, ar[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int i = 0; i < a.items_per_b; i++) {
        const bool used = i < nqi ? i < a.n_qitems : a.n_raw > 0;
        if (!used) continue;
        const float *rec = a.partials + ((static_cast<long long>(b) * a.items_per_b + i) * HQ + qh) * REC;
        const float m = rec[128];
        if (m == -INFINITY) continue;
        const float sc = ex2(m - M);
        L += rec[129] * sc;
        float *dst = i < nqi ? aq : ar;
#pragma unroll
        for (int j = 0; j < 4; j++) dst[j] += rec[4 * lane + j] * sc;
    }
    if (a.rot_v) {
        fwht_warp<4>(aq);
#pragma unroll
        for (int j = 0; j < 4; j++) aq[j] *= a.hscale;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const long long o = (static_cast<long long>(b) * HQ + qh) * 128 + 4 * lane;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float y = (aq[j] + ar[j]) * inv;
        if (a.out_dtype == DQ_F32) reinterpret_cast<float *>(a.out)[o + j] = y;
        else if (a.out_dtype == DQ_F16) reinterpret_cast<__half *>(a.out)[o + j] = __float2half_rn(y);
        else reinterpret_cast<__nv_bfloat16 *>(a.out)[o + j] = __float2bfloat16_rn(y);
    }
}

}  // namespace

size_t rans_attention_smem(int H) {
    switch (H) {
        case 1: return sizeof(RansSmem<1>);
        case 2: return sizeof(RansSmem<2>);
        case 4: return sizeof(RansSmem<4>);
        default: return sizeof(RansSmem<8>);
    }
}

long long rans_partial_floats(int B, int Hq, long long qcap) {
    const long long items = (qcap + ITEM - 1) / ITEM + 1;
    return static_cast<long long>(B) * items * Hq * REC;
}

int launch_attention_rans(const RansAttnArgs &a0, const RansDevTables *tabs, void *stream) {
    RansAttnArgs a = a0;
    a.n_qitems = static_cast<int>((a.n_q + ITEM - 1) / ITEM);
    a.items_per_b = a.n_qitems + 1;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t smem = rans_attention_smem(a.Hkv);
    const unsigned grid = static_cast<unsigned>(a.B * a.items_per_b);
    cudaError_t e = cudaSuccess;
    switch (a.Hkv) {
        case 1:
            e = cudaFuncSetAttribute(attn_rans_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e == cudaSuccess) attn_rans_kernel<1><<<grid, 32 * RW, smem, st>>>(a, tabs);
            break;
        case 2:
            e = cudaFuncSetAttribute(attn_rans_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e == cudaSuccess) attn_rans_kernel<2><<<grid, 32 * RW, smem, st>>>(a, tabs);
            break;
        case 4:
            e = cudaFuncSetAttribute(attn_rans_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e == cudaSuccess) attn_rans_kernel<4><<<grid, 32 * RW, smem, st>>>(a, tabs);
            break;
        case 8:
            e = cudaFuncSetAttribute(attn_rans_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e == cudaSuccess) attn_rans_kernel<8><<<grid, 32 * RW, smem, st>>>(a, tabs);
            break;
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
    if (e != cudaSuccess) return static_cast<int>(e);
    if ((e = cudaGetLastError()) != cudaSuccess) return static_cast<int>(e);
    rans_combine_kernel<<<static_cast<unsigned>(a.B * a.Hkv), 128, 0, st>>>(a);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace dq
