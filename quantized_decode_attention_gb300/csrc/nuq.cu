// Non-uniform (Lloyd-Max) KV-cache quantizer: prefill and decode-time appends (sm_103a).
//
// "KVQuant-NUQ" (VeloxQuant-MLX docs), How it works:
//  * Non-uniform levels (Lloyd-Max): 2^bits levels seeded at evenly spaced
//    quantiles, then assign/update sweeps; codes = nearest level.
//  * Dense-and-Sparse outlier isolation: exactly k = floor(f n + 0.5)
//    elements per vector, the largest |x| by rank (ties to the lower index),
//    leave the fit and keep their fp16 value in a side channel.
//  * Quantization axes: keys per channel over the quantized tokens of the
//    prefill, values per token over its channels.
//  * Attention Sink-Aware quantization: the first n_sink tokens stay exact in
//    16-bit and take no part in the fit.
//  * Decode-time keys keep the prefill's per-channel tables and are screened
//    against the per-channel threshold frozen at prefill (the magnitude of the
//    channel's k-th rank outlier): |x| >= threshold goes to the side channel,
//    appended in token order while it has room.  Decode values are fitted per
//    token like prefill values.
//  * Configuration reference: kvquant_group_size splits a value token's fit
//    into groups of consecutive channels (outliers still ranked over the
//    token); kvquant_refit_interval N gives the key tables blocks of N
//    quantized slots, a block of decode keys fitted on its own keys, as a
//    prefill of them, by the append that completes it.
// The fit follows one fixed arithmetic order so that the tables are bit-exact:
// level sums in the R32 order (lane l = position mod 32 adds its positions in
// increasing order, then a xor butterfly), sum / count in fp32, fp16 table,
// codes re-assigned against the fp16 table.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "dq_internal.h"

namespace dq {

int nuq_outlier_count(float f, int n) {
    const int k = static_cast<int>(std::floor(static_cast<double>(f) * n + 0.5));
    return k < 0 ? 0 : (k > n ? n : k);
}

namespace {

// Order-preserving key of a float (a -0 counts as +0).
__device__ __forceinline__ uint32_t ord_key(float x) {
    const uint32_t b = __float_as_uint(__fadd_rn(x, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_val(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Nearest level, ties to the lower index.
template <int LV>
__device__ __forceinline__ int nearest(float x, const float (&lev)[LV]) {
    int best = 0;
    float bd = fabsf(__fsub_rn(x, lev[0]));
#pragma unroll
    for (int i = 1; i < LV; i++) {
        const float dd = fabsf(__fsub_rn(x, lev[i]));
        if (dd < bd) {
            bd = dd;
            best = i;
        }
    }
    return best;
}

// Block-wide bitonic sort of n2 (a power of two) keys in shared memory.
template <typename K, bool DESCENDING>
__device__ void bitonic_sort(K *keys, int n2) {
    for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = ((i & k) == 0) != DESCENDING;
                    const K a = keys[i], b = keys[l];
                    if ((a > b) == up) {
                        keys[i] = b;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
}

// One warp's Lloyd sweeps over `n` positions of `vals` (skipping the flagged
// outliers), R32 order; lev[] holds the seeds on entry, the levels on exit.
template <int LV>
__device__ __forceinline__ void lloyd_warp_smem(const float *vals, const uint32_t *outmask, int n, int iters,
                                                float (&lev)[LV]) {
    const int lane = threadIdx.x & 31;
    for (int it = 0; it < iters; it++) {
        float sum[LV];
        int cnt[LV];
#pragma unroll
        for (int i = 0; i < LV; i++) {
            sum[i] = 0.f;
            cnt[i] = 0;
        }
        for (int p = lane; p < n; p += 32) {
            if ((outmask[p >> 5] >> (p & 31)) & 1u) continue;
            const float x = vals[p];
            const int a = nearest<LV>(x, lev);
#pragma unroll
            for (int i = 0; i < LV; i++)
                if (a == i) {
                    sum[i] = __fadd_rn(sum[i], x);
                    cnt[i]++;
                }
        }
#pragma unroll
        for (int i = 0; i < LV; i++) {
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                sum[i] = __fadd_rn(sum[i], __shfl_xor_sync(FULL, sum[i], off));
                cnt[i] += __shfl_xor_sync(FULL, cnt[i], off);
            }
            if (cnt[i] > 0) lev[i] = __fdiv_rn(sum[i], static_cast<float>(cnt[i]));
        }
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Key tables: one CTA per (unit, channel).  Sorts (in shared memory) pick the
// rank outliers and the quantile seeds; warp 0 runs the Lloyd sweeps and
// writes the fp16 table.  Outliers are marked in the per-token bitmap that the
// side-channel pass turns into rows.
// ---------------------------------------------------------------------------
template <int D, int BITS>
__global__ void __launch_bounds__(256) nuq_key_fit_kernel(QuantArgs a, Layout L, int n2) {
    constexpr int LV = 1 << BITS;
    extern __shared__ __align__(16) unsigned char sm[];
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(sm);       // [n2]
    float *vals = reinterpret_cast<float *>(keys + n2);                          // [n2]
    uint32_t *outmask = reinterpret_cast<uint32_t *>(vals + n2);                 // [n2 / 32]
    __shared__ float seed[LV];
    const int u = blockIdx.x / D, c = blockIdx.x % D;
    const int n = a.n_fit, k = a.k_out;
    // a refit block the prefill reached keeps the prefill's tables
    if (a.fit_flush && static_cast<long long>(a.fit_blk) * L.refit < a.pq[u]) return;
    if (a.pq && !a.fit_flush && c == 0 && threadIdx.x == 0) a.pq[u] = n;
    const long long base = (static_cast<long long>(u) * a.n_tok + a.fit_t0) * D + c;
    bool finite = true;
    for (int p = threadIdx.x; p < n2; p += blockDim.x) {
        if (p < n) {
            const float x = ld_in(a.x, base + static_cast<long long>(p) * D, a.in_dtype);
            finite = finite && isfinite(x);
            vals[p] = x;
            keys[p] = (static_cast<unsigned long long>(__float_as_uint(fabsf(x))) << 32) | (0xffffffffu - p);
        } else {
            keys[p] = 0ull;
        }
        if ((p & 31) == 0) outmask[p >> 5] = 0u;
    }
    if (!finite) atomicOr(a.status, ST_NONFINITE);
    __syncthreads();
    // outliers: the k largest |x|, lower position first among equals
    bitonic_sort<unsigned long long, true>(keys, n2);
    for (int r = threadIdx.x; r < k; r += blockDim.x) {
        const int p = static_cast<int>(0xffffffffu - static_cast<uint32_t>(keys[r]));
        atomicOr(&outmask[p >> 5], 1u << (p & 31));
        atomicOr(&a.olbits[(static_cast<long long>(u) * L.qcap + a.fit_slot0 + p) * (D / 32) + c / 32], 1u << (c & 31));
    }
    // the threshold decode keys are screened against: the k-th largest magnitude
    if (threadIdx.x == 0 && a.thr && !a.fit_flush)
        a.thr[static_cast<long long>(u) * D + c] = k > 0 ? __uint_as_float(static_cast<uint32_t>(keys[k - 1] >> 32)) : INFINITY;
    __syncthreads();
    // quantile seeds: sort the fit values (outliers and padding sort last)
    uint32_t *k32 = reinterpret_cast<uint32_t *>(keys);
    for (int p = threadIdx.x; p < n2; p += blockDim.x)
        k32[p] = (p < n && !((outmask[p >> 5] >> (p & 31)) & 1u)) ? ord_key(vals[p]) : 0xffffffffu;
    __syncthreads();
    bitonic_sort<uint32_t, false>(k32, n2);
    const int nf = n - k;
    if (threadIdx.x < LV) seed[threadIdx.x] = nf > 0 ? ord_val(k32[static_cast<long long>(2 * threadIdx.x + 1) * nf / (2 * LV)]) : 0.f;
    __syncthreads();
    if (threadIdx.x < 32) {
        float lev[LV];
#pragma unroll
        for (int i = 0; i < LV; i++) lev[i] = seed[i];
        if (nf > 0) lloyd_warp_smem<LV>(vals, outmask, n, a.iters, lev);
        if (threadIdx.x < LV) {
            float mine = lev[0];
#pragma unroll
            for (int i = 1; i < LV; i++)
                if (threadIdx.x == i) mine = lev[i];
            const uint16_t h = __half_as_ushort(__float2half_rn(mine));
            for (int b = a.fit_blk; b < a.fit_blk + a.fit_nblk; b++)
                a.lut[((static_cast<long long>(u) * L.nbk + b) * D + c) * LV + threadIdx.x] = h;
        }
    }
}

// 16-bit region slot of token t (sinks, and the latest n_recent of the prefill), or -1.
__device__ __forceinline__ int raw_slot_of(long long t, long long seq_after, const Layout &L) {
    if (t < L.n_sink) return static_cast<int>(t);
    if (L.n_recent > 0 && t >= seq_after - L.n_recent) return L.n_sink + static_cast<int>(t % L.n_recent);
    return -1;
}

// Raw copy of one token's channels c = lane + 32 j into its 16-bit slot.
template <int V>
__device__ __forceinline__ void copy_raw(const QuantArgs &a, const Layout &L, int u, long long base, int slot,
                                         bool key) {
    constexpr int D = 32 * V;
    const int lane = threadIdx.x & 31;
    const long long ub = static_cast<long long>(u) * L.rcap * D;
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane + 32 * j;
        const long long off = key ? static_cast<long long>(slot) * D + c
                                  : (static_cast<long long>(slot >> 1) * D + c) * 2 + (slot & 1);
        a.raw[ub + off] = raw16_of(a.x, base + c, a.in_dtype);
    }
}

// ---------------------------------------------------------------------------
// Values: one warp per (unit, token).  Lane l holds channels l + 32 j, so its
// positions in the R32 order are its own values in register order.
// ---------------------------------------------------------------------------
template <int V, int BITS>
__global__ void __launch_bounds__(128) nuq_value_kernel(QuantArgs a, Layout L) {
    constexpr int D = 32 * V, LV = 1 << BITS, WPB = 4;
    __shared__ uint32_t wk[WPB][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.n_tok) return;
    const int u = static_cast<int>(gw / a.n_tok);
    const long long ti = gw % a.n_tok, t = a.pos0 + ti;  // row of the input, position in the sequence
    const long long base = (static_cast<long long>(u) * a.n_tok + ti) * D;
    float x[V];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < V; j++) {
        x[j] = ld_in(a.x, base + lane + 32 * j, a.in_dtype);
        finite = finite && isfinite(x[j]);
    }
    if (!__all_sync(FULL, finite) && lane == 0) atomicOr(a.status, ST_NONFINITE);
    const int rs = raw_slot_of(t, a.seq_after, L);
    if (rs >= 0) copy_raw<V>(a, L, u, base, rs, false);
    if (t < L.n_sink) return;
    const long long slot = t - L.n_sink;

    // outliers: k rounds of a warp argmax of (|x|, lower channel first)
    bool out[V];
#pragma unroll
    for (int j = 0; j < V; j++) out[j] = false;
    for (int r = 0; r < a.k_out; r++) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const unsigned long long key =
                (static_cast<unsigned long long>(__float_as_uint(fabsf(x[j]))) << 32) | (0xffffffffu - (lane + 32 * j));
            if (!out[j] && key > best) best = key;
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(FULL, best, off);
            best = o > best ? o : best;
        }
        const int c = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best));
#pragma unroll
        for (int j = 0; j < V; j++)
            if (lane + 32 * j == c) out[j] = true;
    }
    // per group of g = D / gv consecutive channels (the whole token when gv = 1):
    // quantile seeds from the ranks of the group's fit values (equal keys
    // ordered by channel), Lloyd sweeps over the group's positions in the R32
    // order (lane l holds positions l, l + 32, ... of the group in register
    // order), its fp16 table, and the codes of its channels
#pragma unroll
    for (int j = 0; j < V; j++) wk[warp][lane + 32 * j] = out[j] ? 0xffffffffu : ord_key(x[j]);
    __syncwarp();
    const int gv = L.gv, g = D / gv;
    const long long ts = static_cast<long long>(u) * L.qcap + slot;
    uint32_t m[V];
    for (int G = 0; G < gv; G++) {
        bool in[V];
        int nout = 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            in[j] = (lane + 32 * j) / g == G;
            nout += __popc(__ballot_sync(FULL, in[j] && out[j]));
        }
        const int nf = g - nout;
        float lev[LV];
#pragma unroll
        for (int i = 0; i < LV; i++) lev[i] = 0.f;
        if (nf > 0) {
            int rank[V];
#pragma unroll
            for (int j = 0; j < V; j++) {
                const uint32_t kj = wk[warp][lane + 32 * j];
                int r = 0;
                for (int p = G * g; p < G * g + g; p++) {
                    const uint32_t kp = wk[warp][p];
                    r += (kp < kj) || (kp == kj && p < lane + 32 * j);
                }
                rank[j] = (out[j] || !in[j]) ? -1 : r;
            }
#pragma unroll
            for (int i = 0; i < LV; i++) {
                const int target = (2 * i + 1) * nf / (2 * LV);
                float mine = 0.f;
                bool have = false;
#pragma unroll
                for (int j = 0; j < V; j++)
                    if (rank[j] == target) {
                        mine = ord_val(ord_key(x[j]));
                        have = true;
                    }
                const unsigned mk = __ballot_sync(FULL, have);
                lev[i] = __shfl_sync(FULL, mine, __ffs(mk) - 1);
            }
            // Lloyd sweeps, R32 order
            for (int it = 0; it < a.iters; it++) {
                float sum[LV];
                int cnt[LV];
#pragma unroll
                for (int i = 0; i < LV; i++) {
                    sum[i] = 0.f;
                    cnt[i] = 0;
                }
#pragma unroll
                for (int j = 0; j < V; j++) {
                    if (out[j] || !in[j]) continue;
                    const int q = nearest<LV>(x[j], lev);
#pragma unroll
                    for (int i = 0; i < LV; i++)
                        if (q == i) {
                            sum[i] = __fadd_rn(sum[i], x[j]);
                            cnt[i]++;
                        }
                }
#pragma unroll
                for (int i = 0; i < LV; i++) {
#pragma unroll
                    for (int off = 16; off; off >>= 1) {
                        sum[i] = __fadd_rn(sum[i], __shfl_xor_sync(FULL, sum[i], off));
                        cnt[i] += __shfl_xor_sync(FULL, cnt[i], off);
                    }
                    if (cnt[i] > 0) lev[i] = __fdiv_rn(sum[i], static_cast<float>(cnt[i]));
                }
            }
        }
        // fp16 table; codes against it
        float lev16[LV];
#pragma unroll
        for (int i = 0; i < LV; i++) lev16[i] = __half2float(__float2half_rn(lev[i]));
        if (lane < LV) {
            float mine = lev16[0];
#pragma unroll
            for (int i = 1; i < LV; i++)
                if (lane == i) mine = lev16[i];
            a.lut[(ts * gv + G) * LV + lane] = __half_as_ushort(__float2half_rn(mine));
        }
#pragma unroll
        for (int j = 0; j < V; j++)
            if (in[j]) m[j] = static_cast<uint32_t>(nearest<LV>(x[j], lev16));
    }
    // pack this token's half of its value pair record
    constexpr int WV = Rec<D, BITS>::V_WORDS, WLO = 2 * D * 2 / 32;
    const int e = static_cast<int>(slot & 1);
    uint16_t *rec = reinterpret_cast<uint16_t *>(a.codes + (static_cast<long long>(u) * (L.qcap / 2) + slot / 2) * L.pairV);
#pragma unroll
    for (int w = 0; w < WV; w++) {
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int c = lane + 32 * j;
            v |= contrib<D, BITS>(w, v_idx(c, D), e, m[j], WLO);
        }
        v = __reduce_or_sync(FULL, v);
        if (lane == (w & 31)) rec[2 * w + e] = static_cast<uint16_t>(v >> (16 * e));
    }
    // side channel in channel order
    int before = 0;
#pragma unroll
    for (int j = 0; j < V; j++) {
        const unsigned bal = __ballot_sync(FULL, out[j]);
        if (out[j]) {
            const long long idx = ts * a.k_out + before + __popc(bal & ((1u << lane) - 1u));
            a.ol_col[idx] = static_cast<uint16_t>(lane + 32 * j);
            a.ol_val[idx] = __half_as_ushort(__float2half_rn(x[j]));
        }
        before += __popc(bal);
    }
}

// A key row's codes m[j] (channel lane + 32 j) packed into its record.
template <int V, int BITS>
__device__ __forceinline__ void store_key_row(const uint32_t (&m)[V], uint32_t *row) {
    constexpr int D = 32 * V, WK = Rec<D, BITS>::K_WORDS, WLO = D * 2 / 32;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 0; w < WK; w++) {
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            const int c = lane + 32 * j;
            v |= contrib<D, BITS>(w, k_idx(c, D), c & 1, m[j], WLO);
        }
        v = __reduce_or_sync(FULL, v);
        if (lane == w) row[w] = v;
    }
}

// Nearest level of x in channel c's table of block `blk`.
template <int D, int LV>
__device__ __forceinline__ uint32_t key_code(const QuantArgs &a, const Layout &L, int u, long long blk, int c, float x) {
    float lev[LV];
    const uint16_t *t = a.lut + ((static_cast<long long>(u) * L.nbk + blk) * D + c) * LV;
#pragma unroll
    for (int i = 0; i < LV; i++) lev[i] = __half2float(__ushort_as_half(t[i]));
    return static_cast<uint32_t>(nearest<LV>(x, lev));
}

// ---------------------------------------------------------------------------
// Key codes against the per-channel tables: one warp per (unit, token).  With
// refit blocks, a token of a block of decode keys only is not coded here: it
// stays in the 16-bit recent window until its block completes.
// ---------------------------------------------------------------------------
template <int V, int BITS>
__global__ void __launch_bounds__(128) nuq_key_code_kernel(QuantArgs a, Layout L) {
    constexpr int D = 32 * V, LV = 1 << BITS, WPB = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.n_tok) return;
    const int u = static_cast<int>(gw / a.n_tok);
    const long long ti = gw % a.n_tok, t = a.pos0 + ti;  // row of the input, position in the sequence
    const long long base = (static_cast<long long>(u) * a.n_tok + ti) * D;
    const int rs = raw_slot_of(t, a.seq_after, L);
    if (rs >= 0) copy_raw<V>(a, L, u, base, rs, true);
    if (t < L.n_sink) return;
    const long long slot = t - L.n_sink;
    const bool screen = a.pos0 > 0 && a.thr != nullptr;  // decode keys: outliers by the frozen threshold
    const long long blk = L.refit ? slot / L.refit : 0;
    if (L.refit && blk * L.refit >= a.pq[u]) {          // coded when its block completes
        if (screen && lane < V) a.olbits[(static_cast<long long>(u) * L.qcap + slot) * V + lane] = 0u;
        return;
    }
    uint32_t m[V];
#pragma unroll
    for (int j = 0; j < V; j++) {
        const int c = lane + 32 * j;
        const float x = ld_in(a.x, base + c, a.in_dtype);
        m[j] = key_code<D, LV>(a, L, u, blk, c, x);
        if (screen) {
            const unsigned ob = __ballot_sync(FULL, fabsf(x) >= a.thr[static_cast<long long>(u) * D + c]);
            if (lane == 0) a.olbits[(static_cast<long long>(u) * L.qcap + slot) * V + j] = ob;
        }
    }
    store_key_row<V, BITS>(m, reinterpret_cast<uint32_t *>(a.codes + (static_cast<long long>(u) * L.qcap + slot) * L.rowK));
}

// ---------------------------------------------------------------------------
// Key refit blocks.  Gather: the fp32 keys of quantized slots [scr_lo, scr_lo
// + scr_n) of every unit, one warp per (unit, slot), from this call's input or,
// for a token older than the call, from its 16-bit recent-window slot (exact:
// refit caches take 16-bit keys); their outlier bits are cleared for the fit.
// ---------------------------------------------------------------------------
template <int V>
__global__ void __launch_bounds__(128) nuq_gather_kernel(QuantArgs a, Layout L) {
    constexpr int D = 32 * V, WPB = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.scr_n) return;
    const int u = static_cast<int>(gw / a.scr_n);
    const long long j = gw % a.scr_n, slot = a.scr_lo + j, t = slot + L.n_sink;
    float *dst = a.scr + (static_cast<long long>(u) * a.scr_n + j) * D;
#pragma unroll
    for (int i = 0; i < V; i++) {
        const int c = lane + 32 * i;
        float x;
        if (t >= a.pos0) {
            x = ld_in(a.x, (static_cast<long long>(u) * a.n_tok + (t - a.pos0)) * D + c, a.in_dtype);
        } else {
            const uint16_t r = a.raw[(static_cast<long long>(u) * L.rcap + L.n_sink + t % L.n_recent) * D + c];
            x = a.in_dtype == DQ_BF16 ? __bfloat162float(__ushort_as_bfloat16(r)) : __half2float(__ushort_as_half(r));
        }
        dst[c] = x;
    }
    // a block of decode keys only gets its outliers from its fit; the bits of
    // a block the prefill reached stay as they are
    if (lane < V && slot / L.refit * L.refit >= a.pq[u]) a.olbits[(static_cast<long long>(u) * L.qcap + slot) * V + lane] = 0u;
}

// Codes of the gathered slots whose block holds decode keys only, against the
// block's freshly fitted tables: one warp per (unit, slot).
template <int V, int BITS>
__global__ void __launch_bounds__(128) nuq_block_code_kernel(QuantArgs a, Layout L) {
    constexpr int D = 32 * V, LV = 1 << BITS, WPB = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.scr_n) return;
    const int u = static_cast<int>(gw / a.scr_n);
    const long long j = gw % a.scr_n, slot = a.scr_lo + j, blk = slot / L.refit;
    if (blk * L.refit < a.pq[u]) return;               // coded with the prefill's tables
    const float *src = a.scr + (static_cast<long long>(u) * a.scr_n + j) * D;
    uint32_t m[V];
#pragma unroll
    for (int i = 0; i < V; i++) m[i] = key_code<D, LV>(a, L, u, blk, lane + 32 * i, src[lane + 32 * i]);
    store_key_row<V, BITS>(m, reinterpret_cast<uint32_t *>(a.codes + (static_cast<long long>(u) * L.qcap + slot) * L.rowK));
}

// ---------------------------------------------------------------------------
// Key side channel, rows by quantized slot: one CTA per unit, over this
// call's slots [slot_lo, slot_lo + n_slots).  Each thread takes a contiguous
// run of slots; a block scan of the run counts gives the row pointers, which
// continue from the row pointer already stored at slot_lo (0 for a prefill);
// entries follow in channel order.  Entries past the capacity are not stored
// (the row pointers count stored entries only) and latch ST_SIDE_FULL.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) nuq_key_csr_kernel(QuantArgs a, Layout L) {
    constexpr int W = D / 32;
    __shared__ int part[256];
    const int u = blockIdx.x;
    long long s0 = a.slot_lo;
    int n = a.n_slots;
    if (a.scr) {  // refit blocks flushed by this call: rows rebuilt from the first slot they recoded
        const long long f0 = max(a.scr_lo, (static_cast<long long>(a.pq[u]) + L.refit - 1) / L.refit * L.refit);
        if (f0 < s0) {
            n += static_cast<int>(s0 - f0);
            s0 = f0;
        }
    }
    const long long cap = L.nnzk_cap;
    const int chunk = (n + blockDim.x - 1) / blockDim.x;
    const int p0 = min(n, static_cast<int>(threadIdx.x) * chunk), p1 = min(n, p0 + chunk);
    const uint32_t *bits = a.olbits + (static_cast<long long>(u) * L.qcap + s0) * W;
    int local = 0;
    for (int p = p0; p < p1; p++)
#pragma unroll
        for (int w = 0; w < W; w++) local += __popc(bits[p * W + w]);
    part[threadIdx.x] = local;
    __syncthreads();
    for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {  // inclusive scan
        const int v = threadIdx.x >= static_cast<unsigned>(off) ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int *rp = a.ol_rowptr + static_cast<long long>(u) * L.rp_stride;
    const long long run0 = s0 > 0 ? rp[s0] : 0;
    __syncthreads();  // every thread has read rp[s0] before it is rewritten
    long long run = run0 + part[threadIdx.x] - local;
    const long long total = run0 + part[blockDim.x - 1];
    uint16_t *col = a.ol_col + static_cast<long long>(u) * L.nnzk_cap;
    uint16_t *val = a.ol_val + static_cast<long long>(u) * L.nnzk_cap;
    for (int p = p0; p < p1; p++) {
        rp[s0 + p] = static_cast<int>(min(run, cap));
#pragma unroll
        for (int w = 0; w < W; w++) {
            uint32_t b = bits[p * W + w];
            while (b) {
                const int c = 32 * w + __ffs(b) - 1;
                b &= b - 1;
                if (run < cap) {
                    const long long sl = s0 + p;
                    float x;
                    if (a.scr && sl >= a.scr_lo && sl < a.scr_lo + a.scr_n)
                        x = a.scr[(static_cast<long long>(u) * a.scr_n + (sl - a.scr_lo)) * D + c];
                    else
                        x = ld_in(a.x, (static_cast<long long>(u) * a.n_tok + (sl + L.n_sink - a.pos0)) * D + c, a.in_dtype);
                    col[run] = static_cast<uint16_t>(c);
                    val[run] = __half_as_ushort(__float2half_rn(x));
                }
                run++;
            }
        }
    }
    for (long long p = s0 + n + threadIdx.x; p <= L.qcap; p += blockDim.x) rp[p] = static_cast<int>(min(total, cap));
    if (threadIdx.x == 0 && total > cap) atomicOr(a.status, ST_SIDE_FULL);
}

// ---- launchers ----------------------------------------------------------------
template <typename F>
static int nuq_dispatch(const Layout &L, F &&f) {
    if (L.d == 128) {
        if (L.bits_k == 2) return f(std::integral_constant<int, 4>(), std::integral_constant<int, 2>());
        if (L.bits_k == 3) return f(std::integral_constant<int, 4>(), std::integral_constant<int, 3>());
        return f(std::integral_constant<int, 4>(), std::integral_constant<int, 4>());
    }
    if (L.bits_k == 2) return f(std::integral_constant<int, 2>(), std::integral_constant<int, 2>());
    if (L.bits_k == 4) return f(std::integral_constant<int, 2>(), std::integral_constant<int, 4>());
    return static_cast<int>(cudaErrorInvalidValue);
}

int launch_nuq_values(const Layout &L, const QuantArgs &a, void *stream) {
    const long long warps = static_cast<long long>(L.U) * a.n_tok;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    return nuq_dispatch(L, [&](auto v, auto b) {
        nuq_value_kernel<decltype(v)::value, decltype(b)::value>
            <<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, L);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_nuq_key_codes(const Layout &L, const QuantArgs &a, void *stream) {
    const long long warps = static_cast<long long>(L.U) * a.n_tok;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    return nuq_dispatch(L, [&](auto v, auto b) {
        nuq_key_code_kernel<decltype(v)::value, decltype(b)::value>
            <<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, L);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_nuq_key_fit(const Layout &L, const QuantArgs &a, void *stream) {
    int n2 = 32;
    while (n2 < a.n_fit) n2 <<= 1;
    const size_t smem = static_cast<size_t>(n2) * (8 + 4) + static_cast<size_t>(n2 / 32) * 4;
    return nuq_dispatch(L, [&](auto v, auto b) {
        constexpr int D = 32 * decltype(v)::value;
        auto kern = nuq_key_fit_kernel<D, decltype(b)::value>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return static_cast<int>(e);
        kern<<<L.U * D, 256, smem, static_cast<cudaStream_t>(stream)>>>(a, L, n2);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_nuq_gather(const Layout &L, const QuantArgs &a, void *stream) {
    const unsigned grid = static_cast<unsigned>((static_cast<long long>(L.U) * a.scr_n + 3) / 4);
    return nuq_dispatch(L, [&](auto v, auto) {
        nuq_gather_kernel<decltype(v)::value><<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, L);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_nuq_block_codes(const Layout &L, const QuantArgs &a, void *stream) {
    const unsigned grid = static_cast<unsigned>((static_cast<long long>(L.U) * a.scr_n + 3) / 4);
    return nuq_dispatch(L, [&](auto v, auto b) {
        nuq_block_code_kernel<decltype(v)::value, decltype(b)::value>
            <<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, L);
        return static_cast<int>(cudaGetLastError());
    });
}

int launch_nuq_key_csr(const Layout &L, const QuantArgs &a, void *stream) {
    return nuq_dispatch(L, [&](auto v, auto) {
        nuq_key_csr_kernel<32 * decltype(v)::value><<<L.U, 256, 0, static_cast<cudaStream_t>(stream)>>>(a, L);
        return static_cast<int>(cudaGetLastError());
    });
}
}  // namespace dq
