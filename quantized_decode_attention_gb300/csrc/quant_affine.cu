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
#include "quant_row.cuh"

namespace dq {

// ---------------------------------------------------------------------------
// Key channel mean over tokens [t0, t1) of each unit (prefill).  One block per
// unit; thread j < D accumulates channel j over the tokens in order (acc =
// acc + y_tj from 0.0f), then divides by the count.  KM_WARPS warps rotate a
// chunk's rows into shared memory while each holds its rows of the next chunk
// in registers, loaded before the chunk is summed, so no row waits for HBM.
// ---------------------------------------------------------------------------
constexpr int KM_WARPS = 16;
constexpr int KM_ROWS = 4;  // rows per warp per chunk

template <int V>
__device__ __forceinline__ void key_mean_load(const QuantArgs &a, int u, long long c0, long long t1,
                                              float (&xr)[KM_ROWS][V]) {
    constexpr int D = 32 * V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long esz = a.in_dtype == 0 ? 4 : 2;
#pragma unroll
    for (int i = 0; i < KM_ROWS; i++) {
        const long long t = c0 + warp + KM_WARPS * i;
        const long long base = (static_cast<long long>(u) * a.n_tok + (t - a.pos0)) * D;
        const bool ok = t < t1 && in_buf(static_cast<const char *>(a.x) + base * esz, D * esz, a.x, a.sz_x, a.status);
#pragma unroll
        for (int j = 0; j < V; j++) xr[i][j] = ok ? ld_in(a.x, base + lane * V + j, a.in_dtype) : 0.f;
    }
}

template <int V>
__global__ void __launch_bounds__(KM_WARPS * 32) key_mean_kernel(QuantArgs a, int Hkv, long long t0, long long t1) {
    constexpr int D = 32 * V;
    constexpr int CH = KM_WARPS * KM_ROWS;  // tokens per chunk
    __shared__ float ys[CH][D];
    __shared__ float xs[KM_WARPS][D];
    const int u = blockIdx.x, kvh = u % Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *T = a.T ? a.T + static_cast<long long>(kvh) * D * D : nullptr;
    float acc = 0.0f;
    float xr[KM_ROWS][V];
    key_mean_load<V>(a, u, t0, t1, xr);
    for (long long c0 = t0; c0 < t1; c0 += CH) {
        const int n = static_cast<int>(t1 - c0 < CH ? t1 - c0 : CH);
#pragma unroll
        for (int i = 0; i < KM_ROWS; i++) {
            const int r = warp + KM_WARPS * i;
            if (r < n) {
                rotate_row<V>(xr[i], a.rot, a.hscale, T, xs[warp]);
#pragma unroll
                for (int j = 0; j < V; j++) ys[r][lane * V + j] = xr[i][j];
            }
        }
        if (c0 + CH < t1) key_mean_load<V>(a, u, c0 + CH, t1, xr);  // the next chunk's rows, in flight
        __syncthreads();
        if (threadIdx.x < D)
            for (int r = 0; r < n; r++) acc = __fadd_rn(acc, ys[r][threadIdx.x]);
        __syncthreads();
    }
    if (threadIdx.x >= D) return;
    const long long cnt = t1 - t0;
    float *mp = a.mean + static_cast<long long>(u) * D + threadIdx.x;
    if (in_buf(mp, 4, a.mean, a.sz_mean, a.status)) *mp = cnt > 0 ? __fdiv_rn(acc, static_cast<float>(cnt)) : 0.0f;
}

// ---------------------------------------------------------------------------
// Quantize tokens [pos0, pos0 + n_tok): one warp per (unit, token).
// ---------------------------------------------------------------------------
template <int V, int BITS>
__global__ void quantize_kernel(QuantArgs a, RowGeom L) {
    constexpr int D = 32 * V;
    constexpr int WPB = 4;
    __shared__ float xs[WPB][D];
    const int warp = threadIdx.x >> 5;
    const long long gw = static_cast<long long>(blockIdx.x) * WPB + warp;
    if (gw >= static_cast<long long>(L.U) * a.n_tok) return;
    quantize_row<V, BITS>(a, L, static_cast<int>(gw / a.n_tok), gw % a.n_tok, xs[warp]);
}

// ---------------------------------------------------------------------------
// Dequantize export: one warp per (unit, slot).
// ---------------------------------------------------------------------------
template <int D, int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *rec, int idx, int half, int words_lo) {
    if (BITS == 3) {
        const uint32_t lo = (rec[idx / 8] >> (16 * half + 2 * (idx % 8))) & 3u;
        const uint32_t hb = (rec[words_lo + idx / 16] >> (16 * half + bit1_pos(idx % 16))) & 1u;
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
    const long long mbytes = a.meta_f16 ? 4 : 8;
    if (!in_buf(static_cast<const char *>(a.meta) + ms * mbytes, mbytes, a.meta, a.sz_meta, a.status)) return;
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
    if (!in_buf(rec, a.is_key ? L.rowK : L.pairV, a.codes, a.sz_codes, a.status)) return;
    if (a.mean && !in_buf(a.mean + static_cast<long long>(u) * D, D * 4, a.mean, a.sz_mean, a.status)) return;
    if (!in_buf(a.out + (static_cast<long long>(u) * a.n + i) * D, D * 4, a.out, a.sz_out, a.status)) return;
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
    if (L.d == 128) key_mean_kernel<4><<<L.U, KM_WARPS * 32, 0, st>>>(a, L.Hkv, t0, t1);
    else key_mean_kernel<2><<<L.U, KM_WARPS * 32, 0, st>>>(a, L.Hkv, t0, t1);
    return static_cast<int>(cudaGetLastError());
}

template <int V>
static void launch_q_bits(const Layout &L, const QuantArgs &a, cudaStream_t st) {
    const long long warps = static_cast<long long>(L.U) * a.n_tok;
    const unsigned grid = static_cast<unsigned>((warps + 3) / 4);
    const RowGeom g = row_geom(L);
    switch (a.bits) {
        case 2: quantize_kernel<V, 2><<<grid, 128, 0, st>>>(a, g); break;
        case 3: quantize_kernel<V, 3><<<grid, 128, 0, st>>>(a, g); break;
        default: quantize_kernel<V, 4><<<grid, 128, 0, st>>>(a, g); break;
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
