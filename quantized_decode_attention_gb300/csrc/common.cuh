// Device helpers shared by the libdq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace dq {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float ld_in(const void *p, long long i, int dtype) {
    if (dtype == 0) return reinterpret_cast<const float *>(p)[i];
    uint16_t b = reinterpret_cast<const uint16_t *>(p)[i];
    if (dtype == 1) return __half2float(__ushort_as_half(b));
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Bits of the 16-bit value kept in a raw region: the input's own bits for
// fp16/bf16, fp16 round-to-nearest-even for fp32 input.
__device__ __forceinline__ uint16_t raw16_of(const void *p, long long i, int dtype) {
    if (dtype == 0) return __half_as_ushort(__float2half_rn(reinterpret_cast<const float *>(p)[i]));
    return reinterpret_cast<const uint16_t *>(p)[i];
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

// In-warp fast Walsh-Hadamard transform of a d-vector held V = d/32 values per
// lane (lane l holds elements l*V .. l*V+V-1).  Stages h = 1, 2, 4, ... in
// order; the pair (i, i+h) with bit h of i clear becomes (a+b, a-b), each a
// single round-to-nearest fp32 operation, so every element follows the same
// operation sequence as a plain sequential loop over stages.
template <int V>
__device__ __forceinline__ void fwht_warp(float (&x)[V]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 1; h < V; h <<= 1) {
#pragma unroll
        for (int j = 0; j < V; j++)
            if (!(j & h)) {
                float a = x[j], b = x[j + h];
                x[j] = __fadd_rn(a, b);
                x[j + h] = __fsub_rn(a, b);
            }
    }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
        const bool upper = (lane & hl) != 0;
#pragma unroll
        for (int j = 0; j < V; j++) {
            float p = __shfl_xor_sync(FULL, x[j], hl);
            x[j] = upper ? __fsub_rn(p, x[j]) : __fadd_rn(x[j], p);
        }
    }
}

// ---- record format ---------------------------------------------------------
// idx of key channel c / value channel c within a record (see dq.h).
__host__ __device__ __forceinline__ int k_idx(int c, int d) {
    return ((c >> 1) & 3) * (d / 8) + 2 * (c >> 4) + ((c >> 3) & 1);
}
__host__ __device__ __forceinline__ int v_idx(int c, int d) {
    return (c & 7) * (d / 8) + 2 * (c >> 4) + ((c >> 3) & 1);
}

// Power-of-two exponent E carried by an extracted code of register r: the
// kernel reads code m of field f as the fp16 bit pattern m << E, i.e. the value
// m * 2^(E-24) (binary16 subnormals and the first normal binade are evenly
// spaced at 2^-24, so any pattern below 2048 is an exact multiple of it).
__host__ __device__ __forceinline__ int field_exp(int r, int bits) {
    if (bits == 4) {
        int f = r & 3;
        return 4 * (f & 1);
    }
    int f = r & 7;  // bits 2 and 3: 2-bit fields (3-bit adds a plane above)
    return f <= 4 ? 2 * f : 2 * (f - 5);
}

// ---- record packing (writers) -----------------------------------------------
// Number of 32-bit words in a key row / a value pair record.
template <int D, int BITS>
struct Rec {
    static constexpr int K_WORDS = D * BITS / 32;
    static constexpr int V_WORDS = 2 * D * BITS / 32;
};

// Bit of field f (0..15) within a half of a 3-bit record's 1-bit plane: a
// permutation chosen so that the fields a lane turns into operands together
// need few distinct shifts to meet their 2-bit fields.
__host__ __device__ constexpr int bit1_pos(int f) {
    return f <= 6 ? 2 * f + 2 : (f == 7 ? 0 : (f == 15 ? 1 : 2 * f - 13));
}

// OR-contribution of one code to word w of a key row (BITS 2/4: one plane;
// BITS 3: 2-bit plane words first, then the 1-bit plane).
template <int D, int BITS>
__device__ __forceinline__ uint32_t contrib(int w, int idx, int half, uint32_t m, int words_lo) {
    if (BITS == 3) {
        uint32_t v = 0;
        if (w == idx / 8) v |= (m & 3u) << (16 * half + 2 * (idx % 8));
        if (w == words_lo + idx / 16) v |= ((m >> 2) & 1u) << (16 * half + bit1_pos(idx % 16));
        return v;
    }
    constexpr int F = 16 / BITS;
    return (w == idx / F) ? (m << (16 * half + BITS * (idx % F))) : 0u;
}

// ---- mma.sync m16n8k16, fp32 accumulate -----------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Split x into hi + lo 16-bit parts (hi = round(x), lo = round(x - hi)) and
// pack two such parts (for x0, x1) into a 32-bit register.
__device__ __forceinline__ void split_f16(float x, __half &hi, __half &lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) {
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 2^e as an exact fp32 constant, e in [-126, 127].
__host__ __device__ __forceinline__ float pow2i(int e) {
#ifdef __CUDA_ARCH__
    return __int_as_float((127 + e) << 23);
#else
    return e >= 0 ? static_cast<float>(1u << e) : 1.0f / static_cast<float>(1u << (-e));
#endif
}

// ---- bulk async copy (TMA, non-tensor) + mbarrier --------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::);
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// 2^x with the hardware approximation (relative error ~2^-22), flushing
// subnormal results to zero; exp2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- checked build -------------------------------------------------------------
// With DQ_CHECKED defined (the library's bounds-checked build), an access on the
// affine path first tests that its byte range [p, p + bytes) lies inside its
// buffer [base, base + size); one that does not latches ST_OOB and is skipped
// (no trap: the kernel runs on and the host reads the status).  Without it the
// test is a constant true and compiles away.
__device__ __forceinline__ bool in_buf(const void *p, long long bytes, const void *base, long long size,
                                       unsigned *status) {
#ifdef DQ_CHECKED
    const char *a = static_cast<const char *>(p), *b = static_cast<const char *>(base);
    if (b == nullptr || a < b || bytes < 0 || a + bytes > b + size) {
        atomicOr(status, 32u);  // ST_OOB
        return false;
    }
#else
    (void)p; (void)bytes; (void)base; (void)size; (void)status;
#endif
    return true;
}

// Fetch-and-add with acquire-release semantics at GPU scope: writes made
// before it (by the caller, or by its block before a barrier the caller
// passed) are visible to whoever observes the new count, and writes released
// by earlier adds to the same counter are visible to the caller.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Longest a single try_wait may suspend the thread before it reports "not yet"
// (it returns as soon as the phase completes): waiting warps then sleep instead
// of spinning and leave the issue slots to the warps doing arithmetic.
constexpr unsigned WAIT_SUSPEND_NS = 1000000;

// Wait for phase `parity` of an mbarrier for at most `limit_ns` nanoseconds of
// wall time (try_wait may itself suspend for a while, so the bound is taken
// on the global timer, not on the number of polls).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, uint64_t limit_ns) {
    const uint32_t addr = smem_u32(bar);
    uint64_t t0 = 0;
    for (unsigned it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(addr), "r"(parity), "n"(WAIT_SUSPEND_NS)
            : "memory");
        if (done) return true;
        if (it == 0) t0 = global_ns();
        else if (global_ns() - t0 > limit_ns) return false;
    }
}

}  // namespace dq
