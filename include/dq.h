/*
 * dq.h -- C ABI of libdq: quantized KV cache + GQA decode attention on GB300.
 *
 * What it computes
 * ----------------
 * dq_quantize_kv turns each token's key and value (one vector of head_dim
 * values per KV head) into a fixed-size record of low-bit codes:
 *   - an optional normalized Hadamard rotation per head (keys rotated online,
 *     "D-Quant: Driftable Entropy Coding for KV Cache Quantization", Sec. 4.2),
 *     or a dense d x d key transform applied after RoPE ("WUSH-KV: KV Cache
 *     Quantization with Data-Adaptive Transforms", Key Contributions 2);
 *   - removal of the key channel mean (D-Quant Sec. 4.2), frozen at prefill;
 *   - a per-token affine grid x^ = o + s*m (D-Quant Sec. 3.1 Eq. (1) and
 *     Sec. 4.2 Eq. (4)), from min/max or from a two-sided percentile clip
 *     (WUSH-KV, Methodology: OSCAR-style percentile-clipped affine), with s
 *     and o rounded to fp16 before the codes are assigned (D-Quant App. A);
 *   - the first n_sink tokens and the latest n_recent tokens also kept exact
 *     in 16-bit ("KVQuant-NUQ", Attention Sink-Aware quantization; D-Quant
 *     Sec. 5.1: the most recent 128 tokens in BF16).
 * dq_decode_attention computes, for every query head h of every sequence,
 *   out_h = sum_t softmax_t(sm_scale * q_h . k^_t) v^_t
 * over the cache of length seq_len, reading the packed codes and applying the
 * affine terms after the contraction (D-Quant App. A Eq. (7)-(9)).  Query head
 * h reads KV head floor(h * n_kv_heads / n_q_heads) (grouped-query attention).
 *
 * Conventions
 * -----------
 * - Every pointer named "device" is CUDA global memory of the current device;
 *   the caller allocates and owns it.  Nothing here frees caller memory.
 * - Every buffer must be 16-byte aligned (DQ_EALIGN otherwise).
 * - Calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and return without synchronizing.  Argument errors are found on
 *   the host before anything is enqueued and leave all buffers untouched.
 *   Conditions found on the device (non-finite input) are latched in the
 *   context and returned by dq_check().
 * - A context (dq_ctx) is created by the first call that receives a pointer
 *   to a NULL context; it holds the library's workspace on the device that
 *   was current then and is bound to that config.  One context must not be
 *   used from two host threads at once.  Release it with dq_free().
 * - No function throws, aborts, exits or prints.  dq_last_error() gives a
 *   thread-local message for the last failing call.
 */
#ifndef DQ_H
#define DQ_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DQ_OK = 0,
    DQ_EINVAL = 1,        /* bad argument, size or config */
    DQ_EALIGN = 2,        /* a buffer is not 16-byte aligned */
    DQ_EUNSUPPORTED = 3,  /* valid but not implemented combination */
    DQ_EINFEASIBLE = 4,   /* rANS container cannot hold the cheapest stream */
    DQ_ENOMEM = 5,        /* workspace allocation failed */
    DQ_ECUDA = 6,         /* a CUDA runtime call failed */
    DQ_ENONFINITE = 7,    /* a quantized input value was NaN or infinite */
    DQ_ETIMEOUT = 8       /* a bounded device wait ran out */
} dq_status;

typedef enum { DQ_F32 = 0, DQ_F16 = 1, DQ_BF16 = 2 } dq_dtype;
typedef enum { DQ_AFFINE = 0, DQ_NUQ = 1, DQ_RANS = 2 } dq_scheme;
typedef enum { DQ_ROT_NONE = 0, DQ_ROT_HADAMARD = 1, DQ_ROT_DENSE = 2 } dq_rot;
/* Affine grid of a token ("D-Quant", Sec. 4.2 Eq. (4); "WUSH-KV", evaluation). */
typedef enum { DQ_GRID_MINMAX = 0, DQ_GRID_QUEST = 1 } dq_grid;

/* Quantizer settings of one tensor (keys or values). */
typedef struct {
    int scheme;          /* dq_scheme */
    int bits;            /* affine/NUQ code width: 2, 3 or 4 (3 needs head_dim 128) */
    int levels;          /* DQ_RANS: alphabet size M */
    int container_bytes; /* DQ_RANS: record size C */
    int rot;             /* dq_rot; DQ_ROT_DENSE is keys only */
    int mean;            /* keys only: 1 = remove the channel mean frozen at prefill */
    float clip;          /* 0 = min/max grid; kappa in (0.5, 1) = clip to the
                            (1-kappa, kappa) linear-interpolated quantiles */
    int grid;            /* DQ_AFFINE: DQ_GRID_MINMAX (min/max, or the clip above)
                            or DQ_GRID_QUEST, the QuEST integer grid ("WUSH-KV",
                            evaluation: per token, symmetric, clipped from the
                            RMS): 2^bits levels o + s m with s = c_b RMS and
                            o = -((2^bits - 1)/2) s, RMS over the token's
                            rotated (mean-removed) values, c_b from
                            dq_quest_step; needs clip = 0 */
    int lloyd_iters;     /* DQ_NUQ */
    float outlier_frac;  /* DQ_NUQ */
    int group_size;      /* DQ_NUQ values: channels per value table, 0 (the
                            whole token) or 32 ("KVQuant-NUQ", Configuration
                            reference, kvquant_group_size): a token's outliers
                            are ranked over the token, then each group of 32
                            consecutive channels is fitted alone.  32 needs
                            head_dim 128.  Keys: 0 (a key table spans its
                            channel's tokens) */
    int refit_interval;  /* DQ_NUQ keys ("KVQuant-NUQ", Configuration reference,
                            kvquant_refit_interval): 0 = the prefill's tables,
                            frozen; N > 0, a multiple of 128, = key tables per
                            block of N quantized slots, refitted on each block
                            of decode keys when it completes (see
                            dq_quantize_kv).  Values: 0 */
} dq_tensor_cfg;

typedef struct {
    int batch, n_kv_heads, n_q_heads, head_dim, max_seq;
    int kv_dtype;        /* dq_dtype of the K/V handed to dq_quantize_kv */
    int meta_dtype;      /* DQ_F16 or DQ_F32: storage of s and o */
    int out_dtype;       /* dq_dtype of the attention output */
    dq_tensor_cfg k, v;
    int n_sink, n_recent;
    float rans_alpha;    /* DQ_RANS: sharpening exponent */
    int rans_prob_bits;  /* DQ_RANS: frequency precision p */
} dq_config;

/*
 * Cache buffers (device, caller-owned).  dq_kv_sizes() gives the byte size
 * of each, in field order; a field whose size is 0 is unused and may be NULL.
 *
 * U = batch * n_kv_heads units, unit u = b * n_kv_heads + kv_head.
 * Qcap = round_up(max_seq - n_sink, 64) quantized slots per unit; token
 * t >= n_sink lives in quantized slot t - n_sink.
 * Rcap = round_up(n_sink + n_recent, 16) raw slots per unit; token t < n_sink
 * in raw slot t, the latest n_recent tokens in raw slot n_sink + t % n_recent.
 *
 * codes_k  [U][Qcap][Rk]      key records, Rk = head_dim*bits_k/8 bytes
 * codes_v  [U][Qcap/2][2*Rv]  value records, one per token pair
 * meta_k   [U][Qcap][2]       (s, o) per token, meta_dtype
 * meta_v   [U][Qcap][2]
 * mean_k   [U][head_dim]      fp32 key channel mean (rotated space)
 * raw_k    [U][Rcap][head_dim]           16-bit keys (kv dtype; fp16 for fp32 input)
 * raw_v    [U][Rcap/2][head_dim][2]      16-bit values, token pairs interleaved
 * k_transform [n_kv_heads][head_dim][head_dim] fp32 T (DQ_ROT_DENSE keys)
 * q_comp      [n_kv_heads][head_dim][head_dim] fp32 T^{-T} (query compensation)
 *
 * Bit layout of a record: little-endian 32-bit words; with b = 2 or 4 each
 * 16-bit half holds 16/b fields of b bits, field f at bits [b*f, b*f+b); with
 * b = 3 a 2-bit plane (low code bits, laid out as b = 2) is followed by a
 * 1-bit plane (16 fields per half, field f at bit P(f) of its half: P(f) =
 * 2f + 2 for f <= 6, 0 for f = 7, 2f - 13 for 8 <= f <= 14, 1 for f = 15).
 * Key channel c of a token goes to
 *   idx = ((c>>1)&3)*(d/8) + 2*(c>>4) + ((c>>3)&1), half = c&1;
 * value channel c of token t goes to
 *   idx = (c&7)*(d/8) + 2*(c>>4) + ((c>>3)&1), half = t&1,
 * in both cases word idx/F, field idx%F with F = 16/b.
 *
 * Non-uniform scheme (DQ_NUQ on both tensors; "KVQuant-NUQ", How it works:
 * Lloyd-Max levels, keys per channel, values per token, Dense-and-Sparse
 * outliers).  Codes keep the record layout above but index fp16 tables of
 * L = 2^bits levels; meta_v, mean_k and ol_rowptr_v are unused:
 * meta_k      [U][head_dim]       fp32 key outlier threshold of each channel,
 *                                 frozen at prefill (the magnitude of its kk-th
 *                                 rank outlier, +inf when kk = 0); present when
 *                                 kk > 0
 * lut_k       [U][NBK][head_dim][L]  fp16 levels of each key channel for
 *                                 each block of N = refit_interval quantized
 *                                 slots (NBK = ceil(Qcap / N); NBK = 1 when N
 *                                 = 0), then, when N > 0, [U] int32: the
 *                                 prefill's quantized slot count
 * lut_v       [U][Qcap][GV][L]    fp16 levels of each value token (by slot),
 *                                 GV = head_dim / group_size tables, channel c
 *                                 in table c / group_size (GV = 1 for 0)
 * ol_rowptr_k [U][Qcap+4]         int32: key outliers of slot p are entries
 *                                 [rowptr[p], rowptr[p+1]); rowptr[p] for p
 *                                 >= the quantized token count holds the total
 * ol_col_k    [U][NNZk]           uint16 channel of each key outlier, channel
 *                                 order within a slot
 * ol_val_k    [U][NNZk]           its exact fp16 value
 * ol_col_v    [U][Qcap][kv]       uint16 channel of each value outlier of a
 *                                 token, in channel order
 * ol_val_v    [U][Qcap][kv]       its exact fp16 value
 * with kk = floor(k.outlier_frac * (max_seq - n_sink) + 0.5) outliers per key
 * channel, kv = floor(v.outlier_frac * head_dim + 0.5) per value token and
 * NNZk = round_up(2 * head_dim * kk, 8) (the prefill's bound twice: decode
 * keys add entries too).  A code of an outlier element is its
 * nearest level like any other; attention replaces the table value by the
 * stored one.
 *
 * Entropy-coded scheme (DQ_RANS on both tensors; "D-Quant: Driftable Entropy
 * Coding for KV Cache Quantization", Sec. 4.2-4.5 and App. A).  A stream is
 * the n = n_kv_heads * head_dim values of one token's key (or value), KV heads
 * in order; head_dim must be 128 and n_kv_heads 1, 2, 4 or 8.  Here
 * Qcap = round_up(max_seq - n_sink, 128) and quantized slot p of sequence b:
 * codes_k     [B][Qcap][Ck]    rANS containers of Ck = k.container_bytes:
 *                              the final 32-bit state little endian, then the
 *                              emitted bytes (last emitted first), then zeros
 * codes_v     [B][Qcap][Cv]
 * meta_k      [B][Qcap][2]     fp16 (s, o) of the stream's grid o + s m
 * meta_v      [B][Qcap][2]
 * mean_k      [B][Qcap/128][n + 16]  keys with mean = 1: per window of 128
 *                              quantized slots, n INT8 channel means (stream
 *                              order) and at byte n the fp16 scale; the mean
 *                              is q * scale
 * raw_k, raw_v as above; the other buffers are unused.  Symbols are coded with
 * p = 8 bits of probability, state floor L = 2^23, one byte at a time.
 */
typedef struct {
    void *codes_k, *codes_v, *meta_k, *meta_v, *mean_k;
    void *lut_k, *lut_v;
    void *raw_k, *raw_v;
    void *ol_rowptr_k, *ol_col_k, *ol_val_k, *ol_rowptr_v, *ol_col_v, *ol_val_v;
    void *k_transform, *q_comp;
} dq_kv_buffers;

#define DQ_NUM_BUFFERS 17

typedef struct dq_ctx dq_ctx;

/*
 * Byte size of every dq_kv_buffers field for `cfg`, in field order, into
 * bytes[DQ_NUM_BUFFERS].  Host only; enqueues nothing.
 * Errors: DQ_EINVAL (NULL argument or invalid config), DQ_EUNSUPPORTED.
 */
dq_status dq_kv_sizes(const dq_config *cfg, size_t bytes[DQ_NUM_BUFFERS]);

/*
 * Quantize tokens [pos0, pos0 + n_tok) of every sequence into the cache.
 *   k, v : device, [batch][n_kv_heads][n_tok][head_dim] contiguous, kv_dtype.
 * pos0 == 0 is a prefill of n_tok tokens: the key channel mean is computed over
 * tokens [n_sink, n_tok - n_recent) and frozen.  pos0 > 0 appends with the
 * frozen mean.  Every token t >= n_sink is written to its quantized slot;
 * sinks and the latest n_recent tokens (of length pos0 + n_tok) also to their
 * raw slots.  Requires pos0 + n_tok <= max_seq.
 * The dense key transform reads bufs->k_transform.
 * DQ_NUQ ("KVQuant-NUQ", Quantization axes) needs max_seq - n_sink <= 8192:
 * a prefill fits the key tables over every quantized token it has and freezes
 * them with each channel's outlier threshold.  An append (pos0 > n_sink, after
 * such a prefill; else DQ_EUNSUPPORTED) codes its keys against the frozen
 * tables, appends each element with |x| >= its channel's threshold to the key
 * side channel, and fits each value token as a prefill does.  Entries that
 * find the side channel full are not stored (the element keeps its level) and
 * dq_check reports DQ_EINFEASIBLE.  With a key refit_interval N > 0 the key
 * tables live per block of N quantized slots: the blocks a prefill reaches
 * hold its tables and their appended keys are coded as above; an appended key
 * of a later block stays in the 16-bit recent window only, and the append that
 * completes such a block fits that block's tables on its N keys (rank
 * outliers and Lloyd sweeps per channel, as a prefill of those tokens) and
 * codes them, reading the block's older keys from the recent window.  That
 * needs n_recent >= N, a 16-bit kv_dtype and head_dim 128, and appends that
 * follow one another without gaps.  DQ_RANS (D-Quant Sec. 4.2, windowed key mean): a
 * prefill encodes every token t >= n_sink, its last 128-slot window's mean
 * taken over the tokens it has; an append (pos0 > 0) keeps its tokens in the
 * 16-bit recent window only and, for each 128-slot window that it completes,
 * re-encodes the whole window (mean, fit, containers), reading the window's
 * older tokens from the recent window.  Appends therefore need n_recent >= 128
 * and a 16-bit kv_dtype (else DQ_EUNSUPPORTED), and must follow one another
 * without gaps.  A stream whose cheapest coding still exceeds its container
 * latches DQ_EINFEASIBLE (see dq_check).
 * Errors: DQ_EINVAL, DQ_EALIGN, DQ_EUNSUPPORTED, DQ_ENOMEM, DQ_ECUDA (launch).
 */
dq_status dq_quantize_kv(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs,
                         const void *k, const void *v, long long pos0, long long n_tok,
                         void *stream);

/*
 * Decode attention over the first seq_len tokens of every sequence.
 *   q   : device, [batch][n_q_heads][head_dim] fp32
 *   out : device, [batch][n_q_heads][head_dim] out_dtype
 * Requires 1 <= seq_len <= max_seq and that every token < seq_len was
 * quantized; with n_recent > 0, seq_len must be the length after the last
 * dq_quantize_kv call (the recent slots hold that call's latest tokens).  sm_scale multiplies q.k (1/sqrt(head_dim) is usual).  Dense key
 * transforms read bufs->q_comp to form T^{-T} q.
 * Uses the context's workspace for split partials; concurrent calls on one
 * context must be ordered on a stream.  DQ_RANS caches are decoded in place
 * (D-Quant Sec. 4.5: token-centric, each container decoded once, App. A
 * Eq. (8)-(9) for the affine terms); a container that asks for more bytes than
 * it holds (a corrupt cache) stops reading there and latches DQ_EINVAL for
 * dq_check.
 * Errors: DQ_EINVAL, DQ_EALIGN, DQ_EUNSUPPORTED, DQ_ENOMEM, DQ_ECUDA.
 */
dq_status dq_decode_attention(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs,
                              const void *q, void *out, long long seq_len, float sm_scale,
                              void *stream);

/*
 * One decode step: append token seq_len - 1 and attend over the first
 * seq_len tokens -- the same results as dq_quantize_kv(pos0 = seq_len - 1,
 * n_tok = 1) followed by dq_decode_attention(seq_len), cache bytes included
 * ("D-Quant", Sec. 5.1: the newest tokens stay 16-bit in the recent window and
 * enter the quantized region as they leave it; "KVQuant-NUQ", streaming
 * decode).
 *   k_new, v_new : device, [batch][n_kv_heads][1][head_dim] kv_dtype
 *   q, out       : as for dq_decode_attention
 * Requires 2 <= seq_len <= max_seq and a cache holding tokens [0, seq_len - 1).
 * For affine caches with n_recent >= 1 that the affine attention kernel serves
 * (head_dim 128 at 2-4 bits, head_dim 64 at 2 or 4 bits, at most 4 query
 * heads per KV head), the step is one kernel launch: the new token's packed
 * slot lies in the recent window, so nothing the attention reads depends on
 * its quantization, and its 16-bit row is read from k_new / v_new directly.
 * Otherwise the two calls run in order on the stream.
 * Errors: as dq_quantize_kv and dq_decode_attention.
 */
dq_status dq_decode_step(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs,
                         const void *k_new, const void *v_new, const void *q, void *out,
                         long long seq_len, float sm_scale, void *stream);

/*
 * Test export: write the dequantized fp32 values of quantized slots
 * [slot0, slot0 + n) of K (which = 0) or V (which = 1) into
 *   out : device, [batch][n_kv_heads][n][head_dim] fp32
 * in the quantizer's space (rotated; keys with the channel mean added back):
 * x^ = fp32(o + fp32(s*m)) (+ mu).  DQ_NUQ caches give DQ_EUNSUPPORTED (their
 * dequantized values are the table entries and the stored outliers).
 * Errors: DQ_EINVAL, DQ_EALIGN, DQ_EUNSUPPORTED, DQ_ENOMEM, DQ_ECUDA.
 */
dq_status dq_dequantize_kv(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs,
                           int which, long long slot0, long long n, float *out, void *stream);

/*
 * The symbol model of an entropy-coded (DQ_RANS) tensor: which = 0 keys,
 * 1 values.  Writes its number of levels M and the frequencies f[0..M) and
 * cumulative starts c[0..M) (f sums to 2^8; entries past M are 0).  Host only.
 * D-Quant Sec. 4.2 (the model comes from Gaussian order statistics: levels on
 * -a + 2a m/(M-1) with a the expected maximum of n standard normals, each
 * with the normal mass of its bin) and Sec. 4.4 (sharpening p' ~ p^alpha);
 * f_m = max(1, round(256 p'_m)) with the rounding shortfall given to the
 * largest frequency.
 * Errors: DQ_EINVAL, DQ_EUNSUPPORTED, DQ_EINFEASIBLE (as dq_kv_sizes).
 */
dq_status dq_rans_model(const dq_config *cfg, int which, int *levels, int f[16], int c[16]);

/*
 * The analytic symbol probabilities before sharpening: for streams of n
 * values on a per-token grid of `levels` levels, level m sits at normalized
 * position -a + 2a m/(levels-1), a = E[max of n iid N(0,1)], and p[m] is the
 * standard-normal mass of its bin (edges at the midpoints, outer bins open).
 * D-Quant Sec. 4.2 ("Gaussian order statistics"); Sec. 3 Table 1 and App. C
 * (Fig. 6 middle) compare this model with measured symbol frequencies (the
 * "Normal Gap").  Writes p[0..levels) (summing to 1) and zeros up to 16.
 * Host only: no device, stream or context is touched.
 * Errors: DQ_EINVAL (p NULL, n < 1, levels outside [2, 16]).
 */
dq_status dq_symbol_probs(int n, int levels, double p[16]);

/*
 * The QuEST grid's step factor c_b = fp32(2 alpha_b / 2^bits) ("WUSH-KV",
 * evaluation; the near-optimality result assumes Gaussian tails): alpha_b is
 * the clip of the symmetric 2^bits-level grid that minimizes its mean squared
 * error on a standard normal, rounded to 4 decimals (1.9914, 2.3441, 2.6816
 * for 2, 3, 4 bits).  A token's scale is s = c_b * RMS.
 * Host only.  Errors: DQ_EINVAL (c NULL, bits outside [1, 8]).
 */
dq_status dq_quest_step(int bits, float *c);

/*
 * Synchronize `stream`, then return and clear the device-side status latched
 * by earlier calls on this context (DQ_OK, DQ_ENONFINITE, DQ_ETIMEOUT,
 * DQ_EINFEASIBLE for a stream over its container or a full NUQ key side
 * channel, DQ_EINVAL for a container
 * that asked for more bytes than it holds), or
 * DQ_ECUDA if the stream reports an error.  ctx may be NULL (returns DQ_OK).
 * DQ_ETIMEOUT means a kernel stopped waiting after its time limit (2 s) so
 * that it could not hang: that call's output is not valid.  A timed-out
 * attention call may leave a per-unit record count behind; after dq_check has
 * reported DQ_ETIMEOUT, the next attention call on the context clears those
 * counts on its stream first, so the context stays usable.
 */
dq_status dq_check(dq_ctx *ctx, void *stream);

/*
 * Test support for the timeout path.  Enqueues on `stream` one kernel whose
 * bounded mbarrier wait (the same bounded wait the attention kernels use) is
 * on a barrier nothing ever arrives at, so it gives up after limit_ns
 * nanoseconds of wall time (clamped to [1000, 1e9]).  It then latches the
 * same device status and leaves the same stale per-unit record count a
 * timed-out attention call can leave, so that dq_check's DQ_ETIMEOUT report
 * and the context's recovery can be exercised without a fault or a hang.
 * `ctx` must come from an earlier call with a config (it owns the status word
 * and the counts).  Errors: DQ_EINVAL (ctx NULL or without a workspace),
 * DQ_ECUDA (launch).
 */
dq_status dq_test_expire_wait(dq_ctx *ctx, unsigned long long limit_ns, void *stream);

/*
 * Bounds-checked build.  Built with DQ_CHECKED defined (libdq_checked.so next
 * to libdq.so), the library tests every global access of the affine path --
 * the row quantizer and key mean, decode attention with the fused append, the
 * allocation-free entry point, dequantization -- against the byte size of its
 * buffer first; an access outside is skipped and latched, and dq_check then
 * returns DQ_EINVAL ("an access fell outside its buffer").  A skipped bulk copy
 * still completes its pipeline stage, so the call runs to its end.  The
 * non-uniform and entropy-coded kernels are not checked.
 * Test support: dq_test_checked_probe enqueues one range test that lies one
 * byte past a buffer (nothing is accessed): the checked build latches it, the
 * normal build does nothing.  Errors: DQ_EINVAL (ctx without a workspace),
 * DQ_ECUDA.
 */
dq_status dq_test_checked_probe(dq_ctx *ctx, void *stream);

/*
 * Drift statistics of the entropy-coded scheme ("D-Quant", App. C: drift makes
 * only sparse, local corrections).  Accumulated by every prefill and flush on
 * this context since it was created or last read, per tensor: the coded
 * symbols that drift moved off the nearest level of their stream's final
 * fp16 grid o + s m (nearest by |x - (o + s m)| in fp32, ties to the lower
 * level), the symbols coded, and the largest such move in levels.
 * Synchronizes `stream`, writes out[6] = {keys: changed, coded, largest move;
 * values: the same} and clears the counts.
 * Errors: DQ_EINVAL (NULL, or a context of another scheme), DQ_ECUDA.
 */
dq_status dq_drift_stats(dq_ctx *ctx, void *stream, unsigned long long out[6]);

/*
 * Allocation-free decode attention (this library's own addition; the pages
 * have no counterpart).  Computes exactly what dq_decode_attention computes,
 * with the same arguments minus the context, but never calls cudaMalloc,
 * cudaFree or any allocating routine.  It is meant for callers that may not
 * allocate device memory behind their own back: serving engines that hand out
 * all device memory from one pre-reserved pool, decode loops that cannot
 * afford the device-wide synchronization cudaMalloc/cudaFree can cause, and
 * embedders with a fixed device-memory budget.
 *
 * Scratch: the split partials and tickets live in one statically sized device
 * array of DQ_NOALLOC_SCRATCH_BYTES inside this library; every GPU that loads
 * the library holds it until the process exits.
 *   - The first call on a device looks up that array's device address (with
 *     that device current) and caches it; make this first call before any
 *     stream capture.
 *   - All calls share the array and it keeps the last call's contents; each
 *     call clears the part that must start at zero on `stream` first.  Calls
 *     whose work overlaps on the GPU (different streams, or different host
 *     threads without ordering) race on it and give wrong results: order them.
 *   - Limits: batch * n_kv_heads <= 16384 (one ticket each), and the split
 *     partials must fit the array: batch * n_kv_heads * r records of
 *     4 x (head_dim + 4) floats, r being the record slots the plan gives a
 *     unit (r = 2 to 7: one per CTA whose range touches the unit's packed
 *     tokens and one per CTA that takes some of its 16-bit tiles).  Large
 *     batches get r = 4 with 16-bit sink/recent slots and r = 2 without, so
 *     the bound that comes first is the partials one: about 3,960 units at
 *     head_dim 128 and 7,690 at head_dim 64 with 16-bit slots, twice that
 *     without (then the 16384 ticket limit caps head_dim 64).  Where the
 *     kernel can, the grid is narrowed until the partials fit; a config that
 *     still does not fit is refused with DQ_EINVAL and a message naming the
 *     bytes needed and held.
 *   - Device-side conditions (a bounded wait running out) are not reported by
 *     this entry point; use the context-based one with dq_check to see them.
 * DQ_RANS caches are refused (DQ_EUNSUPPORTED): their symbol model lives in a
 * context.
 * Errors: DQ_EINVAL, DQ_EALIGN, DQ_EUNSUPPORTED, DQ_ECUDA.
 */
#define DQ_NOALLOC_SCRATCH_BYTES (32u << 20)
dq_status dq_decode_attention_noalloc(const dq_config *cfg, const dq_kv_buffers *bufs, const void *q,
                                      void *out, long long seq_len, float sm_scale, void *stream);

/* Release a context and its workspace.  NULL-safe.  The caller must make sure
 * no enqueued work still uses it. */
void dq_free(dq_ctx *ctx);

/* Thread-local message of the last error returned on this thread ("" if none). */
const char *dq_last_error(void);

/* Static name of a status code. */
const char *dq_status_name(dq_status s);

#ifdef __cplusplus
}
#endif

#endif /* DQ_H */
