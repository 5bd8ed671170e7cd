// Internal declarations shared by the host API and the CUDA kernels of libdq.
#pragma once

#include <cstddef>
#include <cstdint>

#include "dq.h"

namespace dq {

// Status bits latched on the device (ctx->status word).
enum : unsigned { ST_NONFINITE = 1u, ST_TIMEOUT = 2u, ST_BOUNDS = 4u, ST_INFEASIBLE = 8u, ST_SIDE_FULL = 16u,
                  ST_OOB = 32u };  // ST_OOB: a checked build skipped an access outside its buffer

// Sizes and strides derived from a config (all in bytes unless noted).
struct Layout {
    int B, Hkv, Hq, G, d;
    int U;               // units = B * Hkv
    int bits_k, bits_v;
    int rowK;            // bytes per key record
    int pairV;           // bytes per value pair record
    long long qcap;      // quantized slots per unit (multiple of 16)
    int rcap;            // raw slots per unit (multiple of 16)
    int meta_bytes;      // 2 (fp16) or 4 (fp32) per scale/offset value
    int n_sink, n_recent;
    // non-uniform scheme (scheme == DQ_NUQ)
    int scheme;          // dq_scheme of both tensors
    int levels;          // 2^bits table entries
    int k_out_cap;       // key outliers per channel at the longest prefill
    long long nnzk_cap;  // key side-channel entries per unit (multiple of 8): twice the longest prefill's
    int k_out_v;         // value outliers per token
    long long rp_stride; // ints per unit of the key row pointers (qcap + 4)
    int gv;              // value tables per token (head_dim / group_size)
    int refit;           // key table block in quantized slots (0: one frozen block)
    long long nbk;       // key table blocks per unit
    // entropy-coded scheme (scheme == DQ_RANS): one stream per token and tensor
    int n_stream;        // values per stream = Hkv * d
    int ck, cv;          // container bytes of a key / value stream
    int mk, mv;          // levels of the key / value grid
    long long wcap;      // mean windows per sequence (qcap / 128)
    int mean_rec;        // bytes per window record: n_stream INT8 + fp16 scale, padded to 16
    size_t sz[DQ_NUM_BUFFERS];
};

// Entropy-coded scheme: the symbol model of one tensor (host-built, copied to
// the device context).  dec[z] = m | f_m << 4 | (z - c_m) << 16 for the 2^8
// slots z of the decoder.
constexpr int RANS_MAX_LEVELS = 16;
struct RansTable {
    int M, C;
    int f[RANS_MAX_LEVELS], c[RANS_MAX_LEVELS];
    long long r[RANS_MAX_LEVELS];            // costs, 16 fractional bits, rounded up
    float rf[RANS_MAX_LEVELS];               // r / 2^16 (exact)
    unsigned long long rcp[RANS_MAX_LEVELS]; // ceil(2^40 / f): x / f = (x * rcp) >> 40 for x < 2^31
    uint32_t dec[256];
    long long budget_fx;                     // (8C - 32) * 2^16
    long long min_stream_cost;               // n * min r
};
struct RansDevTables {
    RansTable k, v;
    float F[512];                            // fp32(2^(k/512))
};
// Unsharpened level probabilities p[0..M) of the Gaussian order-statistics model
// for streams of n values (0, or -1 for n < 1 or M outside [2, 16]).
int rans_model_probs(int n, int M, double *p);
int rans_build_table(int n, int M, double alpha, int prob_bits, int C, RansTable *t);
void rans_pow2_table(float *F);

// Per-launch arguments of the entropy-coded prefill kernels.
struct RansQuantArgs {
    const void *x;          // [B][Hkv][n_tok][128] input
    int in_dtype;
    int B, Hkv, n;          // n = Hkv * 128
    long long n_tok;        // prefill length
    int n_sink, n_recent;
    int n_fit;              // quantized tokens n_tok - n_sink
    int is_key, rot;
    float hscale;
    int n_win;              // mean windows covering the quantized tokens
    long long qcap, wcap;
    int rcap, mean_rec;
    uint8_t *mean;          // [B][wcap][mean_rec] or nullptr
    uint8_t *sym;           // scratch [B][n_fit][n] symbols
    uint8_t *codes;         // [B][qcap][C] containers
    void *meta;             // [B][qcap] (s, o) fp16
    uint16_t *raw;          // [U][rcap][128] or [U][rcap/2][128][2]
    unsigned *status;
    // appends (block flush): tokens [pos0, pos0 + n_tok) are this call's input; the
    // quantized slots [slot0, slot0 + n_fit) are (re)encoded, their tokens read from
    // the input or, when older, from the 16-bit recent ring (raw, kv dtype raw_bf16)
    long long pos0, slot0;
    int raw_bf16;
    int raw_ns, raw_nr;     // this call's tokens copied as sinks / into the recent ring
    // drift statistics, accumulated: symbols off the nearest level of their
    // final grid, symbols coded, largest distance (or nullptr)
    unsigned long long *drift_stats;
};
int launch_rans_mean(const RansQuantArgs &a, void *stream);
int launch_rans_drift(const RansQuantArgs &a, const RansTable *tb, const float *F, int M, void *stream);
int launch_rans_encode(const RansQuantArgs &a, const RansTable *tb, int C, void *stream);
int launch_rans_raw(const RansQuantArgs &a, void *stream);

// Per-call arguments of the entropy-coded decode attention.
struct RansAttnArgs {
    const float *q;          // [B][4 Hkv][128]
    void *out;               // [B][4 Hkv][128]
    int out_dtype;
    const uint8_t *codes_k, *codes_v;  // [B][qcap][ck] / [B][qcap][cv]
    const void *meta_k, *meta_v;       // [B][qcap] (s, o) fp16
    const uint8_t *mean;     // [B][wcap][mean_rec] or nullptr
    const uint16_t *raw_k, *raw_v;
    int B, Hkv, ck, cv;
    long long qcap, wcap;
    int mean_rec, rcap;
    long long n_q;           // quantized slots read: [0, n_q)
    int n_sink_eff, n_sink_cfg, n_recent_cfg;
    long long recent_t0;     // first token of the recent window read
    int n_raw;               // 16-bit tokens read
    int rot_k, rot_v, raw_bf16;
    float hscale, sm_log2;
    float *partials;         // [B][items_per_b][4 Hkv][132]
    unsigned *status;
    int n_qitems, items_per_b;  // set by the launcher
};
int launch_attention_rans(const RansAttnArgs &a, const RansDevTables *tabs, void *stream);
long long rans_partial_floats(int B, int Hq, long long qcap);

dq_status make_layout(const dq_config *cfg, Layout *L);

// Record `msg` as this thread's last error (empty for DQ_OK) and return `s`.
dq_status set_last_error(dq_status s, const char *msg);

// Per-launch arguments of the quantize kernels.
struct QuantArgs {
    const void *x;          // [B][Hkv][n_tok][d] input
    int in_dtype;           // dq_dtype
    long long pos0, n_tok;  // tokens [pos0, pos0+n_tok)
    long long seq_after;    // pos0 + n_tok
    int is_key;
    int bits, rot, use_mean, meta_f16;
    float clip;             // 0 or kappa
    float quest_c;          // > 0: the QuEST grid, s = quest_c * RMS (clip is 0)
    int clip_ilo, clip_ihi; // quantile order-statistic indices
    float clip_flo, clip_fhi;
    float hscale;           // fp32(1/sqrt(d))
    uint8_t *codes;         // codes_k or codes_v
    void *meta;
    float *mean;            // [U][d] (keys with mean) or nullptr
    const float *T;         // dense transform [Hkv][d][d] or nullptr
    uint16_t *raw;          // raw_k or raw_v
    unsigned *status;
    // non-uniform scheme
    uint16_t *lut;          // keys [U][nbk][d][L], values [U][Qcap][gv][L] fp16 tables
    uint32_t *olbits;       // keys: [U][Qcap][d/32] outlier bitmap (scratch, zeroed first)
    int *ol_rowptr;         // keys: [U][rp_stride] row pointers by quantized slot
    uint16_t *ol_col, *ol_val;  // keys: [U][nnzk_cap]; values: [U][Qcap][k_out_v]
    int k_out;              // outliers per vector (keys: per channel at this prefill)
    int iters;              // Lloyd sweeps
    int n_fit;              // keys: quantized tokens in the prefill
    float *thr;             // keys: [U][d] outlier thresholds frozen at prefill (fp32 magnitudes)
    long long slot_lo;      // first quantized slot written by this call
    int n_slots;            // quantized slots written by this call
    // key refit blocks (Layout::refit > 0): the prefill's quantized slot count
    // per unit (a block starting at or after it holds decode keys only)
    int *pq;                // [U]
    // key fit: input rows [fit_t0, fit_t0 + n_fit) of each unit are quantized
    // slots [fit_slot0, ...); the table goes to blocks [fit_blk, fit_blk +
    // fit_nblk); fit_flush: a refit block, skipped where the prefill reached it
    long long fit_t0, fit_slot0;
    int fit_blk, fit_nblk, fit_flush;
    // block flush: fp32 keys of quantized slots [scr_lo, scr_lo + scr_n) per
    // unit, [U][scr_n][d], gathered from the input and the recent window
    float *scr;
    long long scr_lo;
    int scr_n;
    // byte sizes of the buffers above (the checked build tests accesses against them)
    long long sz_x, sz_codes, sz_meta, sz_mean, sz_raw;
};

// The geometry a token row's quantizer needs (a slice of Layout).
struct RowGeom {
    int U, Hkv, n_sink, n_recent, rcap, rowK, pairV;
    long long qcap;
};
inline RowGeom row_geom(const Layout &L) {
    return RowGeom{L.U, L.Hkv, L.n_sink, L.n_recent, L.rcap, L.rowK, L.pairV, L.qcap};
}

struct AttnArgs {
    const float *q;         // [B][Hq][d]
    void *out;              // [B][Hq][d]
    int out_dtype;
    const uint8_t *codes_k, *codes_v;
    const void *meta_k, *meta_v;
    const float *mean_k;    // nullptr if no mean
    const uint16_t *raw_k, *raw_v;
    const float *q_comp;    // [Hkv][d][d] T^{-T} or nullptr
    const float *q_tilde;   // [B][Hq][d] T^{-T} q computed beforehand, or nullptr
    int rot_k, rot_v;
    int raw_bf16;           // raw region dtype: 1 bf16, 0 fp16
    long long seq_len;
    long long n_q;          // quantized tokens read: [n_sink, n_sink + n_q)
    int n_sink_eff;         // valid sink slots
    int n_raw_slots;        // raw slots scanned (n_sink + n_recent)
    int n_sink_cfg, n_recent_cfg;
    int has_raw;            // 1 if the unit has 16-bit slots
    int raw_all_valid;      // seq_len >= n_sink + n_recent: every 16-bit slot is in use
    int n_rt;               // 16-slot tiles of 16-bit tokens per unit
    long long n_qc;         // packed pipeline entries per unit (128 tokens each, the last ragged)
    long long items_per_unit, total_items;  // pipeline entries: n_rt + n_qc per unit
    int grid;               // persistent CTAs (one wave)
    int max_slots;          // partial-record slots per unit
    float sm_log2;          // sm_scale * log2(e)
    float hscale;
    float *partials;        // [U][max_slots][2 kinds][4 heads][d + 4]
    int *counters;          // [U] CTAs done with the unit; zero between calls
    unsigned *status;
    // non-uniform scheme
    const uint16_t *lut_k, *lut_v;        // [U][nbk][d][L] / [U][Qcap][gv][L] fp16 tables
    int gv;                               // value tables per token
    int refit;                            // key table block in slots (0: one block)
    long long nbk;                        // key table blocks per unit
    const int *ol_rowptr_k;               // [U][rp_stride] key side-channel rows by slot (or null)
    const uint16_t *ol_col_k, *ol_val_k;  // [U][nnzk_cap]
    const uint16_t *ol_col_v, *ol_val_v;  // [U][Qcap][k_out_v]
    long long rp_stride, nnzk_cap;
    int k_out_v;                          // value outliers per token (0: none)
    // affine kernel schedule (set by plan_affine; affine = 1 routes the
    // launch to it)
    int affine;
    long long n_pt;                       // 16-token packed tiles per unit
    long long cpu;                        // packed chunks per unit
    long long np_total, nr_total;         // packed chunks / 16-bit tiles of all units
    int wp;                               // packed warps per CTA
    int mps;                              // record slots per unit taken by packed CTAs
    // fused decode step: the call first appends token seq_len - 1 (one row per
    // unit of the keys qa[0] and values qa[1]; the 16-bit-tile warp holding its
    // recent-window slot quantizes it and reads its 16-bit row from the input)
    int append;
    QuantArgs qa[2];
    RowGeom rg;
    // byte sizes of the buffers above (the checked build tests accesses against them)
    long long sz_q, sz_out, sz_codes_k, sz_codes_v, sz_meta_k, sz_meta_v, sz_mean_k, sz_raw_k, sz_raw_v, sz_q_comp;
    long long sz_partials, sz_counters;
};

// Byte sizes of the attention call's buffers other than its workspace (the
// checked build tests accesses against them).
inline void attn_extents(const Layout &L, int out_dtype, AttnArgs &a) {
    const long long qo = static_cast<long long>(L.B) * L.Hq * L.d;
    a.sz_q = qo * 4;
    a.sz_out = qo * (out_dtype == DQ_F32 ? 4 : 2);
    a.sz_codes_k = static_cast<long long>(L.sz[0]);
    a.sz_codes_v = static_cast<long long>(L.sz[1]);
    a.sz_meta_k = static_cast<long long>(L.sz[2]);
    a.sz_meta_v = static_cast<long long>(L.sz[3]);
    a.sz_mean_k = static_cast<long long>(L.sz[4]);
    a.sz_raw_k = static_cast<long long>(L.sz[7]);
    a.sz_raw_v = static_cast<long long>(L.sz[8]);
    a.sz_q_comp = static_cast<long long>(L.sz[16]);
}

struct DequantArgs {
    const uint8_t *codes;
    const void *meta;
    const float *mean;
    int is_key, bits, meta_f16;
    long long slot0, n;
    float *out;
    long long sz_codes, sz_meta, sz_mean, sz_out;  // byte sizes (checked build)
    unsigned *status;                               // checked build: ST_OOB
};

struct AttnArgs;
// Fill the non-uniform scheme's table and side-channel pointers (no-op otherwise).
void set_nuq_args(const Layout &L, const dq_kv_buffers *b, AttnArgs &a);

// launchers (return cudaError_t as int)
int launch_key_mean(const Layout &L, const QuantArgs &a, void *stream);
int launch_quantize(const Layout &L, const QuantArgs &a, void *stream);
// non-uniform scheme, prefill: value tables/codes/outliers and raw copies;
// key tables + outlier bitmap; key codes and raw copies; key side channel
int launch_nuq_values(const Layout &L, const QuantArgs &a, void *stream);
int launch_nuq_key_fit(const Layout &L, const QuantArgs &a, void *stream);
int launch_nuq_key_codes(const Layout &L, const QuantArgs &a, void *stream);
int launch_nuq_key_csr(const Layout &L, const QuantArgs &a, void *stream);
// key refit blocks: gather the keys of a.scr's slots, code the gathered blocks
int launch_nuq_gather(const Layout &L, const QuantArgs &a, void *stream);
int launch_nuq_block_codes(const Layout &L, const QuantArgs &a, void *stream);
int nuq_outlier_count(float f, int n);
int launch_dequant(const Layout &L, const DequantArgs &a, void *stream);
int launch_attention(const Layout &L, const AttnArgs &a, int num_sms, void *stream);
// q~ = T^{-T} q of every query head into qt [B][Hq][d] (dense key transforms)
int launch_qcomp(const Layout &L, const float *q, const float *qc, float *qt, void *stream);
// test support: a kernel whose bounded wait runs out (see dq_test_expire_wait)
int launch_expire_wait(unsigned *status, int *counters, unsigned long long limit_ns, void *stream);
// test support: one range test that fails in the checked build (see dq_test_checked_probe)
int launch_checked_probe(unsigned *status, void *stream);
// Fill the work schedule of `a` (items, grid, partial slots) for a launch on a
// device with num_sms SMs whose partial workspace holds cap_floats floats.
int plan_attention(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats);
long long attention_partial_floats(const Layout &L, const AttnArgs &a);
size_t attention_smem_bytes(const Layout &L);
// The affine kernel (attn_affine.cu; 2-4 bit codes at d 128, 2 and 4 at d 64); plan_attention
// routes a call to it when it applies (a supported shape whose packed tokens
// carry at least as many bytes as its 16-bit slots) and marks a.affine.
bool affine_kernel_applies(const Layout &L, const AttnArgs &a);
int plan_affine(const Layout &L, AttnArgs &a, int num_sms, long long cap_floats);
long long affine_partial_floats(const Layout &L, const AttnArgs &a);
int launch_affine(const Layout &L, const AttnArgs &a, void *stream);
size_t affine_smem_bytes(const Layout &L);

}  // namespace dq

struct dq_ctx {
    dq_config cfg;
    dq::Layout L;
    int device;
    int num_sms;
    unsigned *status;    // device word
    float *partials;     // split partials
    size_t partials_cap; // floats
    int *counters;       // [U]
    int counters_dirty;  // set by dq_check after a timeout: clear the counts before the next call
    uint32_t *nuq_bits;  // non-uniform scheme: key outlier bitmap scratch [U][Qcap][d/32]
    float *nuq_scr;      // non-uniform scheme, key refit blocks: gathered keys
    size_t nuq_scr_cap;  // floats
    dq::RansDevTables *rans;  // entropy-coded scheme: symbol models (device)
    uint8_t *rans_sym;   // entropy-coded scheme: symbol scratch of a prefill
    float *rans_partials;  // entropy-coded scheme: attention item records
    float *q_tilde;      // dense key transform: compensated queries [B][Hq][d]
    unsigned long long *drift_stats;  // entropy-coded scheme: [keys, values][changed, coded, largest move]
    size_t rans_sym_cap; // bytes
};
