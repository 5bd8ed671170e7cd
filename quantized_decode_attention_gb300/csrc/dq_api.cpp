// Host side of libdq: validation, buffer sizes, the context, and launches.
// No exceptions cross the C ABI; errors are returned as dq_status with a
// thread-local message.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "dq.h"
#include "dq_internal.h"

namespace {

thread_local char g_err[512] = "";

dq_status fail(dq_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

dq_status ok() {
    g_err[0] = '\0';
    return DQ_OK;
}

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dq_status validate_tensor(const dq_tensor_cfg &t, int d, bool key, const char *name) {
    if (t.scheme != DQ_AFFINE && t.scheme != DQ_NUQ && t.scheme != DQ_RANS)
        return fail(DQ_EINVAL, "%s: unknown scheme %d", name, t.scheme);
    if (t.scheme == DQ_RANS) {
        if (t.levels < 2 || t.levels > dq::RANS_MAX_LEVELS)
            return fail(DQ_EINVAL, "%s: levels must be in [2, %d] (got %d)", name, dq::RANS_MAX_LEVELS, t.levels);
        if (t.container_bytes < 8 || t.container_bytes > 4096)
            return fail(DQ_EINVAL, "%s: container_bytes must be in [8, 4096]", name);
        if (t.rot != DQ_ROT_NONE && t.rot != DQ_ROT_HADAMARD)
            return fail(DQ_EUNSUPPORTED, "%s: the entropy-coded scheme takes no rotation or a Hadamard one", name);
        if (t.clip != 0.0f || t.grid != DQ_GRID_MINMAX)
            return fail(DQ_EUNSUPPORTED, "%s: the entropy-coded scheme takes no clip or grid choice", name);
        if (!key && t.mean) return fail(DQ_EINVAL, "%s: channel mean removal is for keys", name);
        return DQ_OK;
    }
    if (t.bits < 2 || t.bits > 4) return fail(DQ_EINVAL, "%s: bits must be 2, 3 or 4 (got %d)", name, t.bits);
    if (t.scheme == DQ_NUQ) {
        if (t.rot != DQ_ROT_NONE || t.mean || t.clip != 0.0f || t.grid != DQ_GRID_MINMAX)
            return fail(DQ_EUNSUPPORTED, "%s: the non-uniform scheme takes no rotation, mean, clip or grid", name);
        if (t.lloyd_iters < 0 || t.lloyd_iters > 64) return fail(DQ_EINVAL, "%s: lloyd_iters outside [0, 64]", name);
        if (!(t.outlier_frac >= 0.0f && t.outlier_frac < 0.5f))
            return fail(DQ_EINVAL, "%s: outlier_frac outside [0, 0.5)", name);
        if (key && t.group_size != 0)
            return fail(DQ_EUNSUPPORTED, "%s: a key table spans its channel's tokens (group_size 0)", name);
        if (!key && t.group_size != 0 && t.group_size != 32 && t.group_size != d)
            return fail(DQ_EUNSUPPORTED, "%s: group_size must be 0, 32 or head_dim (got %d)", name, t.group_size);
        if (!key && t.refit_interval != 0) return fail(DQ_EINVAL, "%s: refit_interval is for keys", name);
        if (t.refit_interval < 0 || t.refit_interval % 128)
            return fail(DQ_EINVAL, "%s: refit_interval must be 0 or a positive multiple of 128", name);
        if (((t.group_size != 0 && t.group_size != d) || t.refit_interval > 0) && d != 128)
            return fail(DQ_EUNSUPPORTED, "%s: value groups and key refit blocks need head_dim 128", name);
    } else if (t.group_size != 0 || t.refit_interval != 0) {
        return fail(DQ_EINVAL, "%s: group_size and refit_interval are for the non-uniform scheme", name);
    }
    if (t.bits == 3 && d != 128) return fail(DQ_EUNSUPPORTED, "%s: 3-bit records need head_dim 128", name);
    if (t.rot < DQ_ROT_NONE || t.rot > DQ_ROT_DENSE) return fail(DQ_EINVAL, "%s: bad rotation %d", name, t.rot);
    if (!key && t.rot == DQ_ROT_DENSE) return fail(DQ_EUNSUPPORTED, "%s: dense transform is for keys", name);
    if (!key && t.mean) return fail(DQ_EINVAL, "%s: channel mean removal is for keys", name);
    if (!(t.clip == 0.0f || (t.clip > 0.5f && t.clip < 1.0f)))
        return fail(DQ_EINVAL, "%s: clip must be 0 or in (0.5, 1)", name);
    if (t.grid != DQ_GRID_MINMAX && t.grid != DQ_GRID_QUEST) return fail(DQ_EINVAL, "%s: bad grid %d", name, t.grid);
    if (t.grid == DQ_GRID_QUEST && t.clip != 0.0f)
        return fail(DQ_EINVAL, "%s: the QuEST grid takes its clip from the RMS (clip must be 0)", name);
    return DQ_OK;
}

// ---- the QuEST grid's clip ---------------------------------------------------
// The symmetric grid of L levels clipped at +-alpha has step D = 2 alpha / L and
// level k at c_k = alpha (2k + 1 - L) / L, with decision points halfway between.
// Its mean squared error e on N(0,1) has the derivative
//   e'(alpha) = -2 sum_k (2k + 1 - L) / L * E[(X - c_k) ; X in cell k]
// (moving alpha moves level k at rate (2k+1-L)/L; the cell edges move too,
// but the error density is equal on both sides of a midpoint, so they add
// nothing), with E[X - c ; a < X < b] = phi(a) - phi(b) - c (Phi(b) - Phi(a)).
// e' is negative below the minimizing clip and positive above: bisection.
double gauss_cdf(double x) { return 0.5 * std::erfc(-x * 0.70710678118654752440); }
double gauss_pdf(double x) { return 0.39894228040143267794 * std::exp(-0.5 * x * x); }

double quest_clip(int bits) {
    const int L = 1 << bits;
    auto g = [L](double alpha) {
        const double D = 2.0 * alpha / L;
        double acc = 0.0;
        for (int k = 0; k < L; k++) {
            const double c = alpha * (2.0 * k + 1.0 - L) / L;
            const double pa = k == 0 ? 0.0 : gauss_pdf(-alpha + k * D);
            const double pb = k == L - 1 ? 0.0 : gauss_pdf(-alpha + (k + 1) * D);
            const double Pa = k == 0 ? 0.0 : gauss_cdf(-alpha + k * D);
            const double Pb = k == L - 1 ? 1.0 : gauss_cdf(-alpha + (k + 1) * D);
            acc += (2.0 * k + 1.0 - L) / L * ((pa - pb) - c * (Pb - Pa));
        }
        return -2.0 * acc;
    };
    double lo = 0.25, hi = 8.0;
    for (int it = 0; it < 200 && hi - lo > 1e-15; it++) {
        const double mid = 0.5 * (lo + hi);
        (g(mid) < 0.0 ? lo : hi) = mid;
    }
    return std::floor(0.5 * (lo + hi) * 1e4 + 0.5) / 1e4;  // 4 decimals
}

float quest_step_factor(int bits) {
    static float cache[9] = {};
    if (cache[bits] == 0.0f) cache[bits] = static_cast<float>(2.0 * quest_clip(bits) / (1 << bits));
    return cache[bits];
}

// Symbol models are a few milliseconds of host arithmetic; keep the last few.
struct TableCacheEntry {
    int n, M, C, p;
    float alpha;
    int rc;
    dq::RansTable t;
};
std::mutex g_table_mu;
TableCacheEntry g_tables[8];
int g_tables_n = 0, g_tables_next = 0;

int cached_table(int n, int M, float alpha, int p, int C, dq::RansTable *out) {
    std::lock_guard<std::mutex> lk(g_table_mu);
    for (int i = 0; i < g_tables_n; i++) {
        const TableCacheEntry &e = g_tables[i];
        if (e.n == n && e.M == M && e.C == C && e.p == p && e.alpha == alpha) {
            *out = e.t;
            return e.rc;
        }
    }
    TableCacheEntry &e = g_tables[g_tables_next];
    g_tables_next = (g_tables_next + 1) % 8;
    if (g_tables_n < 8) g_tables_n++;
    e.n = n;
    e.M = M;
    e.C = C;
    e.p = p;
    e.alpha = alpha;
    e.rc = dq::rans_build_table(n, M, alpha, p, C, &e.t);
    *out = e.t;
    return e.rc;
}

}  // namespace

namespace dq {

void set_nuq_args(const Layout &L, const dq_kv_buffers *b, AttnArgs &a) {
    if (L.scheme != DQ_NUQ) return;
    a.lut_k = static_cast<const uint16_t *>(b->lut_k);
    a.lut_v = static_cast<const uint16_t *>(b->lut_v);
    if (L.k_out_cap > 0) {
        a.ol_rowptr_k = static_cast<const int *>(b->ol_rowptr_k);
        a.ol_col_k = static_cast<const uint16_t *>(b->ol_col_k);
        a.ol_val_k = static_cast<const uint16_t *>(b->ol_val_k);
    }
    if (L.k_out_v > 0) {
        a.ol_col_v = static_cast<const uint16_t *>(b->ol_col_v);
        a.ol_val_v = static_cast<const uint16_t *>(b->ol_val_v);
        a.k_out_v = L.k_out_v;
    }
    a.rp_stride = L.rp_stride;
    a.nnzk_cap = L.nnzk_cap;
    a.gv = L.gv;
    a.refit = L.refit;
    a.nbk = L.nbk;
}

dq_status set_last_error(dq_status s, const char *msg) {
    if (s == DQ_OK) return ok();
    return fail(s, "%s", msg);
}

dq_status make_layout(const dq_config *cfg, Layout *L) {
    if (!cfg || !L) return fail(DQ_EINVAL, "NULL argument");
    const dq_config &c = *cfg;
    if (c.batch < 1 || c.n_kv_heads < 1 || c.n_q_heads < 1 || c.max_seq < 1)
        return fail(DQ_EINVAL, "batch, heads and max_seq must be positive");
    if (c.n_q_heads % c.n_kv_heads) return fail(DQ_EINVAL, "n_q_heads must be a multiple of n_kv_heads");
    const int G = c.n_q_heads / c.n_kv_heads;
    if (G > 4) return fail(DQ_EUNSUPPORTED, "at most 4 query heads per KV head (got %d)", G);
    if (c.head_dim != 64 && c.head_dim != 128) return fail(DQ_EUNSUPPORTED, "head_dim must be 64 or 128");
    if (c.kv_dtype < DQ_F32 || c.kv_dtype > DQ_BF16 || c.out_dtype < DQ_F32 || c.out_dtype > DQ_BF16)
        return fail(DQ_EINVAL, "bad dtype");
    if (c.meta_dtype != DQ_F16 && c.meta_dtype != DQ_F32) return fail(DQ_EINVAL, "meta_dtype must be F16 or F32");
    if (c.n_sink < 0 || c.n_recent < 0 || c.n_sink > c.max_seq) return fail(DQ_EINVAL, "bad n_sink / n_recent");
    dq_status s;
    if ((s = validate_tensor(c.k, c.head_dim, true, "k")) != DQ_OK) return s;
    if ((s = validate_tensor(c.v, c.head_dim, false, "v")) != DQ_OK) return s;
    if (c.k.scheme != c.v.scheme) return fail(DQ_EUNSUPPORTED, "keys and values must use the same scheme");
    if (c.k.scheme != DQ_RANS && c.k.bits != c.v.bits)
        return fail(DQ_EUNSUPPORTED, "keys and values must use the same code width");
    if (c.k.scheme == DQ_RANS) {
        if (c.head_dim != 128) return fail(DQ_EUNSUPPORTED, "entropy-coded scheme: head_dim must be 128");
        if (c.n_kv_heads != 1 && c.n_kv_heads != 2 && c.n_kv_heads != 4 && c.n_kv_heads != 8)
            return fail(DQ_EUNSUPPORTED, "entropy-coded scheme: 1, 2, 4 or 8 KV heads per stream");
        if (c.n_q_heads != 4 * c.n_kv_heads)
            return fail(DQ_EUNSUPPORTED, "entropy-coded scheme: 4 query heads per KV head");
        if (c.meta_dtype != DQ_F16) return fail(DQ_EINVAL, "entropy-coded scheme: metadata is fp16");
        if (c.rans_prob_bits != 8) return fail(DQ_EUNSUPPORTED, "entropy-coded scheme: prob_bits must be 8");
        if (!(c.rans_alpha > 0.0f && c.rans_alpha <= 8.0f)) return fail(DQ_EINVAL, "rans_alpha outside (0, 8]");
    }
    if (c.k.scheme == DQ_NUQ && c.max_seq - c.n_sink > 8192)
        return fail(DQ_EUNSUPPORTED, "non-uniform key fit: at most 8192 quantized tokens (got %d)",
                    c.max_seq - c.n_sink);
    if (c.k.scheme == DQ_NUQ && c.k.refit_interval > 0) {
        if (c.n_recent < c.k.refit_interval)
            return fail(DQ_EUNSUPPORTED, "key refit blocks: n_recent (%d) must hold a block (%d)", c.n_recent,
                        c.k.refit_interval);
        if (c.kv_dtype == DQ_F32)
            return fail(DQ_EUNSUPPORTED, "key refit blocks read the recent window back: kv_dtype must be 16-bit");
    }

    Layout &l = *L;
    std::memset(&l, 0, sizeof l);
    l.B = c.batch;
    l.Hkv = c.n_kv_heads;
    l.Hq = c.n_q_heads;
    l.G = G;
    l.d = c.head_dim;
    l.U = c.batch * c.n_kv_heads;
    l.bits_k = c.k.bits;
    l.bits_v = c.v.bits;
    l.rowK = c.head_dim * c.k.bits / 8;
    l.pairV = 2 * c.head_dim * c.v.bits / 8;
    l.qcap = round_up(c.max_seq - c.n_sink, c.k.scheme == DQ_RANS ? 128 : 64);
    l.rcap = static_cast<int>(round_up(c.n_sink + c.n_recent, 16));
    l.meta_bytes = c.meta_dtype == DQ_F16 ? 2 : 4;
    l.n_sink = c.n_sink;
    l.n_recent = c.n_recent;
    const size_t U = static_cast<size_t>(l.U), d = static_cast<size_t>(l.d);
    l.scheme = c.k.scheme;
    l.levels = 1 << c.k.bits;
    const bool nuq = l.scheme == DQ_NUQ;
    if (nuq) {
        l.k_out_cap = dq::nuq_outlier_count(c.k.outlier_frac, c.max_seq - c.n_sink);
        l.nnzk_cap = round_up(2LL * static_cast<long long>(d) * l.k_out_cap, 8);  // room for decode keys
        l.k_out_v = dq::nuq_outlier_count(c.v.outlier_frac, c.head_dim);
        l.rp_stride = l.qcap + 4;
        l.gv = c.v.group_size == 0 ? 1 : c.head_dim / c.v.group_size;
        l.refit = c.k.refit_interval;
        l.nbk = l.refit > 0 ? (l.qcap + l.refit - 1) / l.refit : 1;
    }
    l.sz[0] = U * l.qcap * l.rowK;                          // codes_k
    l.sz[1] = U * (l.qcap / 2) * l.pairV;                   // codes_v
    l.sz[2] = nuq ? (l.k_out_cap > 0 ? U * d * 4 : 0)      // meta_k; NUQ: frozen key outlier thresholds
                  : U * l.qcap * 2 * l.meta_bytes;
    l.sz[3] = nuq ? 0 : U * l.qcap * 2 * l.meta_bytes;      // meta_v
    l.sz[4] = c.k.mean ? U * d * 4 : 0;                     // mean_k
    l.sz[5] = nuq ? U * static_cast<size_t>(l.nbk) * d * l.levels * 2 + (l.refit > 0 ? U * 4 : 0) : 0;  // lut_k
    l.sz[6] = nuq ? U * l.qcap * l.gv * l.levels * 2 : 0;   // lut_v
    l.sz[7] = U * l.rcap * d * 2;                           // raw_k
    l.sz[8] = U * l.rcap * d * 2;                           // raw_v
    for (int i = 9; i < 15; i++) l.sz[i] = 0;               // outlier side-channels
    if (nuq && l.k_out_cap > 0) {
        l.sz[9] = U * l.rp_stride * 4;                      // ol_rowptr_k
        l.sz[10] = U * l.nnzk_cap * 2;                      // ol_col_k
        l.sz[11] = l.sz[10];                                // ol_val_k
    }
    if (nuq && l.k_out_v > 0) {
        l.sz[13] = U * l.qcap * l.k_out_v * 2;              // ol_col_v
        l.sz[14] = l.sz[13];                                // ol_val_v
    }
    l.sz[15] = c.k.rot == DQ_ROT_DENSE ? static_cast<size_t>(c.n_kv_heads) * d * d * 4 : 0;  // k_transform
    l.sz[16] = l.sz[15];                                    // q_comp
    if (c.k.scheme == DQ_RANS) {
        l.n_stream = c.n_kv_heads * c.head_dim;
        l.ck = c.k.container_bytes;
        l.cv = c.v.container_bytes;
        l.mk = c.k.levels;
        l.mv = c.v.levels;
        l.wcap = l.qcap / 128;
        l.mean_rec = l.n_stream + 16;
        const size_t B = static_cast<size_t>(c.batch);
        for (int i = 0; i < DQ_NUM_BUFFERS; i++) l.sz[i] = 0;
        l.sz[0] = B * l.qcap * l.ck;                        // codes_k: containers
        l.sz[1] = B * l.qcap * l.cv;                        // codes_v
        l.sz[2] = B * l.qcap * 4;                           // meta_k: (s, o) fp16
        l.sz[3] = B * l.qcap * 4;                           // meta_v
        l.sz[4] = c.k.mean ? B * l.wcap * l.mean_rec : 0;   // mean_k: INT8 window means + scale
        l.sz[7] = U * l.rcap * d * 2;                       // raw_k
        l.sz[8] = U * l.rcap * d * 2;                       // raw_v
        RansTable tk, tv;
        if (cached_table(l.n_stream, l.mk, c.rans_alpha, c.rans_prob_bits, l.ck, &tk) != 0 ||
            cached_table(l.n_stream, l.mv, c.rans_alpha, c.rans_prob_bits, l.cv, &tv) != 0)
            return fail(DQ_EINVAL, "entropy-coded scheme: no valid symbol model for these levels");
        if (tk.min_stream_cost > tk.budget_fx)
            return fail(DQ_EINFEASIBLE, "k: %d levels cannot fit a %d-byte container (cheapest stream %.1f bits)",
                        l.mk, l.ck, tk.min_stream_cost / 65536.0);
        if (tv.min_stream_cost > tv.budget_fx)
            return fail(DQ_EINFEASIBLE, "v: %d levels cannot fit a %d-byte container (cheapest stream %.1f bits)",
                        l.mv, l.cv, tv.min_stream_cost / 65536.0);
    }
    return DQ_OK;
}

}  // namespace dq

using dq::Layout;

static dq_status check_bufs(const Layout &L, const dq_kv_buffers *b) {
    const void *const *p = reinterpret_cast<const void *const *>(b);
    static const char *names[DQ_NUM_BUFFERS] = {"codes_k", "codes_v", "meta_k", "meta_v", "mean_k", "lut_k",
                                                "lut_v", "raw_k", "raw_v", "ol_rowptr_k", "ol_col_k", "ol_val_k",
                                                "ol_rowptr_v", "ol_col_v", "ol_val_v", "k_transform", "q_comp"};
    for (int i = 0; i < DQ_NUM_BUFFERS; i++) {
        if (L.sz[i] == 0) continue;
        if (!p[i]) return fail(DQ_EINVAL, "buffer %s is NULL", names[i]);
        if (!aligned16(p[i])) return fail(DQ_EALIGN, "buffer %s is not 16-byte aligned", names[i]);
    }
    return DQ_OK;
}

static bool same_cfg(const dq_config &a, const dq_config &b) { return std::memcmp(&a, &b, sizeof a) == 0; }

static dq_status get_ctx(dq_ctx **pctx, const dq_config *cfg, const Layout &L) {
    if (!pctx) return fail(DQ_EINVAL, "ctx pointer is NULL");
    if (*pctx) {
        if (!same_cfg((*pctx)->cfg, *cfg)) return fail(DQ_EINVAL, "context was created for a different config");
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev != (*pctx)->device)
            return fail(DQ_EINVAL, "context belongs to device %d", (*pctx)->device);
        return DQ_OK;
    }
    dq_ctx *c = new (std::nothrow) dq_ctx();
    if (!c) return fail(DQ_ENOMEM, "host allocation failed");
    std::memset(c, 0, sizeof *c);
    c->cfg = *cfg;
    c->L = L;
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
        delete c;
        return fail(DQ_ECUDA, "cannot query the current device");
    }
    // split partials for the largest persistent grid the attention kernel can
    // use (at most 8 CTAs per SM): a unit is touched by at most 2G/U + 2 CTAs,
    // each writing two records of 4 heads x (head_dim + 4) floats
    const long long G = 8LL * c->num_sms;
    c->partials_cap = static_cast<size_t>((2 * G + 2LL * L.U) * 2 * 4 * (L.d + 4));
    cudaError_t e1 = cudaMalloc(&c->status, sizeof(unsigned));
    cudaError_t e2 = cudaMalloc(&c->partials, c->partials_cap * sizeof(float));
    cudaError_t e3 = cudaMalloc(&c->counters, sizeof(int) * L.U);
    cudaError_t e4 = cudaSuccess;
    if (L.scheme == DQ_NUQ)
        e4 = cudaMalloc(&c->nuq_bits, static_cast<size_t>(L.U) * L.qcap * (L.d / 32) * sizeof(uint32_t));
    if (e4 == cudaSuccess && cfg->k.rot == DQ_ROT_DENSE)
        e4 = cudaMalloc(&c->q_tilde, sizeof(float) * static_cast<size_t>(L.B) * L.Hq * L.d);
    if (L.scheme == DQ_RANS) {
        e4 = cudaMalloc(&c->drift_stats, 6 * sizeof(unsigned long long));
        if (e4 == cudaSuccess) e4 = cudaMemset(c->drift_stats, 0, 6 * sizeof(unsigned long long));
        if (e4 == cudaSuccess) e4 = cudaMalloc(&c->rans, sizeof(dq::RansDevTables));
        if (e4 == cudaSuccess)
            e4 = cudaMalloc(&c->rans_partials,
                            sizeof(float) * static_cast<size_t>(dq::rans_partial_floats(L.B, L.Hq, L.qcap)));
    }
    if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess) {
        cudaFree(c->status);
        cudaFree(c->partials);
        cudaFree(c->counters);
        cudaFree(c->nuq_bits);
        cudaFree(c->nuq_scr);
        cudaFree(c->rans);
        cudaFree(c->rans_partials);
        cudaFree(c->q_tilde);
        delete c;
        cudaGetLastError();
        return fail(DQ_ENOMEM, "workspace allocation failed");
    }
    if (L.scheme == DQ_RANS) {
        dq::RansDevTables h;
        std::memset(&h, 0, sizeof h);
        if (cached_table(L.n_stream, L.mk, cfg->rans_alpha, cfg->rans_prob_bits, L.ck, &h.k) != 0 ||
            cached_table(L.n_stream, L.mv, cfg->rans_alpha, cfg->rans_prob_bits, L.cv, &h.v) != 0) {
            dq_free(c);
            return fail(DQ_EINVAL, "entropy-coded scheme: no valid symbol model");
        }
        dq::rans_pow2_table(h.F);
        if (cudaMemcpy(c->rans, &h, sizeof h, cudaMemcpyHostToDevice) != cudaSuccess) {
            dq_free(c);
            return fail(DQ_ECUDA, "symbol model upload failed");
        }
    }
    if (cudaMemset(c->status, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(c->counters, 0, sizeof(int) * L.U) != cudaSuccess) {
        dq_free(c);
        return fail(DQ_ECUDA, "workspace initialization failed");
    }
    *pctx = c;
    return DQ_OK;
}

// Non-uniform scheme ("KVQuant-NUQ" page, Quantization axes; Dense-and-Sparse
// outlier isolation).  A prefill (pos0 == 0) fits the key tables per channel
// over its quantized tokens and freezes them with each channel's outlier
// threshold; an append (pos0 > n_sink, after such a prefill) codes its keys
// against the frozen tables, sends |x| >= threshold to the side channel while
// it has room, and fits each value token as the prefill does.
static dq_status quantize_nuq(dq_ctx *c, const dq_config *cfg, const Layout &L, const dq_kv_buffers *bufs,
                              const void *k, const void *v, long long pos0, long long n_tok, void *stream) {
    if (pos0 != 0 && pos0 <= L.n_sink)
        return fail(DQ_EUNSUPPORTED, "non-uniform scheme: appends need a prefill that quantized a token (pos0 > n_sink)");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool append = pos0 > 0;
    dq::QuantArgs a{};
    a.in_dtype = cfg->kv_dtype;
    a.pos0 = pos0;
    a.n_tok = n_tok;
    a.seq_after = pos0 + n_tok;
    a.bits = cfg->k.bits;
    a.status = c->status;
    a.n_fit = append ? 0 : static_cast<int>(n_tok > L.n_sink ? n_tok - L.n_sink : 0);
    a.slot_lo = append ? pos0 - L.n_sink : 0;
    a.n_slots = append ? static_cast<int>(n_tok) : a.n_fit;
    int e;
    // values: per-token tables, codes and side channel; raw copies
    a.x = v;
    a.is_key = 0;
    a.codes = static_cast<uint8_t *>(bufs->codes_v);
    a.raw = static_cast<uint16_t *>(bufs->raw_v);
    a.lut = static_cast<uint16_t *>(bufs->lut_v);
    a.ol_col = static_cast<uint16_t *>(bufs->ol_col_v);
    a.ol_val = static_cast<uint16_t *>(bufs->ol_val_v);
    a.k_out = L.k_out_v;
    a.iters = cfg->v.lloyd_iters;
    if ((e = dq::launch_nuq_values(L, a, stream)) != 0)
        return fail(DQ_ECUDA, "value quantize launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    // keys: per-channel tables, thresholds and outlier bitmap (prefill), codes
    // (and, for an append, the bitmap by threshold), then the side channel
    a.x = k;
    a.is_key = 1;
    a.codes = static_cast<uint8_t *>(bufs->codes_k);
    a.raw = static_cast<uint16_t *>(bufs->raw_k);
    a.lut = static_cast<uint16_t *>(bufs->lut_k);
    a.olbits = c->nuq_bits;
    a.ol_rowptr = static_cast<int *>(bufs->ol_rowptr_k);
    a.ol_col = static_cast<uint16_t *>(bufs->ol_col_k);
    a.ol_val = static_cast<uint16_t *>(bufs->ol_val_k);
    a.thr = L.k_out_cap > 0 ? static_cast<float *>(bufs->meta_k) : nullptr;
    a.k_out = dq::nuq_outlier_count(cfg->k.outlier_frac, a.n_fit);
    a.iters = cfg->k.lloyd_iters;
    const long long N = L.refit;
    if (N > 0)  // the prefill's quantized slot count per unit follows the tables
        a.pq = reinterpret_cast<int *>(static_cast<uint8_t *>(bufs->lut_k) +
                                       static_cast<size_t>(L.U) * L.nbk * L.d * L.levels * 2);
    a.fit_t0 = L.n_sink;
    a.fit_slot0 = 0;
    a.fit_blk = 0;
    a.fit_nblk = N > 0 ? static_cast<int>((a.n_fit + N - 1) / N) : 1;  // every block the prefill reaches
    if (!append) {
        if (cudaMemsetAsync(c->nuq_bits, 0, static_cast<size_t>(L.U) * L.qcap * (L.d / 32) * sizeof(uint32_t), st) !=
            cudaSuccess)
            return fail(DQ_ECUDA, "clearing the key outlier bitmap failed");
        if (a.n_fit > 0 && (e = dq::launch_nuq_key_fit(L, a, stream)) != 0)
            return fail(DQ_ECUDA, "key fit launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    }
    // refit blocks that this append completes: [fb_lo, fb_hi); their keys are
    // gathered before this call's keys overwrite the recent window
    const long long s_lo = pos0 - L.n_sink, s_hi = s_lo + n_tok;
    const long long fb_lo = (append && N > 0) ? s_lo / N : 0, fb_hi = (append && N > 0) ? s_hi / N : 0;
    if (fb_hi > fb_lo) {
        a.scr_lo = fb_lo * N;
        a.scr_n = static_cast<int>((fb_hi - fb_lo) * N);
        const size_t need = static_cast<size_t>(L.U) * a.scr_n * L.d;
        if (c->nuq_scr_cap < need) {
            cudaFree(c->nuq_scr);
            c->nuq_scr = nullptr;
            c->nuq_scr_cap = 0;
            if (cudaMalloc(&c->nuq_scr, need * sizeof(float)) != cudaSuccess)
                return fail(DQ_ENOMEM, "key refit scratch (%zu bytes)", need * sizeof(float));
            c->nuq_scr_cap = need;
        }
        a.scr = c->nuq_scr;
        if ((e = dq::launch_nuq_gather(L, a, stream)) != 0)
            return fail(DQ_ECUDA, "key refit gather launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    }
    if ((e = dq::launch_nuq_key_codes(L, a, stream)) != 0)
        return fail(DQ_ECUDA, "key quantize launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    if (fb_hi > fb_lo) {
        for (long long b = fb_lo; b < fb_hi; b++) {  // per block: rank outliers, Lloyd fit, tables
            dq::QuantArgs f = a;
            f.x = a.scr;
            f.in_dtype = DQ_F32;
            f.n_tok = a.scr_n;
            f.fit_t0 = (b - fb_lo) * N;
            f.fit_slot0 = b * N;
            f.n_fit = static_cast<int>(N);
            f.k_out = dq::nuq_outlier_count(cfg->k.outlier_frac, static_cast<int>(N));
            f.fit_blk = static_cast<int>(b);
            f.fit_nblk = 1;
            f.fit_flush = 1;
            if ((e = dq::launch_nuq_key_fit(L, f, stream)) != 0)
                return fail(DQ_ECUDA, "key refit launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        }
        if ((e = dq::launch_nuq_block_codes(L, a, stream)) != 0)
            return fail(DQ_ECUDA, "key refit codes launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        // the side-channel kernel extends its rows back to the first recoded slot
    }
    if (L.k_out_cap > 0 && (e = dq::launch_nuq_key_csr(L, a, stream)) != 0)
        return fail(DQ_ECUDA, "key side-channel launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    return ok();
}

// Entropy-coded scheme ("D-Quant" page, Sec. 4.2).  A prefill from position 0
// encodes every slot after the sinks, its last window's key mean taken over the
// tokens it has.  An append keeps its tokens in the 16-bit recent window and
// flushes each 128-slot window that it completes: the window's key mean, the
// Drift fit and the rANS containers of all its slots, older tokens read from the
// recent window.  That needs the window's oldest token still there (n_recent of
// at least 128) and exact 16-bit copies (a 16-bit kv dtype).  The flush runs
// before this call's tokens are copied into the recent window.
static dq_status quantize_rans(dq_ctx *c, const dq_config *cfg, const Layout &L, const dq_kv_buffers *bufs,
                               const void *k, const void *v, long long pos0, long long n_tok, void *stream) {
    const long long S = pos0 + n_tok, ns = L.n_sink;
    long long slot0 = 0, n_fit = 0;
    if (pos0 == 0) {
        n_fit = n_tok > ns ? n_tok - ns : 0;
    } else {
        if (L.n_recent < 128)
            return fail(DQ_EUNSUPPORTED, "entropy-coded appends need n_recent >= 128 (has %d)", L.n_recent);
        if (cfg->kv_dtype == DQ_F32)
            return fail(DQ_EUNSUPPORTED, "entropy-coded appends need a 16-bit kv dtype");
        const long long s_lo = (pos0 > ns ? pos0 : ns) - ns, s_hi = S - ns - 1;  // this call's slots
        if (s_hi >= s_lo) {
            const long long wa = s_lo / 128, wb = s_hi >= 127 ? (s_hi - 127) / 128 : -1;
            if (wb >= wa) {
                slot0 = 128 * wa;
                n_fit = 128 * (wb - wa + 1);
            }
        }
    }
    dq::RansQuantArgs a{};
    a.in_dtype = cfg->kv_dtype;
    a.B = L.B;
    a.Hkv = L.Hkv;
    a.n = L.n_stream;
    a.n_tok = n_tok;
    a.n_sink = L.n_sink;
    a.n_recent = L.n_recent;
    a.pos0 = pos0;
    a.slot0 = slot0;
    a.n_fit = static_cast<int>(n_fit);
    a.hscale = static_cast<float>(1.0 / std::sqrt(128.0));
    a.n_win = (a.n_fit + 127) / 128;
    a.qcap = L.qcap;
    a.wcap = L.wcap;
    a.rcap = L.rcap;
    a.mean_rec = L.mean_rec;
    a.raw_bf16 = cfg->kv_dtype == DQ_BF16;
    a.status = c->status;
    // this call's tokens that stay 16-bit: sinks, and those among the latest n_recent
    const long long sink_end = S < ns ? S : ns;
    a.raw_ns = static_cast<int>(sink_end > pos0 ? sink_end - pos0 : 0);
    long long r0 = S - L.n_recent;
    if (r0 < pos0) r0 = pos0;
    if (r0 < ns) r0 = ns;
    a.raw_nr = static_cast<int>(S > r0 ? S - r0 : 0);
    const size_t need = static_cast<size_t>(L.B) * a.n_fit * L.n_stream;
    if (need > c->rans_sym_cap) {
        cudaFree(c->rans_sym);
        c->rans_sym = nullptr;
        c->rans_sym_cap = 0;
        if (cudaMalloc(&c->rans_sym, need) != cudaSuccess) {
            cudaGetLastError();
            return fail(DQ_ENOMEM, "symbol scratch of %zu bytes", need);
        }
        c->rans_sym_cap = need;
    }
    a.sym = c->rans_sym;
    int e;
    for (int which = 0; which < 2 && a.n_fit > 0; which++) {
        const dq_tensor_cfg &t = which == 0 ? cfg->k : cfg->v;
        a.x = which == 0 ? k : v;
        a.is_key = which == 0;
        a.rot = t.rot == DQ_ROT_HADAMARD;
        a.raw = static_cast<uint16_t *>(which == 0 ? bufs->raw_k : bufs->raw_v);
        a.codes = static_cast<uint8_t *>(which == 0 ? bufs->codes_k : bufs->codes_v);
        a.meta = which == 0 ? bufs->meta_k : bufs->meta_v;
        a.mean = which == 0 && t.mean ? static_cast<uint8_t *>(bufs->mean_k) : nullptr;
        a.drift_stats = c->drift_stats + 3 * which;
        const dq::RansTable *tb = which == 0 ? &c->rans->k : &c->rans->v;
        if (a.mean && (e = dq::launch_rans_mean(a, stream)) != 0)
            return fail(DQ_ECUDA, "window mean launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        if ((e = dq::launch_rans_drift(a, tb, c->rans->F, t.levels, stream)) != 0)
            return fail(DQ_ECUDA, "drift launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        if ((e = dq::launch_rans_encode(a, tb, t.container_bytes, stream)) != 0)
            return fail(DQ_ECUDA, "rANS encode launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    }
    for (int which = 0; which < 2 && a.raw_ns + a.raw_nr > 0; which++) {
        a.x = which == 0 ? k : v;
        a.is_key = which == 0;
        a.raw = static_cast<uint16_t *>(which == 0 ? bufs->raw_k : bufs->raw_v);
        if ((e = dq::launch_rans_raw(a, stream)) != 0)
            return fail(DQ_ECUDA, "raw copy launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    }
    return ok();
}

// Arguments of the affine quantizer for tokens [pos0, pos0 + n_tok) of the
// keys (which = 0) or values (which = 1); x is [B][Hkv][n_tok][d].
static void fill_quant_args(const dq_config *cfg, const Layout &L, const dq_kv_buffers *bufs, int which, const void *x,
                            long long pos0, long long n_tok, unsigned *status, dq::QuantArgs &a) {
    const dq_tensor_cfg &t = which == 0 ? cfg->k : cfg->v;
    a.x = x;
    a.in_dtype = cfg->kv_dtype;
    a.pos0 = pos0;
    a.n_tok = n_tok;
    a.seq_after = pos0 + n_tok;
    a.is_key = which == 0;
    a.bits = t.bits;
    a.rot = t.rot;
    a.use_mean = which == 0 && t.mean;
    a.meta_f16 = cfg->meta_dtype == DQ_F16;
    a.clip = t.clip;
    a.quest_c = t.grid == DQ_GRID_QUEST ? quest_step_factor(t.bits) : 0.0f;
    if (t.clip > 0.0f) {
        const double plo = (1.0 - static_cast<double>(t.clip)) * (L.d - 1);
        const double phi = static_cast<double>(t.clip) * (L.d - 1);
        a.clip_ilo = static_cast<int>(std::floor(plo));
        a.clip_flo = static_cast<float>(plo - std::floor(plo));
        a.clip_ihi = static_cast<int>(std::floor(phi));
        a.clip_fhi = static_cast<float>(phi - std::floor(phi));
    }
    a.hscale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(L.d)));
    a.codes = static_cast<uint8_t *>(which == 0 ? bufs->codes_k : bufs->codes_v);
    a.meta = which == 0 ? bufs->meta_k : bufs->meta_v;
    a.mean = which == 0 && t.mean ? static_cast<float *>(bufs->mean_k) : nullptr;
    a.T = which == 0 && t.rot == DQ_ROT_DENSE ? static_cast<const float *>(bufs->k_transform) : nullptr;
    a.raw = static_cast<uint16_t *>(which == 0 ? bufs->raw_k : bufs->raw_v);
    a.status = status;
    a.sz_x = static_cast<long long>(L.U) * n_tok * L.d * (cfg->kv_dtype == DQ_F32 ? 4 : 2);
    a.sz_codes = static_cast<long long>(L.sz[which == 0 ? 0 : 1]);
    a.sz_meta = static_cast<long long>(L.sz[which == 0 ? 2 : 3]);
    a.sz_mean = which == 0 ? static_cast<long long>(L.sz[4]) : 0;
    a.sz_raw = static_cast<long long>(L.sz[which == 0 ? 7 : 8]);
}

// Arguments of an affine or non-uniform decode-attention call (the dense key
// transform's compensated queries are computed here, on the stream).
static dq_status fill_attn_args(const dq_config *cfg, const Layout &L, const dq_kv_buffers *bufs, dq_ctx *c,
                                const void *q, void *out, long long seq_len, float sm_scale, void *stream,
                                dq::AttnArgs &a) {
    a.q = static_cast<const float *>(q);
    a.out = out;
    a.out_dtype = cfg->out_dtype;
    a.codes_k = static_cast<const uint8_t *>(bufs->codes_k);
    a.codes_v = static_cast<const uint8_t *>(bufs->codes_v);
    a.meta_k = bufs->meta_k;
    a.meta_v = bufs->meta_v;
    a.mean_k = cfg->k.mean ? static_cast<const float *>(bufs->mean_k) : nullptr;
    a.raw_k = static_cast<const uint16_t *>(bufs->raw_k);
    a.raw_v = static_cast<const uint16_t *>(bufs->raw_v);
    a.q_comp = cfg->k.rot == DQ_ROT_DENSE ? static_cast<const float *>(bufs->q_comp) : nullptr;
    if (cfg->k.rot == DQ_ROT_DENSE) {
        const int eq = dq::launch_qcomp(L, a.q, a.q_comp, c->q_tilde, stream);
        if (eq != 0) return fail(DQ_ECUDA, "query compensation launch: %s", cudaGetErrorString(static_cast<cudaError_t>(eq)));
        a.q_tilde = c->q_tilde;
    }
    a.rot_k = cfg->k.rot;
    a.rot_v = cfg->v.rot;
    a.raw_bf16 = cfg->kv_dtype == DQ_BF16;
    a.seq_len = seq_len;
    const long long n_s = seq_len < cfg->n_sink ? seq_len : cfg->n_sink;
    long long q_hi = seq_len - cfg->n_recent;
    if (q_hi < n_s) q_hi = n_s;
    a.n_q = q_hi - n_s;
    a.n_sink_eff = static_cast<int>(n_s);
    a.n_sink_cfg = cfg->n_sink;
    a.n_recent_cfg = cfg->n_recent;
    a.n_raw_slots = cfg->n_sink + cfg->n_recent;
    a.has_raw = a.n_raw_slots > 0 ? 1 : 0;
    a.sm_log2 = sm_scale * 1.4426950408889634f;
    a.hscale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(L.d)));
    a.partials = c->partials;
    a.counters = c->counters;
    a.status = c->status;
    dq::attn_extents(L, cfg->out_dtype, a);
    a.sz_partials = static_cast<long long>(c->partials_cap) * 4;
    a.sz_counters = static_cast<long long>(L.U) * 4;
    if (c->counters_dirty) {
        if (cudaMemsetAsync(c->counters, 0, sizeof(int) * L.U, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return fail(DQ_ECUDA, "clearing the record counts failed");
        c->counters_dirty = 0;
    }
    dq::set_nuq_args(L, bufs, a);
    return DQ_OK;
}

static dq_status launch_attn(const Layout &L, dq_ctx *c, dq::AttnArgs &a, void *stream) {
    int e = dq::plan_attention(L, a, c->num_sms, static_cast<long long>(c->partials_cap));
    if (e != 0) return fail(DQ_ECUDA, "attention planning: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    e = dq::launch_attention(L, a, c->num_sms, stream);
    if (e != 0) return fail(DQ_ECUDA, "attention launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    return ok();
}

extern "C" {

const char *dq_last_error(void) { return g_err; }

dq_status dq_rans_model(const dq_config *cfg, int which, int *levels, int f[16], int c[16]) {
    if (!cfg || !levels || !f || !c || (which != 0 && which != 1)) return fail(DQ_EINVAL, "bad argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (L.scheme != DQ_RANS) return fail(DQ_EINVAL, "not an entropy-coded config");
    dq::RansTable t;
    if (cached_table(L.n_stream, which == 0 ? L.mk : L.mv, cfg->rans_alpha, cfg->rans_prob_bits,
                     which == 0 ? L.ck : L.cv, &t) != 0)
        return fail(DQ_EINVAL, "no valid symbol model");
    *levels = t.M;
    for (int m = 0; m < 16; m++) {
        f[m] = m < t.M ? t.f[m] : 0;
        c[m] = m < t.M ? t.c[m] : 0;
    }
    return ok();
}

dq_status dq_symbol_probs(int n, int levels, double p[16]) {
    if (!p) return fail(DQ_EINVAL, "p is NULL");
    if (n < 1) return fail(DQ_EINVAL, "n must be positive (got %d)", n);
    if (levels < 2 || levels > dq::RANS_MAX_LEVELS)
        return fail(DQ_EINVAL, "levels must be in [2, %d] (got %d)", dq::RANS_MAX_LEVELS, levels);
    double q[dq::RANS_MAX_LEVELS];
    if (dq::rans_model_probs(n, levels, q) != 0) return fail(DQ_EINVAL, "no symbol model");
    for (int m = 0; m < 16; m++) p[m] = m < levels ? q[m] : 0.0;
    return ok();
}

dq_status dq_quest_step(int bits, float *c) {
    if (!c) return fail(DQ_EINVAL, "c is NULL");
    if (bits < 1 || bits > 8) return fail(DQ_EINVAL, "bits must be in [1, 8] (got %d)", bits);
    *c = quest_step_factor(bits);
    return ok();
}

const char *dq_status_name(dq_status s) {
    switch (s) {
        case DQ_OK: return "DQ_OK";
        case DQ_EINVAL: return "DQ_EINVAL";
        case DQ_EALIGN: return "DQ_EALIGN";
        case DQ_EUNSUPPORTED: return "DQ_EUNSUPPORTED";
        case DQ_EINFEASIBLE: return "DQ_EINFEASIBLE";
        case DQ_ENOMEM: return "DQ_ENOMEM";
        case DQ_ECUDA: return "DQ_ECUDA";
        case DQ_ENONFINITE: return "DQ_ENONFINITE";
        case DQ_ETIMEOUT: return "DQ_ETIMEOUT";
    }
    return "DQ_UNKNOWN";
}

dq_status dq_kv_sizes(const dq_config *cfg, size_t bytes[DQ_NUM_BUFFERS]) {
    if (!cfg || !bytes) return fail(DQ_EINVAL, "NULL argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    for (int i = 0; i < DQ_NUM_BUFFERS; i++) bytes[i] = L.sz[i];
    return ok();
}

dq_status dq_quantize_kv(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs, const void *k,
                         const void *v, long long pos0, long long n_tok, void *stream) {
    if (!cfg || !bufs || !k || !v) return fail(DQ_EINVAL, "NULL argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (pos0 < 0 || n_tok < 1 || pos0 + n_tok > cfg->max_seq)
        return fail(DQ_EINVAL, "tokens [%lld, %lld) outside [0, max_seq=%d)", pos0, pos0 + n_tok, cfg->max_seq);
    if ((s = check_bufs(L, bufs)) != DQ_OK) return s;
    if (!aligned16(k) || !aligned16(v)) return fail(DQ_EALIGN, "k / v input not 16-byte aligned");
    if ((s = get_ctx(ctx, cfg, L)) != DQ_OK) return s;
    if (L.scheme == DQ_NUQ) return quantize_nuq(*ctx, cfg, L, bufs, k, v, pos0, n_tok, stream);
    if (L.scheme == DQ_RANS) return quantize_rans(*ctx, cfg, L, bufs, k, v, pos0, n_tok, stream);

    for (int which = 0; which < 2; which++) {
        dq::QuantArgs a{};
        fill_quant_args(cfg, L, bufs, which, which == 0 ? k : v, pos0, n_tok, (*ctx)->status, a);
        int e;
        if (a.use_mean && pos0 == 0) {
            if ((e = dq::launch_key_mean(L, a, stream)) != 0)
                return fail(DQ_ECUDA, "key mean launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        }
        if ((e = dq::launch_quantize(L, a, stream)) != 0)
            return fail(DQ_ECUDA, "quantize launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    }
    return ok();
}

dq_status dq_decode_attention(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs, const void *q,
                              void *out, long long seq_len, float sm_scale, void *stream) {
    if (!cfg || !bufs || !q || !out) return fail(DQ_EINVAL, "NULL argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (seq_len < 1 || seq_len > cfg->max_seq) return fail(DQ_EINVAL, "seq_len %lld outside [1, max_seq]", seq_len);
    if (!std::isfinite(sm_scale)) return fail(DQ_EINVAL, "sm_scale is not finite");
    if ((s = check_bufs(L, bufs)) != DQ_OK) return s;
    if (!aligned16(q) || !aligned16(out)) return fail(DQ_EALIGN, "q / out not 16-byte aligned");
    if ((s = get_ctx(ctx, cfg, L)) != DQ_OK) return s;
    dq_ctx *c = *ctx;
    if (L.scheme == DQ_RANS) {
        dq::RansAttnArgs r{};
        r.q = static_cast<const float *>(q);
        r.out = out;
        r.out_dtype = cfg->out_dtype;
        r.codes_k = static_cast<const uint8_t *>(bufs->codes_k);
        r.codes_v = static_cast<const uint8_t *>(bufs->codes_v);
        r.meta_k = bufs->meta_k;
        r.meta_v = bufs->meta_v;
        r.mean = cfg->k.mean ? static_cast<const uint8_t *>(bufs->mean_k) : nullptr;
        r.raw_k = static_cast<const uint16_t *>(bufs->raw_k);
        r.raw_v = static_cast<const uint16_t *>(bufs->raw_v);
        r.B = L.B;
        r.Hkv = L.Hkv;
        r.ck = L.ck;
        r.cv = L.cv;
        r.qcap = L.qcap;
        r.wcap = L.wcap;
        r.mean_rec = L.mean_rec;
        r.rcap = L.rcap;
        const long long n_s = seq_len < cfg->n_sink ? seq_len : cfg->n_sink;
        long long q_hi = seq_len - cfg->n_recent;
        if (q_hi < n_s) q_hi = n_s;
        r.n_q = q_hi - n_s;
        r.n_sink_eff = static_cast<int>(n_s);
        r.n_sink_cfg = cfg->n_sink;
        r.n_recent_cfg = cfg->n_recent;
        r.recent_t0 = q_hi;
        r.n_raw = static_cast<int>(n_s + (seq_len - q_hi));
        r.rot_k = cfg->k.rot == DQ_ROT_HADAMARD;
        r.rot_v = cfg->v.rot == DQ_ROT_HADAMARD;
        r.raw_bf16 = cfg->kv_dtype == DQ_BF16;
        r.hscale = static_cast<float>(1.0 / std::sqrt(128.0));
        r.sm_log2 = sm_scale * 1.4426950408889634f;
        r.partials = c->rans_partials;
        r.status = c->status;
        const int e = dq::launch_attention_rans(r, c->rans, stream);
        if (e != 0) return fail(DQ_ECUDA, "attention launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
        return ok();
    }

    dq::AttnArgs a{};
    if ((s = fill_attn_args(cfg, L, bufs, c, q, out, seq_len, sm_scale, stream, a)) != DQ_OK) return s;
    return launch_attn(L, c, a, stream);
}

dq_status dq_decode_step(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs, const void *k_new,
                         const void *v_new, const void *q, void *out, long long seq_len, float sm_scale, void *stream) {
    if (!cfg || !bufs || !k_new || !v_new || !q || !out) return fail(DQ_EINVAL, "NULL argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (seq_len < 2 || seq_len > cfg->max_seq)
        return fail(DQ_EINVAL, "seq_len %lld outside [2, max_seq]: a step appends to a prefilled cache", seq_len);
    if (!std::isfinite(sm_scale)) return fail(DQ_EINVAL, "sm_scale is not finite");
    if ((s = check_bufs(L, bufs)) != DQ_OK) return s;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out))
        return fail(DQ_EALIGN, "k_new / v_new / q / out not 16-byte aligned");
    if ((s = get_ctx(ctx, cfg, L)) != DQ_OK) return s;
    dq_ctx *c = *ctx;
    // one launch when the affine kernel serves the call and the new token lies
    // in the recent window (so no packed slot this call reads is written by it)
    if (L.scheme == DQ_AFFINE && cfg->n_recent >= 1) {
        dq::AttnArgs a{};
        if ((s = fill_attn_args(cfg, L, bufs, c, q, out, seq_len, sm_scale, stream, a)) != DQ_OK) return s;
        if (dq::affine_kernel_applies(L, a)) {
            a.append = 1;
            for (int which = 0; which < 2; which++)
                fill_quant_args(cfg, L, bufs, which, which == 0 ? k_new : v_new, seq_len - 1, 1, c->status,
                                a.qa[which]);
            a.rg = dq::row_geom(L);
            return launch_attn(L, c, a, stream);
        }
    }
    if ((s = dq_quantize_kv(ctx, cfg, bufs, k_new, v_new, seq_len - 1, 1, stream)) != DQ_OK) return s;
    return dq_decode_attention(ctx, cfg, bufs, q, out, seq_len, sm_scale, stream);
}

dq_status dq_dequantize_kv(dq_ctx **ctx, const dq_config *cfg, const dq_kv_buffers *bufs, int which,
                           long long slot0, long long n, float *out, void *stream) {
    if (!cfg || !bufs || !out) return fail(DQ_EINVAL, "NULL argument");
    Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (which != 0 && which != 1) return fail(DQ_EINVAL, "which must be 0 (K) or 1 (V)");
    if (slot0 < 0 || n < 1 || slot0 + n > L.qcap) return fail(DQ_EINVAL, "slots outside the cache");
    if ((s = check_bufs(L, bufs)) != DQ_OK) return s;
    if (!aligned16(out)) return fail(DQ_EALIGN, "out not 16-byte aligned");
    if ((s = get_ctx(ctx, cfg, L)) != DQ_OK) return s;
    if (L.scheme == DQ_NUQ) return fail(DQ_EUNSUPPORTED, "non-uniform scheme: use the tables and side channel");
    if (L.scheme == DQ_RANS) return fail(DQ_EUNSUPPORTED, "entropy-coded scheme: decode the containers");
    dq::DequantArgs a{};
    a.codes = static_cast<const uint8_t *>(which == 0 ? bufs->codes_k : bufs->codes_v);
    a.meta = which == 0 ? bufs->meta_k : bufs->meta_v;
    a.mean = which == 0 && cfg->k.mean ? static_cast<const float *>(bufs->mean_k) : nullptr;
    a.is_key = which == 0;
    a.bits = which == 0 ? cfg->k.bits : cfg->v.bits;
    a.meta_f16 = cfg->meta_dtype == DQ_F16;
    a.slot0 = slot0;
    a.n = n;
    a.out = out;
    a.sz_codes = static_cast<long long>(L.sz[which == 0 ? 0 : 1]);
    a.sz_meta = static_cast<long long>(L.sz[which == 0 ? 2 : 3]);
    a.sz_mean = which == 0 ? static_cast<long long>(L.sz[4]) : 0;
    a.sz_out = static_cast<long long>(L.U) * n * L.d * 4;
    a.status = (*ctx)->status;
    const int e = dq::launch_dequant(L, a, stream);
    if (e != 0) return fail(DQ_ECUDA, "dequantize launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    return ok();
}

dq_status dq_check(dq_ctx *ctx, void *stream) {
    if (!ctx) return ok();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(DQ_ECUDA, "stream: %s", cudaGetErrorString(e));
    unsigned st = 0;
    if (cudaMemcpy(&st, ctx->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail(DQ_ECUDA, "status read failed");
    if (st && cudaMemset(ctx->status, 0, sizeof st) != cudaSuccess) return fail(DQ_ECUDA, "status clear failed");
    if (st & dq::ST_TIMEOUT) {
        // a wait that ran out may leave a unit's record count behind: the next
        // attention call starts from cleared counts
        ctx->counters_dirty = 1;
        return fail(DQ_ETIMEOUT, "a bounded device wait ran out");
    }
    if (st & dq::ST_OOB) return fail(DQ_EINVAL, "an access fell outside its buffer and was skipped (checked build)");
    if (st & dq::ST_INFEASIBLE) return fail(DQ_EINFEASIBLE, "a stream did not fit its container");
    if (st & dq::ST_SIDE_FULL)
        return fail(DQ_EINFEASIBLE, "the key outlier side channel is full: later decode-key outliers keep their level");
    if (st & dq::ST_BOUNDS) return fail(DQ_EINVAL, "a container asked for more bytes than it holds (corrupt cache)");
    if (st & dq::ST_NONFINITE) return fail(DQ_ENONFINITE, "non-finite K/V input");
    return ok();
}

dq_status dq_test_expire_wait(dq_ctx *ctx, unsigned long long limit_ns, void *stream) {
    if (!ctx || !ctx->status || !ctx->counters) return fail(DQ_EINVAL, "ctx has no workspace yet");
    if (limit_ns < 1000ULL) limit_ns = 1000ULL;
    if (limit_ns > 1000000000ULL) limit_ns = 1000000000ULL;
    const int e = dq::launch_expire_wait(ctx->status, ctx->counters, limit_ns, stream);
    if (e != 0) return fail(DQ_ECUDA, "expire-wait launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    return ok();
}

dq_status dq_drift_stats(dq_ctx *ctx, void *stream, unsigned long long out[6]) {
    if (!ctx || !out) return fail(DQ_EINVAL, "NULL argument");
    if (!ctx->drift_stats) return fail(DQ_EINVAL, "drift statistics belong to the entropy-coded scheme");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(DQ_ECUDA, "stream: %s", cudaGetErrorString(e));
    if (cudaMemcpy(out, ctx->drift_stats, 6 * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(ctx->drift_stats, 0, 6 * sizeof(unsigned long long)) != cudaSuccess)
        return fail(DQ_ECUDA, "drift statistics read failed");
    return ok();
}

dq_status dq_test_checked_probe(dq_ctx *ctx, void *stream) {
    if (!ctx || !ctx->status) return fail(DQ_EINVAL, "ctx has no workspace yet");
    const int e = dq::launch_checked_probe(ctx->status, stream);
    if (e != 0) return fail(DQ_ECUDA, "probe launch: %s", cudaGetErrorString(static_cast<cudaError_t>(e)));
    return ok();
}

void dq_free(dq_ctx *ctx) {
    if (!ctx) return;
    cudaFree(ctx->status);
    cudaFree(ctx->partials);
    cudaFree(ctx->counters);
    cudaFree(ctx->nuq_bits);
    cudaFree(ctx->nuq_scr);
    cudaFree(ctx->rans);
    cudaFree(ctx->drift_stats);
    cudaFree(ctx->rans_sym);
    cudaFree(ctx->rans_partials);
    cudaFree(ctx->q_tilde);
    delete ctx;
}

}  // extern "C"
