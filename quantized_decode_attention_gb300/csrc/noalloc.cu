// dq_decode_attention_noalloc: decode attention that allocates nothing.
//
// Some callers cannot let a library call cudaMalloc: serving engines that
// carve all device memory out of one pre-reserved pool (an allocation behind
// their back breaks their accounting and can fail under memory pressure at an
// arbitrary point), real-time decode loops where cudaMalloc/cudaFree would
// synchronize the device and stall other streams, and embedders with a fixed
// device-memory budget.  The context-based entry point allocates its split
// workspace on first use; this one uses a fixed, statically sized device array
// instead.  The caller still passes the cache buffers, q and out.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "dq.h"
#include "dq_internal.h"

namespace {

constexpr size_t kScratchBytes = DQ_NOALLOC_SCRATCH_BYTES;
constexpr size_t kMaxUnits = 16384;                          // batch * n_kv_heads
constexpr size_t kCountersBytes = kMaxUnits * sizeof(int);   // 64 KiB of split tickets
constexpr size_t kStatusOffset = kCountersBytes;             // one status word
constexpr size_t kPartialsOffset = kCountersBytes + 256;     // split partials after it
constexpr size_t kPartialsBytes = kScratchBytes - kPartialsOffset;

// The scratch itself.  Every GPU that loads this library holds it until the
// process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_addr[kMaxDevices];  // device address of g_scratch, per device
int g_sms[kMaxDevices];

// Host code must not pass g_scratch itself to a kernel: on the host that name
// is a stand-in, not a device address.  Look the address up once per device,
// with that device current.
dq_status scratch_for_device(int dev, unsigned char **addr, int *sms) {
    if (dev < 0 || dev >= kMaxDevices) return dq::set_last_error(DQ_EUNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) {
            char msg[256];
            std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            return dq::set_last_error(DQ_ECUDA, msg);
        }
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return dq::set_last_error(DQ_ECUDA, "cannot query the SM count");
        g_addr[dev] = static_cast<unsigned char *>(p);
        g_sms[dev] = n;
    }
    *addr = g_addr[dev];
    *sms = g_sms[dev];
    return DQ_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dq_status dq_decode_attention_noalloc(const dq_config *cfg, const dq_kv_buffers *bufs, const void *q,
                                                 void *out, long long seq_len, float sm_scale, void *stream) {
    if (!cfg || !bufs || !q || !out) return dq::set_last_error(DQ_EINVAL, "NULL argument");
    dq::Layout L;
    dq_status s = dq::make_layout(cfg, &L);
    if (s != DQ_OK) return s;
    if (L.scheme == DQ_RANS)
        return dq::set_last_error(DQ_EUNSUPPORTED, "entropy-coded caches decode with the symbol model of a context");
    if (seq_len < 1 || seq_len > cfg->max_seq) return dq::set_last_error(DQ_EINVAL, "seq_len outside [1, max_seq]");
    if (!std::isfinite(sm_scale)) return dq::set_last_error(DQ_EINVAL, "sm_scale is not finite");
    const void *const *p = reinterpret_cast<const void *const *>(bufs);
    for (int i = 0; i < DQ_NUM_BUFFERS; i++) {
        if (L.sz[i] == 0) continue;
        if (!p[i]) return dq::set_last_error(DQ_EINVAL, "a cache buffer the config needs is NULL");
        if (!aligned16(p[i])) return dq::set_last_error(DQ_EALIGN, "a cache buffer is not 16-byte aligned");
    }
    if (!aligned16(q) || !aligned16(out)) return dq::set_last_error(DQ_EALIGN, "q / out not 16-byte aligned");
    if (static_cast<size_t>(L.U) > kMaxUnits) {
        char msg[200];
        std::snprintf(msg, sizeof msg, "batch * n_kv_heads = %d exceeds the allocation-free limit of %zu", L.U,
                      kMaxUnits);
        return dq::set_last_error(DQ_EINVAL, msg);
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return dq::set_last_error(DQ_ECUDA, "cannot query the current device");
    unsigned char *scratch = nullptr;
    int num_sms = 0;
    if ((s = scratch_for_device(dev, &scratch, &num_sms)) != DQ_OK) return s;

    dq::AttnArgs a{};
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
    a.counters = reinterpret_cast<int *>(scratch);
    a.status = reinterpret_cast<unsigned *>(scratch + kStatusOffset);
    dq::attn_extents(L, cfg->out_dtype, a);
    a.sz_partials = static_cast<long long>(kPartialsBytes);
    a.sz_counters = static_cast<long long>(kCountersBytes);
    dq::set_nuq_args(L, bufs, a);
    a.partials = reinterpret_cast<float *>(scratch + kPartialsOffset);
    // the partials must fit the static scratch: the plan narrows the grid
    // until they do, and refuses the config if even one CTA's would not
    const long long cap = static_cast<long long>(kPartialsBytes / sizeof(float));
    int pe = dq::plan_attention(L, a, num_sms, cap);
    if (pe == static_cast<int>(cudaErrorMemoryAllocation)) {
        char msg[200];
        std::snprintf(msg, sizeof msg,
                      "split partials need %lld bytes; the allocation-free scratch holds %zu (limit %zu bytes total)",
                      dq::attention_partial_floats(L, a) * 4, kPartialsBytes, kScratchBytes);
        return dq::set_last_error(DQ_EINVAL, msg);
    }
    if (pe != 0) return dq::set_last_error(DQ_ECUDA, cudaGetErrorString(static_cast<cudaError_t>(pe)));

    // the tickets must start at zero; an earlier call leaves them at zero, but
    // clear them anyway so that one aborted call cannot poison the next
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, kPartialsOffset, st) != cudaSuccess)
        return dq::set_last_error(DQ_ECUDA, "clearing the scratch tickets failed");
    const int e = dq::launch_attention(L, a, num_sms, stream);
    if (e != 0) return dq::set_last_error(DQ_ECUDA, cudaGetErrorString(static_cast<cudaError_t>(e)));
    return dq::set_last_error(DQ_OK, "");
}
