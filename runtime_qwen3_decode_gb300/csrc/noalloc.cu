// noalloc.cu - one decode step that needs no device allocation at all.
//
// Some callers cannot allocate device memory when they want to decode: code that
// runs inside another framework's memory pool or a fixed memory budget, or a host
// that must not call cudaMalloc after start-up (its allocations would
// synchronise the device or fail under a cap).  qw_decode_step_noalloc serves them: the
// caller passes the weights, the K/V cache, the input token and the output
// buffers, and every other buffer the decode kernel needs (the tagged exchange
// pages between phases, argmax keys and the arrival counter, the layer pointer table,
// this position's RoPE row, the SM-group tables and the probe scratch) lives in one
// file-scope device array of fixed size, kScratchBytes.  The kernel itself is the
// unchanged decode kernel of decode_kernel.cuh, with the same SM groups as a model
// created on the same device, so both give the same bits.
//
// The array is shared by every call in the process on a given device and keeps the
// last call's contents, so calls whose work overlaps on the GPU (different streams,
// or other threads) race on it and must be serialised by the caller.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "qw.h"
#include "qw_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// Regions of the array (byte offsets; the array itself is 256-aligned)
constexpr size_t kOffFlags = 0;                                   // StepFlags
constexpr size_t kOffStep = 256;                                  // argmax keys [2] + head arrival counter
constexpr size_t kOffRope = 512;                                  // float2 [head_dim / 2], this call's position
constexpr size_t kOffLayers = 1024;                               // DevLayer [n_layers]
constexpr size_t kOffRoles = kOffLayers + 64 * 160;               // uint16 [2][kMaxSmIds]
constexpr size_t kOffPlans = kOffRoles + 2 * qw::kMaxSmIds * 2;   // XPlan [2]
constexpr size_t kOffProbe = 65536;                               // probe scratch (4 KB aligned after rounding)
constexpr size_t kOffXRegion = kOffProbe + qw::kProbeScratchBytes + 4096;  // exchange pages (4 KB aligned)
static_assert(64 * 160 >= qw::kMaxLayers * sizeof(qw::DevLayer), "layer table space");
static_assert(kOffPlans + 2 * sizeof(qw::XPlan) <= kOffProbe, "plan space");
static_assert(kOffXRegion + qw::kXRegionBytes + 4096 <= kScratchBytes, "exchange pages fit the array");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_ptr[kMaxDevices];        // device address of g_scratch, per device (set-up done when non-null)
uint32_t g_seq[kMaxDevices];     // tag sequence of the last call on each device
qw::GroupPlans g_plans[kMaxDevices];

int cuda_rc(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return QW_OK;
    fprintf(stderr, "qw_decode_step_noalloc: %s failed: %s\n", what, cudaGetErrorString(e));
    return QW_CUDA_ERROR;
}

bool aligned16(const void *p) { return p && ((uintptr_t)p % 16) == 0; }

unsigned char *align4k(unsigned char *p) { return (unsigned char *)(((uintptr_t)p + 4095) & ~(uintptr_t)4095); }

}  // namespace

extern "C" int qw_decode_step_noalloc(const qw_config *cfg, const qw_weights *w, void *k_cache, void *v_cache,
                                      int32_t pos, int32_t token, float *logits_dev, int32_t *next_token_dev,
                                      void *cuda_stream, int32_t wait) {
    // configuration and arguments, checked before anything touches the device
    if (!cfg || !w || !w->layers || !k_cache || !v_cache || !logits_dev || !next_token_dev) return QW_INVALID_ARGUMENT;
    if (qw_workspace_bytes(cfg) == 0) return QW_UNSUPPORTED_SHAPE;  // same validation as qw_model_create
    if (token < 0 || token >= cfg->vocab) return QW_INVALID_ARGUMENT;
    if (pos < 0) return QW_INVALID_ARGUMENT;
    if (pos >= cfg->max_ctx) return QW_CONTEXT_EXCEEDED;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(logits_dev) || ((uintptr_t)next_token_dev % 4))
        return QW_ALIGNMENT;
    const bool i8 = cfg->weight_format != QW_W_BF16;
    if (!aligned16(w->embed) || !aligned16(w->final_norm) || (w->lm_head && !aligned16(w->lm_head)))
        return QW_ALIGNMENT;
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qw_layer_weights &lw = w->layers[l];
        const void *norms[4] = {lw.input_norm, lw.q_norm, lw.k_norm, lw.post_norm};
        for (const void *p : norms)
            if (!aligned16(p)) return p ? QW_ALIGNMENT : QW_INVALID_ARGUMENT;
        for (int i = 0; i < 7; ++i) {
            if (!lw.w[i] || (i8 && !lw.s[i])) return QW_INVALID_ARGUMENT;
            if (!aligned16(lw.w[i]) || (i8 && !aligned16(lw.s[i]))) return QW_ALIGNMENT;
        }
    }

    int dev = 0, major = 0, minor = 0, nsm = 0;
    int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= kMaxDevices) return QW_INVALID_ARGUMENT;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
        fprintf(stderr, "qw_decode_step_noalloc: device compute capability %d.%d; built for sm_103a only\n", major, minor);
        return QW_CUDA_ERROR;
    }
    if (cfg->n_layers * sizeof(qw::DevLayer) > kOffRoles - kOffLayers) {
        fprintf(stderr, "qw_decode_step_noalloc: %d layers do not fit the fixed array\n", cfg->n_layers);
        return QW_OUT_OF_MEMORY;
    }

    cudaStream_t stream = (cudaStream_t)cuda_stream;
    int bps = 0;
    rc = cuda_rc(qw::decode_prepare(&bps), "decode_prepare");  // shared-memory attribute of the kernel
    if (rc) return rc;
    if (bps < 1) return QW_CUDA_ERROR;
    unsigned char *base = nullptr;
    uint32_t seq = 0;
    const qw::GroupPlans *gp = nullptr;
    {
        std::lock_guard<std::mutex> g(g_mu);
        if (!g_ptr[dev]) {
            // Once per device, with that device current: find the array's device
            // address (in host code g_scratch is only a stand-in symbol, not an address
            // the GPU can use), zero the array, and measure which SMs and which of its
            // exchange pages sit on which die.  This first call on a device therefore
            // launches kernels and waits for them, and must come before any stream capture.
            void *p = nullptr;
            rc = cuda_rc(cudaGetSymbolAddress(&p, g_scratch), "cudaGetSymbolAddress");
            if (rc) return rc;
            unsigned char *b = (unsigned char *)p;
            rc = cuda_rc(cudaMemsetAsync(b, 0, kScratchBytes, stream), "cudaMemsetAsync");
            if (rc) return rc;
            qw::GroupPlans &pl = g_plans[dev];
            if (qw::plan_groups(dev, align4k(b + kOffProbe), align4k(b + kOffXRegion), cfg->hidden, cfg->n_heads,
                                cfg->n_kv_heads, cfg->intermediate, stream, &pl)) {
                fprintf(stderr, "qw_decode_step_noalloc: measuring the SM groups failed\n");
                return QW_CUDA_ERROR;
            }
            if (pl.ncta != nsm) return QW_CUDA_ERROR;
            rc = cuda_rc(cudaMemcpyAsync(b + kOffRoles, pl.role1, sizeof(pl.role1), cudaMemcpyHostToDevice, stream),
                         "cudaMemcpyAsync");
            if (!rc)
                rc = cuda_rc(cudaMemcpyAsync(b + kOffRoles + sizeof(pl.role1), pl.role2, sizeof(pl.role2),
                                             cudaMemcpyHostToDevice, stream), "cudaMemcpyAsync");
            if (!rc)
                rc = cuda_rc(cudaMemcpyAsync(b + kOffPlans, &pl.plan1, sizeof(qw::XPlan), cudaMemcpyHostToDevice,
                                             stream), "cudaMemcpyAsync");
            if (!rc)
                rc = cuda_rc(cudaMemcpyAsync(b + kOffPlans + sizeof(qw::XPlan), &pl.plan2, sizeof(qw::XPlan),
                                             cudaMemcpyHostToDevice, stream), "cudaMemcpyAsync");
            // the page probe wrote into the exchange pages: clear them (tag 0 is never live)
            if (!rc)
                rc = cuda_rc(cudaMemsetAsync(align4k(b + kOffXRegion), 0, qw::kXRegionBytes, stream), "cudaMemsetAsync");
            if (!rc) rc = cuda_rc(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
            if (rc) return rc;
            g_ptr[dev] = p;
            g_seq[dev] = 0;
        }
        base = (unsigned char *)g_ptr[dev];
        gp = &g_plans[dev];
        g_seq[dev] += 1;
        if (g_seq[dev] >= (1u << 23)) g_seq[dev] = 1;
        seq = g_seq[dev];
    }
    unsigned char *xregion = align4k(base + kOffXRegion);
    if (seq == 1) {
        // tags restart: clear the exchange pages so no stale word carries a live tag
        rc = cuda_rc(cudaMemsetAsync(xregion, 0, qw::kXRegionBytes, stream), "cudaMemsetAsync");
        if (rc) return rc;
    }

    // per call: the layer pointer table and this position's RoPE row (both copied from
    // host memory into the array), and zeroed flags, keys and the arrival counter
    std::vector<qw::DevLayer> layers((size_t)cfg->n_layers);
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qw_layer_weights &lw = w->layers[l];
        qw::DevLayer &d = layers[(size_t)l];
        d.input_norm = (const __nv_bfloat16 *)lw.input_norm;
        d.q_norm = (const __nv_bfloat16 *)lw.q_norm;
        d.k_norm = (const __nv_bfloat16 *)lw.k_norm;
        d.post_norm = (const __nv_bfloat16 *)lw.post_norm;
        for (int i = 0; i < 7; ++i) {
            d.w[i] = lw.w[i];
            d.s[i] = i8 ? (const __half *)lw.s[i] : nullptr;
        }
    }
    const int half = cfg->head_dim / 2;
    std::vector<float2> rope((size_t)half);
    for (int i = 0; i < half; ++i) {
        const double ang = (double)pos * std::pow(cfg->rope_theta, -2.0 * i / (double)cfg->head_dim);
        rope[(size_t)i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
    rc = cuda_rc(cudaMemcpyAsync(base + kOffLayers, layers.data(), layers.size() * sizeof(qw::DevLayer),
                                 cudaMemcpyHostToDevice, stream), "cudaMemcpyAsync");
    if (!rc)
        rc = cuda_rc(cudaMemcpyAsync(base + kOffRope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice,
                                     stream), "cudaMemcpyAsync");
    if (!rc) rc = cuda_rc(cudaMemsetAsync(base + kOffFlags, 0, kOffRope - kOffFlags, stream), "cudaMemsetAsync");
    if (rc) return rc;
    // the two host sources are locals of this call: wait until the copies have run
    rc = cuda_rc(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
    if (rc) return rc;

    qw::DecodeArgs a{};
    a.L = cfg->n_layers;
    a.H = cfg->hidden;
    a.Hq = cfg->n_heads;
    a.Hkv = cfg->n_kv_heads;
    a.I = cfg->intermediate;
    a.V = cfg->vocab;
    a.max_ctx = cfg->max_ctx;
    a.fmt = cfg->weight_format;
    a.eps = cfg->rms_eps;
    a.layers = (const qw::DevLayer *)(base + kOffLayers);
    a.embed = (const __nv_bfloat16 *)w->embed;
    a.lm_head = (const __nv_bfloat16 *)(w->lm_head ? w->lm_head : w->embed);
    a.final_norm = (const __nv_bfloat16 *)w->final_norm;
    a.kc = k_cache;
    a.vc = v_cache;
    a.kv_f32 = cfg->kv_format == QW_KV_F32 ? 1 : 0;
    a.rope = (const float2 *)(base + kOffRope);  // a one-row table holding this position's row
    a.rope_row = 0;
    const bool two = gp->D == 2;
    a.D = two ? 2 : 1;
    a.n_grp[0] = two ? gp->n[0] : gp->ncta;
    a.n_grp[1] = two ? gp->n[1] : 0;
    a.role = (const uint16_t *)(base + kOffRoles) + (two ? qw::kMaxSmIds : 0);
    a.xplan = (const qw::XPlan *)(base + kOffPlans) + (two ? 1 : 0);
    a.xr = (unsigned long long *)xregion;
    a.logits = logits_dev;
    a.hidden = nullptr;
    a.key = (unsigned long long *)(base + kOffStep);
    a.sync = (unsigned *)(base + kOffStep + 16);
    a.flags = (qw::StepFlags *)(base + kOffFlags);
    a.tok_out = next_token_dev;
    a.trace = nullptr;
    a.pos = pos;
    a.token = token;
    a.n_split = qw::attn_splits(pos, cfg->kv_format == QW_KV_F32 ? 4 : 2, a);
    a.debug = 0;
    a.wait_ns = qw::kWaitLimitNs;
    a.step = 1;  // keys and the counter were zeroed for this call
    a.target = (unsigned)gp->ncta;
    a.tag_base = seq * 512u;
    rc = cuda_rc(qw::launch_decode(a, gp->ncta, stream), "decode launch");
    if (rc || !wait) return rc;
    qw::StepFlags f;
    rc = cuda_rc(cudaMemcpyAsync(&f, base + kOffFlags, sizeof(f), cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync");
    if (!rc) rc = cuda_rc(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
    if (rc) return rc;
    return f.err ? (int)f.err : QW_OK;
}
