// qw_api.cu - host side of the C ABI declared in include/qw.h.
//
// Everything here is validation, workspace carving and launch bookkeeping; all
// arithmetic of the decoder runs in the device kernels (decode.cu, prefill.cu).
// Conventions ("Portable WebAssembly Runtime Architecture for TinyRustLM",
// section "Typed host/Wasm API"): status codes, handles checked against a table
// of live models on every call, no exceptions across the boundary.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "qw.h"
#include "qw_internal.h"
#include "qw_batch.h"
#include "qw_prefill.h"
#include "qw_sample.h"

static_assert(qw::kDebugWithhold == QW_DEBUG_WITHHOLD, "debug flag value shared with the kernel");

namespace {

constexpr int kMaxCtas = 1024;  // upper bound on SMs, for the split-attention partials
constexpr size_t kAlign = 256;
constexpr int kPrefillRowsMax = 2048;

struct Layout {
    size_t kc, vc, rope, layers, logits, hidden, step, flags, trace;
    size_t role, xplan1, xplan2, probe, xregion;  // SM roles, exchange plans, probe scratch, exchange pages
    size_t prefill, prefill_bytes;
    size_t sampler, sampler_bytes;  // PCG32 state (16 B) + sampling scratch
    size_t total;
};

bool mul_ok(size_t a, size_t b, size_t *out) {
    if (a != 0 && b > SIZE_MAX / a) return false;
    *out = a * b;
    return true;
}

int validate_config(const qw_config *c) {
    if (!c) return QW_INVALID_ARGUMENT;
    if (c->weight_format != QW_W_BF16 && c->weight_format != QW_W_INT8_G32 && c->weight_format != QW_W_Q8Q8)
        return QW_UNSUPPORTED_QUANTIZATION;
    if (c->kv_format != QW_KV_F32 && c->kv_format != QW_KV_BF16) return QW_INVALID_ARGUMENT;
    if (c->n_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
        c->intermediate < 1 || c->vocab < 1 || c->max_ctx < 1)
        return QW_INVALID_ARGUMENT;
    if (!(c->rms_eps > 0.0f) || !std::isfinite(c->rms_eps) || !(c->rope_theta > 0.0) || !std::isfinite(c->rope_theta))
        return QW_INVALID_ARGUMENT;
    // Q8 blocks are 32 wide and tail groups are not allowed ("Scalar-Native ...", section 3).
    if (c->hidden % 32 || c->intermediate % 32 || (c->n_heads * c->head_dim) % 32) return QW_UNSUPPORTED_QUANTIZATION;
    if (c->head_dim != qw::kHeadDim) return QW_UNSUPPORTED_SHAPE;
    if (c->n_heads % c->n_kv_heads) return QW_UNSUPPORTED_SHAPE;
    const int qd = c->n_heads * c->head_dim;
    for (int k : {c->hidden, qd, c->intermediate})
        if (k % 1024 || k > 3072) return QW_UNSUPPORTED_SHAPE;
    // the decode kernel is built for the Qwen3-0.6B block dims
    if (!qw::block_shape_ok(c->hidden, c->n_heads, c->n_kv_heads, c->intermediate)) return QW_UNSUPPORTED_SHAPE;
    if (c->n_layers > qw::kMaxLayers || c->max_ctx > 131072 || c->vocab > (1 << 24)) return QW_UNSUPPORTED_SHAPE;
    return QW_OK;
}

int make_layout(const qw_config *c, Layout *L) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off += (bytes + kAlign - 1) / kAlign * kAlign;
        return at;
    };
    size_t kv;
    const size_t esz = c->kv_format == QW_KV_F32 ? 4 : 2;
    if (!mul_ok((size_t)c->n_layers * c->n_kv_heads, (size_t)c->max_ctx * c->head_dim * esz, &kv))
        return QW_INTEGER_OVERFLOW;
    L->kc = take(kv);
    L->vc = take(kv);
    L->rope = take((size_t)c->max_ctx * (c->head_dim / 2) * sizeof(float2));
    L->layers = take((size_t)c->n_layers * sizeof(qw::DevLayer));
    L->logits = take((size_t)c->vocab * 4);
    L->hidden = take((size_t)(c->n_layers + 1) * c->hidden * 4);
    L->step = take(qw::kStepBlockBytes);
    L->flags = take(sizeof(qw::StepFlags));
    L->trace = take(((size_t)qw::kPhasesPerLayer * c->n_layers + 1) * kMaxCtas * qw::kTraceStamps * 8);
    L->role = take(2 * (size_t)qw::kMaxSmIds * sizeof(uint16_t));  // one table per layout
    L->xplan1 = take(sizeof(qw::XPlan));
    L->xplan2 = take(sizeof(qw::XPlan));
    // the probe scratch and the exchange pages start on a 4 KB boundary of the device address;
    // the workspace base is only 256-aligned, so each keeps 4 KB of slack
    L->probe = take(qw::kProbeScratchBytes + 4096);
    L->xregion = take(qw::kXRegionBytes + 4096);
    const int rows = c->max_ctx < kPrefillRowsMax ? c->max_ctx : kPrefillRowsMax;
    L->prefill_bytes = qw::prefill_workspace_bytes(*c, rows);
    L->prefill = take(L->prefill_bytes);
    L->sampler_bytes = 256 + qw::sample_scratch_bytes(c->vocab);
    L->sampler = take(L->sampler_bytes);
    L->total = off;
    return QW_OK;
}

std::mutex g_live_mu;
std::unordered_set<const void *> g_live;

}  // namespace

struct qw_model {
    qw_config cfg;
    int ncta = 0, nsm = 0, device = 0;
    int groups = 1;                       // SM groups of the decode step (2 = one per die)
    int n_grp[qw::kMaxGroups] = {0, 0};
    qw::XPlan *xplan_dev[2] = {nullptr, nullptr};  // exchange plans for one group and for two
    cudaStream_t stream = nullptr;
    uint8_t *ws = nullptr;
    Layout lay{};
    qw::DecodeArgs args{};
    qw::StepFlags *flags = nullptr;
    void *step_block = nullptr;
    size_t step_bytes = 0;
    qw::PrefillState pf{};
    int32_t len = 0;
    int has_last = 0;
    int debug = 0;
    int failed = 0;  // device error seen; cleared by qw_kv_reset
    uint32_t step_seq = 0;  // decode steps launched so far (tags of step n use n * 512 + phase + 1)
    uint32_t csteps = 0;    // steps since the arrival counters were last zeroed
    float *logits = nullptr;
    float *hidden = nullptr;
    const uint16_t *role_dev[2] = {nullptr, nullptr};  // role tables (by %smid) for one group and for two
    float rt_near = 0.f, rt_far = 0.f;                 // measured same-die / cross-die round trips (ns)
};

namespace {

bool live(const qw_model *m) {
    std::lock_guard<std::mutex> g(g_live_mu);
    return m && g_live.count(m);
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return QW_OK;
    fprintf(stderr, "qw: CUDA error %d (%s)\n", (int)e, cudaGetErrorString(e));
    return QW_CUDA_ERROR;
}

bool aligned(const void *p, size_t a) { return p && ((uintptr_t)p % a) == 0; }

// The decode arguments for the grouping in use (one group when QW_DEBUG_ONE_GROUP is set).
void set_groups(const qw_model *m, qw::DecodeArgs &a) {
    const bool two = m->groups == 2 && !(m->debug & QW_DEBUG_ONE_GROUP);
    a.D = two ? 2 : 1;
    a.n_grp[0] = two ? m->n_grp[0] : m->ncta;
    a.n_grp[1] = two ? m->n_grp[1] : 0;
    a.xplan = m->xplan_dev[two ? 1 : 0];
    a.role = m->role_dev[two ? 1 : 0];
}

// One decode step at position len; token >= 0 or -1 (device-resident previous pick).
int launch_step(qw_model *m, int32_t token, int32_t *tok_out_dev) {
    qw::DecodeArgs a = m->args;
    a.pos = m->len;
    a.token = token;
    set_groups(m, a);
    a.rope_row = m->len;
    a.n_split = qw::attn_splits(m->len, m->cfg.kv_format == QW_KV_F32 ? 4 : 2, a);
    a.debug = m->debug;
    a.wait_ns = (m->debug & QW_DEBUG_WITHHOLD) ? qw::kDebugWaitLimitNs : qw::kWaitLimitNs;
    a.tok_out = tok_out_dev;
    a.trace = nullptr;
    if (m->debug & QW_DEBUG_TRACE) {  // a fresh timeline per step: stamps a phase does not set stay 0
        a.trace = (unsigned long long *)(m->ws + m->lay.trace);
        const size_t n = ((size_t)qw::kPhasesPerLayer * m->cfg.n_layers + 1) * m->ncta * qw::kTraceStamps * 8;
        const int zr = cuda_status(cudaMemsetAsync(a.trace, 0, n, m->stream));
        if (zr) return zr;
    }
    m->step_seq += 1;
    if (m->step_seq >= (1u << 23)) {  // tag_base stays below 2^32: restart the tags on a clean region
        m->step_seq = 1;
        const int zr = cuda_status(cudaMemsetAsync(m->args.xr, 0, qw::kXRegionBytes, m->stream));
        if (zr) return zr;
    }
    a.step = m->step_seq;
    a.tag_base = m->step_seq * 512u;
    int rc = QW_OK;
    if ((uint64_t)(m->csteps + 1) * (uint64_t)m->ncta >= 0xffffffffull) {  // counters would overflow
        rc = cuda_status(cudaMemsetAsync(m->step_block, 0, m->step_bytes, m->stream));
        if (rc) return rc;
        m->csteps = 0;
    }
    m->csteps += 1;
    a.target = m->csteps * (uint32_t)m->ncta;
    rc = cuda_status(qw::launch_decode(a, m->ncta, m->stream));
    if (rc) return rc;
    m->len += 1;
    m->has_last = 1;
    return QW_OK;
}

// Wait for the stream, read the flags; returns the device error (if any) and the last pick.
int read_flags(qw_model *m, int32_t *tok) {
    qw::StepFlags f;
    int rc = cuda_status(cudaMemcpyAsync(&f, m->flags, sizeof(f), cudaMemcpyDeviceToHost, m->stream));
    if (rc) return rc;
    rc = cuda_status(cudaStreamSynchronize(m->stream));
    if (rc) return rc;
    if (f.err) {
        if (f.err == QW_INTERNAL_INVARIANT && f.diag)
            fprintf(stderr, "qw: a device wait expired (site %u, CTA %u, phase %u)\n", f.diag >> 24,
                    (f.diag >> 12) & 0xfffu, f.diag & 0xfffu);
        m->failed = (int)f.err;
        return (int)f.err;
    }
    if (tok) *tok = f.next_tok;
    return QW_OK;
}

}  // namespace

extern "C" {

int32_t qw_abi_version(void) { return QW_ABI_VERSION; }

const char *qw_status_string(int s) {
    switch (s) {
        case QW_OK: return "ok";
        case QW_INVALID_ARGUMENT: return "invalid argument";
        case QW_INVALID_HANDLE: return "invalid handle";
        case QW_ALIGNMENT: return "pointer misaligned";
        case QW_INTEGER_OVERFLOW: return "size overflow";
        case QW_OUT_OF_MEMORY: return "workspace too small";
        case QW_UNSUPPORTED_QUANTIZATION: return "unsupported quantization (format or a dimension not a multiple of 32)";
        case QW_UNSUPPORTED_SHAPE: return "unsupported shape";
        case QW_CONTEXT_EXCEEDED: return "context exceeded";
        case QW_NUMERICAL_FAILURE: return "non-finite logits";
        case QW_INTERNAL_INVARIANT: return "device wait expired (internal invariant)";
        case QW_CUDA_ERROR: return "CUDA error";
        default: return "unknown status";
    }
}

size_t qw_workspace_bytes(const qw_config *cfg) {
    if (validate_config(cfg) != QW_OK) return 0;
    Layout L;
    if (make_layout(cfg, &L) != QW_OK) return 0;
    return L.total;
}

int qw_model_create(const qw_config *cfg, const qw_weights *w, void *workspace, size_t workspace_bytes,
                    void *cuda_stream, qw_model **out) {
    if (!out) return QW_INVALID_ARGUMENT;
    *out = nullptr;
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!w || !w->layers || !workspace) return QW_INVALID_ARGUMENT;
    Layout L;
    rc = make_layout(cfg, &L);
    if (rc) return rc;
    if (!aligned(workspace, kAlign)) return QW_ALIGNMENT;
    if (workspace_bytes < L.total) return QW_OUT_OF_MEMORY;
    if (!aligned(w->embed, 16) || !aligned(w->final_norm, 16) || (w->lm_head && !aligned(w->lm_head, 16)))
        return w->embed && w->final_norm ? QW_ALIGNMENT : QW_INVALID_ARGUMENT;
    const bool i8 = cfg->weight_format != QW_W_BF16;
    std::vector<qw::DevLayer> host_layers((size_t)cfg->n_layers);
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qw_layer_weights &lw = w->layers[l];
        const void *norms[4] = {lw.input_norm, lw.q_norm, lw.k_norm, lw.post_norm};
        for (const void *p : norms) {
            if (!p) return QW_INVALID_ARGUMENT;
            if (!aligned(p, 16)) return QW_ALIGNMENT;
        }
        for (int i = 0; i < 7; ++i) {
            if (!lw.w[i] || (i8 && !lw.s[i])) return QW_INVALID_ARGUMENT;
            if (!aligned(lw.w[i], 16) || (i8 && !aligned(lw.s[i], 16))) return QW_ALIGNMENT;
        }
        qw::DevLayer &d = host_layers[(size_t)l];
        d.input_norm = (const __nv_bfloat16 *)lw.input_norm;
        d.q_norm = (const __nv_bfloat16 *)lw.q_norm;
        d.k_norm = (const __nv_bfloat16 *)lw.k_norm;
        d.post_norm = (const __nv_bfloat16 *)lw.post_norm;
        for (int i = 0; i < 7; ++i) {
            d.w[i] = lw.w[i];
            d.s[i] = i8 ? (const __half *)lw.s[i] : nullptr;
        }
    }

    int dev = 0;
    rc = cuda_status(cudaGetDevice(&dev));
    if (rc) return rc;
    int major = 0, minor = 0, nsm = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
        fprintf(stderr, "qw: device compute capability %d.%d; this library is built for sm_103a only\n", major, minor);
        return QW_CUDA_ERROR;
    }
    int bps = 0;
    rc = cuda_status(qw::decode_prepare(&bps));
    if (rc) return rc;
    if (bps < 1) {
        fprintf(stderr, "qw: decode kernel does not fit on an SM\n");
        return QW_CUDA_ERROR;
    }
    if (nsm > kMaxCtas) return QW_UNSUPPORTED_SHAPE;
    rc = cuda_status(qw::prefill_prepare());
    if (rc) return rc;

    qw_model *m = new (std::nothrow) qw_model();
    if (!m) return QW_OUT_OF_MEMORY;
    m->cfg = *cfg;
    m->nsm = nsm;
    m->device = dev;
    m->stream = (cudaStream_t)cuda_stream;
    m->ws = (uint8_t *)workspace;
    m->lay = L;
    uint8_t *ws = m->ws;
    auto align4k = [](uint8_t *p) { return (uint8_t *)(((uintptr_t)p + 4095) & ~(uintptr_t)4095); };
    uint8_t *probe = align4k(ws + L.probe), *xregion = align4k(ws + L.xregion);

    // SM groups: which SMs and exchange pages sit on which die (measured once per device for the
    // SMs, once per model for the pages); both layouts are kept, the two-group one is the default
    qw::GroupPlans *gp = new (std::nothrow) qw::GroupPlans();
    if (!gp) {
        delete m;
        return QW_OUT_OF_MEMORY;
    }
    if (qw::plan_groups(dev, probe, xregion, cfg->hidden, cfg->n_heads, cfg->n_kv_heads, cfg->intermediate,
                        m->stream, gp)) {
        fprintf(stderr, "qw: measuring the SM groups failed\n");
        delete gp;
        delete m;
        return QW_CUDA_ERROR;
    }
    m->ncta = gp->ncta;
    m->groups = gp->D;
    m->n_grp[0] = gp->n[0];
    m->n_grp[1] = gp->n[1];
    m->rt_near = gp->rt_near;
    m->rt_far = gp->rt_far;

    // RoPE table: cos/sin of pos * theta^(-2i/d), i < d/2, in double, rounded to f32.
    const int half = cfg->head_dim / 2;
    std::vector<float2> rope((size_t)cfg->max_ctx * half);
    for (int i = 0; i < half; ++i) {
        const double inv_freq = std::pow(cfg->rope_theta, -2.0 * i / (double)cfg->head_dim);
        for (int p = 0; p < cfg->max_ctx; ++p) {
            const double ang = (double)p * inv_freq;
            rope[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    }
    uint16_t *role_dev = (uint16_t *)(ws + L.role);
    rc = cuda_status(cudaMemcpyAsync(ws + L.rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice,
                                     m->stream));
    if (!rc)
        rc = cuda_status(cudaMemcpyAsync(ws + L.layers, host_layers.data(), host_layers.size() * sizeof(qw::DevLayer),
                                         cudaMemcpyHostToDevice, m->stream));
    if (!rc)
        rc = cuda_status(cudaMemcpyAsync(role_dev, gp->role1, sizeof(gp->role1), cudaMemcpyHostToDevice, m->stream));
    if (!rc)
        rc = cuda_status(cudaMemcpyAsync(role_dev + qw::kMaxSmIds, gp->role2, sizeof(gp->role2),
                                         cudaMemcpyHostToDevice, m->stream));
    if (!rc)
        rc = cuda_status(cudaMemcpyAsync(ws + L.xplan1, &gp->plan1, sizeof(qw::XPlan), cudaMemcpyHostToDevice, m->stream));
    if (!rc)
        rc = cuda_status(cudaMemcpyAsync(ws + L.xplan2, &gp->plan2, sizeof(qw::XPlan), cudaMemcpyHostToDevice, m->stream));
    if (!rc) rc = cuda_status(cudaMemsetAsync(ws + L.flags, 0, sizeof(qw::StepFlags), m->stream));
    if (!rc) rc = cuda_status(cudaMemsetAsync(ws + L.sampler, 0, 256, m->stream));
    if (!rc) rc = cuda_status(cudaMemsetAsync(ws + L.step, 0, qw::kStepBlockBytes, m->stream));
    // tagged exchange words start with tag 0, which no step ever uses
    if (!rc) rc = cuda_status(cudaMemsetAsync(xregion, 0, qw::kXRegionBytes, m->stream));
    if (!rc) rc = cuda_status(cudaStreamSynchronize(m->stream));  // host staging buffers go out of scope
    delete gp;
    if (rc) {
        delete m;
        return rc;
    }

    qw::DecodeArgs &a = m->args;
    a.L = cfg->n_layers;
    a.H = cfg->hidden;
    a.Hq = cfg->n_heads;
    a.Hkv = cfg->n_kv_heads;
    a.I = cfg->intermediate;
    a.V = cfg->vocab;
    a.max_ctx = cfg->max_ctx;
    a.fmt = cfg->weight_format;
    a.eps = cfg->rms_eps;
    a.layers = (const qw::DevLayer *)(ws + L.layers);
    a.embed = (const __nv_bfloat16 *)w->embed;
    a.lm_head = (const __nv_bfloat16 *)(w->lm_head ? w->lm_head : w->embed);
    a.final_norm = (const __nv_bfloat16 *)w->final_norm;
    a.kc = ws + L.kc;
    a.vc = ws + L.vc;
    a.kv_f32 = cfg->kv_format == QW_KV_F32 ? 1 : 0;
    a.rope = (const float2 *)(ws + L.rope);
    a.xr = (unsigned long long *)xregion;
    a.logits = (float *)(ws + L.logits);
    a.hidden = (float *)(ws + L.hidden);
    a.key = (unsigned long long *)(ws + L.step);
    a.sync = (unsigned *)(ws + L.step + 16);
    a.flags = (qw::StepFlags *)(ws + L.flags);
    m->role_dev[0] = role_dev;
    m->role_dev[1] = role_dev + qw::kMaxSmIds;
    m->xplan_dev[0] = (qw::XPlan *)(ws + L.xplan1);
    m->xplan_dev[1] = (qw::XPlan *)(ws + L.xplan2);
    m->flags = a.flags;
    m->step_block = ws + L.step;
    m->step_bytes = qw::kStepBlockBytes;
    m->logits = a.logits;
    m->hidden = a.hidden;
    if (qw::prefill_init(&m->pf, *cfg, host_layers.data(), a.rope, ws + L.prefill, L.prefill_bytes,
                         cfg->max_ctx < kPrefillRowsMax ? cfg->max_ctx : kPrefillRowsMax, nsm, m->stream)) {
        fprintf(stderr, "qw: preparing the batched prefill failed\n");
        qw::prefill_destroy(&m->pf);
        delete m;
        return QW_CUDA_ERROR;
    }
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        g_live.insert(m);
    }
    *out = m;
    return QW_OK;
}

void qw_model_destroy(qw_model *m) {
    if (!m) return;
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        if (!g_live.erase(m)) return;
    }
    cudaStreamSynchronize(m->stream);
    qw::prefill_destroy(&m->pf);
    delete m;
}

int qw_decode_step(qw_model *m, int32_t token, int32_t *next_token_host) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (m->failed) return m->failed;
    if (token < -1 || token >= m->cfg.vocab) return QW_INVALID_ARGUMENT;
    if (token == -1 && !m->has_last) return QW_INVALID_ARGUMENT;
    if (m->len + 1 > m->cfg.max_ctx) return QW_CONTEXT_EXCEEDED;
    int rc = launch_step(m, token, nullptr);
    if (rc) return rc;
    if (next_token_host) return read_flags(m, next_token_host);
    return QW_OK;
}

int qw_generate(qw_model *m, int32_t token, int32_t n, int32_t *tokens_dev) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (m->failed) return m->failed;
    if (n < 0 || token < -1 || token >= m->cfg.vocab) return QW_INVALID_ARGUMENT;
    if (n == 0) return QW_OK;
    if (token == -1 && !m->has_last) return QW_INVALID_ARGUMENT;
    if ((int64_t)m->len + n > m->cfg.max_ctx) return QW_CONTEXT_EXCEEDED;
    for (int32_t i = 0; i < n; ++i) {
        int rc = launch_step(m, i == 0 ? token : -1, tokens_dev ? tokens_dev + i : nullptr);
        if (rc) return rc;
    }
    return QW_OK;
}

int qw_prefill(qw_model *m, const int32_t *tokens_host, int32_t n, int32_t *next_token_host) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (m->failed) return m->failed;
    if (n < 0 || (n > 0 && !tokens_host)) return QW_INVALID_ARGUMENT;
    if (n == 0) return QW_OK;
    if ((int64_t)m->len + n > m->cfg.max_ctx) return QW_CONTEXT_EXCEEDED;
    for (int32_t i = 0; i < n; ++i)
        if (tokens_host[i] < 0 || tokens_host[i] >= m->cfg.vocab) return QW_INVALID_ARGUMENT;
    int rc = QW_OK;
    if ((m->debug & QW_DEBUG_PREFILL_BY_TOKEN) || !qw::prefill_supported(m->pf)) {
        for (int32_t i = 0; i < n && !rc; ++i) rc = launch_step(m, tokens_host[i], nullptr);
    } else {
        rc = qw::prefill_run(&m->pf, m->args, m->len, tokens_host, n, m->debug, m->stream);
        if (!rc) {
            m->len += n;
            m->has_last = 1;
        } else {
            rc = QW_CUDA_ERROR;
        }
    }
    if (rc) return rc;
    if (next_token_host) return read_flags(m, next_token_host);
    return QW_OK;
}

int qw_logits(qw_model *m, float *dst_dev, int64_t n) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (!dst_dev || n != m->cfg.vocab) return QW_INVALID_ARGUMENT;
    return cuda_status(cudaMemcpyAsync(dst_dev, m->logits, (size_t)n * 4, cudaMemcpyDeviceToDevice, m->stream));
}

int qw_kv_reset(qw_model *m) {
    if (!live(m)) return QW_INVALID_HANDLE;
    m->len = 0;
    m->has_last = 0;
    m->failed = 0;
    m->csteps = 0;
    int rc = cuda_status(cudaMemsetAsync(m->step_block, 0, m->step_bytes, m->stream));
    if (rc) return rc;
    return cuda_status(cudaMemsetAsync(m->flags, 0, sizeof(qw::StepFlags), m->stream));
}

int qw_kv_length(const qw_model *m, int32_t *out) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (!out) return QW_INVALID_ARGUMENT;
    *out = m->len;
    return QW_OK;
}

int qw_sync(qw_model *m) {
    if (!live(m)) return QW_INVALID_HANDLE;
    return read_flags(m, nullptr);
}

static int kv_copy(qw_model *m, const void *k_src, const void *v_src, void *k_dst, void *v_dst, int32_t n_pos,
                   bool import) {
    const qw_config &c = m->cfg;
    const bool f32 = c.kv_format == QW_KV_F32;
    const size_t row = (size_t)c.head_dim * (f32 ? 4 : 2);
    const size_t width = (size_t)n_pos * row, pitch_cache = (size_t)c.max_ctx * row;
    const size_t height = (size_t)c.n_layers * c.n_kv_heads;
    uint8_t *kc = m->ws + m->lay.kc, *vc = m->ws + m->lay.vc;
    cudaError_t e;
    if (import && f32) {
        e = qw::launch_kv_widen((const __nv_bfloat16 *)k_src, (float *)kc, (long long)height, n_pos, c.max_ctx,
                                m->stream);
        if (e == cudaSuccess)
            e = qw::launch_kv_widen((const __nv_bfloat16 *)v_src, (float *)vc, (long long)height, n_pos, c.max_ctx,
                                    m->stream);
    } else if (import) {
        e = cudaMemcpy2DAsync(kc, pitch_cache, k_src, width, width, height, cudaMemcpyDeviceToDevice, m->stream);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(vc, pitch_cache, v_src, width, width, height, cudaMemcpyDeviceToDevice, m->stream);
    } else {
        e = cudaMemcpy2DAsync(k_dst, width, kc, pitch_cache, width, height, cudaMemcpyDeviceToDevice, m->stream);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(v_dst, width, vc, pitch_cache, width, height, cudaMemcpyDeviceToDevice, m->stream);
    }
    return cuda_status(e);
}

int qw_kv_import(qw_model *m, const void *k_dev, const void *v_dev, int32_t n_pos) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (n_pos < 0 || (n_pos > 0 && (!k_dev || !v_dev))) return QW_INVALID_ARGUMENT;
    if (n_pos > m->cfg.max_ctx) return QW_CONTEXT_EXCEEDED;
    if (!aligned(k_dev, 16) || !aligned(v_dev, 16)) return n_pos ? QW_ALIGNMENT : QW_OK;
    if (n_pos > 0) {
        int rc = kv_copy(m, k_dev, v_dev, nullptr, nullptr, n_pos, true);
        if (rc) return rc;
    }
    m->len = n_pos;
    m->has_last = 0;
    return QW_OK;
}

int qw_kv_export(qw_model *m, void *k_dev, void *v_dev, int32_t n_pos) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (n_pos < 0 || n_pos > m->len || (n_pos > 0 && (!k_dev || !v_dev))) return QW_INVALID_ARGUMENT;
    if (n_pos == 0) return QW_OK;
    return kv_copy(m, nullptr, nullptr, k_dev, v_dev, n_pos, false);
}

int qw_set_debug(qw_model *m, int32_t flags) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (flags & ~(QW_DEBUG_HIDDEN | QW_DEBUG_PREFILL_BY_TOKEN | QW_DEBUG_TRACE | QW_DEBUG_ONE_GROUP |
                  QW_DEBUG_WITHHOLD))
        return QW_INVALID_ARGUMENT;
    m->debug = flags;
    return QW_OK;
}

int qw_debug_hidden(qw_model *m, float *dst_dev, int64_t n) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (!dst_dev || n != (int64_t)(m->cfg.n_layers + 1) * m->cfg.hidden) return QW_INVALID_ARGUMENT;
    return cuda_status(cudaMemcpyAsync(dst_dev, m->hidden, (size_t)n * 4, cudaMemcpyDeviceToDevice, m->stream));
}

int qw_query(const qw_model *m, int32_t what, int64_t *out) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (!out) return QW_INVALID_ARGUMENT;
    switch (what) {
        case QW_QUERY_DECODE_CTAS: *out = m->ncta; return QW_OK;
        case QW_QUERY_TRACE_LEN:
            *out = ((int64_t)qw::kPhasesPerLayer * m->cfg.n_layers + 1) * m->ncta * qw::kTraceStamps;
            return QW_OK;
        case QW_QUERY_WORKSPACE_BYTES: *out = (int64_t)m->lay.total; return QW_OK;
        case QW_QUERY_DECODE_GROUPS: *out = m->groups; return QW_OK;
        case QW_QUERY_GROUP0_CTAS: *out = m->n_grp[0]; return QW_OK;
        case QW_QUERY_RT_NEAR_NS: *out = (int64_t)(m->rt_near + 0.5f); return QW_OK;
        case QW_QUERY_RT_FAR_NS: *out = (int64_t)(m->rt_far + 0.5f); return QW_OK;
        case QW_QUERY_XREGION_OFFSET: *out = (int64_t)((uint8_t *)m->args.xr - m->ws); return QW_OK;
        default: return QW_INVALID_ARGUMENT;
    }
}

int qw_debug_trace(qw_model *m, uint64_t *dst_dev, int64_t n) {
    if (!live(m)) return QW_INVALID_HANDLE;
    const int64_t len = ((int64_t)qw::kPhasesPerLayer * m->cfg.n_layers + 1) * m->ncta * qw::kTraceStamps;
    if (!dst_dev || n != len) return QW_INVALID_ARGUMENT;
    return cuda_status(cudaMemcpyAsync(dst_dev, m->ws + m->lay.trace, (size_t)n * 8, cudaMemcpyDeviceToDevice,
                                       m->stream));
}

static int check_sampling(const qw_sampling *sp, int32_t vocab, int32_t n_history, const int32_t *history) {
    if (!sp || n_history < 0 || (n_history > 0 && !history)) return QW_INVALID_ARGUMENT;
    if (!(sp->temperature >= 0.0f) || !std::isfinite(sp->temperature)) return QW_INVALID_ARGUMENT;
    if (!(sp->repetition_penalty > 0.0f) || !std::isfinite(sp->repetition_penalty)) return QW_INVALID_ARGUMENT;
    if (!(sp->top_p > 0.0f) || !(sp->top_p <= 1.0f)) return QW_INVALID_ARGUMENT;
    if (sp->temperature > 0.0f && (sp->top_k < 1 || sp->top_k > QW_SAMPLE_MAX_TOP_K || sp->top_k > vocab))
        return QW_INVALID_ARGUMENT;
    return QW_OK;
}

size_t qw_sample_scratch_bytes(int32_t vocab) { return vocab > 0 ? qw::sample_scratch_bytes(vocab) : 0; }

int qw_sample_logits(const float *logits_dev, int32_t vocab, const int32_t *history_dev, int32_t n_history,
                     const qw_sampling *params, uint64_t *rng_dev, int32_t *token_dev, void *scratch_dev,
                     size_t scratch_bytes, void *cuda_stream) {
    if (vocab < 1 || vocab > (1 << 24) || !logits_dev || !rng_dev || !token_dev || !scratch_dev)
        return QW_INVALID_ARGUMENT;
    int rc = check_sampling(params, vocab, n_history, history_dev);
    if (rc) return rc;
    if (!aligned(scratch_dev, 256) || !aligned(rng_dev, 16)) return QW_ALIGNMENT;
    if (scratch_bytes < qw::sample_scratch_bytes(vocab)) return QW_OUT_OF_MEMORY;
    return cuda_status(qw::launch_sample(logits_dev, vocab, history_dev, n_history, params->temperature,
                                         params->top_k, params->top_p, params->repetition_penalty, rng_dev,
                                         token_dev, nullptr, nullptr, scratch_dev, (cudaStream_t)cuda_stream));
}

int qw_sampler_seed(qw_model *m, uint64_t seed, uint64_t stream) {
    if (!live(m)) return QW_INVALID_HANDLE;
    // PCG32 seeding of the pages: state 0, increment (stream << 1) | 1, advance, add seed, advance
    uint64_t st = 0, inc = (stream << 1) | 1u;
    st = st * 6364136223846793005ull + inc;
    st += seed;
    st = st * 6364136223846793005ull + inc;
    const uint64_t host[2] = {st, inc};
    int rc = cuda_status(cudaMemcpyAsync(m->ws + m->lay.sampler, host, 16, cudaMemcpyHostToDevice, m->stream));
    if (rc) return rc;
    return cuda_status(cudaStreamSynchronize(m->stream));  // the host source is a local
}

int qw_sampler_state(qw_model *m, uint64_t *state_host) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (!state_host) return QW_INVALID_ARGUMENT;
    int rc = cuda_status(cudaMemcpyAsync(state_host, m->ws + m->lay.sampler, 16, cudaMemcpyDeviceToHost, m->stream));
    if (rc) return rc;
    return cuda_status(cudaStreamSynchronize(m->stream));
}

int qw_sample(qw_model *m, const qw_sampling *params, const int32_t *history_dev, int32_t n_history,
              int32_t *next_token_host) {
    if (!live(m)) return QW_INVALID_HANDLE;
    if (m->failed) return m->failed;
    if (!m->has_last) return QW_INVALID_ARGUMENT;  // no logits yet
    int rc = check_sampling(params, m->cfg.vocab, n_history, history_dev);
    if (rc) return rc;
    uint8_t *base = m->ws + m->lay.sampler;
    rc = cuda_status(qw::launch_sample(m->logits, m->cfg.vocab, history_dev, n_history, params->temperature,
                                       params->top_k, params->top_p, params->repetition_penalty,
                                       reinterpret_cast<uint64_t *>(base), nullptr, &m->flags->next_tok,
                                       &m->flags->err, base + 256, m->stream));
    if (rc) return rc;
    if (next_token_host) return read_flags(m, next_token_host);
    return QW_OK;
}

int qw_debug_gemm_f16(const void *a_dev, const void *b_dev, float *c_dev, int32_t M, int32_t N, int32_t K,
                      int32_t bn, void *cuda_stream) {
    if (M < 1 || N < 1 || K < 64 || K % 64 || (bn != 128 && bn != 256) || N % bn) return QW_INVALID_ARGUMENT;
    if (!a_dev || !b_dev || !c_dev) return QW_INVALID_ARGUMENT;
    if (!aligned(a_dev, 16) || !aligned(b_dev, 16) || !aligned(c_dev, 16)) return QW_ALIGNMENT;
    return qw::prefill_debug_gemm(a_dev, b_dev, c_dev, M, N, K, bn, (cudaStream_t)cuda_stream);
}

// ------------------------------------------------------------------ batched decode

}  // extern "C"

struct qw_batch {
    qw_model *m = nullptr;
    int max_batch = 0, max_ctx = 0;
    size_t seq_elems = 0;                // elements of one sequence's K (or V) cache block
    uint8_t *kc = nullptr, *vc = nullptr;
    int32_t *tok_in = nullptr, *tok = nullptr, *picks = nullptr;
    int *row_pos = nullptr;
    unsigned long long *keys = nullptr;
    qw::StepFlags *flags = nullptr;
    float *part = nullptr, *logits = nullptr, *hidden = nullptr;
    std::vector<int32_t> len;
    std::vector<int> has_last;
    int last_n = 0;                      // sequences of the last step (rows of logits / hidden)
    int failed = 0;
    // A step's launches depend on the sequence count, the attention split count and the debug
    // dump only; each combination is captured once (on a private stream) into a CUDA graph and
    // replayed on the model's stream.
    struct Graph {
        int B, S, hidden;
        cudaGraphExec_t exec;
    };
    std::vector<Graph> graphs;
    cudaStream_t cap = nullptr;
};

namespace {

std::unordered_set<const void *> g_live_batch;

bool live_batch(const qw_batch *b) {
    std::lock_guard<std::mutex> g(g_live_mu);
    return b && g_live_batch.count(b) && g_live.count(b->m);
}

struct BatchLayout {
    size_t kc, vc, small, flags, part, logits, hidden, total;
};

// Regions of a batch workspace (256-byte aligned): the K and V cache blocks of every sequence,
// token / position / pick / key arrays, flags, attention partials, logits, the debug dump.
bool batch_layout(const qw_config &c, int max_batch, int max_ctx, BatchLayout *L) {
    const size_t esz = c.kv_format == QW_KV_F32 ? 4 : 2;
    const size_t block = (size_t)c.n_layers * c.n_kv_heads * max_ctx * c.head_dim * esz;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    L->kc = take(block * max_batch);
    L->vc = take(block * max_batch);
    L->small = take(5 * qw::kBatchMax * 8);
    L->flags = take(sizeof(qw::StepFlags));
    L->part = take((size_t)max_batch * c.n_heads * qw::kBatchMaxSplits * qw::kBatchPartStride * 4);
    L->logits = take((size_t)max_batch * c.vocab * 4);
    L->hidden = take((size_t)(c.n_layers + 1) * max_batch * c.hidden * 4);
    L->total = off;
    return true;
}

int batch_read(qw_batch *b, int32_t *picks_host, int n) {
    qw::StepFlags f;
    int rc = cuda_status(cudaMemcpyAsync(&f, b->flags, sizeof(f), cudaMemcpyDeviceToHost, b->m->stream));
    if (!rc && picks_host)
        rc = cuda_status(cudaMemcpyAsync(picks_host, b->picks, (size_t)n * 4, cudaMemcpyDeviceToHost, b->m->stream));
    if (!rc) rc = cuda_status(cudaStreamSynchronize(b->m->stream));
    if (rc) return rc;
    if (f.err) {
        b->failed = (int)f.err;
        return (int)f.err;
    }
    return QW_OK;
}

}  // namespace

extern "C" {

size_t qw_batch_workspace_bytes(const qw_model *m, int32_t max_batch, int32_t max_ctx) {
    if (!live(m) || max_batch < 1 || max_batch > qw::kBatchMax || max_ctx < 1 || max_ctx > m->cfg.max_ctx) return 0;
    BatchLayout L;
    batch_layout(m->cfg, max_batch, max_ctx, &L);
    return L.total;
}

int qw_batch_create(qw_model *m, int32_t max_batch, int32_t max_ctx, void *workspace_dev, size_t workspace_bytes,
                    qw_batch **out) {
    if (!out) return QW_INVALID_ARGUMENT;
    *out = nullptr;
    if (!live(m)) return QW_INVALID_HANDLE;
    if (max_batch < 1 || max_batch > qw::kBatchMax || max_ctx < 1 || max_ctx > m->cfg.max_ctx)
        return QW_INVALID_ARGUMENT;
    if (!qw::prefill_supported(m->pf) || max_batch > m->pf.rows_max || m->cfg.n_heads != qw::kBatchG * m->cfg.n_kv_heads)
        return QW_UNSUPPORTED_SHAPE;
    const int qd = m->cfg.n_heads * m->cfg.head_dim;  // the skinny projections' row lengths: H, Hq 128, I
    if (!qw::bgemv_supported(m->cfg.hidden) || !qw::bgemv_supported(qd) || !qw::bgemv_supported(m->cfg.intermediate))
        return QW_UNSUPPORTED_SHAPE;
    if (!aligned(workspace_dev, 256)) return QW_ALIGNMENT;
    BatchLayout L;
    batch_layout(m->cfg, max_batch, max_ctx, &L);
    if (workspace_bytes < L.total) return QW_OUT_OF_MEMORY;
    qw_batch *b = new (std::nothrow) qw_batch();
    if (!b) return QW_OUT_OF_MEMORY;
    uint8_t *ws = (uint8_t *)workspace_dev;
    b->m = m;
    b->max_batch = max_batch;
    b->max_ctx = max_ctx;
    b->seq_elems = (size_t)m->cfg.n_layers * m->cfg.n_kv_heads * max_ctx * m->cfg.head_dim;
    b->kc = ws + L.kc;
    b->vc = ws + L.vc;
    b->tok_in = (int32_t *)(ws + L.small);
    b->tok = b->tok_in + qw::kBatchMax;
    b->picks = b->tok + qw::kBatchMax;
    b->row_pos = (int *)(b->picks + qw::kBatchMax);
    b->keys = (unsigned long long *)(ws + L.small + 4 * qw::kBatchMax * 4 + 64);
    b->flags = (qw::StepFlags *)(ws + L.flags);
    b->part = (float *)(ws + L.part);
    b->logits = (float *)(ws + L.logits);
    b->hidden = (float *)(ws + L.hidden);
    b->len.assign(max_batch, 0);
    b->has_last.assign(max_batch, 0);
    int rc = cuda_status(cudaMemsetAsync(ws + L.small, 0, L.part - L.small, m->stream));
    if (!rc) rc = cuda_status(cudaStreamSynchronize(m->stream));
    if (!rc) rc = cuda_status(cudaStreamCreateWithFlags(&b->cap, cudaStreamNonBlocking));
    if (rc) {
        delete b;
        return rc;
    }
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        g_live_batch.insert(b);
    }
    *out = b;
    return QW_OK;
}

void qw_batch_destroy(qw_batch *b) {
    bool model_live;
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        if (!g_live_batch.erase(b)) return;
        model_live = g_live.count(b->m) != 0;
    }
    if (model_live) cudaStreamSynchronize(b->m->stream);
    for (auto &g : b->graphs) cudaGraphExecDestroy(g.exec);
    if (b->cap) cudaStreamDestroy(b->cap);
    delete b;
}

int qw_batch_reset(qw_batch *b, int32_t seq) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    if (seq < -1 || seq >= b->max_batch) return QW_INVALID_ARGUMENT;
    for (int s = 0; s < b->max_batch; ++s)
        if (seq == -1 || s == seq) {
            b->len[s] = 0;
            b->has_last[s] = 0;
        }
    if (seq == -1) {
        b->failed = 0;
        return cuda_status(cudaMemsetAsync(b->flags, 0, sizeof(qw::StepFlags), b->m->stream));
    }
    return QW_OK;
}

int qw_batch_length(const qw_batch *b, int32_t seq, int32_t *out) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    if (!out || seq < 0 || seq >= b->max_batch) return QW_INVALID_ARGUMENT;
    *out = b->len[seq];
    return QW_OK;
}

int qw_batch_prefill(qw_batch *b, int32_t seq, const int32_t *tokens_host, int32_t n, int32_t *next_token_host) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    if (b->failed) return b->failed;
    qw_model *m = b->m;
    if (seq < 0 || seq >= b->max_batch || n < 1 || !tokens_host) return QW_INVALID_ARGUMENT;
    if ((int64_t)b->len[seq] + n > b->max_ctx) return QW_CONTEXT_EXCEEDED;
    for (int32_t i = 0; i < n; ++i)
        if (tokens_host[i] < 0 || tokens_host[i] >= m->cfg.vocab) return QW_INVALID_ARGUMENT;
    qw::DecodeArgs a = m->args;  // the model's weights and RoPE table; this sequence's cache
    const size_t esz = m->cfg.kv_format == QW_KV_F32 ? 4 : 2;
    a.kc = b->kc + (size_t)seq * b->seq_elems * esz;
    a.vc = b->vc + (size_t)seq * b->seq_elems * esz;
    a.max_ctx = b->max_ctx;
    a.logits = b->logits + (size_t)seq * m->cfg.vocab;
    a.flags = b->flags;
    if (qw::prefill_run(&m->pf, a, b->len[seq], tokens_host, n, 0, m->stream)) return QW_CUDA_ERROR;
    b->len[seq] += n;
    b->has_last[seq] = 1;
    int rc = cuda_status(cudaMemcpyAsync(b->picks + seq, &b->flags->next_tok, 4, cudaMemcpyDeviceToDevice, m->stream));
    if (rc) return rc;
    if (next_token_host) {
        rc = batch_read(b, nullptr, 0);
        if (rc) return rc;
        return cuda_status(cudaMemcpy(next_token_host, b->picks + seq, 4, cudaMemcpyDeviceToHost));
    }
    return QW_OK;
}

int qw_batch_step(qw_batch *b, int32_t n_seq, const int32_t *tokens_host, int32_t *next_tokens_host) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    if (b->failed) return b->failed;
    qw_model *m = b->m;
    if (n_seq < 1 || n_seq > b->max_batch) return QW_INVALID_ARGUMENT;
    int32_t tok[qw::kBatchMax];
    int pos[qw::kBatchMax];
    int max_n = 0;
    for (int s = 0; s < n_seq; ++s) {
        tok[s] = tokens_host ? tokens_host[s] : -1;
        if (tok[s] < -1 || tok[s] >= m->cfg.vocab) return QW_INVALID_ARGUMENT;
        if (tok[s] == -1 && !b->has_last[s]) return QW_INVALID_ARGUMENT;
        if (b->len[s] + 1 > b->max_ctx) return QW_CONTEXT_EXCEEDED;
        pos[s] = b->len[s];
        max_n = pos[s] + 1 > max_n ? pos[s] + 1 : max_n;
    }
    int rc = cuda_status(cudaMemcpyAsync(b->tok_in, tok, (size_t)n_seq * 4, cudaMemcpyHostToDevice, m->stream));
    if (!rc) rc = cuda_status(cudaMemcpyAsync(b->row_pos, pos, (size_t)n_seq * 4, cudaMemcpyHostToDevice, m->stream));
    if (rc) return rc;
    qw::BatchStep bs{};
    bs.B = n_seq;
    bs.tokens_in = b->tok_in;
    bs.tokens = b->tok;
    bs.row_pos = b->row_pos;
    bs.max_n = max_n;
    bs.kc = b->kc;
    bs.vc = b->vc;
    bs.seq_elems = b->seq_elems;
    bs.max_ctx = b->max_ctx;
    bs.part = b->part;
    bs.logits = b->logits;
    bs.keys = b->keys;
    bs.picks = b->picks;
    bs.hidden = (m->debug & QW_DEBUG_HIDDEN) ? b->hidden : nullptr;
    qw::DecodeArgs a = m->args;
    a.flags = b->flags;
    const int S = qw::batch_splits(max_n), hid = bs.hidden != nullptr;
    cudaGraphExec_t exec = nullptr;
    for (auto &g : b->graphs)
        if (g.B == n_seq && g.S == S && g.hidden == hid) exec = g.exec;
    if (!exec) {  // capture this combination's launches once
        if (cuda_status(cudaStreamBeginCapture(b->cap, cudaStreamCaptureModeThreadLocal))) return QW_CUDA_ERROR;
        const int frc = qw::prefill_batch_step(&m->pf, a, bs, b->cap);
        cudaGraph_t graph = nullptr;
        const cudaError_t ce = cudaStreamEndCapture(b->cap, &graph);
        if (frc || ce != cudaSuccess || !graph) {
            if (graph) cudaGraphDestroy(graph);
            cudaGetLastError();
            return QW_CUDA_ERROR;
        }
        const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (ie != cudaSuccess) return cuda_status(ie);
        b->graphs.push_back({n_seq, S, hid, exec});
    }
    rc = cuda_status(cudaGraphLaunch(exec, m->stream));
    if (rc) return rc;
    for (int s = 0; s < n_seq; ++s) {
        b->len[s] += 1;
        b->has_last[s] = 1;
    }
    b->last_n = n_seq;
    if (next_tokens_host) return batch_read(b, next_tokens_host, n_seq);
    return QW_OK;
}

int qw_batch_logits(qw_batch *b, float *dst_dev, int64_t n) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    if (!dst_dev || b->last_n == 0 || n != (int64_t)b->last_n * b->m->cfg.vocab) return QW_INVALID_ARGUMENT;
    return cuda_status(
        cudaMemcpyAsync(dst_dev, b->logits, (size_t)n * 4, cudaMemcpyDeviceToDevice, b->m->stream));
}

int qw_batch_debug_hidden(qw_batch *b, float *dst_dev, int64_t n) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    const qw_config &c = b->m->cfg;
    if (!dst_dev || b->last_n == 0 || n != (int64_t)(c.n_layers + 1) * b->last_n * c.hidden) return QW_INVALID_ARGUMENT;
    return cuda_status(
        cudaMemcpyAsync(dst_dev, b->hidden, (size_t)n * 4, cudaMemcpyDeviceToDevice, b->m->stream));
}

int qw_batch_sync(qw_batch *b) {
    if (!live_batch(b)) return QW_INVALID_HANDLE;
    return batch_read(b, nullptr, 0);
}

}  // extern "C"
