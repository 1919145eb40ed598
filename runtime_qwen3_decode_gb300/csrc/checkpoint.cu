// checkpoint.cu - safetensors / SLM2 checkpoint files: header parsing and validation, the
// cross-check against the tensor set a config implies, and the upload of the tensors into the
// device layout qw_model_create takes.  Host code only (compiled with the library).
//
// Format ("Scalar-Native Qwen3 Reference Runtime As The Numerical Authority", section 3 "File
// Layout and Safe Metadata Parsing"; "M1 - Load the weights", section "The safetensors format"):
// [u64 little-endian N][N bytes of UTF-8 JSON][blob].  The JSON object maps each tensor name to
// {"dtype": ..., "shape": [...], "data_offsets": [begin, end]} with offsets into the blob; an
// optional "__metadata__" entry maps strings to strings.  Every entry must satisfy (the pages'
// invariants, failing closed on anything else):
//   end <= blob size                                          (file boundary)
//   spans sorted by begin never overlap                        (monotonic, non-overlapping)
//   8 + N + begin divisible by 8                               (aligned payload)
//   end - begin == bytes of shape x dtype                      (self-consistent entry)
//   Q8_0 tensors hold a whole number of 32-element blocks      (no tail groups)
// Q8_0 (the SLM2 mixed-Q8 matrices) is stored as 34-byte blocks: an fp16 scale, then 32 int8
// codes ("Scalar-Native ...", section 3 "Mixed-Q8 Quantization Definition").
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "qw.h"

struct qw_checkpoint {
    struct Tensor {
        std::string name;
        int32_t dtype;
        std::vector<int64_t> shape;
        uint64_t begin, end;
    };
    const uint8_t *bytes = nullptr;  // borrowed: prefix + header (+ blob when data_ok)
    uint64_t bytes_len = 0, file_size = 0, header_len = 0;
    bool data_ok = false;            // the blob is in memory too
    std::vector<Tensor> tensors;     // sorted by begin
    std::map<std::string, size_t> index;
    const uint8_t *blob() const { return bytes + 8 + header_len; }
};

namespace {

std::mutex g_ck_mu;
std::unordered_set<const void *> g_ck_live;
thread_local std::string g_ck_error;

int fail(int code, const std::string &why) {
    g_ck_error = why;
    return code;
}

bool ck_live(const qw_checkpoint *c) {
    std::lock_guard<std::mutex> g(g_ck_mu);
    return c && g_ck_live.count(c);
}

// ---------------------------------------------------------------- a strict JSON reader
//
// Just what a checkpoint header holds: objects, arrays, strings, non-negative integers.  Anything
// else (floats, negative numbers, true/false/null, duplicate keys, trailing bytes) is an error.
struct Json {
    const char *p, *e;
    std::string err;
    void ws() {
        while (p < e && (*p == ' ' || *p == '\t' || *p == '\n' || *p == '\r')) ++p;
    }
    bool lit(char c) {
        ws();
        if (p < e && *p == c) {
            ++p;
            return true;
        }
        return false;
    }
    bool expect(char c) {
        if (lit(c)) return true;
        err = std::string("expected '") + c + "'";
        return false;
    }
    static int hexv(char c) {
        if (c >= '0' && c <= '9') return c - '0';
        if (c >= 'a' && c <= 'f') return c - 'a' + 10;
        if (c >= 'A' && c <= 'F') return c - 'A' + 10;
        return -1;
    }
    bool str(std::string &out) {
        out.clear();
        ws();
        if (p >= e || *p != '"') {
            err = "expected a string";
            return false;
        }
        ++p;
        while (p < e && *p != '"') {
            const unsigned char c = (unsigned char)*p++;
            if (c < 0x20) {
                err = "control character in a string";
                return false;
            }
            if (c != '\\') {
                out.push_back((char)c);
                continue;
            }
            if (p >= e) break;
            const char k = *p++;
            switch (k) {
                case '"': out.push_back('"'); break;
                case '\\': out.push_back('\\'); break;
                case '/': out.push_back('/'); break;
                case 'b': out.push_back('\b'); break;
                case 'f': out.push_back('\f'); break;
                case 'n': out.push_back('\n'); break;
                case 'r': out.push_back('\r'); break;
                case 't': out.push_back('\t'); break;
                case 'u': {
                    if (e - p < 4) {
                        err = "short \\u escape";
                        return false;
                    }
                    unsigned v = 0;
                    for (int i = 0; i < 4; ++i) {
                        const int h = hexv(p[i]);
                        if (h < 0) {
                            err = "bad \\u escape";
                            return false;
                        }
                        v = v * 16 + (unsigned)h;
                    }
                    p += 4;
                    if (v >= 0xd800 && v < 0xe000) {  // surrogates: names are not expected to need them
                        err = "surrogate \\u escape";
                        return false;
                    }
                    if (v < 0x80) {
                        out.push_back((char)v);
                    } else if (v < 0x800) {
                        out.push_back((char)(0xc0 | (v >> 6)));
                        out.push_back((char)(0x80 | (v & 0x3f)));
                    } else {
                        out.push_back((char)(0xe0 | (v >> 12)));
                        out.push_back((char)(0x80 | ((v >> 6) & 0x3f)));
                        out.push_back((char)(0x80 | (v & 0x3f)));
                    }
                    break;
                }
                default: err = "bad escape"; return false;
            }
        }
        if (p >= e) {
            err = "unterminated string";
            return false;
        }
        ++p;
        return true;
    }
    bool uint(uint64_t &out) {
        ws();
        if (p >= e || *p < '0' || *p > '9') {
            err = "expected a non-negative integer";
            return false;
        }
        if (*p == '0' && p + 1 < e && p[1] >= '0' && p[1] <= '9') {
            err = "leading zero";
            return false;
        }
        uint64_t v = 0;
        while (p < e && *p >= '0' && *p <= '9') {
            const uint64_t d = (uint64_t)(*p - '0');
            if (v > (UINT64_MAX - d) / 10) {
                err = "integer overflow";
                return false;
            }
            v = v * 10 + d;
            ++p;
        }
        if (p < e && (*p == '.' || *p == 'e' || *p == 'E')) {
            err = "not an integer";
            return false;
        }
        out = v;
        return true;
    }
    bool uints(std::vector<uint64_t> &out) {
        out.clear();
        if (!expect('[')) return false;
        if (lit(']')) return true;
        do {
            uint64_t v;
            if (!uint(v)) return false;
            out.push_back(v);
        } while (lit(','));
        return expect(']');
    }
};

int dtype_of(const std::string &s) {
    if (s == "BF16") return QW_DT_BF16;
    if (s == "F16") return QW_DT_F16;
    if (s == "F32") return QW_DT_F32;
    if (s == "I8") return QW_DT_I8;
    if (s == "Q8_0") return QW_DT_Q8_0;
    return -1;
}

// Bytes of a tensor of n elements, or 0 if the count does not fit the dtype (Q8_0 tail groups).
uint64_t dtype_bytes(int dt, uint64_t n) {
    switch (dt) {
        case QW_DT_BF16:
        case QW_DT_F16: return 2 * n;
        case QW_DT_F32: return 4 * n;
        case QW_DT_I8: return n;
        case QW_DT_Q8_0: return n % 32 ? 0 : n / 32 * 34;
        default: return 0;
    }
}

struct Expected {
    std::string name;
    std::vector<int64_t> shape;
    int kind;  // 0 embedding, 1 norm vector, 2 projection matrix, 3 tied head copy
};

// The tensor set a config implies ("M1 - Load the weights", section "Deriving what should be
// there"): embed_tokens [V,H], model.norm [H], an optional lm_head [V,H], and per layer the
// 11-tensor block with matrices stored [out, in].
std::vector<Expected> expected_set(const qw_config &c) {
    const int64_t H = c.hidden, V = c.vocab, d = c.head_dim, I = c.intermediate, QD = (int64_t)c.n_heads * d,
                  KD = (int64_t)c.n_kv_heads * d;
    std::vector<Expected> out;
    out.push_back({"model.embed_tokens.weight", {V, H}, 0});
    for (int l = 0; l < c.n_layers; ++l) {
        const std::string p = "model.layers." + std::to_string(l) + ".";
        out.push_back({p + "input_layernorm.weight", {H}, 1});
        out.push_back({p + "self_attn.q_proj.weight", {QD, H}, 2});
        out.push_back({p + "self_attn.k_proj.weight", {KD, H}, 2});
        out.push_back({p + "self_attn.v_proj.weight", {KD, H}, 2});
        out.push_back({p + "self_attn.q_norm.weight", {d}, 1});
        out.push_back({p + "self_attn.k_norm.weight", {d}, 1});
        out.push_back({p + "self_attn.o_proj.weight", {H, QD}, 2});
        out.push_back({p + "post_attention_layernorm.weight", {H}, 1});
        out.push_back({p + "mlp.gate_proj.weight", {I, H}, 2});
        out.push_back({p + "mlp.up_proj.weight", {I, H}, 2});
        out.push_back({p + "mlp.down_proj.weight", {H, I}, 2});
    }
    out.push_back({"model.norm.weight", {H}, 1});
    out.push_back({"lm_head.weight", {V, H}, 3});
    return out;
}

int64_t numel(const std::vector<int64_t> &s) {
    int64_t n = 1;
    for (int64_t v : s) n *= v;
    return n;
}

bool valid_dims(const qw_config *c) {
    return c && c->n_layers >= 1 && c->n_layers <= 64 && c->hidden > 0 && c->n_heads > 0 && c->n_kv_heads > 0 &&
           c->head_dim > 0 && c->intermediate > 0 && c->vocab > 0 && c->hidden % 32 == 0 &&
           c->intermediate % 32 == 0 && ((int64_t)c->n_heads * c->head_dim) % 32 == 0;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Device bytes of the upload layout: embed, final norm, optional lm_head, then per layer four norm
// vectors and the seven matrices (int8: codes and fp16 scales), every piece 256-byte aligned.
size_t upload_bytes(const qw_config &c, bool head_copy) {
    const size_t H = c.hidden, V = c.vocab, d = c.head_dim, I = c.intermediate, QD = (size_t)c.n_heads * d,
                 KD = (size_t)c.n_kv_heads * d;
    size_t n = up256(V * H * 2) + up256(H * 2) + (head_copy ? up256(V * H * 2) : 0);
    const size_t mats[7][2] = {{QD, H}, {KD, H}, {KD, H}, {H, QD}, {I, H}, {I, H}, {H, I}};
    size_t per = 2 * up256(H * 2) + 2 * up256(d * 2);
    for (const auto &m : mats) {
        const size_t e = m[0] * m[1];
        per += c.weight_format != QW_W_BF16 ? up256(e) + up256(e / 32 * 2) : up256(e * 2);
    }
    return n + per * c.n_layers;
}

}  // namespace

extern "C" {

const char *qw_checkpoint_last_error(void) { return g_ck_error.c_str(); }

int qw_checkpoint_open(const void *bytes, uint64_t bytes_len, uint64_t file_size, qw_checkpoint **out) {
    if (!out) return fail(QW_INVALID_ARGUMENT, "null output");
    *out = nullptr;
    if (!bytes || bytes_len < 8 || file_size < bytes_len) return fail(QW_INVALID_ARGUMENT, "short file");
    const uint8_t *b = (const uint8_t *)bytes;
    uint64_t N = 0;
    for (int i = 7; i >= 0; --i) N = (N << 8) | b[i];  // little-endian u64
    if (N < 2 || N > file_size - 8 || N > bytes_len - 8) return fail(QW_INVALID_ARGUMENT, "header length out of range");
    const uint64_t blob = file_size - 8 - N;
    qw_checkpoint *c = new (std::nothrow) qw_checkpoint();
    if (!c) return fail(QW_OUT_OF_MEMORY, "host allocation");
    c->bytes = b;
    c->bytes_len = bytes_len;
    c->file_size = file_size;
    c->header_len = N;
    c->data_ok = bytes_len == file_size;
    Json j{(const char *)b + 8, (const char *)b + 8 + N, {}};
    auto bad = [&](const std::string &why) {
        delete c;
        return fail(QW_INVALID_ARGUMENT, why);
    };
    if (!j.expect('{')) return bad(j.err);
    if (!j.lit('}')) {
        do {
            std::string name;
            if (!j.str(name)) return bad(j.err);
            if (!j.expect(':')) return bad(j.err);
            if (name == "__metadata__") {  // string -> string
                if (!j.expect('{')) return bad(j.err);
                if (!j.lit('}')) {
                    do {
                        std::string k, v;
                        if (!j.str(k) || !j.expect(':') || !j.str(v)) return bad("__metadata__: " + j.err);
                    } while (j.lit(','));
                    if (!j.expect('}')) return bad(j.err);
                }
                continue;
            }
            if (c->index.count(name)) return bad("duplicate tensor " + name);
            if (!j.expect('{')) return bad(name + ": " + j.err);
            std::string dts;
            std::vector<uint64_t> shape, offs;
            bool have_dt = false, have_shape = false, have_offs = false;
            if (!j.lit('}')) {
                do {
                    std::string key;
                    if (!j.str(key) || !j.expect(':')) return bad(name + ": " + j.err);
                    if (key == "dtype" && !have_dt) {
                        if (!j.str(dts)) return bad(name + ": " + j.err);
                        have_dt = true;
                    } else if (key == "shape" && !have_shape) {
                        if (!j.uints(shape)) return bad(name + ": " + j.err);
                        have_shape = true;
                    } else if (key == "data_offsets" && !have_offs) {
                        if (!j.uints(offs)) return bad(name + ": " + j.err);
                        have_offs = true;
                    } else {
                        return bad(name + ": unexpected or repeated key " + key);
                    }
                } while (j.lit(','));
                if (!j.expect('}')) return bad(name + ": " + j.err);
            }
            if (!have_dt || !have_shape || !have_offs) return bad(name + ": dtype, shape and data_offsets required");
            const int dt = dtype_of(dts);
            if (dt < 0) return bad(name + ": unknown dtype " + dts);
            if (shape.size() > 4 || offs.size() != 2) return bad(name + ": shape rank > 4 or offsets not [begin, end]");
            uint64_t n = 1;
            for (uint64_t s : shape) {
                if (s != 0 && n > UINT64_MAX / s / 4) return bad(name + ": shape overflows");
                n *= s;
            }
            const uint64_t nb = dtype_bytes(dt, n);
            if (dt == QW_DT_Q8_0 && n % 32) return bad(name + ": Q8_0 tensor is not a whole number of 32-element blocks");
            if (offs[1] < offs[0] || offs[1] - offs[0] != nb)
                return bad(name + ": data_offsets span does not match shape x dtype");
            if (offs[1] > blob) return bad(name + ": data ends past the file");
            if ((8 + N + offs[0]) % 8) return bad(name + ": data not 8-byte aligned in the file");
            qw_checkpoint::Tensor t{name, dt, {}, offs[0], offs[1]};
            for (uint64_t s : shape) t.shape.push_back((int64_t)s);
            c->index[name] = c->tensors.size();
            c->tensors.push_back(std::move(t));
        } while (j.lit(','));
        if (!j.expect('}')) return bad(j.err);
    }
    j.ws();
    if (j.p != j.e) return bad("trailing bytes after the header object");
    std::sort(c->tensors.begin(), c->tensors.end(),
              [](const qw_checkpoint::Tensor &a, const qw_checkpoint::Tensor &x) { return a.begin < x.begin; });
    c->index.clear();
    for (size_t i = 0; i < c->tensors.size(); ++i) {
        if (i && c->tensors[i].begin < c->tensors[i - 1].end)
            return bad(c->tensors[i].name + ": overlaps " + c->tensors[i - 1].name);
        c->index[c->tensors[i].name] = i;
    }
    {
        std::lock_guard<std::mutex> g(g_ck_mu);
        g_ck_live.insert(c);
    }
    *out = c;
    g_ck_error.clear();
    return QW_OK;
}

void qw_checkpoint_close(qw_checkpoint *c) {
    {
        std::lock_guard<std::mutex> g(g_ck_mu);
        if (!g_ck_live.erase(c)) return;
    }
    delete c;
}

int32_t qw_checkpoint_count(const qw_checkpoint *c) { return ck_live(c) ? (int32_t)c->tensors.size() : -1; }

int qw_checkpoint_tensor(const qw_checkpoint *c, int32_t i, char *name, int32_t name_cap, int32_t *dtype,
                         int32_t *rank, int64_t *dims, uint64_t *begin, uint64_t *end) {
    if (!ck_live(c)) return QW_INVALID_HANDLE;
    if (i < 0 || i >= (int32_t)c->tensors.size()) return QW_INVALID_ARGUMENT;
    const auto &t = c->tensors[(size_t)i];
    if (name) {
        if (name_cap < (int32_t)t.name.size() + 1) return QW_INVALID_ARGUMENT;
        std::memcpy(name, t.name.c_str(), t.name.size() + 1);
    }
    if (dtype) *dtype = t.dtype;
    if (rank) *rank = (int32_t)t.shape.size();
    if (dims)
        for (size_t k = 0; k < 4; ++k) dims[k] = k < t.shape.size() ? t.shape[k] : 0;
    if (begin) *begin = t.begin;
    if (end) *end = t.end;
    return QW_OK;
}

int qw_checkpoint_check(const qw_checkpoint *c, const qw_config *cfg, qw_checkpoint_report *r) {
    if (!ck_live(c)) return QW_INVALID_HANDLE;
    if (!r || !valid_dims(cfg)) return QW_INVALID_ARGUMENT;
    std::memset(r, 0, sizeof(*r));
    const auto exp = expected_set(*cfg);
    std::unordered_set<std::string> seen;
    auto problem = [&](const std::string &s) {
        if (!r->first_problem[0]) std::snprintf(r->first_problem, sizeof(r->first_problem), "%s", s.c_str());
    };
    for (const auto &e : exp) {
        const auto it = c->index.find(e.name);
        if (e.kind != 3) r->n_expected += 1;
        if (it == c->index.end()) {
            if (e.kind == 3) continue;  // a tied head may be absent
            r->n_missing += 1;
            problem("missing " + e.name);
            continue;
        }
        seen.insert(e.name);
        const auto &t = c->tensors[it->second];
        r->n_found += 1;
        if (t.shape != e.shape) {
            r->n_misshaped += 1;
            std::string s = e.name + ": shape [";
            for (size_t k = 0; k < t.shape.size(); ++k) s += (k ? "," : "") + std::to_string(t.shape[k]);
            s += "], expected [";
            for (size_t k = 0; k < e.shape.size(); ++k) s += (k ? "," : "") + std::to_string(e.shape[k]);
            problem(s + "]");
        }
        const bool vec = e.kind == 1, mat = e.kind == 2;
        const bool dt_ok = vec ? (t.dtype == QW_DT_BF16 || t.dtype == QW_DT_F32)
                           : mat ? (cfg->weight_format != QW_W_BF16 ? t.dtype == QW_DT_Q8_0 : t.dtype == QW_DT_BF16)
                                 : t.dtype == QW_DT_BF16;
        if (!dt_ok) {
            r->n_bad_dtype += 1;
            problem(e.name + ": dtype not loadable for this config");
        }
        r->stored_params += numel(t.shape);
        if (e.kind == 0) r->embedding_params = numel(t.shape);
        if (e.kind == 3) r->lm_head_copy = 1;
        else r->logical_params += numel(t.shape);
    }
    for (const auto &t : c->tensors)
        if (!seen.count(t.name)) {
            r->n_unexpected += 1;
            r->stored_params += numel(t.shape);
            problem("unexpected " + t.name);
        }
    r->n_tensors = (int32_t)c->tensors.size();
    const bool clean = !r->n_missing && !r->n_misshaped && !r->n_unexpected && !r->n_bad_dtype;
    return clean ? QW_OK : QW_UNSUPPORTED_SHAPE;
}

size_t qw_checkpoint_upload_bytes(const qw_checkpoint *c, const qw_config *cfg) {
    if (!ck_live(c) || !valid_dims(cfg)) return 0;
    const auto it = c->index.find("lm_head.weight");
    bool copy = false;
    if (it != c->index.end() && c->data_ok) {  // a head byte-identical to the embedding is tied
        const auto &h = c->tensors[it->second], &e = c->tensors[c->index.at("model.embed_tokens.weight")];
        copy = h.end - h.begin != e.end - e.begin ||
               std::memcmp(c->blob() + h.begin, c->blob() + e.begin, (size_t)(h.end - h.begin)) != 0;
    }
    return upload_bytes(*cfg, copy);
}

int qw_checkpoint_upload(const qw_checkpoint *c, const qw_config *cfg, void *dst_dev, size_t dst_bytes,
                         qw_layer_weights *layers, qw_weights *table, void *cuda_stream) {
    if (!ck_live(c)) return QW_INVALID_HANDLE;
    if (!valid_dims(cfg) || !layers || !table || !dst_dev) return QW_INVALID_ARGUMENT;
    if (!c->data_ok) return fail(QW_INVALID_ARGUMENT, "the checkpoint holds only its header");
    if (((uintptr_t)dst_dev) % 256) return QW_ALIGNMENT;
    qw_checkpoint_report rep;
    int rc = qw_checkpoint_check(c, cfg, &rep);
    if (rc) return fail(rc, rep.first_problem);
    const size_t need = qw_checkpoint_upload_bytes(c, cfg);
    if (dst_bytes < need) return QW_OUT_OF_MEMORY;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    uint8_t *dst = (uint8_t *)dst_dev;
    size_t off = 0;
    std::vector<std::vector<uint8_t>> staging;  // converted host copies, alive until the final sync
    auto put = [&](const void *src, size_t n) -> const void * {
        uint8_t *d = dst + off;
        off += up256(n);
        if (cudaMemcpyAsync(d, src, n, cudaMemcpyHostToDevice, st) != cudaSuccess) return nullptr;
        return d;
    };
    auto tensor = [&](const std::string &name) -> const qw_checkpoint::Tensor & {
        return c->tensors[c->index.at(name)];
    };
    // a norm vector as bf16: bf16 stored, or f32 values that bf16 holds exactly
    auto norm = [&](const std::string &name, const void **out) -> int {
        const auto &t = tensor(name);
        const uint8_t *src = c->blob() + t.begin;
        if (t.dtype == QW_DT_BF16) {
            *out = put(src, (size_t)(t.end - t.begin));
            return *out ? QW_OK : QW_CUDA_ERROR;
        }
        const size_t n = (size_t)numel(t.shape);
        staging.emplace_back(n * 2);
        uint16_t *h = (uint16_t *)staging.back().data();
        for (size_t i = 0; i < n; ++i) {
            uint32_t u;
            std::memcpy(&u, src + 4 * i, 4);
            h[i] = (uint16_t)(u >> 16);
            if (u & 0xffffu) return fail(QW_UNSUPPORTED_QUANTIZATION, name + ": f32 value not representable in bf16");
        }
        *out = put(h, n * 2);
        return *out ? QW_OK : QW_CUDA_ERROR;
    };
    // a projection matrix: bf16 as stored, or Q8_0 blocks split into int8 codes and fp16 scales
    auto matrix = [&](const std::string &name, const void **w, const void **s) -> int {
        const auto &t = tensor(name);
        const uint8_t *src = c->blob() + t.begin;
        if (t.dtype == QW_DT_BF16) {
            *w = put(src, (size_t)(t.end - t.begin));
            *s = nullptr;
            return *w ? QW_OK : QW_CUDA_ERROR;
        }
        const size_t n = (size_t)numel(t.shape), nb = n / 32;
        staging.emplace_back(n);
        uint8_t *codes = staging.back().data();
        staging.emplace_back(nb * 2);
        uint8_t *scales = staging.back().data();
        for (size_t b = 0; b < nb; ++b) {
            std::memcpy(scales + 2 * b, src + 34 * b, 2);
            std::memcpy(codes + 32 * b, src + 34 * b + 2, 32);
        }
        *w = put(codes, n);
        *s = put(scales, nb * 2);
        return *w && *s ? QW_OK : QW_CUDA_ERROR;
    };
    table->embed = put(c->blob() + tensor("model.embed_tokens.weight").begin,
                       (size_t)cfg->vocab * cfg->hidden * 2);
    if (!table->embed) return QW_CUDA_ERROR;
    if ((rc = norm("model.norm.weight", &table->final_norm))) return rc;
    table->lm_head = nullptr;
    if (need != upload_bytes(*cfg, false)) {  // an untied head: its own copy
        table->lm_head = put(c->blob() + tensor("lm_head.weight").begin, (size_t)cfg->vocab * cfg->hidden * 2);
        if (!table->lm_head) return QW_CUDA_ERROR;
    }
    static const char *kMat[7] = {"self_attn.q_proj", "self_attn.k_proj", "self_attn.v_proj", "self_attn.o_proj",
                                  "mlp.gate_proj",    "mlp.up_proj",      "mlp.down_proj"};
    for (int l = 0; l < cfg->n_layers; ++l) {
        const std::string p = "model.layers." + std::to_string(l) + ".";
        qw_layer_weights &L = layers[l];
        std::memset(&L, 0, sizeof(L));
        if ((rc = norm(p + "input_layernorm.weight", &L.input_norm)) ||
            (rc = norm(p + "self_attn.q_norm.weight", &L.q_norm)) ||
            (rc = norm(p + "self_attn.k_norm.weight", &L.k_norm)) ||
            (rc = norm(p + "post_attention_layernorm.weight", &L.post_norm)))
            return rc;
        for (int m = 0; m < 7; ++m)
            if ((rc = matrix(p + kMat[m] + ".weight", &L.w[m], &L.s[m]))) return rc;
    }
    table->layers = layers;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QW_CUDA_ERROR;  // staging copies done
    return QW_OK;
}

}  // extern "C"
