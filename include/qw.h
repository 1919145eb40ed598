/*
 * qw.h - C ABI of the GB300 batch-one Qwen3 decoder (libqw.so).
 *
 * What the library computes: the Qwen3 decoder forward for one sequence,
 * as laid out in "Scalar-Native Qwen3 Reference Runtime As The Numerical
 * Authority", section 2 "Decoder-Layer Mathematical Formulation" steps 1-7:
 * embedding gather, then per layer RMSNorm, bias-free Q/K/V projections,
 * per-head QK-Norm, RoPE, grouped-query causal attention over a K/V cache,
 * o_proj with residual, RMSNorm and the SwiGLU MLP with residual; then the
 * final RMSNorm, the tied lm_head and a greedy argmax (ties to the lowest
 * token id, "Portable WebAssembly Runtime Architecture for TinyRustLM",
 * section "Deterministic sampling contract", sampling order step 6).
 *
 * Interface conventions follow "Portable WebAssembly Runtime Architecture
 * for TinyRustLM", section "Typed host/Wasm API": extern "C", fixed-width
 * integers, an opaque handle checked on every call, status codes instead
 * of exceptions, and borrowed pointers.  Status values reuse that page's
 * TrResult numbering.
 *
 * Ownership.  The caller owns every device buffer: the weights (borrowed
 * for the model's lifetime, never copied or written) and the workspace
 * (sized by qw_workspace_bytes, carved by the library into the K/V cache,
 * activation buffers and bookkeeping).  The library allocates no device
 * memory.  The qw_model handle itself is host memory owned by the library
 * until qw_model_destroy.
 *
 * Streams and synchronisation.  Every call enqueues work on the stream given
 * at creation and returns without waiting, except where it writes a host
 * pointer (next_token_host), which waits for that stream.  Errors raised on
 * the device (non-finite logits, a bounded wait that expired) are recorded
 * in the workspace and reported by the next call that waits on the stream.
 *
 * Device: one GB300 (sm_103a).  There is no CPU fallback: if the device
 * code cannot run, calls fail with QW_CUDA_ERROR.
 */
#ifndef QW_H
#define QW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QW_ABI_VERSION 1

typedef struct qw_model qw_model;

/* Status codes (values from the TrResult table of the typed host API). */
enum qw_status {
    QW_OK = 0,
    QW_INVALID_ARGUMENT = 1,          /* NULL pointer, negative count, token id out of range */
    QW_INVALID_HANDLE = 4,            /* handle not created by qw_model_create, or destroyed */
    QW_ALIGNMENT = 7,                 /* a weight or workspace pointer is not 16/256-byte aligned */
    QW_INTEGER_OVERFLOW = 8,          /* a size computed from the config overflows */
    QW_OUT_OF_MEMORY = 9,             /* workspace smaller than qw_workspace_bytes */
    QW_UNSUPPORTED_QUANTIZATION = 12, /* weight format unknown, or a dimension not a multiple of 32 */
    QW_UNSUPPORTED_SHAPE = 13,        /* dims outside what the kernels are built for (see qw_config) */
    QW_CONTEXT_EXCEEDED = 14,         /* the step would pass max_ctx; the cache is left unchanged */
    QW_NUMERICAL_FAILURE = 18,        /* non-finite logits were produced */
    QW_INTERNAL_INVARIANT = 20,       /* a device-side bounded wait expired; the model must be reset */
    QW_CUDA_ERROR = 21                /* a CUDA runtime call failed (no device, launch failure ...) */
};

/* Weight storage of the seven projection matrices (q, k, v, o, gate, up, down). */
enum qw_weight_format {
    QW_W_BF16 = 0,      /* bf16 [out, in] row-major */
    QW_W_INT8_G32 = 1,  /* int8 codes [out, in] + fp16 scales [out, in/32]; w = f32(q) * f32(s)
                           ("Scalar-Native ...", section 3 "Mixed-Q8 Quantization Definition") */
    QW_W_Q8Q8 = 2       /* weights as QW_W_INT8_G32; every projection's input is quantized per
                           32-element block at run time (d = amax/127, codes round-half-away(a/d)
                           clamped to +-127, scale fp16(d)) and each block contributes
                           f32(i32 dot of the codes) * f32(s_w) * f32(s_a) ("Real-Browser WASM Qwen3
                           Execution", section 5 "Q8_0 Mixed-Precision Matrix Multiplication").
                           Prompts run through the decode path one token at a time; batches
                           (qw_batch_*) are not available for this format. */
};

/*
 * Element type of the K/V cache.  The reference keeps K and V in f32
 * ("Scalar-Native ...", section 6 "Extents and Bytes Formulas"); bf16 halves the
 * cache and its per-token read traffic at the cost of rounding every stored
 * row (about 3e-3 relative L2 on the residual stream after a few hundred
 * freshly computed positions).
 */
enum qw_kv_format {
    QW_KV_F32 = 0,
    QW_KV_BF16 = 1
};

/*
 * Model dimensions.  The decode kernel is built for the Qwen3-0.6B decoder block
 * ("M1 - Load the weights", the layer tensor table): hidden 1024, n_heads 16,
 * n_kv_heads 8, head_dim 128, intermediate 3072.  Free: 1 <= n_layers <= 64,
 * vocab >= 1, 1 <= max_ctx <= 131072, rms_eps (the RMSNorm epsilon, 1e-6 for
 * Qwen3) and rope_theta (the RoPE base, 1e6 for Qwen3).  Any other block returns
 * QW_UNSUPPORTED_SHAPE (QW_UNSUPPORTED_QUANTIZATION when a dimension is not a
 * multiple of 32).
 */
typedef struct {
    int32_t n_layers;
    int32_t hidden;
    int32_t n_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t intermediate;
    int32_t vocab;
    float rms_eps;
    double rope_theta;
    int32_t max_ctx;
    int32_t weight_format; /* enum qw_weight_format */
    int32_t kv_format;     /* enum qw_kv_format */
} qw_config;

/* Matrix slots of qw_layer_weights.w / .s, in checkpoint order. */
enum { QW_Q = 0, QW_K = 1, QW_V = 2, QW_O = 3, QW_GATE = 4, QW_UP = 5, QW_DOWN = 6 };

/*
 * One decoder block's device pointers ("M1 - Load the weights", the 11-tensor
 * block).  Norm weights are bf16 vectors: input_norm and post_norm [hidden],
 * q_norm and k_norm [head_dim].  w[i] is the matrix [out, in] row-major
 * (bf16, or int8 for QW_W_INT8_G32); s[i] its fp16 scales [out, in/32] for
 * QW_W_INT8_G32, else ignored.  Every pointer must be 16-byte aligned.
 */
typedef struct {
    const void *input_norm;
    const void *q_norm;
    const void *k_norm;
    const void *post_norm;
    const void *w[7];
    const void *s[7];
} qw_layer_weights;

/*
 * Whole-model weight table.  embed: bf16 [vocab, hidden] (device);
 * final_norm: bf16 [hidden]; lm_head: bf16 [vocab, hidden] or NULL for a head
 * tied to embed; layers: HOST array of n_layers entries (copied at create).
 */
typedef struct {
    const void *embed;
    const void *final_norm;
    const void *lm_head;
    const qw_layer_weights *layers;
} qw_weights;

/*
 * Bytes of device workspace the model needs: the K/V cache
 * [n_layers][n_kv_heads][max_ctx][head_dim] twice (f32 or bf16 elements), the RoPE table, decode
 * activations and split-attention partials, prefill activations for up to
 * min(max_ctx, 2048) rows, f32 logits [vocab] and bookkeeping.  Returns 0 for
 * an invalid or unsupported config.
 */
size_t qw_workspace_bytes(const qw_config *cfg);

/*
 * Create a model over borrowed weights and a caller-allocated device
 * workspace (256-byte aligned, at least qw_workspace_bytes(cfg) bytes).
 * cuda_stream is a cudaStream_t (NULL = the legacy default stream); every
 * later call is ordered on it.  Validates everything before touching the
 * device; fills the RoPE table and clears the bookkeeping.  On success
 * *out receives the handle and the K/V length is 0.
 */
int qw_model_create(const qw_config *cfg, const qw_weights *weights, void *workspace, size_t workspace_bytes,
                    void *cuda_stream, qw_model **out);

/*
 * Prefill: run n prompt tokens (host array of ids in [0, vocab)) at positions
 * len .. len+n-1, appending their K/V.  The logits and greedy pick of the last
 * prompt position become the model's "last" result (qw_logits; the device-side
 * token that qw_decode_step(-1) consumes).  If next_token_host is not NULL the
 * call waits and writes the greedy pick there.  n == 0 is a no-op.
 * QW_CONTEXT_EXCEEDED if len + n > max_ctx, with nothing changed.
 * The prompt runs in chunks of up to 2048 rows through tensor-core GEMMs and a
 * causal tensor-core attention ("Portable WebAssembly Runtime Architecture for
 * TinyRustLM", section "Prefill versus decode"), with fp16 operands and f32
 * accumulation; the weights were converted to fp16 in the workspace at creation.
 * If a weight does not fit fp16 the model falls back to the decode path, one
 * token at a time (a message on stderr says so).
 */
int qw_prefill(qw_model *m, const int32_t *tokens_host, int32_t n, int32_t *next_token_host);

/*
 * Decode one token at position len.  token >= 0 is fed as given; token == -1
 * feeds the greedy pick of the previous call (already on the device, no host
 * round trip).  If next_token_host is not NULL the call waits and writes this
 * step's greedy pick there; with NULL nothing waits.
 */
int qw_decode_step(qw_model *m, int32_t token, int32_t *next_token_host);

/*
 * Greedy generation of n tokens without host synchronisation: feeds `token`
 * (or the previous pick if -1), then each step's pick into the next.  The n
 * picks are written to tokens_dev (device int32 [n]) if not NULL.
 */
int qw_generate(qw_model *m, int32_t token, int32_t n, int32_t *tokens_dev);

/* Copy the f32 logits [vocab] of the last processed position to dst_dev (device); n must equal vocab. */
int qw_logits(qw_model *m, float *dst_dev, int64_t n);

/* Forget the cache: len = 0 (no memset; "Scalar-Native ...", section 6 "Cancellation and Reset").
 * Also clears a recorded device error. */
int qw_kv_reset(qw_model *m);

/* Current K/V length (number of processed positions). */
int qw_kv_length(const qw_model *m, int32_t *out);

/* Wait for the stream and report any device-side error recorded since the last check. */
int qw_sync(qw_model *m);

/* Release the handle (the caller's device buffers are untouched). NULL is allowed. */
void qw_model_destroy(qw_model *m);

/* ---------------------------------------------------------- batched decode */

/*
 * A batch: up to 8 independent sequences of one model, each with its own K/V cache
 * and length, decoded together one token per sequence per step ("Portable WebAssembly
 * Runtime Architecture for TinyRustLM", sections "Threads, Scheduling" and "Prefill
 * versus decode"; each sequence computes exactly the decode step of the single-sequence
 * calls).  The B rows of a step run through skinny projections that read every weight
 * row once for all B rows (the batched prefill's fp16 weight copy, f32 accumulation),
 * per-sequence split attention over each cache, and one pass of the tied lm_head for
 * all rows; the cache uses the model's format.  Requires the batched prefill
 * (qw_prefill's tensor-core path, which holds that weight copy) to be available and
 * query heads = 2 x KV heads, hidden, query heads x head_dim and intermediate each one
 * of 1024, 2048, 3072, 4096, 6144 (else QW_UNSUPPORTED_SHAPE); max_ctx <= the model's
 * max_ctx.
 *
 * Workspace: caller-owned device memory of qw_batch_workspace_bytes (256-byte aligned),
 * holding every sequence's cache ([n_layers][n_kv_heads][max_ctx][head_dim] K and V
 * blocks), logits [max_batch][vocab] and step scratch.  Calls are stream-ordered on the
 * model's stream and share the model's prefill scratch: do not run batch calls and the
 * model's own calls concurrently from several threads.  A batch becomes invalid when
 * its model is destroyed.
 */
typedef struct qw_batch qw_batch;
enum { QW_BATCH_MAX = 8 };

/* Bytes of device workspace for a batch; 0 for an invalid model or sizes. */
size_t qw_batch_workspace_bytes(const qw_model *m, int32_t max_batch, int32_t max_ctx);
int qw_batch_create(qw_model *m, int32_t max_batch, int32_t max_ctx, void *workspace_dev, size_t workspace_bytes,
                    qw_batch **out);
void qw_batch_destroy(qw_batch *b);
/* Length of sequence seq <- 0 (seq = -1: every sequence, and a recorded device error is
 * cleared). */
int qw_batch_reset(qw_batch *b, int32_t seq);
int qw_batch_length(const qw_batch *b, int32_t seq, int32_t *out);
/* Append n prompt tokens to sequence seq through the batched prefill; its greedy pick
 * becomes the sequence's device-resident last token (and goes to *next_token_host if
 * given, which synchronises). */
int qw_batch_prefill(qw_batch *b, int32_t seq, const int32_t *tokens_host, int32_t n, int32_t *next_token_host);
/* One decode step of sequences 0 .. n_seq-1: tokens_host[s] is sequence s's input token,
 * or -1 (or tokens_host NULL for all) for its device-resident last pick.  Each sequence
 * appends one K/V row at its own length.  next_tokens_host [n_seq] (optional) receives
 * the greedy picks and synchronises; without it the call returns after launching.
 * QW_CONTEXT_EXCEEDED if any sequence is full; a non-finite logit sets
 * QW_NUMERICAL_FAILURE, reported by the next synchronising call, after which the batch
 * refuses work until qw_batch_reset(b, -1). */
int qw_batch_step(qw_batch *b, int32_t n_seq, const int32_t *tokens_host, int32_t *next_tokens_host);
/* f32 logits [n_seq][vocab] of the last step (device), n = n_seq * vocab. */
int qw_batch_logits(qw_batch *b, float *dst_dev, int64_t n);
/* f32 [n_layers + 1][n_seq][hidden] residual stream of the last step (the model's
 * QW_DEBUG_HIDDEN flag must have been set for that step). */
int qw_batch_debug_hidden(qw_batch *b, float *dst_dev, int64_t n);
/* Wait for the batch's work; returns a recorded device error. */
int qw_batch_sync(qw_batch *b);

/* -------------------------------------------------------- checkpoint files */

/*
 * Safetensors / SLM2 checkpoints ("Scalar-Native Qwen3 Reference Runtime As The
 * Numerical Authority", section 3 "File Layout and Safe Metadata Parsing"; "M1 - Load
 * the weights", sections "The loading stack" and "The safetensors format"):
 * [u64 little-endian N][N bytes of UTF-8 JSON][blob].  The JSON maps each tensor name
 * to {"dtype", "shape", "data_offsets": [begin, end]} (offsets into the blob), plus an
 * optional "__metadata__" object of strings.  dtypes: "BF16", "F16", "F32", "I8" and
 * "Q8_0" (SLM2's 34-byte blocks: an fp16 scale, then 32 int8 codes).
 *
 * qw_checkpoint_open parses and validates the header of a file held in host memory
 * (mapped or read by the caller; borrowed until qw_checkpoint_close).  bytes_len may
 * cover only the prefix and header (then the checks run but nothing is uploaded);
 * file_size is the whole file's size.  Every entry must satisfy, else
 * QW_INVALID_ARGUMENT with the reason in qw_checkpoint_last_error(): end <= blob size;
 * spans sorted by begin do not overlap; 8 + N + begin is a multiple of 8;
 * end - begin == the bytes of shape x dtype; a Q8_0 tensor holds whole 32-element
 * blocks; no duplicate names, unknown keys or dtypes, rank <= 4, nothing after the
 * header object.
 */
typedef struct qw_checkpoint qw_checkpoint;
enum qw_dtype { QW_DT_BF16 = 0, QW_DT_F16 = 1, QW_DT_F32 = 2, QW_DT_I8 = 3, QW_DT_Q8_0 = 4 };

int qw_checkpoint_open(const void *bytes, uint64_t bytes_len, uint64_t file_size, qw_checkpoint **out);
void qw_checkpoint_close(qw_checkpoint *c);
/* Reason of the last failed qw_checkpoint_* call of this thread ("" after a success). */
const char *qw_checkpoint_last_error(void);
/* Tensors in the file (-1 for an invalid handle); entry i (sorted by begin): name
 * (NUL-terminated, name_cap bytes available), dtype, rank, dims [4] (0-padded), blob
 * offsets.  Any output pointer may be NULL. */
int32_t qw_checkpoint_count(const qw_checkpoint *c);
int qw_checkpoint_tensor(const qw_checkpoint *c, int32_t i, char *name, int32_t name_cap, int32_t *dtype,
                         int32_t *rank, int64_t *dims, uint64_t *begin, uint64_t *end);

/*
 * Cross-check against the tensor set cfg implies ("M1 - Load the weights", section
 * "Deriving what should be there"): model.embed_tokens.weight [V,H],
 * model.norm.weight [H], an optional lm_head.weight [V,H] (a tied head may be absent or
 * shipped as a copy), and per layer input_layernorm [H], self_attn.{q,k,v}_proj
 * [n_heads*d or n_kv_heads*d, H], self_attn.{q,k}_norm [d], self_attn.o_proj
 * [H, n_heads*d], post_attention_layernorm [H], mlp.{gate,up}_proj [I,H],
 * mlp.down_proj [H,I].  Loadable dtypes: BF16 or F32 norm vectors, BF16 embedding and
 * head, and BF16 (QW_W_BF16) or Q8_0 (QW_W_INT8_G32) matrices.  Parameter counts:
 * stored = every tensor of the file; logical = a shipped head copy not counted.
 * Returns QW_OK when clean, QW_UNSUPPORTED_SHAPE when a tensor is missing, mis-shaped,
 * unexpected or of an unloadable dtype (the first such problem in first_problem).
 */
typedef struct {
    int32_t n_tensors, n_expected, n_found, n_missing, n_misshaped, n_unexpected, n_bad_dtype;
    int32_t lm_head_copy;
    int64_t stored_params, logical_params, embedding_params;
    char first_problem[256];
} qw_checkpoint_report;
int qw_checkpoint_check(const qw_checkpoint *c, const qw_config *cfg, qw_checkpoint_report *report);

/*
 * Device bytes qw_checkpoint_upload needs (0 on error).  The upload copies every tensor
 * of a clean checkpoint (with its blob in memory) into dst_dev (256-byte aligned): the
 * embedding, the final norm, a head only if it differs from the embedding (a byte-equal
 * copy is tied), and per layer the four norm vectors (F32 ones must be exactly
 * representable in bf16, else QW_UNSUPPORTED_QUANTIZATION) and the seven matrices
 * (BF16 as stored; Q8_0 split into int8 codes [out, in] and fp16 scales [out, in/32],
 * the same values).  It fills layers (a host array of n_layers entries) and *table for
 * qw_model_create, and synchronises cuda_stream before returning.
 */
size_t qw_checkpoint_upload_bytes(const qw_checkpoint *c, const qw_config *cfg);
int qw_checkpoint_upload(const qw_checkpoint *c, const qw_config *cfg, void *dst_dev, size_t dst_bytes,
                         qw_layer_weights *layers, qw_weights *table, void *cuda_stream);

/* ---------------------------------------------------------------- testing */

/*
 * Replace the cache with n_pos positions of bf16 K and V, each laid out
 * [n_layers][n_kv_heads][n_pos][head_dim] (device pointers); len = n_pos.
 * An f32 cache receives the exact widening of the bf16 values.  Used to start
 * decode from a pre-filled long context.
 */
int qw_kv_import(qw_model *m, const void *k_dev, const void *v_dev, int32_t n_pos);

/* Copy cache rows back, layout [n_layers][n_kv_heads][n_pos][head_dim], positions
 * [0, n_pos), in the cache's own element type (f32 or bf16). */
int qw_kv_export(qw_model *m, void *k_dev, void *v_dev, int32_t n_pos);

/*
 * Debug flags.  QW_DEBUG_HIDDEN: every decode step also stores the residual
 * stream after the embedding and after each layer, read by qw_debug_hidden.
 * QW_DEBUG_PREFILL_BY_TOKEN: qw_prefill runs the prompt through the decode
 * path one token at a time (the differential baseline of the batched prefill).
 * QW_DEBUG_TRACE: decode steps record a timeline (qw_debug_trace).
 * QW_DEBUG_ONE_GROUP: decode steps run with every SM in one group instead of one
 * group per die (the layout used where no two-die structure is measured; o_proj
 * and down then sum all columns in one dot product instead of two halves).
 * QW_DEBUG_WITHHOLD: the failure path's test.  In each decode step the first SM
 * of group 0 withholds its q|k|v rows of layer 0, and every device-side wait
 * gives up after 1 ms instead of 1 s, so the step ends with
 * QW_INTERNAL_INVARIANT (every CTA returns on its own; nothing faults or hangs).
 * The model then refuses every call with that status until qw_kv_reset.
 */
enum {
    QW_DEBUG_HIDDEN = 1,
    QW_DEBUG_PREFILL_BY_TOKEN = 2,
    QW_DEBUG_TRACE = 4,
    QW_DEBUG_ONE_GROUP = 8,
    QW_DEBUG_WITHHOLD = 16
};
int qw_set_debug(qw_model *m, int32_t flags);

/*
 * f32 [n_layers+1][hidden] residual stream of the last processed position (needs
 * QW_DEBUG_HIDDEN): the last decode step, or the last row of the last prefill.
 */
int qw_debug_hidden(qw_model *m, float *dst_dev, int64_t n);

/*
 * Timeline of the last decode step (needs QW_DEBUG_TRACE): uint64 %globaltimer
 * nanoseconds [phase][cta][16], phase = 5*layer + {0 QKV, 1 attention, 2 o_proj,
 * 3 gate/up, 4 down} and 5*n_layers for the head; stamps 0..3 = consumer entering
 * the phase, its inputs arrived, inputs staged (compute starts), phase done; 4, 5 =
 * producer's first and last copy issue of the phase; 6, 7 = row phases: weight chunks
 * taken, compute done; attention: cached chunks done, merge inputs arrived; 8..14 =
 * SM clock cycles (clock64, comparable within one CTA only) of the first consumer warp
 * in the row phases: 13 compute entered, 8 weights and activation in registers, 9 its
 * rows reduced and stored, 11 further rows done, 12 chunks released, 14 phase done
 * (0 where a stamp does not apply).
 * n must equal QW_QUERY_TRACE_LEN.
 */
int qw_debug_trace(qw_model *m, uint64_t *dst_dev, int64_t n);

/* Integer facts about a created model: CTAs of a decode step, timeline length, workspace
 * bytes, SM groups of the decode step (2 = one per die, 1 = none measured), CTAs in group 0,
 * the measured same-die and cross-die ping-pong round trips in ns (0 when one group), and
 * where the decode step's exchange pages sit in the workspace. */
enum {
    QW_QUERY_DECODE_CTAS = 1,
    QW_QUERY_TRACE_LEN = 2,
    QW_QUERY_WORKSPACE_BYTES = 3,
    QW_QUERY_DECODE_GROUPS = 4,
    QW_QUERY_GROUP0_CTAS = 5,
    QW_QUERY_RT_NEAR_NS = 6,
    QW_QUERY_RT_FAR_NS = 7,
    QW_QUERY_XREGION_OFFSET = 8  /* byte offset of the exchange pages in the workspace (tests) */
};
int qw_query(const qw_model *m, int32_t what, int64_t *out);

/*
 * One decode step with no device allocation (the reference pages have no
 * counterpart; this entry point exists for callers that cannot allocate device
 * memory when they decode, e.g. code running inside another framework's memory
 * pool or under a fixed memory budget, where a cudaMalloc would fail or stall the
 * device).  No handle and no workspace: the caller passes the config, the weight
 * table, the K/V cache planes, the position pos, the input token id, and device
 * outputs logits_dev and next_token_dev.  The caller's buffers must be:
 *   k_cache, v_cache: device, n_layers * n_kv_heads * max_ctx * head_dim elements
 *     each, of the element type cfg->kv_format names (f32 or bf16), laid out
 *     [n_layers][n_kv_heads][max_ctx][head_dim]; rows [0, pos) hold earlier
 *     positions, row pos is written;
 *   logits_dev: device f32 [vocab]; next_token_dev: device int32 (the greedy pick).
 * The library cannot see the sizes of these buffers; smaller ones are read and
 * written out of bounds.  Every other buffer lives in one fixed 4 MiB array in the
 * library's device memory, which holds configs of up to 64 layers; a larger
 * need returns QW_OUT_OF_MEMORY with a message on stderr.  The library calls no
 * allocating routine here.  The first call on a device sets the array up: it looks
 * up the array's device address, zeroes it, and measures which SMs and which of the
 * array's 4 KB pages sit on which die of the GPU (a few short kernels, about 20 ms,
 * waited for); that first call must come before any stream capture.  The array is
 * shared by all calls on a device and keeps the last call's contents (flags, keys
 * and counters are zeroed by every call), so calls that overlap on the GPU race:
 * serialise them.  The call waits for the stream after copying the layer table and
 * the RoPE row; with wait != 0 it also waits for the step and returns any
 * device-side error.  The step runs the same kernel with the same SM groups as a
 * model created on the same device, so the two give identical results.
 */
int qw_decode_step_noalloc(const qw_config *cfg, const qw_weights *weights, void *k_cache, void *v_cache,
                           int32_t pos, int32_t token, float *logits_dev, int32_t *next_token_dev,
                           void *cuda_stream, int32_t wait);

/*
 * On-device sampling ("Portable WebAssembly Runtime Architecture for TinyRustLM",
 * sections "Sampling order" and "Deterministic sampling contract"; repetition
 * penalty of "Scalar-Native Qwen3 Reference Runtime ...", section 7).  Order:
 * repetition penalty (each distinct history token once: positive logit / penalty,
 * negative * penalty), NaN -> -inf, -0 -> +0; temperature 0 takes the greatest logit
 * (lowest id on ties) and draws nothing; otherwise logits / temperature, top-k by
 * descending value then ascending id, max-shifted probabilities over the survivors,
 * the minimal prefix whose cumulative probability reaches top_p, renormalised, and
 * one PCG32 word u = (w >> 8) * 2^-24 picks the first candidate whose cumulative
 * probability exceeds u.
 */
enum { QW_SAMPLE_MAX_TOP_K = 64 };
typedef struct {
    float temperature;        /* >= 0, finite; 0 = greedy */
    int32_t top_k;            /* 1 .. QW_SAMPLE_MAX_TOP_K (and <= vocab) when temperature > 0 */
    float top_p;              /* (0, 1]; 1 keeps every top-k survivor */
    float repetition_penalty; /* > 0, finite; 1 = off */
} qw_sampling;

/* Device scratch bytes qw_sample_logits needs for a vocabulary of this size. */
size_t qw_sample_scratch_bytes(int32_t vocab);

/*
 * Sample one token from device f32 logits [vocab] (not modified).  history_dev:
 * device int32 token ids [n_history] for the repetition penalty (may be NULL when
 * n_history == 0).  rng_dev: device uint64 [2] = PCG32 (state, increment), advanced
 * by one word when temperature > 0.  token_dev: device int32 result, -1 when nothing
 * can be drawn (every logit masked) or a history id is out of range.  scratch_dev:
 * qw_sample_scratch_bytes(vocab) device bytes, 256-byte aligned.  Stream-ordered on
 * cuda_stream; returns after enqueueing (QW_INVALID_ARGUMENT for bad parameters).
 */
int qw_sample_logits(const float *logits_dev, int32_t vocab, const int32_t *history_dev, int32_t n_history,
                     const qw_sampling *params, uint64_t *rng_dev, int32_t *token_dev, void *scratch_dev,
                     size_t scratch_bytes, void *cuda_stream);

/* Seed the model's sampler: PCG32 state 0, increment (stream << 1) | 1, advance, add
 * seed, advance (the pages' seeding).  Stream-ordered. */
int qw_sampler_seed(qw_model *m, uint64_t seed, uint64_t stream);

/* The model's PCG32 (state, increment) after every enqueued call (waits for the stream). */
int qw_sampler_state(qw_model *m, uint64_t *state_host);

/*
 * Sample the next token from the logits of the last processed position with the
 * model's sampler.  The pick becomes the device-resident token that
 * qw_decode_step(-1) consumes; with next_token_host != NULL the call waits and
 * writes it there.  A device-side failure (nothing drawable, a history id out of
 * range) is reported by the next call that waits.
 */
int qw_sample(qw_model *m, const qw_sampling *params, const int32_t *history_dev, int32_t n_history,
              int32_t *next_token_host);

/*
 * Test entry of the tensor-core GEMM the prefill uses: C = A B^T with A fp16
 * [M, K], B fp16 [N, K] (row-major, K contiguous) and C f32 [M, N], all device
 * pointers, 16-byte aligned.  K must be a multiple of 64, N of the tile width bn
 * (128 or 256).  Waits for cuda_stream and returns QW_OK, QW_INTERNAL_INVARIANT
 * (a bounded wait inside the kernel expired) or QW_CUDA_ERROR.
 */
int qw_debug_gemm_f16(const void *a_dev, const void *b_dev, float *c_dev, int32_t M, int32_t N, int32_t K,
                      int32_t bn, void *cuda_stream);

/* Static text for a status code. */
const char *qw_status_string(int status);

/* ABI version the library was built with (QW_ABI_VERSION). */
int32_t qw_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QW_H */
