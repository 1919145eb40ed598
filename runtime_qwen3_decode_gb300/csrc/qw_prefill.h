// qw_prefill.h - batched prefill path (tensor-core GEMMs + causal attention).
#pragma once

#include "qw.h"
#include "qw_internal.h"

namespace qw {

struct PrefillImpl;

struct PrefillState {
    uint8_t *buf;      // prefill region of the model workspace: fp16 weights + activations
    size_t bytes;
    int rows_max;      // prompt rows per chunk
    int nsm;
    int ready;         // batched path available
    PrefillImpl *impl;
};

size_t prefill_workspace_bytes(const qw_config &c, int rows_max);
// Sets kernel attributes and loads the tensor-map encoder; called once per model creation.
cudaError_t prefill_prepare();
// Converts the layer weights to fp16 in buf and encodes their tensor maps (stream-ordered,
// synchronises once).  Returns non-zero on a CUDA failure; ready stays 0 (token-by-token
// prefill) when a weight does not fit fp16.
int prefill_init(PrefillState *st, const qw_config &c, const DevLayer *host_layers, const float2 *rope, uint8_t *buf,
                 size_t bytes, int rows_max, int nsm, cudaStream_t stream);
void prefill_destroy(PrefillState *st);
inline bool prefill_supported(const PrefillState &st) { return st.ready != 0; }
// Runs n prompt tokens at positions pos0.. and leaves logits + greedy pick of the last row
// (flags->next_tok); debug bit 1 dumps the last row's hidden state after every layer.
int prefill_run(PrefillState *st, const DecodeArgs &a, int pos0, const int32_t *tokens_host, int n, int debug,
                cudaStream_t stream);
// One batched decode step: B sequences, one new token each (their tokens resolved on the device:
// -1 takes the sequence's previous pick).  Sequence b's cache is the block of seq_elems elements
// starting seq_elems * b after kc / vc ([L][Hkv][max_ctx][128]); its new row goes to position
// row_pos[b].  The B rows run through the skinny projections (every fp16 weight row of the
// prefill's converted copy read once for all B rows), the batched attention and the head
// kernels of batch.cu; logits [B][V] and picks [B] come out.
struct BatchStep {
    int B;
    const int32_t *tokens_in;  // device [B]: token or -1
    int32_t *tokens;           // device [B] scratch: the resolved tokens
    const int *row_pos;        // device [B]
    int max_n;                 // the longest sequence's cached positions after this step's row
    void *kc, *vc;
    size_t seq_elems;
    int max_ctx;
    float *part;               // attention partials [B][Hq][splits][132]
    float *logits;             // [B][V]
    unsigned long long *keys;  // [B], zero
    int32_t *picks;            // [B] in (previous picks) and out
    float *hidden;             // optional [L + 1][B][H] residual stream dump
};
int prefill_batch_step(PrefillState *st, const DecodeArgs &a, const BatchStep &bs, cudaStream_t stream);

// C = A B^T with fp16 A [M,K], B [N,K] and f32 C [M,N] through the tensor-core GEMM (tests).
int prefill_debug_gemm(const void *a, const void *b, float *c, int M, int N, int K, int bn, cudaStream_t stream);

}  // namespace qw
