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
int prefill_init(PrefillState *st, const qw_config &c, const DevLayer *host_layers, uint8_t *buf, size_t bytes,
                 int rows_max, int nsm, cudaStream_t stream);
void prefill_destroy(PrefillState *st);
inline bool prefill_supported(const PrefillState &st) { return st.ready != 0; }
// Runs n prompt tokens at positions pos0.. and leaves logits + greedy pick of the last row
// (flags->next_tok); debug bit 1 dumps the last row's hidden state after every layer.
int prefill_run(PrefillState *st, const DecodeArgs &a, int pos0, const int32_t *tokens_host, int n, int debug,
                cudaStream_t stream);
// C = A B^T with fp16 A [M,K], B [N,K] and f32 C [M,N] through the tensor-core GEMM (tests).
int prefill_debug_gemm(const void *a, const void *b, float *c, int M, int N, int K, int bn, cudaStream_t stream);

}  // namespace qw
