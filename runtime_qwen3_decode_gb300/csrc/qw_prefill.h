// qw_prefill.h - batched prefill path (tensor-core GEMMs + causal attention).
#pragma once

#include "qw.h"
#include "qw_internal.h"

namespace qw {

struct PrefillState {
    uint8_t *buf;      // prefill activations inside the model workspace
    size_t bytes;
    int rows_max;      // prompt rows per chunk
    int nsm;
    int ready;         // batched path available
};

size_t prefill_workspace_bytes(const qw_config &c, int rows_max);
cudaError_t prefill_prepare();
void prefill_init(PrefillState *st, const DecodeArgs &a, uint8_t *buf, size_t bytes, int rows_max, int nsm);
inline bool prefill_supported(const PrefillState &st) { return st.ready != 0; }
// Runs n prompt tokens at positions pos0.. and leaves logits + greedy pick of the last row.
int prefill_run(PrefillState *st, const DecodeArgs &a, int pos0, const int32_t *tokens_host, int n,
                cudaStream_t stream);

}  // namespace qw
