// qw_sample.h - on-device sampling (sample.cu).
#pragma once

#include "qw_internal.h"

namespace qw {

constexpr int kSampleMaxTopK = 64;  // top-k candidates a sampled step may keep (QW_SAMPLE_MAX_TOP_K)

// Device scratch (bytes) of one sampling launch over a vocabulary of V tokens.
size_t sample_scratch_bytes(int V);
// Stream-ordered sampling of f32 logits [V] (see sample.cu for the order of steps).
// rng: device (state, increment), advanced by one word for temperature > 0.  token:
// optional device int32 (-1 when nothing can be drawn); next_tok: optional device slot
// that also receives a valid pick; err: optional device error word (first error wins).
cudaError_t launch_sample(const float *logits, int V, const int32_t *hist, int n_hist, float temperature,
                          int top_k, float top_p, float penalty, uint64_t *rng, int32_t *token, int32_t *next_tok,
                          unsigned *err, void *scratch, cudaStream_t stream);

}  // namespace qw
