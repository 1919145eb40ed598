// qw_batch.h - batched decode: B sequences, one new token each per step.
#pragma once

#include <cuda_fp16.h>

#include "qw_internal.h"

namespace qw {

constexpr int kBatchMax = 8;            // sequences per batched step
constexpr int kBatchG = 2;              // query heads per KV head (the Qwen3-0.6B block)
constexpr int kBatchPartStride = 132;   // floats per attention partial: acc[128], max, sum, pad
constexpr int kBatchHeadThreads = 256;
constexpr int kBatchSplitRows = 32;     // cached positions per attention split (at most, up to 64 splits)
constexpr int kBatchMaxSplits = 64;

// Skinny projection of the B rows: y[b][r] = sum_k W[r][k] a[b][k] (bgemv_kernel).
enum { BG_STORE = 0, BG_ADD = 1, BG_SWIGLU = 2 };

struct BatchGemv {
    const __half *W;       // [rows][K] fp16; BG_SWIGLU: gate/up rows interleaved in 128-row blocks
    const __half *a;       // [B][K] fp16 activation rows, or null: RMSNorm of x below
    const float *x;        // with a == null: [B][K] f32 residual rows, staged as fp16(w (x r))
    const __nv_bfloat16 *norm_w;  //   r = rsqrt(mean(x^2) + eps), the norm_rows kernel's arithmetic
    float eps;
    int B, N, K;           // N outputs (BG_STORE / BG_ADD: even); K in {1024, 2048, 3072, 4096, 6144}
    float *out;            // BG_STORE: out[b][n] = y; BG_ADD: out[b][n] += y
    int ldo;
    __half *act;           // BG_SWIGLU: act[b][n] = silu(gate_n . a_b) (up_n . a_b)
    int ldh;
};

// QK-Norm, RoPE and the K/V append of the B rows' raw q|k|v projections (bqkv_post_kernel).
struct BatchQkvPost {
    const float *qkv;                        // [B][Hq 128 + 2 Hkv 128]
    const __nv_bfloat16 *q_norm, *k_norm;    // [128] each
    const float2 *rope;                      // [max positions][64] (cos, sin)
    const int *row_pos;                      // [B] each sequence's position this step
    int B, Hq, Hkv;
    float eps;
    __half *q16;                             // [Hq][q_rows][128]: row b = sequence b's query heads
    int q_rows;
    void *kc, *vc;                           // this layer's planes of sequence 0: [Hkv][max_ctx][128]
    size_t seq_elems;                        // elements from one sequence's cache to the next one's
    int max_ctx;
};

struct BatchAttn {
    const __half *q16;    // [Hq][q_rows][128]: row b = sequence b's rotated query heads
    int q_rows;
    const void *kc, *vc;  // this layer's planes of sequence 0: [Hkv][max_ctx][128] (f32 or bf16)
    size_t seq_elems;     // elements from one sequence's cache to the next one's
    int max_ctx;
    const int *row_pos;   // [B] this step's position of each sequence (its row is cached already)
    int S, Hq;            // splits per (sequence, KV head); query heads
    float scale_log2;     // log2(e) / sqrt(head_dim)
    float *part;          // [B][Hq][S][kBatchPartStride]
};

struct BatchHead {
    const float *x;                 // [B][H] residual stream after the last layer
    const __nv_bfloat16 *final_norm, *E;
    int B, V;
    float eps;
    float *logits;                  // [B][V]
    unsigned long long *keys;       // [B] packed argmax keys, zero on entry (left zero)
    int32_t *picks;                 // [B] greedy picks out
    StepFlags *flags;
};

cudaError_t batch_prepare();
// chained: launch with programmatic stream serialization (the previous operation of the
// stream must be a kernel); every batched kernel waits for its predecessor's completion
// before its first memory access.
cudaError_t launch_bgemv(int epi, const BatchGemv &p, int nsm, cudaStream_t st, bool chained);
// Row lengths the skinny projection is built for (launch_bgemv refuses the others).
inline bool bgemv_supported(int K) { return K == 1024 || K == 2048 || K == 3072 || K == 4096 || K == 6144; }
cudaError_t launch_bqkv_post(const BatchQkvPost &p, int kv_f32, cudaStream_t st, bool chained);
cudaError_t launch_batch_tokens(const int32_t *in, const int32_t *picks, int B, int32_t *tokens, cudaStream_t st,
                                bool chained);
cudaError_t launch_batch_attn(const BatchAttn &p, int Hkv, int B, int kv_f32, cudaStream_t st, bool chained);
cudaError_t launch_batch_merge(const float *part, int S, int Hq, int B, __half *o16, int ldo, cudaStream_t st,
                               bool chained);
cudaError_t launch_batch_head(const BatchHead &p, int H, int nsm, cudaStream_t st, bool chained);

// Splits per (sequence, KV head) for a step whose longest sequence caches n positions: at
// most kBatchSplitRows positions per split, the count rounded up to a power of two so that
// the step's captured graph (one per split count) changes only when n doubles.
inline int batch_splits(int n) {
    const int need = (n + kBatchSplitRows - 1) / kBatchSplitRows;
    int s = 1;
    while (s < need && s < kBatchMaxSplits) s *= 2;
    return s;
}

}  // namespace qw
