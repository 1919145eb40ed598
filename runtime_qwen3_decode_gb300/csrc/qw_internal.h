// qw_internal.h - structures shared by the host ABI (qw_api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qw {

constexpr int kHeadDim = 128;
constexpr int kMaxLayers = 64;
constexpr int kPhasesPerLayer = 5;  // QKV, ATTN, OPROJ, GATEUP, DOWN; then one LMHEAD phase per step
enum { PH_QKV = 0, PH_ATTN = 1, PH_OPROJ = 2, PH_GATEUP = 3, PH_DOWN = 4 };

// Persistent decode kernel geometry: 8 consumer warps + 1 producer warp per CTA,
// one CTA per SM, a ring of shared-memory slots filled by bulk async copies.
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kDecodeThreads = kConsumerThreads + 32;
constexpr int kSlotBytes = 32768;
constexpr int kSlots = 6;
constexpr int kPartStride = kHeadDim + 2;    // split-attention partial: acc[128], max, sum

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // every device-side wait gives up after 1 s

// Status values written by device code (same numbers as qw.h).
constexpr unsigned kErrInvalidArgument = 1;
constexpr unsigned kErrNumerical = 18;
constexpr unsigned kErrInvariant = 20;

struct DevLayer {
    const __nv_bfloat16 *input_norm, *q_norm, *k_norm, *post_norm;
    const void *w[7];      // q, k, v, o, gate, up, down: bf16 or int8 [out, in]
    const __half *s[7];    // fp16 scales [out, in/32] (int8 format)
};

// Error word, abort flag and the device-resident greedy token, read back together.
struct StepFlags {
    unsigned err;
    unsigned abort;
    int next_tok;
    int pad;
};

struct DecodeArgs {
    // dims
    int L, H, Hq, Hkv, I, V, max_ctx, fmt;
    float eps;
    // weights
    const DevLayer *layers;          // device [L]
    const __nv_bfloat16 *embed;      // [V, H]
    const __nv_bfloat16 *lm_head;    // [V, H]
    const __nv_bfloat16 *final_norm; // [H]
    // state (workspace)
    void *kc, *vc;                   // [L][Hkv][max_ctx][128] of f32 (kv_f32) or bf16
    int kv_f32;
    const float2 *rope;              // [max_ctx][64] (cos, sin)
    float *x;                        // residual [H]
    float *qkv;                      // [(Hq + 2 Hkv) * 128]
    float *o;                        // attention output [Hq * 128]
    float *act;                      // SwiGLU output [I]
    float *part;                     // split partials [Hkv][S][G][kPartStride]
    float *logits;                   // [V]
    float *hidden;                   // [(L + 1) H] debug dump
    unsigned *sync;                  // per-step counters: phases [5L+1], attention merges [L*Hkv], zeroed per step
    unsigned long long *key;         // packed argmax key, zeroed per step
    StepFlags *flags;
    int *tok_out;                    // optional device slot for this step's greedy pick
    // step
    int pos, token, n_split, debug;
    int phase_begin, phase_end;
};

// Size of the per-step bookkeeping block (counters + key), zeroed before each decode step.
inline size_t step_block_bytes(int L, int Hkv) {
    size_t counters = (size_t)kPhasesPerLayer * L + 1 + (size_t)L * Hkv;
    return ((counters * 4 + 7) / 8) * 8 + 8;
}

size_t decode_smem_bytes();
cudaError_t decode_prepare(int group, int *blocks_per_sm);
cudaError_t launch_decode(const DecodeArgs &a, int group, int ncta, cudaStream_t stream);
// Widen bf16 K/V rows [heads][n_pos][128] into an f32 cache [heads][max_ctx][128].
cudaError_t launch_kv_widen(const __nv_bfloat16 *src, float *dst, long long heads, int n_pos, int max_ctx,
                            cudaStream_t stream);

}  // namespace qw
