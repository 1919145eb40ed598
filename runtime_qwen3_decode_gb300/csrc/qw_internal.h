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

// Persistent decode kernel geometry: 7 consumer warps + 1 producer warp per CTA (8
// warps: two per SM sub-partition, so a thread may use up to 255 registers), one CTA
// per SM, a ring of shared-memory slots filled by bulk async copies.
constexpr int kConsumerWarps = 7;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kDecodeThreads = kConsumerThreads + 32;
constexpr int kSlotBytes = 32768;
constexpr int kSlots = 6;
// Cached positions per attention slot: one pass of 4 positions per consumer warp for
// f32 rows (512 B), two passes for bf16 rows; K rows then V rows at half the slot.
__host__ __device__ constexpr int kv_chunk_rows(int elem_bytes) { return 4 * kConsumerWarps * (4 / elem_bytes); }
constexpr int kPartStride = kHeadDim + 4;    // split-attention partial: acc[128], max, sum, 2 pad (16-B rows)
constexpr int kMaxOwnRows = 64;             // residual rows per CTA kept in shared memory
constexpr int kMaxKvHeads = 32;             // split-merge counters per layer
constexpr int kMaxSplits = 21;              // attention splits per KV head (3 per consumer warp in the merge)
// Cached-row chunks per attention split.  A split streams its chunks through the
// CTA's ring back to back; every extra split adds a tagged partial that the merge
// must wait for, so splits are only worth it once a split's own stream takes longer
// than that round trip.
constexpr int kSplitChunks = 2;
// Attention splits for a step at position pos: kSplitChunks chunks of cached rows per
// split, at most one split per CTA and KV head, at most kMaxSplits.
inline int attn_splits(int pos, int kv_elem_bytes, int ncta, int n_kv_heads) {
    const int ch = kv_chunk_rows(kv_elem_bytes) * kSplitChunks;
    int s = (pos + ch - 1) / ch;
    const int cap = ncta / n_kv_heads < kMaxSplits ? ncta / n_kv_heads : kMaxSplits;
    if (s > cap) s = cap;
    if (s > pos) s = pos;
    if (s < 1) s = 1;
    return s;
}

// Debug timeline stamps per (phase, CTA): consumer before wait, after wait, after
// compute, after arrive; producer first issue, last issue of the phase.
constexpr int kTraceStamps = 8;

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
    // tagged exchange words (tag << 32 | f32 bits) between phases
    unsigned long long *xa;          // residual after down [H]
    unsigned long long *xb;          // residual after o_proj [H]
    unsigned long long *qkvt;        // [(Hq + 2 Hkv) * 128]
    unsigned long long *actt;        // SwiGLU output [I]
    unsigned long long *partt;       // split-attention partials [Hkv][S][G][kPartStride]
    unsigned long long *ot;          // attention output, the merged partials [Hq * 128]
    unsigned *merge;                 // finished splits per (layer, KV head) [L][kMaxKvHeads]; the
                                     // merging CTA sets its counter back to 0
    float *logits;                   // [V]
    float *hidden;                   // [(L + 1) H] debug dump
    unsigned *sync;                  // arrivals per phase [5L+1]; each step adds the CTA count
    unsigned target;                 // arrivals that mean "this step's phase is done" (steps * CTAs)
    unsigned long long *key;         // packed argmax keys [2], one per step parity
    StepFlags *flags;
    int *tok_out;                    // optional device slot for this step's greedy pick
    unsigned long long *trace;       // debug timeline [phase][cta][kTraceStamps] (%globaltimer ns) or null
    // step
    int pos, token, n_split, debug;
    unsigned step;                   // step sequence number (never 0 after creation)
    unsigned tag_base;               // step * 512: tags of this step are tag_base + phase + 1
};

// Step bookkeeping: two argmax keys then the per-phase arrival counters (zeroed at
// creation, by qw_kv_reset and when the counters would overflow).
inline size_t step_block_bytes(int L) { return 16 + 4 * ((size_t)kPhasesPerLayer * L + 1); }
inline size_t merge_block_bytes(int L) { return 4 * (size_t)kMaxKvHeads * L; }

size_t decode_smem_bytes();
cudaError_t decode_prepare(int group, int *blocks_per_sm);
cudaError_t launch_decode(const DecodeArgs &a, int group, int ncta, cudaStream_t stream);
// Widen bf16 K/V rows [heads][n_pos][128] into an f32 cache [heads][max_ctx][128].
cudaError_t launch_kv_widen(const __nv_bfloat16 *src, float *dst, long long heads, int n_pos, int max_ctx,
                            cudaStream_t stream);

}  // namespace qw
