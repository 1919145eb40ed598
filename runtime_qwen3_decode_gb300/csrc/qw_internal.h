// qw_internal.h - structures shared by the host ABI (qw_api.cu, noalloc.cu), the GPU
// topology probe (topology.cu) and the kernels.
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

// The decoder block the decode kernel is built for: the Qwen3-0.6B block ("M1 - Load the
// weights", the layer-0 tensor table): hidden 1024, 16 query heads and 8 KV heads of 128,
// SwiGLU width 3072.  Layer count, vocabulary, context, epsilon and RoPE base are free.
constexpr int kBlockH = 1024, kBlockHq = 16, kBlockHkv = 8, kBlockI = 3072, kBlockG = kBlockHq / kBlockHkv;

// Persistent decode kernel geometry: 7 consumer warps + 1 producer warp per CTA (two warps per
// SM sub-partition, so up to 255
// registers a thread, enough to hold a warp's weight rows of a phase), one CTA per SM, a ring
// of shared-memory slots filled by bulk async copies.
constexpr int kConsumerWarps = 7;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kDecodeThreads = kConsumerThreads + 32;
constexpr int kSlotBytes = 32768;
constexpr int kSlots = 6;
// Cached positions per attention chunk: 16 lanes per position, so one pass covers 2 positions
// per consumer warp; f32 rows (512 B) take one pass per chunk, bf16 rows two.  K rows then V
// rows at half the slot, with room for one more row (the step's own position).
__host__ __device__ constexpr int kv_chunk_rows(int elem_bytes) { return 2 * kConsumerWarps * (4 / elem_bytes); }
constexpr int kPartStride = kHeadDim + 4;  // split-attention partial: acc[128], max, sum, 2 pad (16-B rows)
constexpr int kMaxSplits = 21;             // attention splits per KV head
// Cached-row chunks per attention split.  A split streams its chunks through the CTA's ring
// back to back; every extra split adds a partial that the merge must wait for.
constexpr int kSplitChunks = 2;

// Two-group ("die") layout of the decode step.  A GB300 is two dies; a store becomes visible
// to an SM of the die that homes the line about twice as fast as to an SM of the other die,
// and every 4 KB page of device memory is homed by one die.  The decode step therefore splits
// its work into D groups of SMs (D = 2: one per die, D = 1: the whole GPU as one group): group
// g owns KV heads [g Hkv/D, (g+1) Hkv/D) and their query heads, the gate/up rows
// [g I/D, (g+1) I/D), and the matching column halves of o_proj and down.  Exchange buffers
// written and read inside a group sit in pages its die homes.
constexpr int kMaxGroups = 2;
constexpr int kMaxSmIds = 1024;     // role table length (%smid < this)
constexpr int kPageWords = 512;     // 4 KB pages of 64-bit tagged words
constexpr int kMaxXPages = 160;     // exchange pages per group
constexpr size_t kXRegionBytes = (size_t)2 << 20;  // candidate pages for the exchange buffers

// Exchange buffers of one group (tagged 64-bit words: tag << 32 | f32 bits).
enum {
    XB_QKV = 0,   // q|k|v rows of the group's heads            [(Hq + 2 Hkv)/D * 128]
    XB_PART = 1,  // split-attention partials                    [Hkv/D][Smax][G][kPartStride]
    XB_O = 2,     // merged attention output of the group        [Hq/D * 128]
    XB_ACT = 3,   // SwiGLU output of the group's rows            [I/D]
    XB_PO = 4,    // o_proj partial sum over the group's columns  [H]  (read by every group)
    XB_PD = 5,    // down partial sum over the group's columns    [H]  (read by every group)
    XB_POX = 6,   // copy of XB_PO in pages the other group's die homes (two groups only)
    XB_PDX = 7,   // copy of XB_PD in pages the other group's die homes (two groups only)
    kXBufs = 8
};
constexpr int kXFar = XB_POX - XB_PO;  // a partial-sum buffer's far copy: b + kXFar

// Where each group's exchange buffers live: word i of buffer b of group g is at
// region + page[g][first[g][b] + i / kPageWords] * 4096 + (i % kPageWords) * 8.
struct XPlan {
    uint32_t page[kMaxGroups][kMaxXPages];  // page offsets (4 KB units) from the region base
    uint16_t first[kMaxGroups][kXBufs];
};
static_assert(sizeof(XPlan) % 16 == 0, "XPlan is copied in 16-byte units");

// Host view of the SM groups of one device.
struct Topology {
    int D;                        // groups: 2 (one per die) or 1
    int n[kMaxGroups];            // SMs per group
    uint16_t role[kMaxSmIds];     // per %smid: group << 12 | rank within the group; 0xffff = absent
    float rt_near, rt_far;        // measured ping-pong round trips (ns), for reports
};
constexpr uint16_t kNoRole = 0xffff;

// Debug timeline stamps per (phase, CTA): consumer before wait, after wait, after
// compute, after its outputs are written; producer first issue, last issue of the phase.
constexpr int kTraceStamps = 16;

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // every device-side wait gives up after 1 s
constexpr unsigned long long kDebugWaitLimitNs = 1000000ull; // ... or after 1 ms under the withholding debug flag
constexpr int kDebugWithhold = 16;                            // QW_DEBUG_WITHHOLD

// Status values written by device code (same numbers as qw.h).
constexpr unsigned kErrInvalidArgument = 1;
constexpr unsigned kErrNumerical = 18;
constexpr unsigned kErrInvariant = 20;

struct DevLayer {
    const __nv_bfloat16 *input_norm, *q_norm, *k_norm, *post_norm;
    const void *w[7];      // q, k, v, o, gate, up, down: bf16 or int8 [out, in]
    const __half *s[7];    // fp16 scales [out, in/32] (int8 format)
};

// Error word, abort flag and the device-resident greedy token, read back together; diag holds
// where the first device wait gave up (site << 24 | CTA << 12 | phase), 0 if none did.
struct StepFlags {
    unsigned err;
    unsigned abort;
    int next_tok;
    unsigned diag;
};
// Wait sites recorded in StepFlags::diag.
enum { WS_SLOT = 1, WS_RING = 2, WS_VEC = 3, WS_HEAD = 4, WS_MERGE = 5, WS_ROLE = 6, WS_DRAIN = 7 };

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
    const float2 *rope;              // rows of (cos, sin) [64]; the step reads row rope_row
    int rope_row;
    // groups and exchange buffers
    int D;                           // 1 or 2
    int n_grp[kMaxGroups];           // CTAs per group
    const uint16_t *role;            // [kMaxSmIds] group << 12 | rank, by %smid
    unsigned long long *xr;          // exchange region base (4 KB aligned)
    const XPlan *xplan;              // device copy of the buffer placement
    float *logits;                   // [V]
    float *hidden;                   // [(L + 1) H] debug dump
    unsigned *sync;                  // arrivals of the head phase; each step adds the CTA count
    unsigned target;                 // arrivals that mean "this step's head is done" (steps * CTAs)
    unsigned long long *key;         // packed argmax keys [2], one per step parity
    StepFlags *flags;
    int *tok_out;                    // optional device slot for this step's greedy pick
    unsigned long long *trace;       // debug timeline [phase][cta][kTraceStamps] (%globaltimer ns) or null
    // step
    int pos, token, n_split, debug;
    unsigned long long wait_ns;      // limit of every device-side wait of the step
    unsigned step;                   // step sequence number (never 0 after creation)
    unsigned tag_base;               // step * 512: tags of this step are tag_base + 8 layer + kind + 1
};

// Attention splits per KV head for a step at position pos: kSplitChunks chunks of cached rows
// per split, at most one split per CTA of the smaller group and KV head of that group, at most
// kMaxSplits.
inline int attn_splits(int pos, int kv_elem_bytes, const DecodeArgs &a) {
    const int ch = kv_chunk_rows(kv_elem_bytes) * kSplitChunks;
    int s = (pos + ch - 1) / ch;
    int nmin = a.n_grp[0];
    if (a.D > 1 && a.n_grp[1] < nmin) nmin = a.n_grp[1];
    int cap = nmin / (a.Hkv / a.D);
    if (cap > kMaxSplits) cap = kMaxSplits;
    if (s > cap) s = cap;
    if (s > pos) s = pos;
    if (s < 1) s = 1;
    return s;
}

// Largest split count any step can use with this grouping (sizes the partial buffers).
inline int max_attn_splits(int Hkv, int D, const int *n_grp) {
    int nmin = n_grp[0];
    if (D > 1 && n_grp[1] < nmin) nmin = n_grp[1];
    int cap = nmin / (Hkv / D);
    if (cap > kMaxSplits) cap = kMaxSplits;
    return cap < 1 ? 1 : cap;
}

// Words of each exchange buffer of one group.
inline void xbuf_words(int H, int Hq, int Hkv, int I, int D, int smax, size_t *words) {
    const int G = Hq / Hkv;
    words[XB_QKV] = (size_t)(Hq + 2 * Hkv) / D * kHeadDim;
    words[XB_PART] = (size_t)(Hkv / D) * smax * G * kPartStride;
    words[XB_O] = (size_t)Hq / D * kHeadDim;
    words[XB_ACT] = (size_t)I / D;
    words[XB_PO] = (size_t)H;
    words[XB_PD] = (size_t)H;
    words[XB_POX] = D == 2 ? (size_t)H : 0;
    words[XB_PDX] = D == 2 ? (size_t)H : 0;
}

// Step bookkeeping: two argmax keys then the head-phase arrival counter (zeroed at creation,
// by qw_kv_reset and when the counter would overflow).
constexpr size_t kStepBlockBytes = 256;

// Whether a config is the block the decode kernel is built for (head_dim 128 is checked
// separately).
inline bool block_shape_ok(int H, int Hq, int Hkv, int I) {
    return H == kBlockH && Hq == kBlockHq && Hkv == kBlockHkv && I == kBlockI;
}

size_t decode_smem_bytes();
// Sets the shared-memory attribute of every decode instantiation; *blocks_per_sm = the fewest
// CTAs of any of them that fit an SM (1 expected).
cudaError_t decode_prepare(int *blocks_per_sm);
// One cooperative launch of ncta CTAs (one per SM) of the instantiation for (a.D, a.fmt, a.kv_f32).
cudaError_t launch_decode(const DecodeArgs &a, int ncta, cudaStream_t stream);
// Widen bf16 K/V rows [heads][n_pos][128] into an f32 cache [heads][max_ctx][128].
cudaError_t launch_kv_widen(const __nv_bfloat16 *src, float *dst, long long heads, int n_pos, int max_ctx,
                            cudaStream_t stream);

// The SM groups of the current device (probed once per device and cached; D = 1 when the
// two-die structure cannot be seen).  scratch: kProbeScratchBytes of device memory, 4 KB aligned.
constexpr size_t kProbeScratchBytes = 65536;
int probe_topology(int device, uint8_t *scratch, cudaStream_t stream, Topology *out);
// Home group of each 4 KB page of [region, region + npages * 4096) (0 or 1; all 0 when D == 1),
// npages <= 4096; the region's contents are overwritten.
int probe_pages(const Topology &t, uint8_t *region, int npages, int8_t *page_group, uint8_t *scratch,
                cudaStream_t stream);
// Both layouts of the decode step for one device and one exchange region: one group of every
// SM (role1, plan1) and, when the device shows two dies, two groups (role2, plan2; D == 2).
struct GroupPlans {
    int D;                          // 2 when the two-group layout is available
    int ncta;                       // SMs (CTAs of a decode launch)
    int n[kMaxGroups];              // SMs per group of the two-group layout
    uint16_t role1[kMaxSmIds], role2[kMaxSmIds];
    XPlan plan1, plan2;
    float rt_near, rt_far;          // measured round trips (ns)
};
// probe_scratch: kProbeScratchBytes, xregion: kXRegionBytes, both 4 KB aligned device memory.
int plan_groups(int device, uint8_t *probe_scratch, uint8_t *xregion, int H, int Hq, int Hkv, int I,
                cudaStream_t stream, GroupPlans *out);

// Place every group's exchange buffers on pages of its own home group; returns false if the
// region holds too few pages of a group.
bool plan_exchange(const Topology &t, const int8_t *page_group, int npages, const size_t *words, XPlan *plan);

// Launches kernel k on stream st; chained = true adds programmatic stream serialization,
// letting k start while the stream's previous kernel finishes (k must call chain_wait()
// before touching memory that kernel used).  Use it only when the previous operation of
// the stream is a kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool chained, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace qw
