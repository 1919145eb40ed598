// decode_kernel.cuh - one batch-one decode step of the Qwen3 decoder as a single persistent
// kernel for sm_103a (GB300).  Device code only; the instantiations live in decode_g1.cu and
// decode_g2.cu, the host glue in decode.cu.
//
// The step ("Scalar-Native Qwen3 Reference Runtime As The Numerical Authority", section 2
// steps 1-7; the decode schedule of "Portable WebAssembly Runtime Architecture for TinyRustLM",
// section "Prefill versus decode") runs as 5 phases per layer plus one head phase:
//   QKV     x += the previous layer's down partial sums; h = RMSNorm(x); q|k|v = W h
//   ATTN    per (KV head, split): QK-Norm + RoPE of the group's queries and of the new key,
//           append k, v at this position, online softmax over a slice of the cache, a partial
//           (acc, max, sum) per query head; then every split merges a slice of the outputs
//   OPROJ   partial o_proj over the group's columns: Wo[:, group] o[group]
//   GATEUP  x += both groups' o_proj partials; h2 = RMSNorm(x); a = silu(Wg h2) * (Wu h2)
//   DOWN    partial down over the group's columns: Wd[:, group] a[group]
//   LMHEAD  x += both groups' down partials; logits = E RMSNorm(x); packed-key argmax
//
// Layout on the GPU: one CTA per SM (cooperative launch, so all CTAs are resident), 7
// consumer warps and 1 producer warp (two warps per SM sub-partition, so each thread may
// hold 255 registers); the kernel is built for the Qwen3-0.6B block dims
// (kBlockH ... in qw_internal.h), one instantiation per (group count, weight format, cache
// element type).  The SMs form D groups (one per die of the GB300, or a
// single group): group g owns the KV heads [g Hkv/D, (g+1) Hkv/D) with their query heads, the
// gate/up rows [g I/D, (g+1) I/D), and computes o_proj and down as partial sums over the
// matching column halves.  So per layer only two exchanges cross groups (the partial sums of
// o_proj and of down, which every CTA adds into its own full copy of the residual stream, in
// the same order everywhere); q|k|v, the attention partials, the attention output and the
// SwiGLU output stay inside the group, in pages of device memory its die homes.  The two
// partial sums are written twice, once into pages each die homes, so every reader polls
// words on its own die.
//
// The producer streams, with bulk async copies (cp.async.bulk + mbarrier transaction counts),
// every weight row (segment) and cached K/V row its CTA will consume during the whole step into
// a ring of shared-memory slots.  Weights do not depend on the step's data, so the ring keeps
// HBM busy across phase boundaries while consumers wait for the previous phase.  Every output
// element is owned by one warp, so results do not depend on timing.  Every wait is bounded in
// time: on expiry the kernel records QW_INTERNAL_INVARIANT, raises an abort flag that every
// other wait also watches, drains its own copies in flight and returns.
//
// Data between phases travels as tagged words: 64-bit stores of (tag << 32 | f32 bits), tag =
// step sequence * 512 + 8 layer + kind + 1.  Readers poll the words themselves; a naturally
// aligned 64-bit access is single-copy atomic, so a matching tag guarantees the value and no
// fence or counter is needed.  A buffer is rewritten once per layer; a writer never overwrites
// words a reader still needs, because each write of a buffer for layer l+1 comes after its
// writer has seen every CTA's partial sums of a later phase of layer l, which every CTA
// produces only after its reads of that buffer for layer l.
#pragma once

#include <cstddef>

#include "qw_internal.h"

namespace qw {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxVec = kBlockI;  // longest activation row: the whole SwiGLU output (one group)

enum { TK_QKV = 0, TK_PART = 1, TK_O = 2, TK_PO = 3, TK_ACT = 4, TK_PD = 5 };
enum { T_QKV = 0, T_ATTN = 1, T_OPROJ = 2, T_GATEUP = 3, T_DOWN = 4, T_LMHEAD = 5 };

constexpr int kMaxPartials = 512;  // rows (x2 for gate/up) x K slices of one phase

struct AttnScratch {
    float wacc[kConsumerWarps][kBlockG][kHeadDim];  // per-warp accumulators
    float wml[kConsumerWarps][kBlockG][2];          // per-warp running max, sum
    float sq[kBlockG][kHeadDim];                    // normalised, rotated queries
    float sk[kHeadDim];                             // this position's key (cache element type)
    float sv[kHeadDim];                             // this position's value (cache element type)
    float mrg[384];                                 // merge staging: (max, sum) per split and head, then acc values
};

// Every array member is 16-byte aligned: slots are bulk-copy destinations, x and vec are read
// with 16-byte vector loads.
struct __align__(16) Smem {
    alignas(16) uint8_t slot[kSlots][kSlotBytes];
    alignas(16) float x[kBlockH];  // the full residual stream (every CTA keeps its own copy)
    alignas(16) union {
        float vec[kMaxVec];  // the phase's activation vector (staged once per CTA)
        AttnScratch at;
    } u;
    alignas(16) XPlan plan;
    alignas(16) unsigned long long full[kSlots];
    alignas(16) unsigned long long empty[kSlots];
    alignas(16) unsigned long long best[kConsumerWarps];  // head: per-warp argmax keys
    alignas(16) float red[kConsumerWarps];                // block reductions
    alignas(16) float part[kMaxPartials];                 // K-slice partial dot products of a phase
    int fail;                                             // a consumer thread's poll gave up
    int flag;
    int tok;
    int bad;
    int g, r, cidx, ok;                                   // group, rank in the group, index for the head
    int ph, pph;                                          // consumer's and producer's current phase
    alignas(16) DecodeArgs args;                          // this launch's arguments
};
static_assert(sizeof(Smem) <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ Smem &smem() {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    return *reinterpret_cast<Smem *>(smem_raw);
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned smid() {
    unsigned s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

__device__ __forceinline__ void mbar_init(unsigned long long *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_test(unsigned long long *b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, unsigned long long *bar,
                                          unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ unsigned long long policy_evict_first() {
    unsigned long long p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ unsigned long long policy_evict_normal() {
    unsigned long long p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Polls use relaxed loads at gpu scope: the data and flags live in this GPU's memory.
__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void raise_error(StepFlags *f, unsigned code, bool abort) {
    atomicCAS(&f->err, 0u, code);
    if (abort) atomicExch(&f->abort, 1u);
}

__device__ __forceinline__ Smem &smem();

// Bounded poll bookkeeping: true to keep polling, false on abort or timeout.  The first wait of
// the step to expire records its site, CTA and phase in flags->diag.
__device__ __forceinline__ bool poll_more(unsigned i, unsigned long long &t0, StepFlags *f, int site,
                                          bool watch_abort = true) {
    if ((i & 15u) != 15u) return true;
    if (watch_abort && ld_relaxed(&f->abort)) return false;
    const unsigned long long t = gtime();
    if (t0 == 0) {
        t0 = t;
    } else if (t - t0 > smem().args.wait_ns) {
        const Smem &sm = smem();
        const int ph = threadIdx.x >= kConsumerThreads ? sm.pph : sm.ph;
        atomicCAS(&f->diag, 0u, ((unsigned)site << 24) | ((blockIdx.x & 0xfffu) << 12) | ((unsigned)ph & 0xfffu));
        raise_error(f, kErrInvariant, true);
        return false;
    }
    return true;
}

// Bounded wait for an mbarrier phase; watch_abort = false only while draining.
__device__ __forceinline__ bool mbar_wait(unsigned long long *b, unsigned parity, StepFlags *f, int site,
                                          bool watch_abort = true) {
    unsigned long long t0 = 0;
    for (unsigned i = 0; !mbar_test(b, parity); ++i)
        if (!poll_more(i, t0, f, site, watch_abort)) return false;
    return true;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float i8f(uint32_t word, int byte) {
    return (float)((int)(word << (24 - 8 * byte)) >> 24);
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    if (v == 0.0f) v = 0.0f;  // -0 and +0 compare equal: lowest id wins
    uint32_t u = __float_as_uint(v);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

// ----------------------------------------------------------------- tagged words

__device__ __forceinline__ unsigned xtag(const DecodeArgs &a, int l, int kind) {
    return a.tag_base + 8u * (unsigned)l + (unsigned)kind + 1u;
}

// Word i of exchange buffer b of group g.
__device__ __forceinline__ unsigned long long *xw(const Smem &sm, int g, int b, int i) {
    return sm.args.xr + (size_t)sm.plan.page[g][sm.plan.first[g][b] + (i >> 9)] * kPageWords + (i & (kPageWords - 1));
}

__device__ __forceinline__ void st_tag(unsigned long long *p, float v, unsigned tag) {
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ void ld_tag2(const unsigned long long *p, unsigned long long &x, unsigned long long &y) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long ld_tag(const unsigned long long *p) {
    unsigned long long x;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
    return x;
}

__device__ __forceinline__ bool tag_is(unsigned long long w, unsigned tag) { return (unsigned)(w >> 32) == tag; }
__device__ __forceinline__ float tag_val(unsigned long long w) { return __uint_as_float((unsigned)w); }

// --------------------------------------------------------------- phase geometry

struct Phase {
    int type, l;
    // row-streaming phases: rows [r0, r1) of a phase with R rows (pairs for gate/up) of K
    // stored elements each, rpc rows per slot
    int K, i8, pair, rpc, r0, r1;
    // attention
    int kvh, s, p0, p1;
    int nchunks;
};

__device__ __forceinline__ int phase_type(const DecodeArgs &a, int ph) {
    return ph / kPhasesPerLayer >= a.L ? T_LMHEAD : ph % kPhasesPerLayer;
}

__device__ __forceinline__ Phase describe(const DecodeArgs &a, int ph, int g, int r, int cidx, int ncta) {
    Phase p;
    p.l = ph / kPhasesPerLayer;
    p.type = phase_type(a, ph);
    p.i8 = 0;
    p.pair = 0;
    p.nchunks = 0;
    p.kvh = p.s = p.p0 = p.p1 = 0;
    p.K = p.rpc = p.r0 = p.r1 = 0;
    const int D = a.D, n = a.n_grp[g];
    if (p.type == T_ATTN) {
        const int S = a.n_split, hk = a.Hkv / D;
        if (r < hk * S) {
            p.kvh = g * hk + r / S;
            p.s = r % S;
            p.p0 = (int)((long long)a.pos * p.s / S);
            p.p1 = (int)((long long)a.pos * (p.s + 1) / S);
            const int ch = kv_chunk_rows(a.kv_f32 ? 4 : 2);
            p.nchunks = (p.p1 - p.p0 + ch - 1) / ch;
        } else {
            p.kvh = -1;
        }
        return p;
    }
    int R;
    switch (p.type) {
        case T_QKV: R = (a.Hq + 2 * a.Hkv) / D * kHeadDim; p.K = a.H; break;
        case T_OPROJ: R = a.H; p.K = a.Hq * kHeadDim / D; break;
        case T_GATEUP: R = a.I / D; p.K = a.H; p.pair = 1; break;
        case T_DOWN: R = a.H; p.K = a.I / D; break;
        default: R = a.V; p.K = a.H; break;
    }
    p.i8 = (p.type != T_LMHEAD) && a.fmt != 0;  // int8 storage for both int8 formats
    const int bpr = (p.pair ? 2 : 1) * (p.i8 ? p.K + p.K / 16 : 2 * p.K);
    int fit = kSlotBytes / bpr;
    if (fit > 64) fit = 64;
    if (p.type == T_LMHEAD) {
        // streamed chunk by chunk: a whole number of rows per consumer warp
        p.rpc = fit >= kConsumerWarps ? fit - fit % kConsumerWarps : fit;
        p.r0 = (int)((long long)R * cidx / ncta);
        p.r1 = (int)((long long)R * (cidx + 1) / ncta);
    } else {
        p.rpc = fit;
        p.r0 = (int)((long long)R * r / n);
        p.r1 = (int)((long long)R * (r + 1) / n);
    }
    p.nchunks = (p.r1 - p.r0 + p.rpc - 1) / p.rpc;
    return p;
}

// ---------------------------------------------------------------------- producer

struct Issuer {
    uint8_t *slot;
    unsigned long long *bar;
    unsigned long long pol;
    unsigned bytes;
    bool go;  // false: only count bytes
    __device__ void copy(void *dst, const void *src, unsigned n) {
        if (go) bulk_load(dst, src, n, bar, pol);
        else bytes += n;
    }
};

// rows [row, row+count) (whole rows of K elements) of one matrix into stored rows
// [j0, j0+count) of a slot holding ns rows
__device__ __forceinline__ void copy_rows(Issuer &is, const Phase &p, int ns, int j0, const void *w, const __half *s,
                                          long long row, int count) {
    if (count <= 0) return;
    if (p.i8) {
        is.copy(is.slot + (size_t)j0 * p.K, (const uint8_t *)w + row * p.K, (unsigned)(count * p.K));
        is.copy(is.slot + (size_t)ns * p.K + (size_t)j0 * (p.K / 16), (const uint8_t *)s + row * (p.K / 16),
                (unsigned)(count * (p.K / 16)));
    } else {
        is.copy(is.slot + (size_t)j0 * 2 * p.K, (const uint8_t *)w + row * 2 * p.K, (unsigned)(count * 2 * p.K));
    }
}

// columns [col0, col0 + K) of row `row` of a matrix with `width` columns into stored row j
__device__ __forceinline__ void copy_seg(Issuer &is, const Phase &p, int ns, int j, const void *w, const __half *s,
                                         long long row, int width, int col0) {
    if (p.i8) {
        is.copy(is.slot + (size_t)j * p.K, (const uint8_t *)w + row * width + col0, (unsigned)p.K);
        is.copy(is.slot + (size_t)ns * p.K + (size_t)j * (p.K / 16),
                (const uint8_t *)s + (row * (width / 32) + col0 / 32) * 2, (unsigned)(p.K / 16));
    } else {
        is.copy(is.slot + (size_t)j * 2 * p.K, (const uint8_t *)w + (row * width + col0) * 2, (unsigned)(2 * p.K));
    }
}

__device__ __forceinline__ void issue_chunk(Issuer &is, const DecodeArgs &a, const Phase &p, int g, int c) {
    if (p.type == T_ATTN) {
        const int esz = a.kv_f32 ? 4 : 2, ch = kv_chunk_rows(esz);
        const int q0 = p.p0 + c * ch;
        const int n = min(ch, p.p1 - q0);
        const size_t off = ((((size_t)p.l * a.Hkv + p.kvh) * a.max_ctx + q0) * kHeadDim) * esz;
        is.copy(is.slot, (const uint8_t *)a.kc + off, (unsigned)(n * kHeadDim * esz));
        is.copy(is.slot + kSlotBytes / 2, (const uint8_t *)a.vc + off, (unsigned)(n * kHeadDim * esz));
        return;
    }
    const int a0 = p.r0 + c * p.rpc;
    const int n = min(p.rpc, p.r1 - a0);
    if (p.type == T_LMHEAD) {
        copy_rows(is, p, n, 0, a.lm_head, nullptr, a0, n);
        return;
    }
    const DevLayer &Ly = a.layers[p.l];
    const int D = a.D;
    if (p.type == T_QKV) {
        // local rows: q rows of the group's query heads, then its k rows, then its v rows
        const int qr = a.Hq / D * kHeadDim, kr = a.Hkv / D * kHeadDim, b = a0 + n;
        int lo = a0, hi = min(b, qr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[0], Ly.s[0], (long long)g * qr + lo, hi - lo);
        lo = max(a0, qr);
        hi = min(b, qr + kr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[1], Ly.s[1], (long long)g * kr + lo - qr, hi - lo);
        lo = max(a0, qr + kr);
        hi = b;
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[2], Ly.s[2], (long long)g * kr + lo - qr - kr, hi - lo);
    } else if (p.type == T_OPROJ) {
        const int width = a.Hq * kHeadDim;
        for (int j = 0; j < n; ++j) copy_seg(is, p, n, j, Ly.w[3], Ly.s[3], a0 + j, width, g * p.K);
    } else if (p.type == T_GATEUP) {
        const long long row = (long long)g * (a.I / D) + a0;
        copy_rows(is, p, 2 * n, 0, Ly.w[4], Ly.s[4], row, n);
        copy_rows(is, p, 2 * n, n, Ly.w[5], Ly.s[5], row, n);
    } else {
        for (int j = 0; j < n; ++j) copy_seg(is, p, n, j, Ly.w[6], Ly.s[6], a0 + j, a.I, g * p.K);
    }
}

__device__ __noinline__ void producer() {
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int ncta = gridDim.x, g = sm.g, r = sm.r, cidx = sm.cidx;
    const unsigned long long pol_w = policy_evict_first();
    const unsigned long long pol_kv = policy_evict_normal();
    unsigned it = 0;
    bool ok = true;
    const int nph = kPhasesPerLayer * a.L + 1;
    for (int ph = 0; ph < nph && ok; ++ph) {
        const Phase p = describe(a, ph, g, r, cidx, ncta);
        sm.pph = ph;
        unsigned long long *tr = a.trace ? a.trace + ((size_t)ph * ncta + blockIdx.x) * kTraceStamps : nullptr;
        for (int c = 0; c < p.nchunks; ++c) {
            const unsigned slot = it % kSlots, par = ((it / kSlots) & 1u) ^ 1u;
            if (!mbar_wait(&sm.empty[slot], par, a.flags, WS_RING)) {
                ok = false;
                break;
            }
            if (tr) {
                if (c == 0) tr[4] = gtime();
                if (c == p.nchunks - 1) tr[5] = gtime();
            }
            Issuer is{sm.slot[slot], &sm.full[slot], p.type == T_ATTN ? pol_kv : pol_w, 0u, false};
            issue_chunk(is, a, p, g, c);
            mbar_expect_tx(&sm.full[slot], is.bytes);
            is.go = true;
            issue_chunk(is, a, p, g, c);
            ++it;
        }
    }
    if (!ok) {
        // drain: the last chunk issued into each slot must land before the CTA exits
        for (unsigned s = 0; s < (unsigned)kSlots && s < it; ++s) {
            const unsigned last = ((it - 1 - s) / kSlots) * kSlots + s;
            mbar_wait(&sm.full[s], (last / kSlots) & 1u, a.flags, WS_DRAIN, false);
        }
    }
}

// ---------------------------------------------------------------------- consumer

constexpr int kFailed = -1;                 // uniform: the step is aborting
constexpr unsigned kDeadBit = 0x80000000u;  // this warp gave up inside a chunk loop
constexpr int kHeadBatch = 1;               // head chunks a warp holds at once (the rest stay in flight)
// rows (gate/up: pairs) a warp keeps in registers in the row phases: the Qwen3-0.6B block over
// 76 SMs per group (152 in one group) gives q|k|v 27, gate/up 21 pairs, o_proj and down 14 rows
// per CTA, i.e. at most 4, 3 and 2 per warp
constexpr int kPreQkv = 4;
constexpr int kPreGateUp = 3;
constexpr int kPreDown = 2;

__device__ __forceinline__ int ctid() { return threadIdx.x; }
__device__ __forceinline__ int cwarp() { return threadIdx.x >> 5; }
__device__ __forceinline__ int clane() { return threadIdx.x & 31; }

__device__ __forceinline__ unsigned long long *trace_of(const DecodeArgs &a, int ph) {
    return a.trace ? a.trace + ((size_t)ph * gridDim.x + blockIdx.x) * kTraceStamps : nullptr;
}

// Wait for a slot to fill; warp-uniform result.
__device__ __forceinline__ bool take_slot(unsigned slot, unsigned par) {
    Smem &sm = smem();
    const bool ok = mbar_wait(&sm.full[slot], par, sm.args.flags, WS_SLOT);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void release_slot(unsigned slot) {
    __syncwarp();
    if (clane() == 0) mbar_arrive(&smem().empty[slot]);
}

// The staging hook of phases with nothing to overlap with the input barrier.
struct NoPre {
    __device__ __forceinline__ void operator()() const {}
};

// Make a per-thread poll result uniform over the consumer threads (one barrier).
__device__ __forceinline__ bool all_ok(bool ok) {
    Smem &sm = smem();
    if (!ok) sm.fail = 1;
    bar_consumers();
    return sm.fail == 0;
}

// Poll the float4 slots tid + NT i (i < NI, slot < n4) of NB tagged buffers.
template <int NB, int NI>
__device__ __forceinline__ bool poll_vec_n(const int (&gg)[NB], int b, int n4, unsigned tag, float4 (&v)[NB][NI],
                                           StepFlags *f) {
    const Smem &sm = smem();
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
        bool ok = true;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int idx = ctid() + kConsumerThreads * k;
            if (idx < n4) {
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    const unsigned long long *p = xw(sm, gg[q], b, 4 * idx);
                    unsigned long long w0, w1, w2, w3;
                    ld_tag2(p, w0, w1);
                    ld_tag2(p + 2, w2, w3);
                    ok &= tag_is(w0, tag) & tag_is(w1, tag) & tag_is(w2, tag) & tag_is(w3, tag);
                    v[q][k] = make_float4(tag_val(w0), tag_val(w1), tag_val(w2), tag_val(w3));
                }
            }
        }
        if (ok) break;
        if (!poll_more(i, t0, f, WS_VEC)) return false;
    }
    return true;
}

// Float4 slots per consumer thread for a vector of K floats.
template <int K>
__host__ __device__ constexpr int vec_iters() { return (K / 4 + kConsumerThreads - 1) / kConsumerThreads; }

// Poll the float4 slots tid + NT i (< K/4) of NB tagged buffers (buffer kind bb[k] of groups gg[k]).
// Each word's value is taken as it is loaded, so only floats stay live across the retries.
template <int NB, int K>
__device__ __forceinline__ bool poll_vec(const int (&gg)[NB], const int (&bb)[NB], unsigned tag,
                                         float4 (&v)[NB][vec_iters<K>()], StepFlags *f) {
    constexpr int NI = vec_iters<K>();
    const Smem &sm = smem();
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
        bool ok = true;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int idx = ctid() + kConsumerThreads * k;
            if (idx < K / 4) {
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    const unsigned long long *p = xw(sm, gg[q], bb[q], 4 * idx);
                    unsigned long long w0, w1, w2, w3;
                    ld_tag2(p, w0, w1);
                    ld_tag2(p + 2, w2, w3);
                    ok &= tag_is(w0, tag) & tag_is(w1, tag) & tag_is(w2, tag) & tag_is(w3, tag);
                    v[q][k] = make_float4(tag_val(w0), tag_val(w1), tag_val(w2), tag_val(w3));
                }
            }
        }
        if (ok) break;
        if (!poll_more(i, t0, f, WS_VEC)) return false;
    }
    return true;
}

// Raw weight piece (8 columns, piece index pi counted in 8-column units from the row start)
// of one stored row: 16 bytes of bf16, or 8 bytes of int8 codes plus their group's fp16 scale.
template <bool I8>
struct WPiece;
template <>
struct WPiece<false> {
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *row, const uint8_t *, int pi) {
        v = reinterpret_cast<const uint4 *>(row)[pi];
    }
    // w[k] = columns (2k, 2k+1) of the piece as f32
    __device__ __forceinline__ void unpack(float2 (&w)[4]) const {
        w[0] = make_float2(bf_lo(v.x), bf_hi(v.x));
        w[1] = make_float2(bf_lo(v.y), bf_hi(v.y));
        w[2] = make_float2(bf_lo(v.z), bf_hi(v.z));
        w[3] = make_float2(bf_lo(v.w), bf_hi(v.w));
    }
};
template <>
struct WPiece<true> {
    uint2 v;
    __half s;
    __device__ __forceinline__ void load(const uint8_t *row, const uint8_t *srow, int pi) {
        v = reinterpret_cast<const uint2 *>(row)[pi];
        s = reinterpret_cast<const __half *>(srow)[pi >> 2];
    }
    // int8 group-32 codes dequantised in registers: w = f32(q) * f32(s), an exact product
    __device__ __forceinline__ void unpack(float2 (&w)[4]) const {
        const float sf = __half2float(s);
        w[0] = make_float2(i8f(v.x, 0) * sf, i8f(v.x, 1) * sf);
        w[1] = make_float2(i8f(v.x, 2) * sf, i8f(v.x, 3) * sf);
        w[2] = make_float2(i8f(v.y, 0) * sf, i8f(v.y, 1) * sf);
        w[3] = make_float2(i8f(v.y, 2) * sf, i8f(v.y, 3) * sf);
    }
};

// Stored row j of a slot holding ns rows of K elements: weights, and (int8) scales.
template <bool I8>
__device__ __forceinline__ const uint8_t *slot_row(const uint8_t *sp, int K, int j) {
    return sp + (size_t)j * (I8 ? K : 2 * K);
}
template <bool I8>
__device__ __forceinline__ const uint8_t *slot_scales(const uint8_t *sp, int K, int ns, int j) {
    return I8 ? sp + (size_t)ns * K + (size_t)j * (K / 16) : nullptr;
}

// The activation vector is staged in shared memory lane-interleaved by 256-column slice: the 8
// columns 256 s + 8 L .. + 7 that lane L multiplies with its 16-byte weight piece of slice s sit
// as two float4 at float4 index 64 s + L (columns + 0..3) and 64 s + 32 + L (+ 4..7), so the
// lanes of a warp read consecutive 16-byte words (no bank conflicts).
__device__ __forceinline__ int vec_slot(int c4) {  // float4 index of columns 4 c4 .. 4 c4 + 3
    const int s = c4 >> 6, w = c4 & 63;
    return 64 * s + ((w & 1) ? 32 : 0) + (w >> 1);
}

// Lane L's 8 activation columns of slice s as 4 pairs.
__device__ __forceinline__ void load_slice(const float *vec, int s, int lane, float2 (&act)[4]) {
    const float4 *v4 = reinterpret_cast<const float4 *>(vec) + 64 * s;
    const float4 a0 = v4[lane], a1 = v4[32 + lane];
    act[0] = make_float2(a0.x, a0.y);
    act[1] = make_float2(a0.z, a0.w);
    act[2] = make_float2(a1.x, a1.y);
    act[3] = make_float2(a1.z, a1.w);
}

// acc += weight piece (columns 8 L .. of slice s of a stored row) . act, two columns per paired FMA.
template <bool I8>
__device__ __forceinline__ void piece_fma(const WPiece<I8> &wp, const float2 (&act)[4], float2 &acc) {
    float2 w[4];
    wp.unpack(w);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc = __ffma2_rn(w[k], act[k], acc);
}

// Q8 x Q8 (weight format 2): the lane's 8 activation columns of one slice times mul, quantized
// as part of their 32-column block (lanes 4j .. 4j + 3 of a slice share one): d = amax / 127,
// codes round-half-away(a / d) clamped to +-127 (0 when amax is 0), the scale rounded to fp16;
// lo / hi hold the codes of columns 0..3 / 4..7 as bytes, matching a weight piece's layout.
struct QAct {
    uint32_t lo, hi;
    float d;
};
__device__ __forceinline__ QAct quant8(const float2 (&a)[4], float mul) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = a[k].x * mul;
        v[2 * k + 1] = a[k].y * mul;
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const float d = m / 127.0f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float t = d > 0.f ? roundf(v[i] / d) : 0.f;  // halves away from zero
        t = fminf(fmaxf(t, -127.f), 127.f);
        w[i >> 2] |= ((uint32_t)(int)t & 0xffu) << (8 * (i & 3));
    }
    return QAct{w[0], w[1], __half2float(__float2half_rn(d))};
}

// acc += (integer dot of a weight piece with the lane's activation codes) * (s_w * s_a)
__device__ __forceinline__ void piece_dot_q8(const WPiece<true> &wp, const QAct &qa, float &acc) {
    const int isum = __dp4a((int)wp.v.x, (int)qa.lo, __dp4a((int)wp.v.y, (int)qa.hi, 0));
    acc = fmaf((float)isum, __half2float(wp.s) * qa.d, acc);
}

__device__ __forceinline__ float warp_sum2(float2 v) {
    float s = v.x + v.y;
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// Stage the input of a row-streaming phase into sm.u.vec (K columns, lane-interleaved).  The
// residual-stream phases (QKV, gate/up, head) first add the previous phase's partial sums of
// every group to their copy of x (in group order, so every CTA holds the same x) and stage
// w (.) x, the RMSNorm weight times x; the normalisation factor r = 1/sqrt(mean(x^2) + eps) is
// returned in *scale and applied to each row's dot product (W (w (.) x r) = r W (w (.) x)), so
// the sum of squares needs no barrier of its own.  o_proj and down copy their group's exchange
// buffer (*scale = 1).  Returns false (uniformly) if a wait gave up.
template <int D, int NI, typename Pre>
__device__ __forceinline__ bool stage_input(int kind, int l, int K, const DecodeArgs &a, unsigned long long *tr,
                                            float *scale, Pre &&before_barrier) {
    Smem &sm = smem();
    const int tid = ctid(), warp = cwarp(), lane = clane();
    float4 *vec4 = reinterpret_cast<float4 *>(sm.u.vec);
    float4 *x4 = reinterpret_cast<float4 *>(sm.x);
    bool ok = true;
    if (tr && tid == 0) tr[10] = clock64();
    if (kind == T_QKV || kind == T_GATEUP || kind == T_LMHEAD) {
        const __nv_bfloat16 *nwp = kind == T_QKV ? a.layers[l].input_norm
                                   : kind == T_GATEUP ? a.layers[l].post_norm
                                                      : a.final_norm;
        constexpr int NH = vec_iters<kBlockH>();  // float4 slots of x per thread
        float4 nw[NH];
        float4 pv[D][NH];
        if (!(kind == T_QKV && l == 0)) {  // at layer 0 x is the embedding, already staged
            const int b = kind == T_GATEUP ? XB_PO : XB_PD;
            const unsigned tg = kind == T_GATEUP ? xtag(a, l, TK_PO) : xtag(a, l - 1, TK_PD);
            // every group's partial sums, each from the copy in pages this CTA's die homes
            int gg[D], bb[D];
#pragma unroll
            for (int q = 0; q < D; ++q) {
                gg[q] = q;
                bb[q] = q == sm.g ? b : b + kXFar;
            }
            ok = poll_vec<D, kBlockH>(gg, bb, tg, pv, a.flags);
        }
        if (tr && tid == 0) {
            tr[1] = gtime();
            tr[15] = clock64();
        }
#pragma unroll
        for (int i = 0; i < NH; ++i) {
            const int idx = tid + kConsumerThreads * i;
            if (idx < kBlockH / 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(nwp) + idx);
                nw[i] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NH; ++i) {
            const int idx = tid + kConsumerThreads * i;
            if (idx >= kBlockH / 4) continue;
            float4 x = x4[idx];
            if (!(kind == T_QKV && l == 0)) {
#pragma unroll
                for (int q = 0; q < D; ++q) {  // groups in order: the same sum in every CTA
                    const float4 pq = pv[q][i];
                    x.x += pq.x; x.y += pq.y; x.z += pq.z; x.w += pq.w;
                }
                x4[idx] = x;
                if ((a.debug & 1) && sm.cidx == 0 && kind != T_GATEUP)
                    reinterpret_cast<float4 *>(a.hidden + (size_t)l * kBlockH)[idx] = x;
            }
            ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
            vec4[vec_slot(idx)] = make_float4(nw[i].x * x.x, nw[i].y * x.y, nw[i].z * x.z, nw[i].w * x.w);
        }
        ss = warp_sum(ss);
        if (lane == 0) sm.red[warp] = ss;
        before_barrier();
        if (!all_ok(ok)) return false;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += sm.red[w];
        *scale = rsqrtf(tot * (1.0f / (float)kBlockH) + a.eps);
        return true;
    }
    const int b = kind == T_OPROJ ? XB_O : XB_ACT;
    const unsigned tg = xtag(a, l, kind == T_OPROJ ? TK_O : TK_ACT);
    const int gg[1] = {sm.g};
    float4 v[1][NI];
    ok = poll_vec_n<1, NI>(gg, b, K / 4, tg, v, a.flags);
    if (tr && tid == 0) {
        tr[1] = gtime();
        tr[15] = clock64();
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int idx = tid + kConsumerThreads * i;
        if (idx < K / 4) vec4[vec_slot(idx)] = v[0][i];
    }
    *scale = 1.0f;
    before_barrier();
    return all_ok(ok);
}

// Where a phase's output words go: rows [r0, r1) of one exchange buffer of the CTA's group (and,
// for the two partial sums with two groups, of its far-die copy), resolved to at most two page
// runs before the phase waits for its input, so storing a result needs no table lookup.
struct OutRows {
    unsigned long long *lo, *hi, *flo, *fhi;  // first page run, the next one; far copy (or null)
    int split;                                // rows of the first run
    bool mute;                                // failure-path test: this CTA withholds its rows
    __device__ __forceinline__ void init(const Smem &sm, int buf, int r0, int r1) {
        const int first = kPageWords - (r0 & (kPageWords - 1));
        split = first;
        lo = xw(sm, sm.g, buf, r0);
        hi = r1 - r0 > first ? xw(sm, sm.g, buf, r0 + first) : lo;
        const bool far = sm.args.D == 2 && (buf == XB_PO || buf == XB_PD);
        flo = far ? xw(sm, sm.g, buf + kXFar, r0) : nullptr;
        fhi = far && r1 - r0 > first ? xw(sm, sm.g, buf + kXFar, r0 + first) : flo;
        mute = (sm.args.debug & kDebugWithhold) && sm.ph == 0 && sm.g == 0 && sm.r == 0;
    }
    __device__ __forceinline__ void put(int jl, float v, unsigned tag) const {
        if (mute) return;
        const bool a = jl < split;
        st_tag(a ? lo + jl : hi + (jl - split), v, tag);
        if (flo) st_tag(a ? flo + jl : fhi + (jl - split), v, tag);
    }
};

// Warp sums of RP values at once (RP a power of two, at most 32): the first log2(RP) exchange
// levels halve the values each lane carries, so the whole reduction takes RP - 1 + 5 - log2(RP)
// shuffles instead of 5 RP.  Afterwards every lane holds the total of value lane / (32 / RP).
template <int RP>
__device__ __forceinline__ float warp_sum_many(float (&v)[RP], int lane) {
#pragma unroll
    for (int h = RP / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h], keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 / RP; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

template <int N>
__host__ __device__ constexpr int pow2_at_least(int n = 1) { return n >= N ? n : pow2_at_least<N>(2 * n); }

// A layer phase over rows [p.r0, p.r1) with K = 256 NP columns (K <= 1536), all chunks taken and
// the input staged (scale: the deferred RMSNorm factor): warp w owns rows w, w + 7, ... (gate/up:
// pairs).  It loads the weight pieces of its first PR rows from the ring into registers at once,
// reads the activation, runs the paired FMAs of all its rows and one transposed warp reduction
// for all of them, and stores the results through precomputed addresses.  Rows beyond PR per
// warp (only with fewer SMs than the block is laid out for) follow one at a time.
template <int NP, int WF, bool PAIR, int PR>
__device__ __forceinline__ void gemv_rows(const Phase &p, int kind, unsigned it0, unsigned out_tag, float scale,
                                          unsigned long long *tr) {
    constexpr bool I8 = WF != 0, Q8A = WF == 2;
    constexpr int NR = PAIR ? 2 : 1;
    constexpr int NV = PR * NR;               // values a lane accumulates
    constexpr int RP = pow2_at_least<NV>();   // padded to a power of two for the reduction
    constexpr int LW = 32 / RP;               // lanes per reduced value
    constexpr int K = 256 * NP;
    Smem &sm = smem();
    const int warp = cwarp(), lane = clane();
    const int R = p.r1 - p.r0;
    const int buf = kind == T_QKV ? XB_QKV : kind == T_OPROJ ? XB_PO : kind == T_GATEUP ? XB_ACT : XB_PD;
    auto piece_rows = [&](int j, const uint8_t *(&rp)[NR], const uint8_t *(&sc)[NR]) {
        const int c = j / p.rpc, jj = j - c * p.rpc;
        const int n = min(p.rpc, R - c * p.rpc), ns = PAIR ? 2 * n : n;
        const uint8_t *sp = sm.slot[(it0 + c) % kSlots];
        rp[0] = slot_row<I8>(sp, K, jj);
        sc[0] = slot_scales<I8>(sp, K, ns, jj);
        if constexpr (PAIR) {
            rp[1] = slot_row<I8>(sp, K, n + jj);
            sc[1] = slot_scales<I8>(sp, K, ns, n + jj);
        }
    };
    if (tr && ctid() == 0) tr[13] = clock64();
    WPiece<I8> pre[PR][NR][NP];
#pragma unroll
    for (int q = 0; q < PR; ++q) {
        const int j = warp + q * kConsumerWarps;
        const uint8_t *rp[NR], *sc[NR];
        piece_rows(j < R ? j : 0, rp, sc);
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int s = 0; s < NP; ++s) pre[q][r][s].load(rp[r], sc[r], 32 * s + lane);
    }
    OutRows out;
    out.init(sm, buf, p.r0, p.r1);
    float2 act[NP][4];
#pragma unroll
    for (int s = 0; s < NP; ++s) load_slice(sm.u.vec, s, lane, act[s]);
    QAct qa[Q8A ? NP : 1];
    if constexpr (Q8A) {  // the normalised input quantized per block; the scale is inside the codes' d
#pragma unroll
        for (int s = 0; s < NP; ++s) qa[s] = quant8(act[s], scale);
    }
    const float oscale = Q8A ? 1.0f : scale;
    if (tr && ctid() == 0) tr[8] = clock64();
    {
        float v[RP];  // value q NR + r = this lane's part of row (q, r)
#pragma unroll
        for (int q = 0; q < PR; ++q)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if constexpr (Q8A) {
                    float acc = 0.f;
#pragma unroll
                    for (int s = 0; s < NP; ++s) piece_dot_q8(pre[q][r][s], qa[s], acc);
                    v[q * NR + r] = acc;
                } else {
                    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int s = 0; s < NP; ++s) piece_fma<I8>(pre[q][r][s], act[s], acc[s & 1]);
                    v[q * NR + r] = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                }
            }
#pragma unroll
        for (int i = NV; i < RP; ++i) v[i] = 0.f;
        const float t = warp_sum_many<RP>(v, lane) * oscale;
        const int vi = lane / LW;  // the value this lane now holds
        if constexpr (PAIR) {
            const float up = __shfl_xor_sync(0xffffffffu, t, LW);  // value vi + 1: the pair's up row
            const int j = warp + (vi >> 1) * kConsumerWarps;
            if ((lane & (2 * LW - 1)) == 0 && vi < NV && j < R)
                out.put(j, (t / (1.0f + __expf(-t))) * up, out_tag);  // silu(gate) * up
        } else {
            const int j = warp + vi * kConsumerWarps;
            if ((lane & (LW - 1)) == 0 && vi < NV && j < R) out.put(j, t, out_tag);
        }
        if (tr && ctid() == 0) tr[9] = clock64();
    }
    // any further rows of this warp (fewer SMs than the block is laid out for)
#pragma unroll 1
    for (int j = warp + PR * kConsumerWarps; j < R; j += kConsumerWarps) {
        const uint8_t *rp[NR], *sc[NR];
        piece_rows(j, rp, sc);
        float o[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int s = 0; s < NP; ++s) {
                WPiece<I8> wp;
                wp.load(rp[r], sc[r], 32 * s + lane);
                if constexpr (Q8A) piece_dot_q8(wp, qa[s], acc[0].x);
                else piece_fma<I8>(wp, act[s], acc[s & 1]);
            }
            o[r] = warp_sum((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) * oscale;
        }
        if (lane == 0) {
            float val = o[0];
            if constexpr (PAIR) val = (o[0] / (1.0f + __expf(-o[0]))) * o[1];
            out.put(j, val, out_tag);
        }
    }
    if (tr && ctid() == 0) tr[11] = clock64();
}

// A layer phase over rows [p.r0, p.r1) of K stored columns whose chunks (all of them) are
// already taken: split K into F = K/256 slices; each warp works on whole slices (slice w % F for
// every W-th row when there are at least as many warps as slices), so it reads only its slices
// of the activation.
// Each (row, slice) dot product goes to sm.part; then one thread per row adds the F slices in
// order and writes the row's tagged result (silu(gate) * up for gate/up pairs).
template <int WF, bool PAIR>
__device__ __forceinline__ void gemv_ksplit(const Phase &p, int kind, unsigned it0, unsigned out_tag) {
    constexpr bool I8 = WF != 0, Q8A = WF == 2;
    constexpr int NR = PAIR ? 2 : 1;
    Smem &sm = smem();
    const int warp = cwarp(), lane = clane(), tid = ctid(), g = sm.g;
    const int K = p.K, F = K >> 8, R = p.r1 - p.r0;
    // the (row, slice) dot products of slice s for rows j0, j0 + step, ...
    auto slice_rows = [&](int s, int j0, int step) {
        float2 act[4];
        load_slice(sm.u.vec, s, lane, act);
        QAct qa{};
        if constexpr (Q8A) qa = quant8(act, 1.0f);  // o_proj / down inputs carry no deferred scale
        for (int j = j0; j < R; j += step) {
            const int c = j / p.rpc, jj = j - c * p.rpc;
            const int n = min(p.rpc, R - c * p.rpc), ns = PAIR ? 2 * n : n;
            const uint8_t *sp = sm.slot[(it0 + c) % kSlots];
            WPiece<I8> wp[NR];
            wp[0].load(slot_row<I8>(sp, K, jj), slot_scales<I8>(sp, K, ns, jj), 32 * s + lane);
            if constexpr (PAIR) wp[1].load(slot_row<I8>(sp, K, n + jj), slot_scales<I8>(sp, K, ns, n + jj), 32 * s + lane);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                float2 acc = make_float2(0.f, 0.f);
                if constexpr (Q8A) piece_dot_q8(wp[r], qa, acc.x);
                else piece_fma<I8>(wp[r], act, acc);
                const float v = warp_sum2(acc);
                if (lane == 0) sm.part[(j * NR + r) * F + s] = v;
            }
        }
    };
    if (F <= kConsumerWarps) {  // warp w: slice w % F, every W-th row from w / F
        const int s = warp % F;
        slice_rows(s, warp / F, (kConsumerWarps - s + F - 1) / F);
    } else {  // more slices than warps: warp w takes slices w, w + NW, ... for every row
        for (int s = warp; s < F; s += kConsumerWarps) slice_rows(s, 0, 1);
    }
    bar_consumers();
    const int buf = kind == T_QKV ? XB_QKV : kind == T_OPROJ ? XB_PO : kind == T_GATEUP ? XB_ACT : XB_PD;
    for (int j = tid; j < R; j += kConsumerThreads) {
        float o[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float *pp = sm.part + (j * NR + r) * F;
            float v = pp[0];
            for (int q = 1; q < F; ++q) v += pp[q];
            o[r] = v;
        }
        float v = o[0];
        if constexpr (PAIR) v = (o[0] / (1.0f + __expf(-o[0]))) * o[1];  // silu(gate) * up
        st_tag(xw(sm, g, buf, p.r0 + j), v, out_tag);
    }
}

// The head: rows [p.r0, p.r1) of the tied lm_head streamed through the ring in batches of
// kHeadBatch chunks, which each warp takes and releases on its own, so the other slots stay in
// flight; each warp owns whole rows (full K = H, the activation in registers) and
// keeps the best packed (logit, id) key it has seen.  Returns the new ring position (kDeadBit
// set if this warp gave up).
__device__ __forceinline__ int gemv_head(const Phase &p, unsigned it, float scale) {
    constexpr int NS = kBlockH / 256;  // slices of a row
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int warp = cwarp(), lane = clane();
    const int R = p.r1 - p.r0;
    float2 act[NS][4];
#pragma unroll
    for (int s = 0; s < NS; ++s) load_slice(sm.u.vec, s, lane, act[s]);
    unsigned long long best = 0;
    bool bad = false, dead = false;
    for (int c0 = 0; c0 < p.nchunks && !dead; c0 += kHeadBatch) {
        const int nb = min(kHeadBatch, p.nchunks - c0);
        for (int c = 0; c < nb && !dead; ++c) dead = !take_slot((it + c) % kSlots, ((it + c) / kSlots) & 1u);
        if (dead) break;
        const int g1 = min(R, (c0 + nb) * p.rpc);
        for (int gi = c0 * p.rpc + warp; gi < g1; gi += kConsumerWarps) {
            const int c = gi / p.rpc, j = gi - c * p.rpc;
            const uint8_t *row = slot_row<false>(sm.slot[(it + c - c0) % kSlots], kBlockH, j);
            WPiece<false> wp[NS];
#pragma unroll
            for (int s = 0; s < NS; ++s) wp[s].load(row, nullptr, 32 * s + lane);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int s = 0; s < NS; ++s) piece_fma<false>(wp[s], act[s], acc);
            const float o = warp_sum2(acc) * scale;
            if (lane == 0) {
                const int row_id = p.r0 + gi;
                a.logits[row_id] = o;
                if (isfinite(o)) {
                    const unsigned long long k = argmax_key(o, row_id);
                    best = k > best ? k : best;
                } else {
                    bad = true;
                }
            }
        }
        for (int c = 0; c < nb; ++c) release_slot((it + c) % kSlots);
        it += nb;
    }
    if (lane == 0) {
        sm.best[warp] = best;
        if (bad) atomicOr(&sm.bad, 1);
    }
    return (int)(it | (dead ? kDeadBit : 0u));
}

// One row-streaming phase (QKV, o_proj, gate/up, down or the head) of layer l.  The phase kind
// is a runtime value, so one copy of each core serves every phase that shares its row shape.  A
// layer phase takes its weight chunks from the ring before it waits for its input (they do not
// depend on it), then stages the input, computes and releases the chunks.
template <int D, int WF>
__device__ __forceinline__ int gemv_phase(int ph, unsigned it) {
    constexpr int KO = kBlockHq * kHeadDim / D, KD = kBlockI / D;
    constexpr int KMAX = KO > KD ? KO : KD;
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const Phase p = describe(a, ph, sm.g, sm.r, sm.cidx, gridDim.x);
    const int kind = p.type, l = p.l;
    unsigned long long *tr = trace_of(a, ph);
    if (tr && ctid() == 0) tr[0] = gtime();
    if (kind == T_LMHEAD) {
        float scale;
        if (!stage_input<D, vec_iters<KMAX>()>(kind, l, p.K, a, tr, &scale, NoPre{})) return kFailed;
        if (tr && ctid() == 0) tr[2] = gtime();
        return gemv_head(p, it, scale);
    }
    // every chunk of a layer phase fits the ring at once
    bool dead = false;
    for (int c = 0; c < p.nchunks && !dead; ++c) dead = !take_slot((it + c) % kSlots, ((it + c) / kSlots) & 1u);
    if (tr && ctid() == 0) tr[6] = gtime();
    if (!all_ok(!dead)) return kFailed;
    const unsigned out_tag =
        xtag(a, l, kind == T_QKV ? TK_QKV : kind == T_OPROJ ? TK_PO : kind == T_GATEUP ? TK_ACT : TK_PD);
    // one staging copy for every row phase (and the head): the phase's input vector in shared memory
    float scale;
    const bool ok = stage_input<D, vec_iters<KMAX>()>(kind, l, p.K, a, tr, &scale, NoPre{});
    if (ok) {
        if (tr && ctid() == 0) tr[2] = gtime();
        if (kind == T_GATEUP) {
            gemv_rows<4, WF, true, kPreGateUp>(p, kind, it, out_tag, scale, tr);
        } else if (kind == T_QKV || (kind == T_OPROJ && KO == kBlockH)) {
            gemv_rows<4, WF, false, kPreQkv>(p, kind, it, out_tag, scale, tr);
        } else if (kind == T_DOWN && KD == 1536) {
            gemv_rows<6, WF, false, kPreDown>(p, kind, it, out_tag, scale, tr);
        } else if constexpr (D == 1) {  // one group: o_proj and down rows of 2048 / 3072 columns, split over the warps
            gemv_ksplit<WF, false>(p, kind, it, out_tag);
        }
    }
    if (!ok) return kFailed;
    if (tr && ctid() == 0) tr[7] = gtime();
    for (int c = 0; c < p.nchunks; ++c) release_slot((it + c) % kSlots);
    if (tr && ctid() == 0) tr[12] = clock64();
    it += p.nchunks;
    return (int)it;
}

// QK-Norm then RoPE of one head held as dims (lane, lane+32, lane+64, lane+96);
// w and cs are the lane's norm weights and (cos, sin) for dims lane and lane+32.
__device__ __forceinline__ void qk_norm_rope(float (&v)[4], const float (&w)[4], const float2 (&cs)[2], float eps) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.0f / kHeadDim) + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = w[i] * (v[i] * r);
    const float a0 = v[0], a1 = v[1], b0 = v[2], b1 = v[3];
    v[0] = a0 * cs[0].x - b0 * cs[0].y;
    v[2] = b0 * cs[0].x + a0 * cs[0].y;
    v[1] = a1 * cs[1].x - b1 * cs[1].y;
    v[3] = b1 * cs[1].x + a1 * cs[1].y;
}

// Poll a head's 128 tagged values (words src[lane + 32 k]) as dims (lane, lane+32, lane+64, lane+96).
__device__ __forceinline__ bool poll_head(const unsigned long long *src, int lane, unsigned tag, float (&v)[4],
                                          StepFlags *f) {
    unsigned long long w[4];
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = ld_tag(src + lane + 32 * k);
        if (tag_is(w[0], tag) && tag_is(w[1], tag) && tag_is(w[2], tag) && tag_is(w[3], tag)) break;
        if (!poll_more(i, t0, f, WS_HEAD)) return false;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = tag_val(w[k]);
    return true;
}

// K/V element type of the cache: f32 (default) or bf16.  Sixteen lanes share a position;
// lane o16 = lane % 16 holds dims dim(o16, r, e) of piece r (16 bytes at byte off(o16, r) of
// the row), so the 16 lanes of a position read 256 contiguous bytes per piece.
template <typename KT>
struct KvTraits;
template <>
struct KvTraits<float> {
    static constexpr int kPieces = 2;  // a lane's 8 dims = 2 x 16-byte pieces, 256 B apart
    static constexpr int kPer = 4;     // elements per piece
    __device__ static __forceinline__ int off(int o16, int r) { return 16 * o16 + 256 * r; }
    __device__ static __forceinline__ int dim(int o16, int r, int e) { return 4 * o16 + 64 * r + e; }
    __device__ static __forceinline__ void load(const uint8_t *p, float (&o)[4]) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ static __forceinline__ float store(float v) { return v; }
};
template <>
struct KvTraits<__nv_bfloat16> {
    static constexpr int kPieces = 1;
    static constexpr int kPer = 8;
    __device__ static __forceinline__ int off(int o16, int) { return 16 * o16; }
    __device__ static __forceinline__ int dim(int o16, int, int e) { return 8 * o16 + e; }
    __device__ static __forceinline__ void load(const uint8_t *p, float (&o)[8]) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        o[0] = bf_lo(v.x); o[1] = bf_hi(v.x); o[2] = bf_lo(v.y); o[3] = bf_hi(v.y);
        o[4] = bf_lo(v.z); o[5] = bf_hi(v.z); o[6] = bf_lo(v.w); o[7] = bf_hi(v.w);
    }
    __device__ static __forceinline__ __nv_bfloat16 store(float v) { return __float2bfloat16_rn(v); }
};

// Online-softmax update over n positions whose K and V rows (128 elements of KT each) sit at
// kb and vb.  Lane (jj = lane / 16, o16 = lane % 16) of warp w takes position
// base + 2 w + jj for base = 0, 2 NW, ... and its dims (KvTraits::dim).
template <int G, typename KT>
__device__ __forceinline__ void attn_block(const uint8_t *kb, const uint8_t *vb, int n, int warp, int lane,
                                           const float (&qr)[G][KvTraits<KT>::kPieces][KvTraits<KT>::kPer],
                                           float (&acc)[G][KvTraits<KT>::kPieces][KvTraits<KT>::kPer],
                                           float (&M)[G], float (&Ls)[G]) {
    using T = KvTraits<KT>;
    constexpr int NP = T::kPieces, PER = T::kPer, ROWB = kHeadDim * (int)sizeof(KT);
    const int jj = lane >> 4, o16 = lane & 15;
    for (int base = 0; base < n; base += 2 * kConsumerWarps) {
        const int jpos = base + 2 * warp + jj;
        const bool valid = jpos < n;
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
        if (valid) {
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                float kv[PER];
                T::load(kb + (size_t)jpos * ROWB + T::off(o16, r), kv);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < PER; ++e) sc[h] = fmaf(qr[h][r][e], kv[e], sc[h]);
            }
        }
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = sc[h];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            s += __shfl_xor_sync(0xffffffffu, s, 8);
            const float s2 = valid ? s : -INFINITY;
            const float mx = fmaxf(s2, __shfl_xor_sync(0xffffffffu, s2, 16));
            const float mn = fmaxf(M[h], mx);
            if (mn != M[h]) {  // warp-uniform
                const float alpha = (M[h] == -INFINITY) ? 0.f : exp2f(M[h] - mn);
                Ls[h] *= alpha;
#pragma unroll
                for (int r = 0; r < NP; ++r)
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[h][r][e] *= alpha;
                M[h] = mn;
            }
            pr[h] = valid ? exp2f(s2 - mn) : 0.f;
            Ls[h] += pr[h];
        }
        if (valid) {
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                float vv[PER];
                T::load(vb + (size_t)jpos * ROWB + T::off(o16, r), vv);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[h][r][e] = fmaf(pr[h], vv[e], acc[h][r][e]);
            }
        }
    }
}

// One (KV head, split) item: QK-Norm + RoPE of the group's queries and of the new key,
// append k, v at this position (the last split owns it), online softmax over the split's
// cached positions (+ the new one), and the split's tagged partial (acc, max, sum) for each
// query head.  Then every split of the KV head merges a slice of the head's outputs from all
// partials; a single split writes the outputs directly.
template <int G, typename KT>
__device__ __forceinline__ int attn_phase(int ph, unsigned it) {
    using T = KvTraits<KT>;
    constexpr int NP = T::kPieces, PER = T::kPer, CH = kv_chunk_rows((int)sizeof(KT));
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int tid = ctid(), warp = cwarp(), lane = clane();
    const int g = sm.g;
    const Phase p = describe(a, ph, g, sm.r, sm.cidx, gridDim.x);
    unsigned long long *tr = trace_of(a, ph);
    if (p.kvh < 0) {  // no attention item on this CTA
        if (tr && tid == 0) tr[0] = tr[1] = tr[2] = gtime();
        return (int)it;
    }
    AttnScratch &at = sm.u.at;
    const int S = a.n_split, P = a.pos, kvh = p.kvh, l = p.l;
    const int hk = a.Hkv / a.D, kvl = kvh - g * hk, qrows = a.Hq / a.D * kHeadDim;
    const bool owner = (p.s == S - 1);
    const DevLayer &Ly = a.layers[l];
    const unsigned in_tag = xtag(a, l, TK_QKV);
    // read-only inputs before the wait: norm weights and this position's rotation
    float w4[4];
    float2 cs[2];
    if (warp <= G) {
        const __nv_bfloat16 *nw = warp < G ? Ly.q_norm : Ly.k_norm;
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = __bfloat162float(nw[lane + 32 * i]);
        const float2 *rope = a.rope + (size_t)a.rope_row * (kHeadDim / 2);
        cs[0] = rope[lane];
        cs[1] = rope[lane + 32];
    }
    if (tr && tid == 0) tr[0] = gtime();
    KT *snew_k = reinterpret_cast<KT *>(at.sk), *snew_v = reinterpret_cast<KT *>(at.sv);
    const size_t row_off = (((size_t)l * a.Hkv + kvh) * a.max_ctx + P) * kHeadDim;
    bool ok = true;
    if (warp < G) {
        float v[4];
        ok = poll_head(xw(sm, g, XB_QKV, (kvl * G + warp) * kHeadDim), lane, in_tag, v, a.flags);
        qk_norm_rope(v, w4, cs, a.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) at.sq[warp][lane + 32 * i] = v[i];
    } else if (warp == G) {
        float v[4];
        ok = poll_head(xw(sm, g, XB_QKV, qrows + kvl * kHeadDim), lane, in_tag, v, a.flags);
        qk_norm_rope(v, w4, cs, a.eps);
        KT *dst = reinterpret_cast<KT *>(a.kc) + row_off;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const KT b = T::store(v[i]);
            snew_k[lane + 32 * i] = b;
            if (owner && ok) dst[lane + 32 * i] = b;
        }
    } else if (warp == G + 1) {
        float v[4];
        ok = poll_head(xw(sm, g, XB_QKV, qrows + hk * kHeadDim + kvl * kHeadDim), lane, in_tag, v, a.flags);
        KT *dst = reinterpret_cast<KT *>(a.vc) + row_off;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const KT b = T::store(v[i]);
            snew_v[lane + 32 * i] = b;
            if (owner && ok) dst[lane + 32 * i] = b;
        }
    }
    if (tr && tid == 0) tr[1] = gtime();
    if (!all_ok(ok)) return kFailed;

    const int jj = lane >> 4, o16 = lane & 15;
    const float qscale = 0.08838834764831845f * kLog2e;  // 1/sqrt(128), log2 domain
    float qr[G][NP][PER], acc[G][NP][PER], M[G], Ls[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        Ls[h] = 0.f;
#pragma unroll
        for (int r = 0; r < NP; ++r)
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                qr[h][r][e] = at.sq[h][T::dim(o16, r, e)] * qscale;
                acc[h][r][e] = 0.f;
            }
    }
    if (tr && tid == 0) tr[2] = gtime();
    bool dead = false, folded = false;
    for (int ch = 0; ch < p.nchunks; ++ch) {
        const unsigned slot = it % kSlots, par = (it / kSlots) & 1u;
        ++it;
        if (!take_slot(slot, par)) {
            dead = true;
            break;
        }
        uint8_t *sp = sm.slot[slot];
        int n = min(CH, p.p1 - (p.p0 + ch * CH));
        if (owner && ch == p.nchunks - 1) {
            // the owner appends this position's K and V rows to its last chunk (a slot half
            // holds one row more than a chunk), so the new position costs no separate pass
            constexpr int W16 = kHeadDim * (int)sizeof(KT) / 16;
            if (tid < 2 * W16) {
                const bool isv = tid >= W16;
                const uint4 *src = reinterpret_cast<const uint4 *>(isv ? (const void *)snew_v : (const void *)snew_k);
                reinterpret_cast<uint4 *>(sp + (isv ? kSlotBytes / 2 : 0) + (size_t)n * (W16 * 16))[tid % W16] =
                    src[tid % W16];
                fence_async_smem();  // ordered before the producer's next bulk copy into this slot
            }
            bar_consumers();
            ++n;
            folded = true;
        }
        attn_block<G, KT>(sp, sp + kSlotBytes / 2, n, warp, lane, qr, acc, M, Ls);
        release_slot(slot);
    }
    if (owner && !dead && !folded)
        attn_block<G, KT>(reinterpret_cast<const uint8_t *>(snew_k), reinterpret_cast<const uint8_t *>(snew_v), 1,
                          warp, lane, qr, acc, M, Ls);
    if (tr && tid == 0) tr[6] = gtime();
    // combine the two positions of each warp (lanes with equal o16 share dims)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        Ls[h] += __shfl_xor_sync(0xffffffffu, Ls[h], 16);
#pragma unroll
        for (int r = 0; r < NP; ++r)
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[h][r][e] += __shfl_xor_sync(0xffffffffu, acc[h][r][e], 16);
    }
    if (jj == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int r = 0; r < NP; ++r)
#pragma unroll
                for (int e = 0; e < PER; ++e) at.wacc[warp][h][T::dim(o16, r, e)] = acc[h][r][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            at.wml[warp][h][0] = M[h];
            at.wml[warp][h][1] = Ls[h];
        }
    }
    bar_consumers();
    // combine the warps into this split's tagged partial (exact rescaling to the common max)
    const unsigned part_tag = xtag(a, l, TK_PART), o_tag = xtag(a, l, TK_O);
    for (int t = tid; t < G * kHeadDim; t += kConsumerThreads) {
        const int h = t / kHeadDim, dim = t % kHeadDim;
        float mx = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, at.wml[w][h][0]);
        float av = 0.f, ls = 0.f;
        if (mx != -INFINITY) {
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = at.wml[w][h][0];
                if (mw == -INFINITY) continue;
                const float sc = exp2f(mw - mx);
                av = fmaf(at.wacc[w][h][dim], sc, av);
                ls = fmaf(at.wml[w][h][1], sc, ls);
            }
        }
        if (S == 1) {  // the only split: its result is the group's output
            st_tag(xw(sm, g, XB_O, (kvl * G + h) * kHeadDim + dim), av / ls, o_tag);
            continue;
        }
        const int pb = ((kvl * S + p.s) * G + h) * kPartStride;
        st_tag(xw(sm, g, XB_PART, pb + dim), av, part_tag);
        if (dim == 0) {
            st_tag(xw(sm, g, XB_PART, pb + kHeadDim), mx, part_tag);
            st_tag(xw(sm, g, XB_PART, pb + kHeadDim + 1), ls, part_tag);
        }
    }
    if (S == 1) return (int)(it | (dead ? kDeadBit : 0u));
    // Split s merges outputs [G 128 s / S, G 128 (s+1) / S) of the KV head from all S partials:
    // o = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s, splits in order.
    const int o0 = G * kHeadDim * p.s / S, o1 = G * kHeadDim * (p.s + 1) / S, cnt = o1 - o0;
    const int n_ml = 2 * G * S, items = n_ml + S * cnt;
    float *mrg = at.mrg;
    bool pok = true;
    for (int t = tid; t < items && pok; t += kConsumerThreads) {
        int word;
        if (t < n_ml) {
            const int sp = t / (2 * G), h = (t / 2) % G, which = t & 1;
            word = ((kvl * S + sp) * G + h) * kPartStride + kHeadDim + which;
        } else {
            const int t2 = t - n_ml, sp = t2 / cnt, oo = o0 + t2 % cnt;
            word = ((kvl * S + sp) * G + oo / kHeadDim) * kPartStride + oo % kHeadDim;
        }
        const unsigned long long *src = xw(sm, g, XB_PART, word);
        unsigned long long w;
        unsigned long long t0 = 0;
        for (unsigned i = 0;; ++i) {
            w = ld_tag(src);
            if (tag_is(w, part_tag)) break;
            if (!poll_more(i, t0, a.flags, WS_MERGE)) {
                pok = false;
                break;
            }
        }
        mrg[t] = tag_val(w);
    }
    if (!all_ok(pok)) return kFailed;
    if (tr && tid == 0) tr[7] = gtime();
    for (int t = tid; t < cnt; t += kConsumerThreads) {
        const int oo = o0 + t, h = oo / kHeadDim;
        float mx = -INFINITY;
        for (int sp = 0; sp < S; ++sp) mx = fmaxf(mx, mrg[sp * 2 * G + 2 * h]);
        float av = 0.f, ls = 0.f;
        for (int sp = 0; sp < S; ++sp) {
            const float ms = mrg[sp * 2 * G + 2 * h];
            if (ms == -INFINITY) continue;
            const float sc = exp2f(ms - mx);
            av = fmaf(mrg[n_ml + sp * cnt + t], sc, av);
            ls = fmaf(mrg[sp * 2 * G + 2 * h + 1], sc, ls);
        }
        st_tag(xw(sm, g, XB_O, kvl * G * kHeadDim + oo), av / ls, o_tag);
    }
    return (int)(it | (dead ? kDeadBit : 0u));
}

template <int D, int WF, typename KT>
__device__ void consumer() {
    constexpr int G = kBlockG;
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int tid = ctid();
    if (tid == 0) {
        const int tok = a.token >= 0 ? a.token : a.flags->next_tok;
        sm.tok = tok;
        sm.bad = 0;
        sm.fail = 0;
        const bool valid = tok >= 0 && tok < a.V;
        sm.flag = valid && !ld_relaxed(&a.flags->abort);
        if (!valid) raise_error(a.flags, kErrInvalidArgument, true);
    }
    bar_consumers();
    if (!sm.flag) return;
    // the residual stream starts as the embedding of the input token (every CTA keeps all of it)
    for (int j = tid; j < kBlockH / 2; j += kConsumerThreads) {
        const uint32_t u = reinterpret_cast<const uint32_t *>(a.embed + (size_t)sm.tok * kBlockH)[j];
        sm.x[2 * j] = bf_lo(u);
        sm.x[2 * j + 1] = bf_hi(u);
        if ((a.debug & 1) && sm.cidx == 0) {
            a.hidden[2 * j] = bf_lo(u);
            a.hidden[2 * j + 1] = bf_hi(u);
        }
    }
    if (tid == 0) sm.ph = 0;
    bar_consumers();
    unsigned it = 0;
    // one phase: stamp the trace, fold its status into the ring position
    auto step = [&](int ph, int r) -> bool {
        if (r == kFailed) return false;  // uniform: decided at a barrier
        if (((unsigned)r & kDeadBit) && clane() == 0) raise_error(a.flags, kErrInvariant, true);
        it = (unsigned)r & ~kDeadBit;
        // the barrier guards the shared vector (and attention scratch) the next phase restages
        bar_consumers();
        if (tid == 0) {
            sm.ph = ph + 1;  // read by expiring waits of the next phase
            unsigned long long *tr = trace_of(a, ph);
            if (tr) {
                tr[3] = gtime();
                tr[14] = clock64();
            }
        }
        return true;
    };
    // every row-streaming phase (and the head) runs through one call site, so one copy of the
    // code serves them all and stays in the instruction cache
    const int nph = kPhasesPerLayer * a.L + 1;
#pragma unroll 1
    for (int ph = 0; ph < nph; ++ph) {
        const int r = phase_type(a, ph) == T_ATTN ? attn_phase<G, KT>(ph, it) : gemv_phase<D, WF>(ph, it);
        if (!step(ph, r)) return;
    }
    if (tid == 0) {
        unsigned long long b = 0;
        for (int w = 0; w < kConsumerWarps; ++w) b = sm.best[w] > b ? sm.best[w] : b;
        if (sm.bad) raise_error(a.flags, kErrNumerical, false);
        unsigned long long *key = a.key + (a.step & 1u);
        if (b) atomicMax(key, b);
        __threadfence();
        const unsigned old = atomicAdd(a.sync, 1u);
        if (old + 1u == a.target) {  // the last CTA of this step
            __threadfence();
            const unsigned long long k = atomicAdd(key, 0ull);
            const int tok = k ? (int)(0xffffffffu - (unsigned)(k & 0xffffffffull)) : 0;
            a.flags->next_tok = tok;
            if (a.tok_out) *a.tok_out = tok;
            a.key[(a.step + 1u) & 1u] = 0ull;  // ready for the next step
        }
    }
}

template <int D, int WF, typename KT>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
    Smem &sm = smem();
    const int tid = threadIdx.x;
    if (tid == 0) {
        sm.args = a;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const unsigned s = smid();
        const uint16_t role = s < (unsigned)kMaxSmIds ? a.role[s] : kNoRole;
        const int g = role >> 12, r = role & 0xfff;
        sm.ok = role != kNoRole && g < D && a.D == D && r < a.n_grp[g];
        sm.g = sm.ok ? g : 0;
        sm.r = sm.ok ? r : 0;
        sm.cidx = sm.g == 0 ? sm.r : a.n_grp[0] + sm.r;
    }
    // the exchange plan, read on every exchange access
    for (int i = tid; i < (int)(sizeof(XPlan) / 4); i += kDecodeThreads)
        reinterpret_cast<uint32_t *>(&sm.plan)[i] = reinterpret_cast<const uint32_t *>(a.xplan)[i];
    __syncthreads();
    if (!sm.ok) {
        if (tid == 0) {
            atomicCAS(&a.flags->diag, 0u, ((unsigned)WS_ROLE << 24) | ((blockIdx.x & 0xfffu) << 12));
            raise_error(a.flags, kErrInvariant, true);
        }
        return;
    }
    if (tid >= kConsumerThreads) {
        if (tid == kConsumerThreads) producer();
        return;
    }
    consumer<D, WF, KT>();
}

}  // namespace
}  // namespace qw
