// decode.cu - one batch-one decode step of the Qwen3 decoder as a single
// persistent kernel for sm_103a (GB300).
//
// The step ("Scalar-Native Qwen3 Reference Runtime As The Numerical Authority",
// section 2 steps 1-7; the decode schedule of "Portable WebAssembly Runtime
// Architecture for TinyRustLM", section "Prefill versus decode") is split into
// 5 phases per layer plus one head phase:
//   QKV     h = RMSNorm(x) (folded into the activation staging), q|k|v = W h
//   ATTN    per (KV head, split): QK-Norm + RoPE of the group's queries and of the
//           new key, append k,v at this position, online softmax over a slice of
//           the cache, a partial (acc, max, sum) per query head
//   OPROJ   merge the partials, x = x + Wo o
//   GATEUP  h2 = RMSNorm(x), a = silu(Wg h2) * (Wu h2)
//   DOWN    x = x + Wd a
//   LMHEAD  logits = E RMSNorm(x), packed-key atomicMax argmax (ties -> lowest id)
//
// Layout on the GPU: one CTA per SM (cooperative launch, so all CTAs are
// resident), 7 consumer warps and 1 producer warp.  The producer streams, with
// bulk async copies (cp.async.bulk + mbarrier transaction counts), every weight
// row and cached K/V row its CTA will consume during the whole step into a ring
// of shared-memory slots.  Weights do not depend on the step's data, so the ring
// keeps HBM busy across phase boundaries while consumers wait for the previous
// phase.  Every output row is owned by one warp, so results do not depend on
// timing.  Every wait is bounded in time: on expiry the kernel records
// QW_INTERNAL_INVARIANT, raises an abort flag that every other wait also
// watches, drains its own copies in flight and returns.
//
// Data between phases travels as tagged words: 64-bit stores of (tag << 32 |
// f32 bits), tag = step sequence * 512 + producing phase + 1.  One thread per
// CTA waits on a per-phase arrival counter, then the CTA reads the words it needs
// and re-polls any whose tag does not match yet; a naturally aligned 64-bit
// access is single-copy atomic, so a matching tag guarantees the value and the
// producer needs no release fence before its arrival.  Buffers are reused every
// layer; a writer never overwrites words a reader still needs, because every
// phase reads the whole output of the phase before it: e.g. down(l) rewrites xa
// only after reading all of gate/up(l), which every CTA produces after its own
// qkv(l) read of xa.  The residual stream alternates between xa (written by down,
// read by qkv and the head) and xb (written by o_proj, read by gate/up).
//
// The kernel arguments are copied to shared memory at start, so phase bodies read
// them with shared loads; each lane keeps its columns of the phase's activation in
// registers while it streams rows.
#include <cstddef>

#include "qw_internal.h"

namespace qw {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxVec = 3072;  // longest activation vector staged in shared memory

// Every array member is 16-byte aligned: slots are bulk-copy destinations, vec, sk and
// sv are read with 16-byte vector loads.
struct __align__(16) Smem {
    alignas(16) uint8_t slot[kSlots][kSlotBytes];
    alignas(16) float wacc[kConsumerWarps][2][kHeadDim];  // attention: per-warp accumulators (group <= 2)
    alignas(16) float wml[kConsumerWarps][2][2];          // attention: per-warp running max, sum
    alignas(16) float sq[2][kHeadDim];                    // attention: normalised, rotated queries
    alignas(16) float sk[kHeadDim];                       // attention: this position's key (cache element type)
    alignas(16) float sv[kHeadDim];                       // attention: this position's value (cache element type)
    alignas(16) float vec[kMaxVec];                       // the phase's activation vector (staged once per CTA)
    alignas(16) float xown[kMaxOwnRows];                  // this CTA's residual rows, kept for the whole step
    alignas(16) unsigned long long full[kSlots];
    alignas(16) unsigned long long empty[kSlots];
    alignas(16) unsigned long long best[kConsumerWarps];  // head: per-warp argmax keys
    alignas(16) float red[kConsumerWarps];                // block reductions
    int fail;                                             // a consumer thread's poll gave up
    int flag;
    int tok;
    int bad;
    alignas(16) DecodeArgs args;                          // this launch's arguments
};
static_assert(offsetof(Smem, vec) % 16 == 0 && offsetof(Smem, sk) % 16 == 0 && offsetof(Smem, sv) % 16 == 0,
              "vector-accessed shared arrays must be 16-byte aligned");
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

// Polls use relaxed loads at gpu scope: the data and flags live in this GPU's memory, and
// system-scope (volatile) loads would also have to stay coherent with the host side.
__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_add(unsigned *p, unsigned v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void raise_error(StepFlags *f, unsigned code, bool abort) {
    atomicCAS(&f->err, 0u, code);
    if (abort) atomicExch(&f->abort, 1u);
}

// Bounded poll bookkeeping: true to keep polling, false on abort or timeout.
__device__ __forceinline__ bool poll_more(unsigned i, unsigned long long &t0, StepFlags *f, bool watch_abort = true) {
    if ((i & 15u) != 15u) return true;
    if (watch_abort && ld_relaxed(&f->abort)) return false;
    const unsigned long long t = gtime();
    if (t0 == 0) {
        t0 = t;
    } else if (t - t0 > kWaitLimitNs) {
        raise_error(f, kErrInvariant, true);
        return false;
    }
    return true;
}

// Bounded wait for an mbarrier phase; watch_abort = false only while draining.
__device__ __forceinline__ bool mbar_wait(unsigned long long *b, unsigned parity, StepFlags *f,
                                          bool watch_abort = true) {
    unsigned long long t0 = 0;
    for (unsigned i = 0; !mbar_test(b, parity); ++i)
        if (!poll_more(i, t0, f, watch_abort)) return false;
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

__device__ __forceinline__ unsigned phase_tag(const DecodeArgs &a, int ph) { return a.tag_base + (unsigned)ph + 1u; }

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

enum { T_QKV = 0, T_ATTN = 1, T_OPROJ = 2, T_GATEUP = 3, T_DOWN = 4, T_LMHEAD = 5 };

struct Phase {
    int type, l;
    // row-streaming phases
    int R, K, i8, pair, rpc, r0, r1;
    // attention
    int kvh, s, p0, p1;
    int nchunks;
};

__device__ __forceinline__ int phase_type(const DecodeArgs &a, int ph) {
    return ph / kPhasesPerLayer >= a.L ? T_LMHEAD : ph % kPhasesPerLayer;
}

__device__ __forceinline__ Phase describe(const DecodeArgs &a, int ph, int cta, int ncta) {
    Phase p;
    p.l = ph / kPhasesPerLayer;
    p.type = phase_type(a, ph);
    p.i8 = 0;
    p.pair = 0;
    p.nchunks = 0;
    p.kvh = p.s = p.p0 = p.p1 = 0;
    p.R = p.K = p.rpc = p.r0 = p.r1 = 0;
    if (p.type == T_ATTN) {
        int S = a.n_split;
        if (cta < a.Hkv * S) {
            p.kvh = cta / S;
            p.s = cta % S;
            p.p0 = (int)((long long)a.pos * p.s / S);
            p.p1 = (int)((long long)a.pos * (p.s + 1) / S);
            const int ch = kv_chunk_rows(a.kv_f32 ? 4 : 2);
            p.nchunks = (p.p1 - p.p0 + ch - 1) / ch;
        } else {
            p.kvh = -1;
        }
        return p;
    }
    switch (p.type) {
        case T_QKV: p.R = (a.Hq + 2 * a.Hkv) * kHeadDim; p.K = a.H; break;
        case T_OPROJ: p.R = a.H; p.K = a.Hq * kHeadDim; break;
        case T_GATEUP: p.R = a.I; p.K = a.H; p.pair = 1; break;
        case T_DOWN: p.R = a.H; p.K = a.I; break;
        default: p.R = a.V; p.K = a.H; break;
    }
    p.i8 = (p.type != T_LMHEAD) && a.fmt == 1;
    // output rows per slot; a multiple of 2 x the consumer warps when possible, as each
    // warp takes two rows per pass
    const int bpr = (p.pair ? 2 : 1) * (p.i8 ? p.K + p.K / 16 : 2 * p.K);
    p.rpc = kSlotBytes / bpr;
    if (p.rpc > 32) p.rpc = 32;
    if (p.rpc >= 2 * kConsumerWarps) p.rpc -= p.rpc % (2 * kConsumerWarps);
    else if (p.rpc >= kConsumerWarps) p.rpc = kConsumerWarps;
    p.r0 = (int)((long long)p.R * cta / ncta);
    p.r1 = (int)((long long)p.R * (cta + 1) / ncta);
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

// rows [row, row+count) of one [out, K] matrix into stored rows [j0, j0+count) of a slot holding ns rows
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

__device__ __forceinline__ void issue_chunk(Issuer &is, const DecodeArgs &a, const Phase &p, int c) {
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
    if (p.type == T_QKV) {
        const int qr = a.Hq * kHeadDim, kr = a.Hkv * kHeadDim, b = a0 + n;
        // q rows [0, qr), k rows [qr, qr+kr), v rows [qr+kr, qr+2kr)
        int lo = a0, hi = min(b, qr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[0], Ly.s[0], lo, hi - lo);
        lo = max(a0, qr);
        hi = min(b, qr + kr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[1], Ly.s[1], lo - qr, hi - lo);
        lo = max(a0, qr + kr);
        hi = b;
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[2], Ly.s[2], lo - qr - kr, hi - lo);
    } else if (p.type == T_OPROJ) {
        copy_rows(is, p, n, 0, Ly.w[3], Ly.s[3], a0, n);
    } else if (p.type == T_GATEUP) {
        copy_rows(is, p, 2 * n, 0, Ly.w[4], Ly.s[4], a0, n);
        copy_rows(is, p, 2 * n, n, Ly.w[5], Ly.s[5], a0, n);
    } else {
        copy_rows(is, p, n, 0, Ly.w[6], Ly.s[6], a0, n);
    }
}

__device__ __noinline__ void producer() {
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const unsigned long long pol_w = policy_evict_first();
    const unsigned long long pol_kv = policy_evict_normal();
    unsigned it = 0;
    bool ok = true;
    const int nph = kPhasesPerLayer * a.L + 1;
    for (int ph = 0; ph < nph && ok; ++ph) {
        const Phase p = describe(a, ph, cta, ncta);
        unsigned long long *tr = a.trace ? a.trace + ((size_t)ph * ncta + cta) * kTraceStamps : nullptr;
        for (int c = 0; c < p.nchunks; ++c) {
            const unsigned slot = it % kSlots, par = ((it / kSlots) & 1u) ^ 1u;
            if (!mbar_wait(&sm.empty[slot], par, a.flags)) {
                ok = false;
                break;
            }
            if (tr) {
                if (c == 0) tr[4] = gtime();
                if (c == p.nchunks - 1) tr[5] = gtime();
            }
            Issuer is{sm.slot[slot], &sm.full[slot], p.type == T_ATTN ? pol_kv : pol_w, 0u, false};
            issue_chunk(is, a, p, c);
            mbar_expect_tx(&sm.full[slot], is.bytes);
            is.go = true;
            issue_chunk(is, a, p, c);
            ++it;
        }
    }
    if (!ok) {
        // drain: the last chunk issued into each slot must land before the CTA exits
        for (unsigned s = 0; s < (unsigned)kSlots && s < it; ++s) {
            const unsigned last = ((it - 1 - s) / kSlots) * kSlots + s;
            mbar_wait(&sm.full[s], (last / kSlots) & 1u, a.flags, false);
        }
    }
}

// ---------------------------------------------------------------------- consumer

constexpr int kFailed = -1;                 // uniform: the step is aborting
constexpr unsigned kDeadBit = 0x80000000u;  // this warp gave up inside a chunk loop
constexpr int kFusedChunks = kSlots - 2;     // phases with at most this many chunks take them all at once

__device__ __forceinline__ int ctid() { return threadIdx.x; }
__device__ __forceinline__ int cwarp() { return threadIdx.x >> 5; }
__device__ __forceinline__ int clane() { return threadIdx.x & 31; }

__device__ __forceinline__ unsigned long long *trace_of(const DecodeArgs &a, int ph) {
    return a.trace ? a.trace + ((size_t)ph * gridDim.x + blockIdx.x) * kTraceStamps : nullptr;
}

// Wait for a slot to fill; warp-uniform result.
__device__ __forceinline__ bool take_slot(unsigned slot, unsigned par) {
    Smem &sm = smem();
    const bool ok = mbar_wait(&sm.full[slot], par, sm.args.flags);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void release_slot(unsigned slot) {
    __syncwarp();
    if (clane() == 0) mbar_arrive(&smem().empty[slot]);
}

// Thread 0 polls (bounded) until every CTA has arrived at phase ph - 1 of this step;
// the data itself is then read with tag checks, so the arrival needs no release fence.
__device__ __forceinline__ bool phase_wait(int ph) {
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    if (ctid() == 0) {
        bool ok = !ld_relaxed(&a.flags->abort);
        if (ok && ph > 0) {
            const unsigned *ctr = a.sync + ph - 1;
            unsigned long long t0 = 0;
            for (unsigned i = 0; ld_relaxed(ctr) < a.target; ++i)
                if (!poll_more(i, t0, a.flags)) {
                    ok = false;
                    break;
                }
        }
        sm.flag = ok;
    }
    bar_consumers();
    return sm.flag != 0;
}

// Make a per-thread poll result uniform over the consumer threads (one barrier).
__device__ __forceinline__ bool all_ok(bool ok) {
    Smem &sm = smem();
    if (!ok) sm.fail = 1;
    bar_consumers();
    return sm.fail == 0;
}

// Float4 slots per consumer thread for a vector of 1024*KM floats (index tid + NT*i).
template <int KM>
__host__ __device__ constexpr int vec_iters() { return (256 * KM + kConsumerThreads - 1) / kConsumerThreads; }

// Poll the thread's float4 slots tid + NT*i (< 256 KM) of a tagged vector of 1024*KM words.
template <int KM>
__device__ __forceinline__ bool poll_vec(const unsigned long long *src, unsigned tag, float4 (&v)[vec_iters<KM>()],
                                         StepFlags *f) {
    constexpr int NI = vec_iters<KM>();
    unsigned long long w[NI][4];
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
        bool ok = true;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int idx = ctid() + kConsumerThreads * k;
            if (idx < 256 * KM) {
                const unsigned long long *p = src + 4 * idx;
                ld_tag2(p, w[k][0], w[k][1]);
                ld_tag2(p + 2, w[k][2], w[k][3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) ok &= tag_is(w[k][e], tag);
            }
        }
        if (ok) break;
        if (!poll_more(i, t0, f)) return false;
    }
#pragma unroll
    for (int k = 0; k < NI; ++k)
        v[k] = make_float4(tag_val(w[k][0]), tag_val(w[k][1]), tag_val(w[k][2]), tag_val(w[k][3]));
    return true;
}

// Raw weight piece m (8 columns 8*(lane + 32 m) ..) of one stored row: 16 bytes of
// bf16, or 8 bytes of int8 codes plus their group's fp16 scale.  row points at the
// row's weights in a slot; srow at its scales (int8 only).
template <int KM, bool I8>
struct WPiece;
template <int KM>
struct WPiece<KM, false> {
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *row, const uint8_t *, int lane, int m) {
        v = reinterpret_cast<const uint4 *>(row)[lane + 32 * m];
    }
    __device__ __forceinline__ void unpack(float (&w)[8]) const {
        w[0] = bf_lo(v.x); w[1] = bf_hi(v.x); w[2] = bf_lo(v.y); w[3] = bf_hi(v.y);
        w[4] = bf_lo(v.z); w[5] = bf_hi(v.z); w[6] = bf_lo(v.w); w[7] = bf_hi(v.w);
    }
};
template <int KM>
struct WPiece<KM, true> {
    uint2 v;
    __half s;
    __device__ __forceinline__ void load(const uint8_t *row, const uint8_t *srow, int lane, int m) {
        v = reinterpret_cast<const uint2 *>(row)[lane + 32 * m];
        s = reinterpret_cast<const __half *>(srow)[(lane + 32 * m) >> 2];
    }
    // int8 group-32 codes dequantised in registers: w = f32(q) * f32(s), an exact product
    __device__ __forceinline__ void unpack(float (&w)[8]) const {
        const float sf = __half2float(s);
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = i8f(v.x, e) * sf;
#pragma unroll
        for (int e = 0; e < 4; ++e) w[4 + e] = i8f(v.y, e) * sf;
    }
};

// Stored row j of a slot holding ns rows: weights, and (int8) scales.
template <int KM, bool I8>
__device__ __forceinline__ const uint8_t *slot_row(const uint8_t *sp, int j) {
    return sp + (size_t)j * (I8 ? 1024 * KM : 2048 * KM);
}
template <int KM, bool I8>
__device__ __forceinline__ const uint8_t *slot_scales(const uint8_t *sp, int ns, int j) {
    return I8 ? sp + (size_t)ns * (1024 * KM) + (size_t)j * (64 * KM) : nullptr;
}

// Dot products of NR stored rows with the activation held in registers
// (act[8 m + e] = activation column 8*(lane + 32 m) + e).  All weight loads of the
// row group are issued before any arithmetic, and the accumulation chains of the
// rows are interleaved; rows must be valid (callers repeat a valid row for unused ones).
template <int KM, bool I8, int NR>
__device__ __forceinline__ void dot_rows(const uint8_t *const (&rp)[NR], const uint8_t *const (&sc)[NR], int lane,
                                         const float *act, float (&out)[NR]) {
    WPiece<KM, I8> wp[NR][4 * KM];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < 4 * KM; ++m) wp[r][m].load(rp[r], sc[r], lane, m);
    float acc[NR][2];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float w[8];
            wp[r][m].unpack(w);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][0] = fmaf(w[e], act[8 * m + e], acc[r][0]);
#pragma unroll
            for (int e = 4; e < 8; ++e) acc[r][1] = fmaf(w[e], act[8 * m + e], acc[r][1]);
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) out[r] = acc[r][0] + acc[r][1];
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int r = 0; r < NR; ++r) out[r] += __shfl_xor_sync(0xffffffffu, out[r], o);
}

// Row-streaming phase PT: stage the activation vector in shared memory once per CTA
// (RMSNorm folded in where the phase normalises), then each warp owns whole rows
// (two at a time) of each chunk.  Thread t stages float4 slots t + NT*i.
// Returns the new ring position (kDeadBit set if this warp gave up) or kFailed.
template <int PT, int KM, bool I8, int G>
__device__ __forceinline__ int gemv_phase(int ph, unsigned it) {
    constexpr bool norm = PT == T_QKV || PT == T_GATEUP || PT == T_LMHEAD;
    constexpr bool pair = PT == T_GATEUP;
    constexpr int NI = vec_iters<KM>();
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int tid = ctid(), warp = cwarp(), lane = clane();
    const Phase p = describe(a, ph, blockIdx.x, gridDim.x);
    const bool embed = PT == T_QKV && p.l == 0;
    const int own0 = (int)((long long)a.H * blockIdx.x / gridDim.x);
    const unsigned in_tag = ph ? phase_tag(a, ph - 1) : 0u, out_tag = phase_tag(a, ph);
    unsigned long long *tr = trace_of(a, ph);
    // read-only inputs first: they do not depend on the previous phase, so their
    // latency overlaps the wait
    float4 nw[NI], v[NI];
    if constexpr (norm) {
        const __nv_bfloat16 *w = PT == T_QKV    ? a.layers[p.l].input_norm
                                 : PT == T_GATEUP ? a.layers[p.l].post_norm
                                                  : a.final_norm;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int idx = tid + kConsumerThreads * i;
            if (idx < 256 * KM) {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(w) + idx);
                nw[i] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
            }
        }
    }
    if (tr && tid == 0) tr[0] = gtime();
    if (!phase_wait(ph)) return kFailed;
    bool ok = true;
    float4 *vec4 = reinterpret_cast<float4 *>(sm.vec);
    {
        if (embed) {
            const uint2 *row = reinterpret_cast<const uint2 *>(a.embed + (size_t)sm.tok * a.H);
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int idx = tid + kConsumerThreads * i;
                v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (idx < 256 * KM) {
                    const uint2 u = __ldg(row + idx);
                    v[i] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
                    if ((a.debug & 1) && blockIdx.x == 0) reinterpret_cast<float4 *>(a.hidden)[idx] = v[i];
                }
            }
        } else {
            const unsigned long long *src = PT == T_GATEUP ? a.xb : PT == T_DOWN ? a.actt : PT == T_OPROJ ? a.ot : a.xa;
            ok = poll_vec<KM>(src, in_tag, v, a.flags);
        }
    }
    if (tr && tid == 0) tr[1] = gtime();
    if constexpr (norm) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i)
            if (tid + kConsumerThreads * i < 256 * KM)
                ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        ss = warp_sum(ss);
        if (lane == 0) sm.red[warp] = ss;
        if (!all_ok(ok)) return kFailed;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += sm.red[w];
        const float r = rsqrtf(tot * (1.0f / (1024.0f * KM)) + a.eps);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int idx = tid + kConsumerThreads * i;
            if (idx < 256 * KM)
                vec4[idx] = make_float4(nw[i].x * (v[i].x * r), nw[i].y * (v[i].y * r), nw[i].z * (v[i].z * r),
                                        nw[i].w * (v[i].w * r));
        }
    } else {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int idx = tid + kConsumerThreads * i;
            if (idx < 256 * KM) vec4[idx] = v[i];
        }
    }
    if (!all_ok(ok)) return kFailed;
    // each lane keeps its 32*KM activation columns in registers for the whole phase
    float areg[8 * 4 * KM];
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m) {
        reinterpret_cast<float4 *>(areg)[2 * m] = reinterpret_cast<const float4 *>(sm.vec + 8 * (lane + 32 * m))[0];
        reinterpret_cast<float4 *>(areg)[2 * m + 1] = reinterpret_cast<const float4 *>(sm.vec + 8 * (lane + 32 * m))[1];
    }
    unsigned long long best = 0;
    bool bad = false, dead = false;
    // the value of output row (CTA-local index g) -> its destination (lane 0 only)
    auto emit = [&](int g, float v, float up) {
        const int row = p.r0 + g;
        if constexpr (PT == T_GATEUP) {
            st_tag(a.actt + row, (v / (1.0f + __expf(-v))) * up, out_tag);
        } else if constexpr (PT == T_QKV) {
            st_tag(a.qkvt + row, v, out_tag);
        } else if constexpr (PT == T_OPROJ || PT == T_DOWN) {
            // the residual rows of this CTA live in shared memory for the whole step
            const float nx = sm.xown[row - own0] + v;
            sm.xown[row - own0] = nx;
            st_tag((PT == T_OPROJ ? a.xb : a.xa) + row, nx, out_tag);
            if (PT == T_DOWN && (a.debug & 1)) a.hidden[(size_t)(p.l + 1) * a.H + row] = nx;
        } else {
            a.logits[row] = v;
            if (isfinite(v)) {
                const unsigned long long k = argmax_key(v, row);
                best = k > best ? k : best;
            } else {
                bad = true;
            }
        }
    };
    if (PT != T_LMHEAD && p.nchunks <= kFusedChunks) {
        // Every chunk of the phase fits in the ring at once: take them all, then each warp
        // computes its rows g = warp, warp + 7, ... in as few passes as possible (the rows
        // of one pass may sit in different slots), then release every chunk.
        const unsigned it0 = it;
        for (int ch = 0; ch < p.nchunks && !dead; ++ch)
            dead = !take_slot((it0 + ch) % kSlots, ((it0 + ch) / kSlots) & 1u);
        it += p.nchunks;
        if (!dead) {
            constexpr int NRW = pair ? 3 : (KM == 1 ? 4 : 1);  // rows (gate/up pairs) per pass
            constexpr int NR = pair ? 2 * NRW : NRW;
            const int R = p.r1 - p.r0;
            for (int g0 = warp; g0 < R; g0 += NRW * kConsumerWarps) {
                const uint8_t *rp[NR], *sc[NR];
                int cnt = 0;
#pragma unroll
                for (int i = 0; i < NRW; ++i) {
                    int g = g0 + i * kConsumerWarps;
                    if (g < R) cnt = i + 1;
                    else g = g0;  // an unused row repeats a valid one
                    const int c = g / p.rpc, j = g - c * p.rpc;
                    const int n = min(p.rpc, R - c * p.rpc), ns = pair ? 2 * n : n;
                    const uint8_t *sp = sm.slot[(it0 + c) % kSlots];
                    if constexpr (pair) {
                        rp[2 * i] = slot_row<KM, I8>(sp, j);
                        sc[2 * i] = slot_scales<KM, I8>(sp, ns, j);
                        rp[2 * i + 1] = slot_row<KM, I8>(sp, n + j);
                        sc[2 * i + 1] = slot_scales<KM, I8>(sp, ns, n + j);
                    } else {
                        rp[i] = slot_row<KM, I8>(sp, j);
                        sc[i] = slot_scales<KM, I8>(sp, ns, j);
                    }
                }
                float o[NR];
                dot_rows<KM, I8, NR>(rp, sc, lane, areg, o);
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < NRW; ++i)
                        if (i < cnt) {
                            if constexpr (pair)
                                emit(g0 + i * kConsumerWarps, o[2 * i], o[2 * i + 1]);
                            else
                                emit(g0 + i * kConsumerWarps, o[i], 0.f);
                        }
                }
            }
            for (int ch = 0; ch < p.nchunks; ++ch) release_slot((it0 + ch) % kSlots);
        }
    } else {
        for (int ch = 0; ch < p.nchunks; ++ch) {
            const unsigned slot = it % kSlots, par = (it / kSlots) & 1u;
            ++it;
            if (!take_slot(slot, par)) {
                dead = true;
                break;
            }
            const uint8_t *sp = sm.slot[slot];
            const int c0 = ch * p.rpc;
            const int n = min(p.rpc, p.r1 - p.r0 - c0);
            const int ns = pair ? 2 * n : n;
            for (int j = warp; j < n; j += 2 * kConsumerWarps) {
                const int j2 = j + kConsumerWarps;
                const int cnt = j2 < n ? 2 : 1;
                const int j2c = cnt == 2 ? j2 : j;  // an unused second row repeats the first
                if constexpr (pair) {
                    // gate row j, up row j (stored at n + j), and the same for j2
                    const uint8_t *rp[4] = {slot_row<KM, I8>(sp, j), slot_row<KM, I8>(sp, n + j),
                                            slot_row<KM, I8>(sp, j2c), slot_row<KM, I8>(sp, n + j2c)};
                    const uint8_t *sc[4] = {slot_scales<KM, I8>(sp, ns, j), slot_scales<KM, I8>(sp, ns, n + j),
                                            slot_scales<KM, I8>(sp, ns, j2c), slot_scales<KM, I8>(sp, ns, n + j2c)};
                    float o[4];
                    dot_rows<KM, I8, 4>(rp, sc, lane, areg, o);
                    if (lane == 0) {
                        emit(c0 + j, o[0], o[1]);
                        if (cnt == 2) emit(c0 + j2, o[2], o[3]);
                    }
                } else {
                    const uint8_t *rp[2] = {slot_row<KM, I8>(sp, j), slot_row<KM, I8>(sp, j2c)};
                    const uint8_t *sc[2] = {slot_scales<KM, I8>(sp, ns, j), slot_scales<KM, I8>(sp, ns, j2c)};
                    float o[2];
                    dot_rows<KM, I8, 2>(rp, sc, lane, areg, o);
                    if (lane == 0) {
                        emit(c0 + j, o[0], 0.f);
                        if (cnt == 2) emit(c0 + j2, o[1], 0.f);
                    }
                }
            }
            release_slot(slot);
        }
    }
    if constexpr (PT == T_LMHEAD) {
        if (lane == 0) {
            sm.best[warp] = best;
            if (bad) atomicOr(&sm.bad, 1);
        }
    }
    return (int)(it | (dead ? kDeadBit : 0u));
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

// Poll a head's 128 tagged values as dims (lane, lane+32, lane+64, lane+96).
__device__ __forceinline__ bool poll_head(const unsigned long long *src, int lane, unsigned tag, float (&v)[4],
                                          StepFlags *f) {
    unsigned long long w[4];
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = ld_tag(src + lane + 32 * k);
        if (tag_is(w[0], tag) && tag_is(w[1], tag) && tag_is(w[2], tag) && tag_is(w[3], tag)) break;
        if (!poll_more(i, t0, f)) return false;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = tag_val(w[k]);
    return true;
}

// K/V element type of the cache: f32 (default) or bf16.
template <typename KT>
struct KvTraits;
template <>
struct KvTraits<float> {
    static constexpr int kPieces = 4;  // a lane's 16 dims = 4 x 16-byte pieces
    static constexpr int kPer = 4;     // elements per piece
    __device__ static __forceinline__ void load(const uint8_t *p, float (&o)[4]) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ static __forceinline__ float store(float v) { return v; }
};
template <>
struct KvTraits<__nv_bfloat16> {
    static constexpr int kPieces = 2;
    static constexpr int kPer = 8;
    __device__ static __forceinline__ void load(const uint8_t *p, float (&o)[8]) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        o[0] = bf_lo(v.x); o[1] = bf_hi(v.x); o[2] = bf_lo(v.y); o[3] = bf_hi(v.y);
        o[4] = bf_lo(v.z); o[5] = bf_hi(v.z); o[6] = bf_lo(v.w); o[7] = bf_hi(v.w);
    }
    __device__ static __forceinline__ __nv_bfloat16 store(float v) { return __float2bfloat16_rn(v); }
};

// Online-softmax update over n positions whose K and V rows (128 elements of KT each)
// sit at kb and vb.  Eight lanes share a position: lane (jj = lane/8, o8 = lane%8)
// takes dims [16*o8, 16*o8 + 16) of positions base + 4*warp + jj for base = 0, 4*NCW, ...
// Each lane visits its 16-byte pieces in an order rotated by f(o8), so the eight
// lanes of a shared-memory phase hit distinct banks; lanes with equal o8 share f,
// which keeps their accumulators aligned for the reduction over jj.
template <int G, typename KT>
__device__ __forceinline__ void attn_block(const uint8_t *kb, const uint8_t *vb, int n, int warp, int lane,
                                           const float (&qr)[G][KvTraits<KT>::kPieces][KvTraits<KT>::kPer],
                                           float (&acc)[G][KvTraits<KT>::kPieces][KvTraits<KT>::kPer],
                                           float (&M)[G], float (&Ls)[G]) {
    using T = KvTraits<KT>;
    constexpr int NP = T::kPieces, PER = T::kPer, ROWB = kHeadDim * (int)sizeof(KT);
    const int jj = lane >> 3, o8 = lane & 7, f = (o8 / (8 / NP)) % NP;
    for (int base = 0; base < n; base += 4 * kConsumerWarps) {
        const int jpos = base + 4 * warp + jj;
        const bool valid = jpos < n;
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
        if (valid) {
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                float kv[PER];
                T::load(kb + (size_t)jpos * ROWB + (size_t)(16 * o8 + ((r + f) % NP) * PER) * sizeof(KT), kv);
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
            const float s2 = valid ? s : -INFINITY;
            float mx = fmaxf(s2, __shfl_xor_sync(0xffffffffu, s2, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
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
                T::load(vb + (size_t)jpos * ROWB + (size_t)(16 * o8 + ((r + f) % NP) * PER) * sizeof(KT), vv);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[h][r][e] = fmaf(pr[h], vv[e], acc[h][r][e]);
            }
        }
    }
}

// One (KV head, split) item: QK-Norm + RoPE of the group's queries and of the new key,
// append k, v at this position (the last split owns it), online softmax over the
// split's cached positions (+ the new one), and the split's tagged partial (acc, max,
// sum) for each query head of the group; the CTA that finishes a KV head's last split
// merges the partials into the group's output.  A single split writes the output
// directly.
template <int G, typename KT>
__device__ __forceinline__ int attn_phase(int ph, unsigned it) {
    using T = KvTraits<KT>;
    constexpr int NP = T::kPieces, PER = T::kPer, CH = kv_chunk_rows((int)sizeof(KT));
    Smem &sm = smem();
    const DecodeArgs &a = sm.args;
    const int tid = ctid(), warp = cwarp(), lane = clane();
    const Phase p = describe(a, ph, blockIdx.x, gridDim.x);
    unsigned long long *tr = trace_of(a, ph);
    if (p.kvh < 0) {  // no attention item on this CTA
        if (tr && tid == 0) tr[0] = tr[1] = gtime();
        return (int)it;
    }
    const int S = a.n_split, P = a.pos, kvh = p.kvh, l = p.l;
    const bool owner = (p.s == S - 1);
    const DevLayer &Ly = a.layers[l];
    const unsigned in_tag = phase_tag(a, ph - 1), out_tag = phase_tag(a, ph);
    // read-only inputs before the wait: norm weights and this position's rotation
    float w4[4];
    float2 cs[2];
    if (warp <= G) {
        const __nv_bfloat16 *nw = warp < G ? Ly.q_norm : Ly.k_norm;
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = __bfloat162float(nw[lane + 32 * i]);
        const float2 *rope = a.rope + (size_t)P * (kHeadDim / 2);
        cs[0] = rope[lane];
        cs[1] = rope[lane + 32];
    }
    if (tr && tid == 0) tr[0] = gtime();
    if (!phase_wait(ph)) return kFailed;
    KT *snew_k = reinterpret_cast<KT *>(sm.sk), *snew_v = reinterpret_cast<KT *>(sm.sv);
    const size_t row_off = (((size_t)l * a.Hkv + kvh) * a.max_ctx + P) * kHeadDim;
    bool ok = true;
    if (warp < G) {
        float v[4];
        ok = poll_head(a.qkvt + (size_t)(kvh * G + warp) * kHeadDim, lane, in_tag, v, a.flags);
        qk_norm_rope(v, w4, cs, a.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.sq[warp][lane + 32 * i] = v[i];
    } else if (warp == G) {
        float v[4];
        ok = poll_head(a.qkvt + (size_t)(a.Hq + kvh) * kHeadDim, lane, in_tag, v, a.flags);
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
        ok = poll_head(a.qkvt + (size_t)(a.Hq + a.Hkv + kvh) * kHeadDim, lane, in_tag, v, a.flags);
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

    const int jj = lane >> 3, o8 = lane & 7, f = (o8 / (8 / NP)) % NP;
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
                qr[h][r][e] = sm.sq[h][16 * o8 + ((r + f) % NP) * PER + e] * qscale;
                acc[h][r][e] = 0.f;
            }
    }
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
        if (owner && ch == p.nchunks - 1 && n < CH) {
            // the owner appends this position's K and V rows to its last chunk (a slot half
            // holds more rows than a chunk), so the new position costs no separate pass
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
    // combine the four positions of each warp (lanes with equal o8 share a dim order)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        Ls[h] += __shfl_xor_sync(0xffffffffu, Ls[h], 8);
        Ls[h] += __shfl_xor_sync(0xffffffffu, Ls[h], 16);
#pragma unroll
        for (int r = 0; r < NP; ++r)
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                float v = acc[h][r][e];
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                acc[h][r][e] = v;
            }
    }
    if (jj == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int r = 0; r < NP; ++r)
#pragma unroll
                for (int e = 0; e < PER; ++e) sm.wacc[warp][h][16 * o8 + ((r + f) % NP) * PER + e] = acc[h][r][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            sm.wml[warp][h][0] = M[h];
            sm.wml[warp][h][1] = Ls[h];
        }
    }
    bar_consumers();
    // combine the warps into this split's tagged partial (exact rescaling to the common max)
    for (int t = tid; t < G * kHeadDim; t += kConsumerThreads) {
        const int h = t / kHeadDim, dim = t % kHeadDim;
        float mx = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm.wml[w][h][0]);
        float av = 0.f, ls = 0.f;
        if (mx != -INFINITY) {
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = sm.wml[w][h][0];
                if (mw == -INFINITY) continue;
                const float sc = exp2f(mw - mx);
                av = fmaf(sm.wacc[w][h][dim], sc, av);
                ls = fmaf(sm.wml[w][h][1], sc, ls);
            }
        }
        if (S == 1) {  // the only split: its result is the group's output
            st_tag(a.ot + (size_t)(kvh * G + h) * kHeadDim + dim, av / ls, out_tag);
            continue;
        }
        unsigned long long *pp = a.partt + ((size_t)(kvh * S + p.s) * G + h) * kPartStride;
        st_tag(pp + dim, av, out_tag);
        if (dim == 0) {
            st_tag(pp + kHeadDim, mx, out_tag);
            st_tag(pp + kHeadDim + 1, ls, out_tag);
        }
    }
    if (S == 1) return (int)(it | (dead ? kDeadBit : 0u));
    // The CTA that finishes the last split of this KV head merges all S partials into the
    // group's attention output (once, instead of in every o_proj CTA):
    // o = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s.
    // The count needs no fence: the merging CTA checks every word's tag and re-polls any
    // partial that is not visible yet.
    bar_consumers();
    if (tid == 0) {
        unsigned *ctr = a.merge + (size_t)l * kMaxKvHeads + kvh;
        sm.flag = atomicAdd(ctr, 1u) + 1u == (unsigned)S;
        if (sm.flag) *ctr = 0u;  // every split has counted; the next use is the next step
    }
    bar_consumers();
    if (sm.flag) {
        // warp w folds splits w, w + 7, w + 14 (one polling round), lane holds dims lane + 32 k
        constexpr int KS = kMaxSplits / kConsumerWarps;  // splits per warp
        static_assert(KS * kConsumerWarps >= kMaxSplits, "every split has a merging warp");
        float mw[G], lw[G], aw[G][4];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mw[h] = -INFINITY;
            lw[h] = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) aw[h][k] = 0.f;
        }
        unsigned long long w[KS][G][6];
        unsigned long long t0 = 0;
        bool ok = true;
        for (unsigned i = 0;; ++i) {
            bool got = true;
#pragma unroll
            for (int q = 0; q < KS; ++q) {
                const int sidx = warp + kConsumerWarps * q;
                if (sidx >= S) break;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const unsigned long long *pp = a.partt + ((size_t)(kvh * S + sidx) * G + h) * kPartStride;
                    ld_tag2(pp + kHeadDim, w[q][h][0], w[q][h][1]);
#pragma unroll
                    for (int k = 0; k < 4; ++k) w[q][h][2 + k] = ld_tag(pp + lane + 32 * k);
#pragma unroll
                    for (int e = 0; e < 6; ++e) got &= tag_is(w[q][h][e], out_tag);
                }
            }
            if (__all_sync(0xffffffffu, got)) break;
            if (!poll_more(i, t0, a.flags)) {
                ok = false;
                break;
            }
        }
        if (ok) {
#pragma unroll
            for (int q = 0; q < KS; ++q) {
                if (warp + kConsumerWarps * q >= S) break;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float ms = tag_val(w[q][h][0]);
                    if (ms == -INFINITY) continue;
                    const float mn = fmaxf(mw[h], ms);
                    const float sa = (mw[h] == -INFINITY) ? 0.f : exp2f(mw[h] - mn), sb = exp2f(ms - mn);
                    lw[h] = lw[h] * sa + tag_val(w[q][h][1]) * sb;
#pragma unroll
                    for (int k = 0; k < 4; ++k) aw[h][k] = aw[h][k] * sa + tag_val(w[q][h][2 + k]) * sb;
                    mw[h] = mn;
                }
            }
        }
        if (!all_ok(ok)) return kFailed;  // its barrier also ends every read of wacc / wml
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < 4; ++k) sm.wacc[warp][h][lane + 32 * k] = aw[h][k];
            if (lane == 0) {
                sm.wml[warp][h][0] = mw[h];
                sm.wml[warp][h][1] = lw[h];
            }
        }
        bar_consumers();
        for (int t = tid; t < G * kHeadDim; t += kConsumerThreads) {
            const int h = t / kHeadDim, dim = t % kHeadDim;
            float mx = -INFINITY;
            for (int w2 = 0; w2 < kConsumerWarps; ++w2) mx = fmaxf(mx, sm.wml[w2][h][0]);
            float av = 0.f, ls = 0.f;
            for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
                const float m2 = sm.wml[w2][h][0];
                if (m2 == -INFINITY) continue;
                const float sc = exp2f(m2 - mx);
                av = fmaf(sm.wacc[w2][h][dim], sc, av);
                ls = fmaf(sm.wml[w2][h][1], sc, ls);
            }
            st_tag(a.ot + (size_t)(kvh * G + h) * kHeadDim + dim, av / ls, out_tag);
        }
    }
    return (int)(it | (dead ? kDeadBit : 0u));
}

template <int PT, bool I8, int G>
__device__ __forceinline__ int gemv_km(int K, int ph, unsigned it) {
    switch (K >> 10) {
        case 1: return gemv_phase<PT, 1, I8, G>(ph, it);
        case 2: return gemv_phase<PT, 2, I8, G>(ph, it);
        default: return gemv_phase<PT, 3, I8, G>(ph, it);
    }
}

template <bool I8, int G>
__device__ __forceinline__ int gemv_dispatch(const DecodeArgs &a, int type, int ph, unsigned it) {
    switch (type) {
        case T_QKV: return gemv_km<T_QKV, I8, G>(a.H, ph, it);
        case T_OPROJ: return gemv_km<T_OPROJ, I8, G>(a.Hq * kHeadDim, ph, it);
        case T_GATEUP: return gemv_km<T_GATEUP, I8, G>(a.H, ph, it);
        case T_DOWN: return gemv_km<T_DOWN, I8, G>(a.I, ph, it);
        default: return gemv_km<T_LMHEAD, false, G>(a.H, ph, it);
    }
}

// One kernel per (group size, weight format, cache element type), so each carries only
// the phase code it runs.
template <int G, bool I8, typename KT>
__device__ void consumer() {
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
    // residual rows owned by this CTA start as the embedding of the input token
    const int own0 = (int)((long long)a.H * blockIdx.x / gridDim.x);
    const int own1 = (int)((long long)a.H * (blockIdx.x + 1) / gridDim.x);
    for (int j = tid; j < own1 - own0; j += kConsumerThreads)
        sm.xown[j] = __bfloat162float(a.embed[(size_t)sm.tok * a.H + own0 + j]);
    unsigned it = 0;
    const int nph = kPhasesPerLayer * a.L + 1;
    for (int ph = 0; ph < nph; ++ph) {
        const int type = phase_type(a, ph);
        int r;
        if (type == T_ATTN)
            r = attn_phase<G, KT>(ph, it);
        else
            r = gemv_dispatch<I8, G>(a, type, ph, it);
        unsigned long long *tr = trace_of(a, ph);
        if (tr && tid == 0) tr[2] = gtime();
        if (r == kFailed) return;  // uniform: decided at a barrier
        if (((unsigned)r & kDeadBit) && clane() == 0) raise_error(a.flags, kErrInvariant, true);
        it = (unsigned)r & ~kDeadBit;
        // arrive; the barrier also guards the shared activation vector the next phase restages
        bar_consumers();
        if (tid == 0) {
            if (type != T_LMHEAD) {
                red_add(a.sync + ph, 1u);
            } else {
                unsigned long long b = 0;
                for (int w = 0; w < kConsumerWarps; ++w) b = sm.best[w] > b ? sm.best[w] : b;
                if (sm.bad) raise_error(a.flags, kErrNumerical, false);
                unsigned long long *key = a.key + (a.step & 1u);
                if (b) atomicMax(key, b);
                __threadfence();
                const unsigned old = atomicAdd(a.sync + ph, 1u);
                if (old + 1u == a.target) {  // the last CTA of this step
                    __threadfence();
                    const unsigned long long k = atomicAdd(key, 0ull);
                    const int tok = k ? (int)(0xffffffffu - (unsigned)(k & 0xffffffffull)) : 0;
                    a.flags->next_tok = tok;
                    if (a.tok_out) *a.tok_out = tok;
                    a.key[(a.step + 1u) & 1u] = 0ull;  // ready for the next step
                }
            }
            if (tr) tr[3] = gtime();
        }
    }
}

template <int G, bool I8, typename KT>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
    Smem &sm = smem();
    if (threadIdx.x == 0) {
        sm.args = a;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= kConsumerThreads) {
        if (threadIdx.x == kConsumerThreads) producer();
        return;
    }
    consumer<G, I8, KT>();
}

// The kernel instantiation for (group, weight format, cache element type).
const void *decode_fn(int group, int fmt, int kv_f32) {
    if (group == 1) {
        if (fmt == 1) return kv_f32 ? (const void *)decode_kernel<1, true, float> : (const void *)decode_kernel<1, true, __nv_bfloat16>;
        return kv_f32 ? (const void *)decode_kernel<1, false, float> : (const void *)decode_kernel<1, false, __nv_bfloat16>;
    }
    if (fmt == 1) return kv_f32 ? (const void *)decode_kernel<2, true, float> : (const void *)decode_kernel<2, true, __nv_bfloat16>;
    return kv_f32 ? (const void *)decode_kernel<2, false, float> : (const void *)decode_kernel<2, false, __nv_bfloat16>;
}

__global__ void kv_widen_kernel(const __nv_bfloat16 *__restrict__ src, float *__restrict__ dst, long long heads,
                                int n_pos, int max_ctx) {
    const long long total = heads * n_pos * (kHeadDim / 8);  // 8 elements per thread step
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / (kHeadDim / 8), piece = i % (kHeadDim / 8);
        const long long h = row / n_pos, p = row % n_pos;
        const uint4 u = *reinterpret_cast<const uint4 *>(src + row * kHeadDim + piece * 8);
        float4 *o = reinterpret_cast<float4 *>(dst + (h * max_ctx + p) * kHeadDim + piece * 8);
        o[0] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
        o[1] = make_float4(bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w));
    }
}

}  // namespace

cudaError_t launch_kv_widen(const __nv_bfloat16 *src, float *dst, long long heads, int n_pos, int max_ctx,
                            cudaStream_t stream) {
    const long long total = heads * n_pos * (kHeadDim / 8);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 65536) blocks = 65536;
    if (blocks < 1) return cudaSuccess;
    kv_widen_kernel<<<(unsigned)blocks, threads, 0, stream>>>(src, dst, heads, n_pos, max_ctx);
    return cudaGetLastError();
}

size_t decode_smem_bytes() { return sizeof(Smem); }

cudaError_t decode_prepare(int group, int *blocks_per_sm) {
    const int bytes = (int)decode_smem_bytes();
    *blocks_per_sm = 1 << 30;
    for (int fmt = 0; fmt < 2; ++fmt)
        for (int kv = 0; kv < 2; ++kv) {
            const void *fn = decode_fn(group, fmt, kv);
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kDecodeThreads, bytes);
            if (e != cudaSuccess) return e;
            if (n < *blocks_per_sm) *blocks_per_sm = n;
        }
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &a, int group, int ncta, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ncta);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = decode_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<DecodeArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, decode_fn(group, a.fmt, a.kv_f32), args);
}

}  // namespace qw
