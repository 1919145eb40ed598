// decode.cu - one batch-one decode step of the Qwen3 decoder as a single
// persistent kernel for sm_103a (GB300).
//
// The step ("Scalar-Native Qwen3 Reference Runtime As The Numerical Authority",
// section 2 steps 1-7; the decode schedule of "Portable WebAssembly Runtime
// Architecture for TinyRustLM", section "Prefill versus decode") is split into
// 5 phases per layer plus one head phase:
//   QKV     h = RMSNorm(x) (folded into the activation load), q|k|v = W h
//   ATTN    per (KV head, split): QK-Norm + RoPE of the head's queries and of
//           the new key, append k,v at this position, online-softmax attention
//           over a slice of the cache; the last split to finish merges
//   OPROJ   x = x + Wo o
//   GATEUP  h2 = RMSNorm(x), a = silu(Wg h2) * (Wu h2)
//   DOWN    x = x + Wd a
//   LMHEAD  logits = E RMSNorm(x), packed-key atomicMax argmax (ties -> lowest id)
//
// Layout on the GPU: one CTA per SM (cooperative launch, so all CTAs are
// resident).  Warp 8 of each CTA is a producer that streams, with bulk async
// copies (cp.async.bulk + mbarrier transaction counts), every weight row and
// cached K/V row this CTA will consume during the whole step into a ring of
// shared-memory slots.  Weights do not depend on the step's data, so the ring
// keeps HBM busy across phase boundaries while the 8 consumer warps wait for
// the previous phase's outputs.  Phase order between CTAs is a set of global
// arrival counters (release add / acquire load).  Every output row is owned by
// one warp, so results do not depend on timing.  Every wait is bounded in time:
// on expiry the kernel records QW_INTERNAL_INVARIANT, raises an abort flag that
// every other wait also watches, drains its own copies in flight and returns.
#include "qw_internal.h"

namespace qw {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct __align__(128) Smem {
    uint8_t slot[kSlots][kSlotBytes];
    unsigned long long full[kSlots];
    unsigned long long empty[kSlots];
    float wacc[kConsumerWarps][2][kHeadDim];  // attention: per-warp accumulators (group <= 2)
    float wml[kConsumerWarps][2][2];          // attention: per-warp running max, sum
    float sq[2][kHeadDim];                    // attention: normalised, rotated queries
    float sk[kHeadDim];                       // attention: this position's key (cache element type)
    float sv[kHeadDim];                       // attention: this position's value (cache element type)
    unsigned long long best[kConsumerWarps];  // head: per-warp argmax keys
    int flag;
    int tok;
    int merge;
    int bad;
};

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

__device__ __forceinline__ void bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_volatile(const unsigned *p) { return *(volatile const unsigned *)p; }

__device__ __forceinline__ void raise_error(StepFlags *f, unsigned code, bool abort) {
    atomicCAS(&f->err, 0u, code);
    if (abort) atomicExch(&f->abort, 1u);
}

// Bounded wait for a phase counter; false on abort or timeout (timeout raises the error).
__device__ bool wait_count(const unsigned *ctr, unsigned target, StepFlags *f) {
    unsigned long long t0 = 0;
    for (unsigned i = 0;; ++i) {
        if (ld_acquire(ctr) >= target) return true;
        if ((i & 31u) == 31u) {
            if (ld_volatile(&f->abort)) return false;
            unsigned long long t = gtime();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > kWaitLimitNs) {
                raise_error(f, kErrInvariant, true);
                return false;
            }
        }
    }
}

// Bounded wait for an mbarrier phase; watch_abort = false only while draining.
__device__ bool mbar_wait(unsigned long long *b, unsigned parity, StepFlags *f, bool watch_abort = true) {
    if (mbar_test(b, parity)) return true;
    unsigned long long t0 = gtime();
    for (unsigned i = 0;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 15u) == 15u) {
            if (watch_abort && ld_volatile(&f->abort)) return false;
            if (gtime() - t0 > kWaitLimitNs) {
                raise_error(f, kErrInvariant, true);
                return false;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float dot8_bf16(uint4 v, const float (&a)[8], float acc) {
    acc = fmaf(bf_lo(v.x), a[0], acc);
    acc = fmaf(bf_hi(v.x), a[1], acc);
    acc = fmaf(bf_lo(v.y), a[2], acc);
    acc = fmaf(bf_hi(v.y), a[3], acc);
    acc = fmaf(bf_lo(v.z), a[4], acc);
    acc = fmaf(bf_hi(v.z), a[5], acc);
    acc = fmaf(bf_lo(v.w), a[6], acc);
    acc = fmaf(bf_hi(v.w), a[7], acc);
    return acc;
}

__device__ __forceinline__ float i8f(uint32_t word, int byte) {
    return (float)((int)(word << (24 - 8 * byte)) >> 24);
}

// int8 group-32 dequantisation in registers: w = f32(q) * f32(s) (an exact product).
__device__ __forceinline__ float dot8_i8(uint2 v, float s, const float (&a)[8], float acc) {
#pragma unroll
    for (int e = 0; e < 4; ++e) acc = fmaf(a[e], i8f(v.x, e) * s, acc);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc = fmaf(a[4 + e], i8f(v.y, e) * s, acc);
    return acc;
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    if (v == 0.0f) v = 0.0f;  // -0 and +0 compare equal: lowest id wins
    uint32_t u = __float_as_uint(v);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

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

__device__ __forceinline__ Phase describe(const DecodeArgs &a, int ph, int cta, int ncta) {
    Phase p;
    p.l = ph / kPhasesPerLayer;
    p.type = (p.l >= a.L) ? T_LMHEAD : ph % kPhasesPerLayer;
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
            const int ch = kSlotBytes / (2 * kHeadDim * (a.kv_f32 ? 4 : 2));
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
    int bpr = (p.pair ? 2 : 1) * (p.i8 ? p.K + p.K / 16 : 2 * p.K);
    p.rpc = kSlotBytes / bpr;
    if (p.rpc > 32) p.rpc = 32;
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

__device__ void issue_chunk(Issuer &is, const DecodeArgs &a, const Phase &p, int c) {
    if (p.type == T_ATTN) {
        const int esz = a.kv_f32 ? 4 : 2, ch = kSlotBytes / (2 * kHeadDim * esz);
        int q0 = p.p0 + c * ch;
        int n = min(ch, p.p1 - q0);
        size_t off = ((((size_t)p.l * a.Hkv + p.kvh) * a.max_ctx + q0) * kHeadDim) * esz;
        is.copy(is.slot, (const uint8_t *)a.kc + off, (unsigned)(n * kHeadDim * esz));
        is.copy(is.slot + kSlotBytes / 2, (const uint8_t *)a.vc + off, (unsigned)(n * kHeadDim * esz));
        return;
    }
    int a0 = p.r0 + c * p.rpc;
    int n = min(p.rpc, p.r1 - a0);
    if (p.type == T_LMHEAD) {
        copy_rows(is, p, n, 0, a.lm_head, nullptr, a0, n);
        return;
    }
    const DevLayer &Ly = a.layers[p.l];
    if (p.type == T_QKV) {
        int qr = a.Hq * kHeadDim, kr = a.Hkv * kHeadDim;
        int b = a0 + n;
        // q rows [0, qr), k rows [qr, qr+kr), v rows [qr+kr, qr+2kr)
        int lo = a0, hi = min(b, qr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[0], Ly.s[0], lo, hi - lo);
        lo = max(a0, qr); hi = min(b, qr + kr);
        if (hi > lo) copy_rows(is, p, n, lo - a0, Ly.w[1], Ly.s[1], lo - qr, hi - lo);
        lo = max(a0, qr + kr); hi = b;
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

__device__ void producer(const DecodeArgs &a, Smem &sm) {
    const int cta = blockIdx.x, ncta = gridDim.x;
    const unsigned long long pol_w = policy_evict_first();
    const unsigned long long pol_kv = policy_evict_normal();
    unsigned it = 0;
    bool ok = true;
    for (int ph = a.phase_begin; ph < a.phase_end && ok; ++ph) {
        Phase p = describe(a, ph, cta, ncta);
        for (int c = 0; c < p.nchunks; ++c) {
            unsigned slot = it % kSlots, par = ((it / kSlots) & 1u) ^ 1u;
            if (!mbar_wait(&sm.empty[slot], par, a.flags)) {
                ok = false;
                break;
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
            unsigned last = ((it - 1 - s) / kSlots) * kSlots + s;
            mbar_wait(&sm.full[s], (last / kSlots) & 1u, a.flags, false);
        }
    }
}

// ---------------------------------------------------------------------- consumer

// Activation for lanes' columns 8*(lane + 32 m) + e, m < 4*KM.
template <int KM>
__device__ __forceinline__ void load_plain(const float *src, int lane, float (&v)[4 * KM][8]) {
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m) {
        const float4 *p = reinterpret_cast<const float4 *>(src + 8 * (lane + 32 * m));
        float4 lo = __ldcg(p), hi = __ldcg(p + 1);
        v[m][0] = lo.x; v[m][1] = lo.y; v[m][2] = lo.z; v[m][3] = lo.w;
        v[m][4] = hi.x; v[m][5] = hi.y; v[m][6] = hi.z; v[m][7] = hi.w;
    }
}

template <int KM>
__device__ __forceinline__ void load_bf16_row(const __nv_bfloat16 *src, int lane, float (&v)[4 * KM][8]) {
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(src + 8 * (lane + 32 * m)));
        v[m][0] = bf_lo(u.x); v[m][1] = bf_hi(u.x); v[m][2] = bf_lo(u.y); v[m][3] = bf_hi(u.y);
        v[m][4] = bf_lo(u.z); v[m][5] = bf_hi(u.z); v[m][6] = bf_lo(u.w); v[m][7] = bf_hi(u.w);
    }
}

// In-place RMSNorm over the warp's full vector (each lane holds 32*KM of the K = 1024*KM entries).
template <int KM>
__device__ __forceinline__ void rmsnorm_regs(float (&v)[4 * KM][8], const __nv_bfloat16 *w, int lane, float eps) {
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[m][e], v[m][e], ss);
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.0f / (1024.0f * KM)) + eps);
#pragma unroll
    for (int m = 0; m < 4 * KM; ++m) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(w + 8 * (lane + 32 * m)));
        const float wv[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y),
                             bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[m][e] = wv[e] * (v[m][e] * r);
    }
}

template <int KM, bool I8>
__device__ __forceinline__ float row_dot(const uint8_t *slot, int ns, int j, int lane, const float (&a)[4 * KM][8]) {
    float acc = 0.f;
    if constexpr (!I8) {
        const uint4 *row = reinterpret_cast<const uint4 *>(slot + (size_t)j * (2048 * KM));
#pragma unroll
        for (int m = 0; m < 4 * KM; ++m) acc = dot8_bf16(row[lane + 32 * m], a[m], acc);
    } else {
        const uint2 *row = reinterpret_cast<const uint2 *>(slot + (size_t)j * (1024 * KM));
        const __half *sc = reinterpret_cast<const __half *>(slot + (size_t)ns * (1024 * KM) + (size_t)j * (64 * KM));
#pragma unroll
        for (int m = 0; m < 4 * KM; ++m) acc = dot8_i8(row[lane + 32 * m], __half2float(sc[(lane + 32 * m) >> 2]), a[m], acc);
    }
    return warp_sum(acc);
}

struct Ctx {
    const DecodeArgs &a;
    Smem &sm;
    int tid, warp, lane, cta, ncta;
    unsigned it;
    bool dead;  // this warp saw an abort inside a chunk loop
};

// Wait for a slot to fill; warp-uniform result.
__device__ __forceinline__ bool take_slot(Ctx &c, unsigned slot, unsigned par) {
    bool ok = mbar_wait(&c.sm.full[slot], par, c.a.flags);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void release_slot(Ctx &c, unsigned slot) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.sm.empty[slot]);
}

// Row-streaming phase: each warp owns whole rows of each chunk (row j -> warp j % 8).
template <int KM, bool I8>
__device__ void gemv_phase(Ctx &c, const Phase &p) {
    const DecodeArgs &a = c.a;
    float act[4 * KM][8];
    const DevLayer *Ly = p.type == T_LMHEAD ? nullptr : &a.layers[p.l];
    // activation of this phase, every warp holds the whole vector across its lanes
    if (p.type == T_QKV || p.type == T_GATEUP || p.type == T_LMHEAD) {
        if (p.type == T_QKV && p.l == 0) {
            load_bf16_row<KM>(a.embed + (size_t)c.sm.tok * a.H, c.lane, act);
            if ((a.debug & 1) && c.cta == 0 && c.warp == 0) {
#pragma unroll
                for (int m = 0; m < 4 * KM; ++m)
#pragma unroll
                    for (int e = 0; e < 8; ++e) a.hidden[8 * (c.lane + 32 * m) + e] = act[m][e];
            }
        } else {
            load_plain<KM>(a.x, c.lane, act);
        }
        const __nv_bfloat16 *nw =
            p.type == T_QKV ? Ly->input_norm : (p.type == T_GATEUP ? Ly->post_norm : a.final_norm);
        rmsnorm_regs<KM>(act, nw, c.lane, a.eps);
    } else if (p.type == T_OPROJ) {
        load_plain<KM>(a.o, c.lane, act);
    } else {
        load_plain<KM>(a.act, c.lane, act);
    }
    unsigned long long best = 0;
    bool bad = false;
    for (int ch = 0; ch < p.nchunks; ++ch) {
        const unsigned slot = c.it % kSlots, par = (c.it / kSlots) & 1u;
        ++c.it;
        if (!take_slot(c, slot, par)) {
            c.dead = true;
            break;
        }
        const uint8_t *sp = c.sm.slot[slot];
        const int a0 = p.r0 + ch * p.rpc;
        const int n = min(p.rpc, p.r1 - a0);
        const int ns = p.pair ? 2 * n : n;
        for (int j = c.warp; j < n; j += kConsumerWarps) {
            const int row = a0 + j;
            if (p.pair) {
                float g = row_dot<KM, I8>(sp, ns, j, c.lane, act);
                float u = row_dot<KM, I8>(sp, ns, j + n, c.lane, act);
                if (c.lane == 0) a.act[row] = (g / (1.0f + __expf(-g))) * u;
            } else {
                float v = row_dot<KM, I8>(sp, ns, j, c.lane, act);
                if (c.lane == 0) {
                    switch (p.type) {
                        case T_QKV: a.qkv[row] = v; break;
                        case T_OPROJ: {
                            float r = p.l == 0 ? __bfloat162float(a.embed[(size_t)c.sm.tok * a.H + row]) : __ldcg(a.x + row);
                            a.x[row] = r + v;
                            break;
                        }
                        case T_DOWN: {
                            float nx = __ldcg(a.x + row) + v;
                            a.x[row] = nx;
                            if (a.debug & 1) a.hidden[(size_t)(p.l + 1) * a.H + row] = nx;
                            break;
                        }
                        default: {
                            a.logits[row] = v;
                            if (isfinite(v)) {
                                unsigned long long k = argmax_key(v, row);
                                best = k > best ? k : best;
                            } else {
                                bad = true;
                            }
                        }
                    }
                }
            }
        }
        release_slot(c, slot);
    }
    if (p.type == T_LMHEAD && c.lane == 0) {
        c.sm.best[c.warp] = best;
        if (bad) atomicOr(&c.sm.bad, 1);
    }
}

// QK-Norm then RoPE of one head held as dims (lane, lane+32, lane+64, lane+96).
__device__ __forceinline__ void qk_norm_rope(float (&v)[4], const __nv_bfloat16 *w, const float2 *rope, int lane,
                                             float eps) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.0f / kHeadDim) + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __bfloat162float(w[lane + 32 * i]) * (v[i] * r);
    const float2 cs0 = rope[lane], cs1 = rope[lane + 32];
    const float a0 = v[0], a1 = v[1], b0 = v[2], b1 = v[3];
    v[0] = a0 * cs0.x - b0 * cs0.y;
    v[2] = b0 * cs0.x + a0 * cs0.y;
    v[1] = a1 * cs1.x - b1 * cs1.y;
    v[3] = b1 * cs1.x + a1 * cs1.y;
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

template <typename KT>
constexpr int attn_chunk() { return kSlotBytes / (2 * kHeadDim * (int)sizeof(KT)); }

// Online-softmax update over n positions whose K and V rows (128 elements of KT each)
// sit at kb and vb.  Eight lanes share a position: lane (jj = lane/8, o8 = lane%8)
// takes dims [16*o8, 16*o8 + 16) of positions base + 4*warp + jj for base = 0, 32, ...
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

template <int G, typename KT>
__device__ void attn_phase(Ctx &c, const Phase &p) {
    using T = KvTraits<KT>;
    constexpr int NP = T::kPieces, PER = T::kPer, CH = attn_chunk<KT>();
    const DecodeArgs &a = c.a;
    Smem &sm = c.sm;
    if (p.kvh < 0) return;
    const int S = a.n_split, P = a.pos, kvh = p.kvh, l = p.l;
    const bool owner = (p.s == S - 1);
    const DevLayer &Ly = a.layers[l];
    const float2 *rope = a.rope + (size_t)P * (kHeadDim / 2);
    const int warp = c.warp, lane = c.lane;
    KT *snew_k = reinterpret_cast<KT *>(sm.sk), *snew_v = reinterpret_cast<KT *>(sm.sv);
    const size_t row_off = (((size_t)l * a.Hkv + kvh) * a.max_ctx + P) * kHeadDim;
    if (warp < G) {
        const float *src = a.qkv + (size_t)(kvh * G + warp) * kHeadDim;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldcg(src + lane + 32 * i);
        qk_norm_rope(v, Ly.q_norm, rope, lane, a.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.sq[warp][lane + 32 * i] = v[i];
    } else if (warp == G) {
        const float *src = a.qkv + (size_t)(a.Hq + kvh) * kHeadDim;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldcg(src + lane + 32 * i);
        qk_norm_rope(v, Ly.k_norm, rope, lane, a.eps);
        KT *dst = reinterpret_cast<KT *>(a.kc) + row_off;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const KT b = T::store(v[i]);
            snew_k[lane + 32 * i] = b;
            if (owner) dst[lane + 32 * i] = b;
        }
    } else if (warp == G + 1) {
        const float *src = a.qkv + (size_t)(a.Hq + a.Hkv + kvh) * kHeadDim;
        KT *dst = reinterpret_cast<KT *>(a.vc) + row_off;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const KT b = T::store(__ldcg(src + lane + 32 * i));
            snew_v[lane + 32 * i] = b;
            if (owner) dst[lane + 32 * i] = b;
        }
    }
    bar_consumers();

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
    for (int ch = 0; ch < p.nchunks; ++ch) {
        const unsigned slot = c.it % kSlots, par = (c.it / kSlots) & 1u;
        ++c.it;
        if (!c.dead && !take_slot(c, slot, par)) c.dead = true;
        if (c.dead) break;
        const uint8_t *sp = sm.slot[slot];
        const int n = min(CH, p.p1 - (p.p0 + ch * CH));
        attn_block<G, KT>(sp, sp + kSlotBytes / 2, n, warp, lane, qr, acc, M, Ls);
        release_slot(c, slot);
    }
    if (owner && !c.dead)
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
    // combine the eight warps: exact split-softmax merge
    for (int t = c.tid; t < G * kHeadDim; t += kConsumerThreads) {
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
        if (S == 1) {
            a.o[(size_t)(kvh * G + h) * kHeadDim + dim] = av / ls;
        } else {
            float *pp = a.part + ((size_t)(kvh * S + p.s) * G + h) * kPartStride;
            pp[dim] = av;
            if (dim == 0) {
                pp[kHeadDim] = mx;
                pp[kHeadDim + 1] = ls;
            }
        }
    }
    if (S == 1) return;
    __threadfence();
    bar_consumers();
    if (c.tid == 0) {
        const unsigned old = atomicAdd(&a.sync[kPhasesPerLayer * a.L + 1 + l * a.Hkv + kvh], 1u);
        __threadfence();
        sm.merge = (old == (unsigned)(S - 1));
    }
    bar_consumers();
    if (!sm.merge) return;
    for (int t = c.tid; t < G * kHeadDim; t += kConsumerThreads) {
        const int h = t / kHeadDim, dim = t % kHeadDim;
        float mx = -INFINITY;
        for (int s = 0; s < S; ++s) mx = fmaxf(mx, __ldcg(a.part + ((size_t)(kvh * S + s) * G + h) * kPartStride + kHeadDim));
        float av = 0.f, ls = 0.f;
        for (int s = 0; s < S; ++s) {
            const float *pp = a.part + ((size_t)(kvh * S + s) * G + h) * kPartStride;
            const float ms = __ldcg(pp + kHeadDim);
            if (ms == -INFINITY) continue;
            const float sc = exp2f(ms - mx);
            av = fmaf(__ldcg(pp + dim), sc, av);
            ls = fmaf(__ldcg(pp + kHeadDim + 1), sc, ls);
        }
        a.o[(size_t)(kvh * G + h) * kHeadDim + dim] = av / ls;
    }
}

template <bool I8>
__device__ void gemv_dispatch(Ctx &c, const Phase &p) {
    switch (p.K >> 10) {
        case 1: gemv_phase<1, I8>(c, p); break;
        case 2: gemv_phase<2, I8>(c, p); break;
        default: gemv_phase<3, I8>(c, p); break;
    }
}

template <int G>
__device__ void consumer(const DecodeArgs &a, Smem &sm) {
    Ctx c{a, sm, (int)threadIdx.x, (int)threadIdx.x >> 5, (int)threadIdx.x & 31, (int)blockIdx.x, (int)gridDim.x, 0u,
          false};
    if (c.tid == 0) {
        int tok = a.token >= 0 ? a.token : a.flags->next_tok;
        sm.tok = tok;
        sm.bad = 0;
        sm.flag = (tok >= 0 && tok < a.V) ? 1 : 0;
        if (!sm.flag) raise_error(a.flags, kErrInvalidArgument, true);
    }
    bar_consumers();
    if (!sm.flag) return;
    for (int ph = a.phase_begin; ph < a.phase_end; ++ph) {
        if (c.tid == 0) sm.flag = (ph == 0) ? !ld_volatile(&a.flags->abort) : wait_count(&a.sync[ph - 1], c.ncta, a.flags);
        bar_consumers();
        if (!sm.flag) return;
        const Phase p = describe(a, ph, c.cta, c.ncta);
        if (!c.dead) {
            if (p.type == T_ATTN) {
                if (a.kv_f32) attn_phase<G, float>(c, p);
                else attn_phase<G, __nv_bfloat16>(c, p);
            }
            else if (p.i8) gemv_dispatch<true>(c, p);
            else gemv_dispatch<false>(c, p);
        }
        __threadfence();
        bar_consumers();
        if (c.tid == 0) {
            if (p.type == T_LMHEAD) {
                unsigned long long b = 0;
                for (int w = 0; w < kConsumerWarps; ++w) b = sm.best[w] > b ? sm.best[w] : b;
                if (sm.bad) raise_error(a.flags, kErrNumerical, false);
                if (b) atomicMax(a.key, b);
                __threadfence();
                const unsigned old = atomicAdd(&a.sync[ph], 1u);
                if (old == (unsigned)(c.ncta - 1)) {
                    __threadfence();
                    const unsigned long long k = atomicAdd(a.key, 0ull);
                    const int tok = k ? (int)(0xffffffffu - (unsigned)(k & 0xffffffffull)) : 0;
                    a.flags->next_tok = tok;
                    if (a.tok_out) *a.tok_out = tok;
                }
            } else {
                red_release_add(&a.sync[ph], 1u);
            }
        }
        if (c.dead) {
            if (c.lane == 0) raise_error(a.flags, kErrInvariant, true);
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= kConsumerThreads) {
        if (threadIdx.x == kConsumerThreads) producer(a, sm);
        return;
    }
    consumer<G>(a, sm);
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

size_t decode_smem_bytes() { return sizeof(Smem) + 128; }

cudaError_t decode_prepare(int group, int *blocks_per_sm) {
    const int bytes = (int)decode_smem_bytes();
    const void *fn = group == 1 ? (const void *)decode_kernel<1> : (const void *)decode_kernel<2>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kDecodeThreads, bytes);
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
    switch (group) {
        case 1: return cudaLaunchKernelEx(&cfg, decode_kernel<1>, a);
        default: return cudaLaunchKernelEx(&cfg, decode_kernel<2>, a);
    }
}

}  // namespace qw
