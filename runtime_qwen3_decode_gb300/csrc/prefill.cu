// prefill.cu - batched prefill of a prompt chunk on the sm_103a tensor cores.
//
// The prompt's T rows go through every layer together ("Portable WebAssembly Runtime
// Architecture for TinyRustLM", section "Prefill versus decode": prefill is the
// matrix-matrix form of the same decoder; "Scalar-Native Qwen3 Reference Runtime As
// The Numerical Authority", section 2 steps 1-7 give the per-row arithmetic):
//
//   embed+norm   x = f32(E[tok]), h = fp16(RMSNorm(x) * w_in)            row kernel
//   QKV GEMM     qkv = h Wqkv^T, epilogue: QK-Norm + RoPE of q (fp16 out)
//                and k, K/V rows -> cache, fp16 K / V^T shadows           tcgen05
//   attention    causal GQA, S = Q K^T, online softmax, O += P V          tcgen05
//   O GEMM       x += o Wo^T                       (residual epilogue)    tcgen05
//   norm         h = fp16(RMSNorm(x) * w_post)                            row kernel
//   GU GEMM      a = fp16(silu(h Wg^T) * (h Wu^T)) (SwiGLU epilogue)      tcgen05
//   down GEMM    x += a Wd^T                       (residual epilogue)    tcgen05
//   head         last row only: final RMSNorm, logits = E hf, argmax      GEMV kernel
//
// Operands of the tensor-core steps are fp16 with f32 accumulation (kind::f16); the
// weights are converted to fp16 once, when the model is created (exact for every
// bf16 value of magnitude >= 2^-14; smaller ones round to fp16 subnormals).  Gate and
// up rows are interleaved in blocks of 128 so that one 256-wide output tile holds a
// gate block and its matching up block and the SwiGLU product happens in the epilogue.
//
// GEMM kernel: persistent, one CTA per SM, warp-specialised: 2 or 3 producer warps take
// turns issuing the TMA tile loads of a ring of shared-memory stages, one warp owns the
// TMEM allocation and issues tcgen05.mma from one thread, and 4 (q|k|v: 8) epilogue
// warps drain the double-buffered TMEM accumulator (tcgen05.ld) and apply the epilogue
// while the next tile accumulates.  Every wait is bounded: on expiry the CTA records
// QW_INTERNAL_INVARIANT, raises a shared abort flag, waits (bounded) for its own copies
// and MMAs in flight, frees TMEM and returns.
//
// Every kernel of a chunk after its first is launched chained (programmatic dependent
// launch): it waits with griddepcontrol.wait before touching memory an earlier kernel
// used, so its launch and setup overlap the previous kernel's tail.  The batched decode
// step (prefill_batch_step) reuses the fp16 weight copy and the row kernel here, with the
// skinny projections of batch.cu.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdio>
#include <vector>

#include "qw_batch.h"
#include "qw_prefill.h"
#include "tc.cuh"

namespace qw {
namespace {

using namespace tc;

constexpr int BM = 128;  // GEMM tile rows (prompt rows) = TMEM lanes
constexpr int BK = 64;   // K elements per stage: one 128-byte swizzle span of fp16
constexpr float kLog2e = 1.4426950408889634f;

enum { EPI_STORE = 0, EPI_ADD = 1, EPI_SWIGLU = 2, EPI_QKV = 3 };

// Where the q|k|v epilogue puts a row's heads (QK-Norm + RoPE of q and k first).
struct QkvOut {
    const __nv_bfloat16 *q_norm, *k_norm;  // [128] each
    const float2 *rope;                    // [max_ctx][64] (cos, sin)
    const float2 *rope_t;                  // the same table frequency-major: [64][rope_ld]
    int rope_ld;
    int pos0, Hq, Hkv;
    float eps;
    __half *q16;                           // [Hq][q_rows][128]
    int q_rows;
    void *kc, *vc;                         // this layer's cache planes [Hkv][max_ctx][128]
    int kv_f32, max_ctx;
    __half *k16, *v16t;                    // fp16 shadows [Hkv][kv_rows][128] and [Hkv][128][kv_rows] (or null)
    int kv_rows;
};

struct GemmParams {
    int M, N, K;       // rows, output columns, reduction length
    float *out;        // EPI_STORE: out[M][ldo] = acc; EPI_ADD: out[M][ldo] += acc
    int ldo;
    __half *act;       // EPI_SWIGLU: act[M][ldh], column block nt * BN/2
    int ldh;
    QkvOut qkv;        // EPI_QKV
    StepFlags *flags;
};

// Warp roles of a GEMM CTA: kProducers TMA warps (one issuing lane each, taking turns
// over the stages: one thread's issue cost per stage would otherwise exceed the MMA time
// of a stage), one MMA warp, kEpiWarps epilogue warps.  The q|k|v tile has eight epilogue
// warps, one per (TMEM lane quarter, head); the others four.  A stage holds kKbPerStage
// 64-deep k-blocks: with 128-wide tiles one thread's wait + issue + commit per 64-deep
// block (measured ~430 cycles) exceeds the block's 256 tensor cycles, so those tiles
// take 128-deep stages (8 MMAs per wait and commit).
template <int BN, int EPI>
struct GemmCfg {
    static constexpr int kProducers = BN == 256 ? 2 : 3;
    static constexpr int kMmaWarp = kProducers;
    static constexpr int kEpi0 = kProducers + 1;  // first epilogue warp
    static constexpr int kEpiWarps = EPI == EPI_QKV ? 8 : 4;
    static constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
    static constexpr int kStgCols = EPI == EPI_QKV ? 16 : 32;  // columns per staged block
    static constexpr int kStgStride = kStgCols + 4;            // floats per staged row
    static constexpr int kStgWarpFloats = 32 * kStgStride;
    static constexpr int kKbPerStage = BN == 256 ? 1 : 2;
    static constexpr int kStages = BN == 256 ? 4 : 3;
    static constexpr int kABytes = BM * BK * 2;  // one 64-deep k-block of A
    static constexpr int kBBytes = BN * BK * 2;  // one 64-deep k-block of B
    static constexpr int kStageA = kKbPerStage * kABytes;
    static constexpr int kStageB = kKbPerStage * kBBytes;
    static constexpr int kTmemCols = 2 * BN;  // two accumulator buffers
    static constexpr int kBarBytes = 256;
    static constexpr int kStgBytes = kEpiWarps * kStgWarpFloats * 4;
    static constexpr int kNormBytes = EPI == EPI_QKV ? 2 * kHeadDim * 4 : 0;  // q_norm, k_norm as f32
    static constexpr size_t kSmem =
        1024 + (size_t)kStages * (kStageA + kStageB) + kStgBytes + kNormBytes + kBarBytes;
    static_assert(kTmemCols <= 512, "TMEM has 512 columns");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert(kProducers <= kStages, "each producer owns at most one stage at a time");
    static_assert(EPI != EPI_QKV || BN == 2 * kHeadDim, "the q|k|v tile is two heads wide");
};

__device__ __forceinline__ void raise(StepFlags *f, unsigned code) {
    atomicCAS(&f->err, 0u, code);
    atomicExch(&f->abort, 1u);
}

// 1024-byte aligned start of dynamic shared memory (swizzled tiles need it).
__device__ __forceinline__ uint8_t *smem_base1024() {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t off = (1024u - (su32(smem_raw) & 1023u)) & 1023u;
    return smem_raw + off;
}

__device__ __forceinline__ uint4 pack_half8(const float *v) {
    uint4 u;
    __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
    __half2 h2 = __floats2half2_rn(v[4], v[5]), h3 = __floats2half2_rn(v[6], v[7]);
    u.x = *reinterpret_cast<uint32_t *>(&h0);
    u.y = *reinterpret_cast<uint32_t *>(&h1);
    u.z = *reinterpret_cast<uint32_t *>(&h2);
    u.w = *reinterpret_cast<uint32_t *>(&h3);
    return u;
}

// ------------------------------------------------------------------ GEMM epilogues
//
// An epilogue warp holds 32 output rows, one per lane (TMEM lane = tile row).  Stores
// straight from that layout would make every instruction touch 32 cache lines, so each
// block of SC columns goes through a per-warp shared-memory staging area (32 rows x
// (SC + 4) floats) and leaves transposed, every store instruction covering whole row
// segments.  The padding keeps both directions free of bank conflicts: writing, the
// eight lanes of a quarter warp store the same 16-byte chunk of eight rows (row pitch
// = 4 banks mod 32 x odd); reading, a quarter warp takes one row's eight chunks (SC = 32)
// or one chunk of eight rows (SC = 16).

// Lane l's SC values -> staging row l.
template <int SC>
__device__ __forceinline__ void stage_rows(float *stg, const float *v) {
    const int lane = threadIdx.x & 31;
    float4 *d = reinterpret_cast<float4 *>(stg + lane * (SC + 4));
#pragma unroll
    for (int k = 0; k < SC / 4; ++k) d[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    __syncwarp();
}

// Visit the staged block transposed: f(r, c4, x) for row r (0..31) and columns
// 4 c4 .. 4 c4 + 3.  Ends with a __syncwarp so the area can be restaged.
template <int SC, typename F>
__device__ __forceinline__ void unstage(const float *stg, F &&f) {
    static_assert(SC == 16 || SC == 32, "staging block width");
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int it = 0; it < SC / 4; ++it) {
        const int r = SC == 32 ? 4 * it + (lane >> 3) : 8 * it + (lane & 7);
        const int c4 = SC == 32 ? lane & 7 : lane >> 3;
        f(r, c4, *reinterpret_cast<const float4 *>(stg + r * (SC + 4) + 4 * c4));
    }
    __syncwarp();
}

__device__ __forceinline__ uint2 pack_half4(float4 x) {
    __half2 h0 = __floats2half2_rn(x.x, x.y), h1 = __floats2half2_rn(x.z, x.w);
    return make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
}

__device__ __forceinline__ uint2 pack_bf164(float4 x) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y), h1 = __floats2bfloat162_rn(x.z, x.w);
    return make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
}

__device__ __forceinline__ float4 round_bf16(float4 x) {
    return make_float4(__bfloat162float(__float2bfloat16_rn(x.x)), __bfloat162float(__float2bfloat16_rn(x.y)),
                       __bfloat162float(__float2bfloat16_rn(x.z)), __bfloat162float(__float2bfloat16_rn(x.w)));
}

// 32 columns d0 .. d0 + 31 of one q|k|v head for the warp's 32 prompt rows (lane = row):
// q -> q16, k and v -> the cache plus their fp16 shadows.
template <typename KT>
__device__ __forceinline__ void qkv_put32(const QkvOut &o, float (&v)[32], int d0, int slot, bool is_q, bool is_k,
                                          int kvh, KT *cache, int t, int r0, int M, float *stg) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        stage_rows<16>(stg, v + 16 * h);
        unstage<16>(stg, [&](int r, int c4, float4 x) {
            const int tr = r0 + r;  // prompt row
            if (tr >= M) return;
            const int d = d0 + 16 * h + 4 * c4;
            if (is_q) {
                *reinterpret_cast<uint2 *>(o.q16 + ((size_t)slot * o.q_rows + tr) * kHeadDim + d) = pack_half4(x);
                return;
            }
            const size_t prow = (size_t)(o.pos0 + tr) * kHeadDim + d;
            if constexpr (sizeof(KT) == 4) {
                *reinterpret_cast<float4 *>(cache + prow) = x;
            } else {
                *reinterpret_cast<uint2 *>(cache + prow) = pack_bf164(x);
                x = round_bf16(x);  // the shadows hold the cached value
            }
            if (is_k && o.k16)
                *reinterpret_cast<uint2 *>(o.k16 + ((size_t)kvh * o.kv_rows + o.pos0 + tr) * kHeadDim + d) =
                    pack_half4(x);
        });
    }
    // V^T shadow: for each dim the warp's 32 rows are 32 consecutive positions (64 B)
    if (!is_q && !is_k && t < M && o.v16t) {
        __half *dst = o.v16t + (size_t)kvh * kHeadDim * o.kv_rows + o.pos0 + t + (size_t)d0 * o.kv_rows;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float x = v[i];
            if constexpr (sizeof(KT) == 2) x = __bfloat162float(__float2bfloat16_rn(x));
            dst[(size_t)i * o.kv_rows] = __float2half_rn(x);
        }
    }
}

// One 128-wide head of the q|k|v tile (TMEM columns tcol .. tcol + 127) for the warp's
// 32 prompt rows (lane = row, t = the lane's row): QK-Norm and RoPE of q and k heads (the
// decode kernel's arithmetic: r = rsqrt(mean(v^2) + eps), v = w * (v * r), then dims
// (i, i + 64) rotated by the position's angle), then the stores of qkv_put32.  The head
// is read from TMEM twice (sum of squares, then the rotation pairs) so that at most 64
// of its values are live.  snorm: q_norm then k_norm as f32 in shared memory.
template <typename KT>
__device__ __forceinline__ void qkv_head_out(const QkvOut &o, uint32_t tcol, int slot, int t, int r0, int M,
                                             float *stg, const float *snorm) {
    const bool is_q = slot < o.Hq, is_k = !is_q && slot < o.Hq + o.Hkv;
    const int kvh = is_q ? 0 : is_k ? slot - o.Hq : slot - o.Hq - o.Hkv;
    KT *cache = reinterpret_cast<KT *>(is_k ? o.kc : o.vc) + (size_t)kvh * o.max_ctx * kHeadDim;
    if (!is_q && !is_k) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tcol + 32 * c, v);
            qkv_put32<KT>(o, v, 32 * c, slot, false, false, kvh, cache, t, r0, M, stg);
        }
        return;
    }
    float ss = 0.f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tcol + 32 * c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) ss += v[i] * v[i];
    }
    const float r = rsqrtf(ss * (1.0f / kHeadDim) + o.eps);
    const int P = o.pos0 + t;
    // frequency-major table: for each frequency the warp's 32 rows read 32 consecutive
    // positions (one coalesced request) instead of 32 rows 512 bytes apart
    const float2 *cs = o.rope_t + min(P, o.max_ctx - 1);
    const float *w = snorm + (is_q ? 0 : kHeadDim);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
        float a[32], b[32];
        tmem_ld32(tcol + 32 * j, a);
        tmem_ld32(tcol + 64 + 32 * j, b);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 wa = reinterpret_cast<const float4 *>(w + 32 * j)[k];
            const float4 wb = reinterpret_cast<const float4 *>(w + 64 + 32 * j)[k];
            const float wav[4] = {wa.x, wa.y, wa.z, wa.w}, wbv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * k + u;
                const float2 c = cs[(size_t)(32 * j + i) * o.rope_ld];
                const float x = wav[u] * (a[i] * r), y = wbv[u] * (b[i] * r);
                a[i] = x * c.x - y * c.y;
                b[i] = y * c.x + x * c.y;
            }
        }
        qkv_put32<KT>(o, a, 32 * j, slot, is_q, is_k, kvh, cache, t, r0, M, stg);
        qkv_put32<KT>(o, b, 64 + 32 * j, slot, is_q, is_k, kvh, cache, t, r0, M, stg);
    }
}

// The residual block an EPI_ADD epilogue warp updates (rows r0 .. r0 + 31, the tile's BN
// columns) in the transposed staging order: y[c][it] = row 4 it + lane / 8, columns
// c 32 + 4 (lane % 8) .. + 3.  Loaded before the accumulator is ready, it overlaps the
// mainloop; the tile's region of out is written only by this epilogue.
template <int BN>
__device__ __forceinline__ void load_residual(const GemmParams &p, int r0, int nt, float4 (&y)[BN / 32][8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int r = 4 * it + (lane >> 3);
            y[c][it] = r0 + r < p.M ? reinterpret_cast<const float4 *>(p.out + (size_t)(r0 + r) * p.ldo +
                                                                        (size_t)nt * BN + 32 * c)[lane & 7]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
}

// r0: the warp's first row (tile rows r0 .. r0 + 31); tacc: the accumulator buffer at the
// warp's TMEM lane quarter; e: the warp's epilogue index; stg: its staging area; y: the
// residual block (EPI_ADD).
template <int BN, int EPI>
__device__ __forceinline__ void gemm_epilogue(const GemmParams &p, uint32_t tacc, int r0, int nt, int e, float *stg,
                                              const float *snorm, const float4 (&y)[BN / 32][8]) {
    using C = GemmCfg<BN, EPI>;
    constexpr int SC = C::kStgCols;
    const int lane = threadIdx.x & 31;
    if constexpr (EPI == EPI_QKV) {
        const int hl = e >> 2;  // warps e and e + 4 share a lane quarter and split the two heads
        const int slot = nt * (BN / kHeadDim) + hl;
        if (p.qkv.kv_f32)
            qkv_head_out<float>(p.qkv, tacc + hl * kHeadDim, slot, r0 + lane, r0, p.M, stg, snorm);
        else
            qkv_head_out<__nv_bfloat16>(p.qkv, tacc + hl * kHeadDim, slot, r0 + lane, r0, p.M, stg, snorm);
    } else if constexpr (EPI == EPI_SWIGLU) {
        constexpr int HB = BN / 2;  // gate columns [0, HB), matching up columns [HB, BN)
#pragma unroll 1
        for (int c = 0; c < HB; c += 32) {
            float g[32], u[32];
            tmem_ld32(tacc + c, g);
            tmem_ld32(tacc + HB + c, u);
#pragma unroll
            // SiLU(g) u with the fast exp and divide (a few ulp, far below the fp16 rounding
            // of the output); the accurate forms made this epilogue ~2.3x longer than the
            // tile's mainloop.  g -> -inf gives g / inf = -0, g -> +inf gives g.
            for (int i = 0; i < 32; ++i) g[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
            stage_rows<SC>(stg, g);
            unstage<SC>(stg, [&](int r, int c4, float4 x) {
                if (r0 + r < p.M)
                    *reinterpret_cast<uint2 *>(p.act + (size_t)(r0 + r) * p.ldh + (size_t)nt * HB + c + 4 * c4) =
                        pack_half4(x);
            });
        }
    } else {
        static_assert(SC == 32, "the store / add epilogue reads 32-column blocks");
#pragma unroll
        for (int c = 0; c < BN; c += 32) {
            float v[32];
            tmem_ld32(tacc + c, v);
            stage_rows<SC>(stg, v);
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = 4 * it + (lane >> 3), c4 = lane & 7;
                float4 x = *reinterpret_cast<const float4 *>(stg + r * C::kStgStride + 4 * c4);
                if (r0 + r >= p.M) continue;
                if constexpr (EPI == EPI_ADD) {
                    const float4 yv = y[c / 32][it];
                    x.x += yv.x;
                    x.y += yv.y;
                    x.z += yv.z;
                    x.w += yv.w;
                }
                reinterpret_cast<float4 *>(p.out + (size_t)(r0 + r) * p.ldo + (size_t)nt * BN + c)[c4] = x;
            }
            __syncwarp();
        }
    }
}

// ------------------------------------------------------------------ GEMM kernel
//
// C[M, N] = A[M, K] * B[N, K]^T, A and B fp16 row-major (K contiguous), read by TMA
// with 128-byte swizzle.  Tiles BM x BN, tile index -> (m tile fastest, n tile).

template <int BN, int EPI>
__global__ void __launch_bounds__(GemmCfg<BN, EPI>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                const GemmParams p) {
    using C = GemmCfg<BN, EPI>;
    uint8_t *base = smem_base1024();
    uint8_t *sa = base;
    uint8_t *sb = base + C::kStages * C::kStageA;
    float *stg_all = reinterpret_cast<float *>(sb + C::kStages * C::kStageB);
    float *snorm = stg_all + C::kEpiWarps * C::kStgWarpFloats;
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(snorm) + C::kNormBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (p.M + BM - 1) / BM;
    const int ntiles = tiles_m * (p.N / BN);
    const int nkb = p.K / BK;
    const int nst = (nkb + C::kKbPerStage - 1) / C::kKbPerStage;  // stages per tile (the last may be short)

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], C::kEpiWarps);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort = 0;
        mbar_fence_init();
    }
    if constexpr (EPI == EPI_QKV) {
        for (int i = threadIdx.x; i < 2 * kHeadDim; i += C::kThreads)
            snorm[i] = __bfloat162float(i < kHeadDim ? p.qkv.q_norm[i] : p.qkv.k_norm[i - kHeadDim]);
    }
    if (warp == C::kMmaWarp) tmem_alloc(tslot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the setup above overlaps the previous kernel's tail; A and the outputs are its products
    chain_wait();
    chain_release();

    if (warp < C::kProducers) {
        if (lane == 0) {
            // ---- TMA producers: producer `warp` fills stages warp, warp + kProducers, ...
            // of the CTA's sequence (slot and phase advance over every stage)
            int s = 0, turn = 0;
            unsigned ph = 0;
            int last_par[C::kStages];
            for (int i = 0; i < C::kStages; ++i) last_par[i] = -1;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
                const int m0 = (tile % tiles_m) * BM, n0 = (tile / tiles_m) * BN;
                for (int st = 0; st < nst; ++st) {
                    if (turn == warp) {
                        if (!mbar_wait(&empty[s], ph ^ 1u, abort, true, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        const int kb0 = st * C::kKbPerStage;
                        const int nk = min(C::kKbPerStage, nkb - kb0);
                        mbar_expect_tx(&full[s], (unsigned)(nk * (C::kABytes + C::kBBytes)));
                        for (int j = 0; j < nk; ++j) {
                            tma_load_2d(sa + s * C::kStageA + j * C::kABytes, &tma, (kb0 + j) * BK, m0, &full[s]);
                            tma_load_2d(sb + s * C::kStageB + j * C::kBBytes, &tmb, (kb0 + j) * BK, n0, &full[s]);
                        }
                        last_par[s] = (int)ph;
                    }
                    if (++turn == C::kProducers) turn = 0;
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort = 1;
                raise(p.flags, kErrInvariant);
                // no copy may land in shared memory after this CTA has exited
                for (int i = 0; i < C::kStages; ++i)
                    if (last_par[i] >= 0) mbar_wait(&full[i], (unsigned)last_par[i], abort, false, kWaitLimitNs);
            }
        }
    } else if (warp == C::kMmaWarp) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            int s = 0, acc = 0;
            unsigned ph = 0, aph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], aph ^ 1u, abort, true, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN);
                for (int st = 0; st < nst; ++st) {
                    if (!mbar_wait(&full[s], ph, abort, true, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(C::kKbPerStage, nkb - st * C::kKbPerStage);
                    for (int j = 0; j < nk; ++j) {
                        const uint64_t ad = desc_sw128(su32(sa + s * C::kStageA + j * C::kABytes));
                        const uint64_t bd = desc_sw128(su32(sb + s * C::kStageB + j * C::kBBytes));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)  // +32 bytes along K per step (address field >> 4)
                            mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, (st | j | k) != 0);
                    }
                    mma_commit(&empty[s]);
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
            if (!ok) {
                *abort = 1;
                raise(p.flags, kErrInvariant);
            }
            // every MMA this thread issued completes before TMEM is released
            mma_commit(drain);
            mbar_wait(drain, 0, abort, false, kWaitLimitNs);
        }
    } else {
        // ---- epilogue warps: TMEM lane quarter = warp % 4
        const int e = warp - C::kEpi0, q = warp & 3;
        float *stg = stg_all + e * C::kStgWarpFloats;
        int acc = 0;
        unsigned aph = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int mt = tile % tiles_m, nt = tile / tiles_m;
            float4 y[BN / 32][8];
            if constexpr (EPI == EPI_ADD) load_residual<BN>(p, mt * BM + q * 32, nt, y);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], aph, abort, true, kWaitLimitNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort = 1;
                    raise(p.flags, kErrInvariant);
                }
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            gemm_epilogue<BN, EPI>(p, tacc, mt * BM + q * 32, nt, e, stg, snorm, y);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ row kernels

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read by a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
    return t;
}

// h[t] = fp16(w * (x[t] * rsqrt(mean(x[t]^2) + eps))); with tokens, x[t] = f32(E[tok[t]]) first.
// One warp per row of H = 1024 KM; lane l holds the 8-element chunks l + 32 c.
template <int KM>
__global__ void __launch_bounds__(kRowThreads) norm_rows_kernel(float *x, const int32_t *tokens,
                                                                const __nv_bfloat16 *embed,
                                                                const __nv_bfloat16 *w, __half *h, int rows,
                                                                float eps) {
    constexpr int H = 1024 * KM, NC = 4 * KM;
    chain_wait();
    chain_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kRowThreads / 32) + warp;
    if (t >= rows) return;
    float4 *xr = reinterpret_cast<float4 *>(x + (size_t)t * H);
    float v[NC][8];
    if (tokens) {
        const uint4 *er = reinterpret_cast<const uint4 *>(embed + (size_t)tokens[t] * H);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 u = er[lane + 32 * c];
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(b2[i]);
                v[c][2 * i] = f.x;
                v[c][2 * i + 1] = f.y;
            }
            xr[2 * (lane + 32 * c)] = make_float4(v[c][0], v[c][1], v[c][2], v[c][3]);
            xr[2 * (lane + 32 * c) + 1] = make_float4(v[c][4], v[c][5], v[c][6], v[c][7]);
        }
    } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float4 a0 = xr[2 * (lane + 32 * c)], a1 = xr[2 * (lane + 32 * c) + 1];
            v[c][0] = a0.x, v[c][1] = a0.y, v[c][2] = a0.z, v[c][3] = a0.w;
            v[c][4] = a1.x, v[c][5] = a1.y, v[c][6] = a1.z, v[c][7] = a1.w;
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += v[c][i] * v[c][i];
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / (float)H + eps);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    uint4 *hr = reinterpret_cast<uint4 *>(h + (size_t)t * H);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 u = wr[lane + 32 * c];
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
        float o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b2[i]);
            o[2 * i] = f.x * (v[c][2 * i] * r);
            o[2 * i + 1] = f.y * (v[c][2 * i + 1] * r);
        }
        hr[lane + 32 * c] = pack_half8(o);
    }
}

cudaError_t launch_norm_rows(float *x, const int32_t *tokens, const __nv_bfloat16 *embed, const __nv_bfloat16 *w,
                             __half *h, int rows, int H, float eps, cudaStream_t st, bool chained) {
    const dim3 grid((rows + kRowThreads / 32 - 1) / (kRowThreads / 32)), block(kRowThreads);
    auto k = H >> 10 == 1 ? norm_rows_kernel<1> : H >> 10 == 2 ? norm_rows_kernel<2> : norm_rows_kernel<3>;
    return launch_k(chained, k, grid, block, 0, st, x, tokens, embed, w, h, rows, eps);
}

// ------------------------------------------------------------------ K/V fp16 shadows
//
// The attention reads K as fp16 [Hkv][kv_rows][128] and V transposed, V^T fp16
// [Hkv][128][kv_rows], both with TMA.  kv_shadow_kernel fills positions [0, n_pos) of
// one layer from the cache (f32 or bf16) and zeroes [n_pos, n_fill), so every key a
// 128-key block can touch holds a finite value (a masked key still meets p = 0 in P V).

constexpr int kShadowPos = 64;

template <typename KT>
__device__ __forceinline__ void load8(const KT *src, float (&f)[8]) {
    if constexpr (sizeof(KT) == 4) {
        const float4 a = reinterpret_cast<const float4 *>(src)[0], b = reinterpret_cast<const float4 *>(src)[1];
        f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(src);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = __bfloat1622float2(h[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

template <typename KT>
__global__ void __launch_bounds__(256) kv_shadow_kernel(const KT *kc, const KT *vc, int max_ctx, int n_pos, int n_fill,
                                                       __half *k16, __half *v16t, int kv_rows) {
    __shared__ __align__(16) __half vt[kHeadDim][kShadowPos + 8];  // padded rows (144 B, 16-B aligned)
    chain_wait();
    chain_release();
    const int p0 = blockIdx.x * kShadowPos, kvh = blockIdx.y;
    const KT *ks = kc + (size_t)kvh * max_ctx * kHeadDim;
    const KT *vs = vc + (size_t)kvh * max_ctx * kHeadDim;
    __half *kd = k16 + (size_t)kvh * kv_rows * kHeadDim;
    // thread -> (position, 8 dims): K straight through, V into shared memory transposed
    for (int c = threadIdx.x; c < kShadowPos * 16; c += 256) {
        const int j = c >> 4, d0 = (c & 15) * 8, p = p0 + j;
        float fk[8], fv[8];
        if (p < n_pos) {
            load8(ks + (size_t)p * kHeadDim + d0, fk);
            load8(vs + (size_t)p * kHeadDim + d0, fv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) fk[i] = fv[i] = 0.f;
        }
        if (p < n_fill) *reinterpret_cast<uint4 *>(kd + (size_t)p * kHeadDim + d0) = pack_half8(fk);
#pragma unroll
        for (int i = 0; i < 8; ++i) vt[d0 + i][j] = __float2half_rn(fv[i]);
    }
    __syncthreads();
    // thread -> (dim, 8 positions): rows of V^T
    __half *vd = v16t + (size_t)kvh * kHeadDim * kv_rows;
    for (int c = threadIdx.x; c < kHeadDim * (kShadowPos / 8); c += 256) {
        const int d = c >> 3, j0 = (c & 7) * 8;
        if (p0 + j0 < n_fill)
            *reinterpret_cast<uint4 *>(vd + (size_t)d * kv_rows + p0 + j0) =
                *reinterpret_cast<const uint4 *>(&vt[d][j0]);
    }
}

// ------------------------------------------------------------------ causal attention
//
// CTA = (query tile, KV head).  The 128 MMA rows are the G query heads of the KV head
// stacked over 128/G positions: row r -> head kvh*G + r/(128/G), position
// t0 + r%(128/G), so both heads of a group share every K/V tile.  Per 128-key block j:
//   S_j = Q K_j^T into one of two TMEM buffers (the tensor core computes S_{j+1} while
//   the softmax warps work on S_j);
//   one softmax lane per row applies the causal mask and the online softmax in the log2
//   domain over the block's 128 keys (a whole row per lane: no partial maxima or sums
//   cross warps) and writes P_j (fp16) over the first half of S_j's buffer, so that P is
//   double-buffered with S and softmax j never waits for P_{j-1} V_{j-1};
//   O += P_j V_j accumulates in TMEM.  The tensor core runs S_{j+1} during softmax j
//   and P_j V_j right after it.
// Both A operands live in tensor memory (Q copied there once by the softmax warps, P
// written by them per block), so the tensor core reads only K and V^T from shared
// memory.  Per block, shared memory then carries the two 32 KB TMA writes and the two
// 32 KB operand reads; staging Q and P there as well doubled that traffic, and it was
// shared-memory bandwidth, not the tensor core or the softmax, that set the block time.
// O is rescaled only when a row's running max grows by more than 8 (factor 256): O and
// the row sum l always refer to the same reference max, so O / l is unaffected, and
// p <= 2^8 stays well inside fp16.
// Warp 0 issues the TMA loads of Q once and K per block, warp 6 those of V^T per block,
// into two independent 3-stage rings (K of block j+3 streams in as soon as S_j is done,
// V of block j+3 once P_j V_j is; under load a 32 KB tile takes about 3000 cycles to
// arrive, more than one block's softmax).  The third V stage is the Q tile's shared
// memory, refilled only after Q has been copied into TMEM.  The two producers sit in different warps: two
// spinning branches of one warp are not guaranteed to interleave, and a K load held
// behind a V wait delays S_{j+2} past the end of softmax j+1.  Warp 1 owns TMEM and
// issues the MMAs; warps 2-5 copy Q into TMEM, run the softmax and the output epilogue.

constexpr int kFaSoftmaxWarps = 4;
constexpr int kFaVWarp = 2 + kFaSoftmaxWarps;
constexpr int kFaThreads = 32 * (kFaVWarp + 1);
constexpr int kFaKeys = 128;
constexpr int kFaStages = 3;

// Each tile (Q, a K block, a V^T block) is 2 regions x [128 rows][128 B] = 32 KB.
struct FaSmem {
    static constexpr int kTile = 2 * 16384;
    static constexpr int kQ = 0;                              // Q, later V^T stage 2
    static constexpr int kK = kTile;                          // K stages 0..2
    static constexpr int kV = kK + kFaStages * kTile;         // V^T stages 0, 1
    static constexpr int kBar = kV + (kFaStages - 1) * kTile;
    static constexpr int kBytes = kBar + 256;
    static constexpr size_t kDyn = 1024 + kBytes;
};
// TMEM columns: S buffers 0 and 128 (f32; P_j as fp16 pairs over the first 64 columns
// of S_j's buffer), O 256 (f32), Q 448 (fp16 pairs).
constexpr uint32_t kFaColO = 256, kFaColQ = 448;
static_assert(FaSmem::kDyn <= 227 * 1024, "shared memory budget");
static_assert(kFaStages == 3, "the last V^T stage is the Q tile");

struct FaParams {
    int n, pos0, G, Hq;
    int q_rows, kv_rows;  // rows per head of the q16 and k16 buffers (V^T: columns)
    float scale_log2;     // log2(e) / sqrt(128)
    __half *o16;          // [n][Hq * 128]
    StepFlags *flags;
};

// Lane 0 waits (bounded) and the verdict is shared with the warp.
__device__ __forceinline__ bool warp_wait(uint64_t *b, unsigned parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(b, parity, abort, true, kWaitLimitNs);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2^x on the special-function unit (ex2.approx: about 2 ulp; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kFaThreads, 1)
    fa_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const FaParams p) {
    uint8_t *base = smem_base1024();
    uint8_t *sQ = base + FaSmem::kQ, *sK = base + FaSmem::kK, *sV = base + FaSmem::kV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + FaSmem::kBar);
    uint64_t *q_full = bars, *q_tm = bars + 1, *k_full = bars + 2, *k_empty = bars + 5, *v_full = bars + 8,
             *v_empty = bars + 11, *s_full = bars + 14, *p_full = bars + 18, *pv_done = bars + 19,
             *drain = bars + 24;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 25);
    volatile int *abort = reinterpret_cast<volatile int *>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, QT = 128 / G;
    const int ntq = (p.n + QT - 1) / QT;
    // block i: query tile ntq-1-i/Hkv of KV head i%Hkv.  Blocks start in index order, so
    // the longest (latest) tiles of every head go first and the short ones fill the tail;
    // a (tile, head) grid would start all tiles of the first heads before the longest
    // tiles of the last ones.
    const int Hkv = p.Hq / G;
    const int qt = ntq - 1 - (int)blockIdx.x / Hkv;
    const int g = (int)blockIdx.x % Hkv;
    const int t0 = qt * QT;
    const int nkb = (p.pos0 + min(t0 + QT, p.n) - 1) / kFaKeys + 1;
    const int first_masked = (p.pos0 + t0) / kFaKeys;  // blocks from here on cross the diagonal

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_tm, kFaSoftmaxWarps);
        for (int i = 0; i < kFaStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&s_full[i], 1);
        mbar_init(p_full, kFaSoftmaxWarps);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tO = tmem + kFaColO;  // S buffers at columns 0 and 128
    chain_wait();
    chain_release();

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer of Q, then K per block
            int par[kFaStages] = {-1, -1, -1};
            bool ok = true;
            mbar_expect_tx(q_full, 4 * 8192);
            for (int half = 0; half < 2; ++half) {
                const int head = g * G + (G == 2 ? half : 0);
                const int row = head * p.q_rows + t0 + (G == 2 ? 0 : 64 * half);
                for (int reg = 0; reg < 2; ++reg)
                    tma_load_2d(sQ + reg * 16384 + half * 8192, &tq, reg * 64, row, q_full);
            }
            for (int j = 0; j < nkb; ++j) {
                const int st = j % kFaStages;
                const unsigned ph = (unsigned)(j / kFaStages) & 1u;
                if (!mbar_wait(&k_empty[st], ph ^ 1u, abort, true, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&k_full[st], 2 * 16384);
                uint8_t *sk = sK + st * FaSmem::kTile;
                for (int reg = 0; reg < 2; ++reg)
                    tma_load_2d(sk + reg * 16384, &tk, reg * 64, g * p.kv_rows + j * kFaKeys, &k_full[st]);
                par[st] = (int)ph;
            }
            if (!ok) {
                *abort = 1;
                raise(p.flags, kErrInvariant);
                // no copy may land in shared memory after this CTA has exited
                mbar_wait(q_full, 0, abort, false, kWaitLimitNs);
                for (int i = 0; i < kFaStages; ++i)
                    if (par[i] >= 0) mbar_wait(&k_full[i], (unsigned)par[i], abort, false, kWaitLimitNs);
            }
        }
    } else if (warp == kFaVWarp) {
        if (lane == 0) {
            // ---- TMA producer of V^T per block
            int par[kFaStages] = {-1, -1, -1};
            bool ok = true;
            for (int j = 0; j < nkb; ++j) {
                const int st = j % kFaStages;
                const unsigned ph = (unsigned)(j / kFaStages) & 1u;
                // stage 2 is Q's tile: its first fill waits until Q sits in TMEM
                if (!mbar_wait(&v_empty[st], ph ^ 1u, abort, true, kWaitLimitNs) ||
                    (j == 2 && !mbar_wait(q_tm, 0, abort, true, kWaitLimitNs))) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&v_full[st], 2 * 16384);
                uint8_t *sv = st == 2 ? sQ : sV + st * FaSmem::kTile;
                for (int reg = 0; reg < 2; ++reg)
                    tma_load_2d(sv + reg * 16384, &tv, j * kFaKeys + reg * 64, g * kHeadDim, &v_full[st]);
                par[st] = (int)ph;
            }
            if (!ok) {
                *abort = 1;
                raise(p.flags, kErrInvariant);
                for (int i = 0; i < kFaStages; ++i)
                    if (par[i] >= 0) mbar_wait(&v_full[i], (unsigned)par[i], abort, false, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer, A operands (Q, P) in TMEM.  Iteration j issues S_{j+1} (it only
            // needs K_{j+1}, so the tensor core computes it while the softmax warps work on
            // block j) and then P_j V_j (after softmax j).  P_j sits in the first 64 columns of
            // S_j's buffer; S_{j+2} overwrites that buffer only after P_j V_j, which the
            // in-order tensor pipe guarantees by issue order.
            constexpr uint32_t idesc = idesc_f16_f32(128, 128);
            bool ok = mbar_wait(q_tm, 0, abort, true, kWaitLimitNs);
            for (int j = -1; ok && j < nkb; ++j) {
                if (j + 1 < nkb) {
                    const int jn = j + 1, st = jn % kFaStages;
                    if (!mbar_wait(&k_full[st], (unsigned)(jn / kFaStages) & 1u, abort, true, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sk = su32(sK + st * FaSmem::kTile);
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k) {
                        const uint64_t bd = desc_sw128(sk + (k >> 2) * 16384) + 2u * (k & 3);
                        mma_f16_ts(tmem + 128u * (jn & 1), tmem + kFaColQ + 8u * k, bd, idesc, k != 0);
                    }
                    mma_commit(&s_full[jn & 1]);
                    mma_commit(&k_empty[st]);
                }
                if (j >= 0) {
                    const int st = j % kFaStages;
                    if (!mbar_wait(&v_full[st], (unsigned)(j / kFaStages) & 1u, abort, true, kWaitLimitNs) ||
                        !mbar_wait(p_full, (unsigned)j & 1u, abort, true, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sv = su32(st == 2 ? sQ : sV + st * FaSmem::kTile);
#pragma unroll
                    for (int k = 0; k < kFaKeys / 16; ++k) {
                        const uint64_t bd = desc_sw128(sv + (k >> 2) * 16384) + 2u * (k & 3);
                        mma_f16_ts(tO, tmem + 128u * (j & 1) + 8u * k, bd, idesc, j > 0 || k > 0);
                    }
                    mma_commit(pv_done);
                    mma_commit(&v_empty[st]);
                }
            }
            if (!ok) {
                *abort = 1;
                raise(p.flags, kErrInvariant);
            }
            // every MMA this thread issued completes before TMEM is released
            mma_commit(drain);
            mbar_wait(drain, 0, abort, false, kWaitLimitNs);
        }
    } else {
        // ---- softmax warps 2..5: lane quarter q = warp % 4, row r = 32 q + lane; each lane
        // owns its row's whole block (128 keys), so no partial maxima or sums cross warps
        const int q = warp & 3, r = 32 * q + lane;
        const int t = G == 2 ? t0 + (r & 63) : t0 + r;
        const int head = g * G + (G == 2 ? (r >> 6) : 0);
        const int pr = p.pos0 + t;
        const uint32_t lb0 = (uint32_t)(32 * q) << 16;
        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        // Q row r: sixteen 16-byte chunks of the swizzled tile (two 64-dim regions), already
        // fp16 pairs in K order, into 64 TMEM columns
        bool ok = warp_wait(q_full, 0, abort);
        if (ok) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t qv[32];
                const uint8_t *src = sQ + hf * 16384;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(src + swz128(r, c));
                    qv[4 * c] = u.x;
                    qv[4 * c + 1] = u.y;
                    qv[4 * c + 2] = u.z;
                    qv[4 * c + 3] = u.w;
                }
                tmem_st32u(tmem + lb0 + kFaColQ + 32u * hf, qv);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_tm);
        }
        for (int j = 0; ok && j < nkb; ++j) {
            const int b = j & 1;
            if (!warp_wait(&s_full[b], (unsigned)(j >> 1) & 1u, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lb0 + 128u * b + 32u * c, s[c]);
            const int k0 = j * kFaKeys;
            float mb = -INFINITY;
            if (j >= first_masked) {
#pragma unroll
                for (int i = 0; i < kFaKeys; ++i) {
                    float &v = s[i >> 5][i & 31];
                    v = k0 + i <= pr ? v : -INFINITY;
                    mb = fmaxf(mb, v);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kFaKeys; ++i) mb = fmaxf(mb, s[i >> 5][i & 31]);
            }
            mb *= sc;
            const bool resc = mb > m_used + 8.f;
            const float m_new = resc ? mb : m_used;
            const float factor = resc ? fast_exp2(m_used - m_new) : 1.f;
            // O must hold P_{j-1} V_{j-1} before it is rescaled
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
                if (!warp_wait(pv_done, (unsigned)(j - 1) & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float o[32];
                    tmem_ld32(tO + lb0 + 32u * c, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= factor;
                    tmem_st32(tO + lb0 + 32u * c, o);
                }
            }
            l *= factor;
            m_used = m_new;
            // P_j (keys 2c, 2c + 1 in column c) over the first 64 columns of S_j's buffer: this
            // lane's S values are in registers, and P_{j-2} V_{j-2} (the buffer's previous P)
            // completed before S_j was written
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float e0 = fast_exp2(fmaf(s[2 * hf + (c >> 4)][2 * (c & 15)], sc, -m_used));
                    const float e1 = fast_exp2(fmaf(s[2 * hf + (c >> 4)][2 * (c & 15) + 1], sc, -m_used));
                    l += e0;
                    l += e1;
                    __half2 h = __floats2half2_rn(e0, e1);
                    pk[c] = *reinterpret_cast<uint32_t *>(&h);
                }
                tmem_st32u(tmem + lb0 + 128u * b + 32u * hf, pk);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && !warp_wait(pv_done, (unsigned)(nkb - 1) & 1u, abort)) ok = false;
        if (ok) {
            tc_fence_after();
            const float inv = 1.0f / l;
            __half *dst = p.o16 + (size_t)t * p.Hq * kHeadDim + (size_t)head * kHeadDim;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tmem_ld32(tO + lb0 + 32u * c, o);
                if (t < p.n) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= inv;
#pragma unroll
                    for (int i = 0; i < 4; ++i) reinterpret_cast<uint4 *>(dst + 32 * c)[i] = pack_half8(o + 8 * i);
                }
            }
        } else if (lane == 0) {
            *abort = 1;
            raise(p.flags, kErrInvariant);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ head (last row)

constexpr int kHeadThreads = 256;

__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
    const uint32_t u = __float_as_uint(v);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (0xffffffffu - (uint32_t)id);
}

// logits[v] = E[v] . (final_norm * RMSNorm(x)), packed-key argmax (ties -> lowest id);
// the last CTA to finish publishes the token and re-arms the key for the next call.
template <int KM>
__global__ void __launch_bounds__(kHeadThreads) head_kernel(const float *x, const __nv_bfloat16 *final_norm,
                                                            const __nv_bfloat16 *E, int V, int H, float eps,
                                                            float *logits, unsigned long long *key,
                                                            unsigned *count, StepFlags *flags) {
    __shared__ __align__(16) float hf[3072];
    __shared__ float red[kHeadThreads / 32];
    __shared__ unsigned long long best[kHeadThreads / 32];
    __shared__ int bad_any;
    chain_wait();
    chain_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) bad_any = 0;
    float ss = 0.f;
    for (int c = threadIdx.x; c < H; c += kHeadThreads) ss += x[c] * x[c];
    const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
    for (int c = threadIdx.x; c < H; c += kHeadThreads) hf[c] = __bfloat162float(final_norm[c]) * (x[c] * r);
    __syncthreads();
    unsigned long long kbest = 0;
    bool bad = false;
    constexpr int NC = 4 * KM;  // 16-byte chunks of 8 bf16 per lane and row
    const int gw = blockIdx.x * (kHeadThreads / 32) + warp, nw = gridDim.x * (kHeadThreads / 32);
    // two rows per pass, every load of both rows issued before the arithmetic
    for (int v0 = gw; v0 < V; v0 += 2 * nw) {
        const int v1 = v0 + nw < V ? v0 + nw : v0;
        const uint4 *r0 = reinterpret_cast<const uint4 *>(E + (size_t)v0 * H);
        const uint4 *r1 = reinterpret_cast<const uint4 *>(E + (size_t)v1 * H);
        uint4 u0[NC], u1[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            u0[i] = __ldg(r0 + lane + 32 * i);
            u1[i] = __ldg(r1 + lane + 32 * i);
        }
        float acc[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const int c = lane + 32 * i;
            const float4 h0 = *reinterpret_cast<const float4 *>(hf + 8 * c);
            const float4 h1 = *reinterpret_cast<const float4 *>(hf + 8 * c + 4);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(r ? &u1[i] : &u0[i]);
                float2 f;
                f = __bfloat1622float2(b[0]);
                acc[r] += f.x * h0.x + f.y * h0.y;
                f = __bfloat1622float2(b[1]);
                acc[r] += f.x * h0.z + f.y * h0.w;
                f = __bfloat1622float2(b[2]);
                acc[r] += f.x * h1.x + f.y * h1.y;
                f = __bfloat1622float2(b[3]);
                acc[r] += f.x * h1.z + f.y * h1.w;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
            acc[1] += __shfl_xor_sync(0xffffffffu, acc[1], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r == 1 && v1 == v0) break;
                const int v = r ? v1 : v0;
                logits[v] = acc[r];
                if (!isfinite(acc[r])) bad = true;
                const unsigned long long k = argmax_key(acc[r], v);
                kbest = k > kbest ? k : kbest;
            }
        }
    }
    if (lane == 0) {
        best[warp] = kbest;
        if (bad) bad_any = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = 0;
        for (int w = 0; w < kHeadThreads / 32; ++w) b = best[w] > b ? best[w] : b;
        if (bad_any) atomicCAS(&flags->err, 0u, kErrNumerical);
        if (b) atomicMax(key, b);
        __threadfence();
        const unsigned old = atomicAdd(count, 1u);
        if (old + 1u == gridDim.x) {
            __threadfence();
            const unsigned long long k = atomicAdd(key, 0ull);
            flags->next_tok = k ? (int)(0xffffffffu - (unsigned)(k & 0xffffffffull)) : 0;
            *key = 0ull;
            *count = 0u;
        }
    }
}

// ------------------------------------------------------------------ weight conversion

// dst row mapping of source row i: mode 0 -> off + i; mode 1 (gate) / 2 (up) ->
// (i / 128) * 256 + (mode == 2 ? 128 : 0) + i % 128.
__global__ void convert_kernel(const void *src, const __half *scales, int int8, int rows, int cols, __half *dst,
                               int mode, int off, unsigned *overflow) {
    const long long n = (long long)rows * cols;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(e / cols), c = (int)(e % cols);
        float w;
        if (int8) {
            w = (float)reinterpret_cast<const int8_t *>(src)[e] * __half2float(scales[(size_t)i * (cols / 32) + c / 32]);
        } else {
            w = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[e]);
        }
        const int drow = mode == 0 ? off + i : (i / 128) * 256 + (mode == 2 ? 128 : 0) + i % 128;
        const __half h = __float2half_rn(w);
        if (__hisinf(h)) atomicAdd(overflow, 1u);
        dst[(size_t)drow * cols + c] = h;
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

cudaError_t load_encoder() {
    if (g_encode) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = (EncodeTiledFn)fn;
    return cudaSuccess;
}

// fp16 row-major [rows][cols] read in boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int rows, int cols, int box_rows) {
    if (!g_encode || rows < 1 || cols % 64 || ((uintptr_t)ptr & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI>
cudaError_t set_gemm_attr() {
    return cudaFuncSetAttribute(gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GemmCfg<BN, EPI>::kSmem);
}

template <int BN, int EPI>
cudaError_t launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &p, int nsm,
                        cudaStream_t st, bool chained = false) {
    const int tiles = (p.M + BM - 1) / BM * (p.N / BN);
    const int grid = tiles < nsm ? tiles : nsm;
    return launch_k(chained, gemm_kernel<BN, EPI>, dim3(grid), dim3(GemmCfg<BN, EPI>::kThreads),
                    GemmCfg<BN, EPI>::kSmem, st, ma, mb, p);
}

size_t align_up(size_t v) { return (v + 255) / 256 * 256; }

struct PrefillLayout {
    size_t w16, x, h, q16, o16, act, k16, v16t, tok, misc, rope_t, bqkv, total;
    size_t w_layer;  // fp16 weight elements per layer
    int kv_rows;     // positions per head in the fp16 K / V^T shadows (max_ctx rounded up to 128)
};

PrefillLayout prefill_layout(const qw_config &c, int rows) {
    PrefillLayout L{};
    const size_t H = c.hidden, QD = (size_t)c.n_heads * c.head_dim, KD = (size_t)c.n_kv_heads * c.head_dim,
                 I = c.intermediate;
    L.w_layer = (QD + 2 * KD) * H + H * QD + 2 * I * H + H * I;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align_up(bytes);
        return at;
    };
    L.w16 = take((size_t)c.n_layers * L.w_layer * 2);
    L.x = take((size_t)rows * H * 4);
    L.h = take((size_t)rows * (H > I ? H : I) * 2);
    L.q16 = take((size_t)rows * QD * 2);
    L.o16 = take((size_t)rows * QD * 2);
    L.act = take((size_t)rows * I * 2);
    L.kv_rows = (c.max_ctx + kFaKeys - 1) / kFaKeys * kFaKeys;
    L.k16 = take((size_t)c.n_kv_heads * L.kv_rows * c.head_dim * 2);
    L.v16t = take((size_t)c.n_kv_heads * L.kv_rows * c.head_dim * 2);
    L.tok = take((size_t)rows * 4);
    L.misc = take(64);
    L.rope_t = take((size_t)c.max_ctx * (c.head_dim / 2) * sizeof(float2));
    L.bqkv = take((size_t)kBatchMax * (QD + 2 * KD) * 4);  // batched decode: raw q|k|v rows (f32)
    L.total = off;
    return L;
}

}  // namespace

struct PrefillImpl {
    PrefillLayout lay;
    qw_config cfg;
    std::vector<DevLayer> host_layers;  // the model's layer table (device pointers)
    std::vector<CUtensorMap> wmaps;     // per layer: qkv, o, gate/up, down
    CUtensorMap tq, tk, tv;             // attention operands: q16, k16, v16t
};

size_t prefill_workspace_bytes(const qw_config &c, int rows_max) { return prefill_layout(c, rows_max).total; }

cudaError_t prefill_prepare() {
    cudaError_t e = load_encoder();
    if (e != cudaSuccess) return e;
    if ((e = set_gemm_attr<256, EPI_STORE>()) != cudaSuccess) return e;
    if ((e = set_gemm_attr<256, EPI_QKV>()) != cudaSuccess) return e;
    if ((e = set_gemm_attr<256, EPI_SWIGLU>()) != cudaSuccess) return e;
    if ((e = set_gemm_attr<128, EPI_ADD>()) != cudaSuccess) return e;
    if ((e = set_gemm_attr<128, EPI_STORE>()) != cudaSuccess) return e;
    if ((e = batch_prepare()) != cudaSuccess) return e;
    return cudaFuncSetAttribute(fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FaSmem::kDyn);
}

namespace {
// rope_t[i][p] = rope[p][i]: the RoPE table frequency-major for the q|k|v epilogue
__global__ void rope_transpose_kernel(const float2 *rope, int ctx, int half, float2 *rope_t) {
    const long long n = (long long)ctx * half;
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(k / ctx), p = (int)(k % ctx);
        rope_t[k] = rope[(size_t)p * half + i];
    }
}
}  // namespace

int prefill_init(PrefillState *st, const qw_config &c, const DevLayer *host_layers, const float2 *rope, uint8_t *buf,
                 size_t bytes, int rows_max, int nsm, cudaStream_t stream) {
    st->buf = buf;
    st->bytes = bytes;
    st->rows_max = rows_max;
    st->nsm = nsm;
    st->ready = 0;
    st->impl = nullptr;
    PrefillImpl *im = new (std::nothrow) PrefillImpl();
    if (!im) return 1;
    im->cfg = c;
    im->lay = prefill_layout(c, rows_max);
    // int8 activations are a different arithmetic from the fp16 tensor-core prefill: such a model
    // prefills through the decode path, one token at a time (ready stays 0)
    if (c.weight_format == QW_W_Q8Q8) {
        st->impl = im;
        return 0;
    }
    if (im->lay.total > bytes) {
        delete im;
        return 1;
    }
    rope_transpose_kernel<<<2 * nsm, 256, 0, stream>>>(rope, c.max_ctx, c.head_dim / 2,
                                                        reinterpret_cast<float2 *>(buf + im->lay.rope_t));
    if (cudaGetLastError() != cudaSuccess) {
        delete im;
        return 1;
    }
    st->impl = im;
    im->host_layers.assign(host_layers, host_layers + c.n_layers);
    const PrefillLayout &L = im->lay;
    const int H = c.hidden, QD = c.n_heads * c.head_dim, KD = c.n_kv_heads * c.head_dim, I = c.intermediate;
    unsigned *overflow = reinterpret_cast<unsigned *>(buf + L.misc + 16);
    if (cudaMemsetAsync(buf + L.misc, 0, 64, stream) != cudaSuccess) return 1;
    // attention operand rows past the prompt are read (and masked); they must hold finite values
    if (cudaMemsetAsync(buf + L.q16, 0, L.o16 - L.q16, stream) != cudaSuccess ||
        cudaMemsetAsync(buf + L.k16, 0, L.tok - L.k16, stream) != cudaSuccess)
        return 1;
    if (!make_map(&im->tq, buf + L.q16, c.n_heads * rows_max, kHeadDim, 64) ||
        !make_map(&im->tk, buf + L.k16, c.n_kv_heads * L.kv_rows, kHeadDim, kFaKeys) ||
        !make_map(&im->tv, buf + L.v16t, c.n_kv_heads * kHeadDim, L.kv_rows, kFaKeys))
        return 1;
    const int int8 = c.weight_format == QW_W_INT8_G32 ? 1 : 0;
    im->wmaps.resize((size_t)c.n_layers * 4);
    for (int l = 0; l < c.n_layers; ++l) {
        __half *w = reinterpret_cast<__half *>(buf + L.w16) + (size_t)l * L.w_layer;
        __half *wqkv = w, *wo = wqkv + (size_t)(QD + 2 * KD) * H, *wgu = wo + (size_t)H * QD,
               *wd = wgu + (size_t)2 * I * H;
        const DevLayer &Ly = host_layers[l];
        struct Job {
            int m, rows, cols, mode, off;
            __half *dst;
        } jobs[7] = {{0, QD, H, 0, 0, wqkv},  {1, KD, H, 0, QD, wqkv}, {2, KD, H, 0, QD + KD, wqkv},
                     {3, H, QD, 0, 0, wo},     {4, I, H, 1, 0, wgu},    {5, I, H, 2, 0, wgu},
                     {6, H, I, 0, 0, wd}};
        for (const Job &j : jobs) {
            convert_kernel<<<4 * nsm, 256, 0, stream>>>(Ly.w[j.m], Ly.s[j.m], int8, j.rows, j.cols, j.dst, j.mode,
                                                        j.off, overflow);
            if (cudaGetLastError() != cudaSuccess) return 1;
        }
        CUtensorMap *m = &im->wmaps[(size_t)l * 4];
        if (!make_map(&m[0], wqkv, QD + 2 * KD, H, 256) || !make_map(&m[1], wo, H, QD, 128) ||
            !make_map(&m[2], wgu, 2 * I, H, 256) || !make_map(&m[3], wd, H, I, 128))
            return 1;
    }
    unsigned ovf = 0;
    if (cudaMemcpyAsync(&ovf, overflow, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return 1;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return 1;
    if (ovf) {
        fprintf(stderr, "qw: %u weights exceed the fp16 range; prefill runs token by token\n", ovf);
        return 0;
    }
    st->ready = 1;
    return 0;
}

void prefill_destroy(PrefillState *st) {
    delete st->impl;
    st->impl = nullptr;
    st->ready = 0;
}

int prefill_run(PrefillState *st, const DecodeArgs &a, int pos0, const int32_t *tokens_host, int n, int debug,
                cudaStream_t stream) {
    PrefillImpl *im = st->impl;
    if (!im || !st->ready) return 1;
    const qw_config &c = im->cfg;
    const PrefillLayout &L = im->lay;
    uint8_t *buf = st->buf;
    const int H = c.hidden, Hq = c.n_heads, Hkv = c.n_kv_heads, QD = Hq * kHeadDim, KD = Hkv * kHeadDim,
              I = c.intermediate, G = Hq / Hkv;
    float *x = reinterpret_cast<float *>(buf + L.x);
    __half *h = reinterpret_cast<__half *>(buf + L.h);
    __half *q16 = reinterpret_cast<__half *>(buf + L.q16);
    __half *o16 = reinterpret_cast<__half *>(buf + L.o16);
    __half *act = reinterpret_cast<__half *>(buf + L.act);
    int32_t *tok = reinterpret_cast<int32_t *>(buf + L.tok);
    unsigned long long *key = reinterpret_cast<unsigned long long *>(buf + L.misc);
    unsigned *count = reinterpret_cast<unsigned *>(buf + L.misc + 8);
    const size_t kv_plane = (size_t)Hkv * a.max_ctx * kHeadDim * (a.kv_f32 ? 4 : 2);
    const DevLayer *hl = im->host_layers.data();

    // argmax key and finishing counter of the head kernel start at zero every call
    if (cudaMemsetAsync(key, 0, 16, stream) != cudaSuccess) return 1;
    for (int done = 0; done < n;) {
        const int m = n - done < st->rows_max ? n - done : st->rows_max;
        const int p0 = pos0 + done;
        cudaError_t e = cudaMemcpyAsync(tok, tokens_host + done, (size_t)m * 4, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return 1;
        CUtensorMap mh, mo, ma;
        if (!make_map(&mh, h, m, H, BM) || !make_map(&mo, o16, m, QD, BM) || !make_map(&ma, act, m, I, BM))
            return 1;
        launch_norm_rows(x, tok, a.embed, hl[0].input_norm, h, m, H, a.eps, stream, false);
        // chained launches (programmatic dependent launch) only directly after a kernel
        bool ch = true;
        if (debug & 1) {
            cudaMemcpyAsync(a.hidden, x + (size_t)(m - 1) * H, (size_t)H * 4, cudaMemcpyDeviceToDevice, stream);
            ch = false;
        }
        for (int l = 0; l < c.n_layers; ++l) {
            const CUtensorMap *wm = &im->wmaps[(size_t)l * 4];
            GemmParams gp{};
            gp.flags = a.flags;
            gp.M = m;
            uint8_t *kc = reinterpret_cast<uint8_t *>(a.kc) + (size_t)l * kv_plane;
            uint8_t *vc = reinterpret_cast<uint8_t *>(a.vc) + (size_t)l * kv_plane;
            __half *k16 = reinterpret_cast<__half *>(buf + L.k16), *v16t = reinterpret_cast<__half *>(buf + L.v16t);
            // fp16 shadows of cache rows written before this chunk (earlier chunks, decode
            // steps or an import); the chunk's own rows come from the q|k|v epilogue below
            if (p0 > 0) {
                const dim3 sg((p0 + kShadowPos - 1) / kShadowPos, Hkv);
                cudaError_t se;
                if (a.kv_f32)
                    se = launch_k(ch, kv_shadow_kernel<float>, sg, dim3(256), 0, stream,
                                  reinterpret_cast<const float *>(kc), reinterpret_cast<const float *>(vc), a.max_ctx,
                                  p0, p0, k16, v16t, L.kv_rows);
                else
                    se = launch_k(ch, kv_shadow_kernel<__nv_bfloat16>, sg, dim3(256), 0, stream,
                                  reinterpret_cast<const __nv_bfloat16 *>(kc),
                                  reinterpret_cast<const __nv_bfloat16 *>(vc), a.max_ctx, p0, p0, k16, v16t,
                                  L.kv_rows);
                if (se != cudaSuccess) return 1;
                ch = true;
            }
            // q | k | v with QK-Norm, RoPE, the K/V append and the shadows in the epilogue
            gp.N = QD + 2 * KD;
            gp.K = H;
            QkvOut &qo = gp.qkv;
            qo.q_norm = hl[l].q_norm;
            qo.k_norm = hl[l].k_norm;
            qo.rope = a.rope;
            qo.rope_t = reinterpret_cast<const float2 *>(buf + L.rope_t);
            qo.rope_ld = c.max_ctx;
            qo.pos0 = p0;
            qo.Hq = Hq;
            qo.Hkv = Hkv;
            qo.eps = a.eps;
            qo.q16 = q16;
            qo.q_rows = st->rows_max;
            qo.kc = kc;
            qo.vc = vc;
            qo.kv_f32 = a.kv_f32;
            qo.max_ctx = a.max_ctx;
            qo.k16 = k16;
            qo.v16t = v16t;
            qo.kv_rows = L.kv_rows;
            if (launch_gemm<256, EPI_QKV>(mh, wm[0], gp, st->nsm, stream, ch) != cudaSuccess) return 1;
            FaParams fp{};
            fp.n = m;
            fp.pos0 = p0;
            fp.G = G;
            fp.Hq = Hq;
            fp.q_rows = st->rows_max;
            fp.kv_rows = L.kv_rows;
            fp.scale_log2 = kLog2e / sqrtf((float)kHeadDim);
            fp.o16 = o16;
            fp.flags = a.flags;
            const dim3 ag((m + 128 / G - 1) / (128 / G) * Hkv);
            if (launch_k(true, fa_kernel, ag, dim3(kFaThreads), FaSmem::kDyn, stream, im->tq, im->tk, im->tv, fp) !=
                cudaSuccess)
                return 1;
            // x += o Wo^T
            gp.N = H;
            gp.K = QD;
            gp.out = x;
            gp.ldo = H;
            if (launch_gemm<128, EPI_ADD>(mo, wm[1], gp, st->nsm, stream, true) != cudaSuccess) return 1;
            if (launch_norm_rows(x, nullptr, nullptr, hl[l].post_norm, h, m, H, a.eps, stream, true) != cudaSuccess)
                return 1;
            // a = silu(h Wg^T) * (h Wu^T)
            gp.N = 2 * I;
            gp.K = H;
            gp.act = act;
            gp.ldh = I;
            if (launch_gemm<256, EPI_SWIGLU>(mh, wm[2], gp, st->nsm, stream, true) != cudaSuccess) return 1;
            // x += a Wd^T
            gp.N = H;
            gp.K = I;
            gp.out = x;
            gp.ldo = H;
            if (launch_gemm<128, EPI_ADD>(ma, wm[3], gp, st->nsm, stream, true) != cudaSuccess) return 1;
            ch = true;
            if (debug & 1) {
                cudaMemcpyAsync(a.hidden + (size_t)(l + 1) * H, x + (size_t)(m - 1) * H, (size_t)H * 4,
                                cudaMemcpyDeviceToDevice, stream);
                ch = false;
            }
            if (l + 1 < c.n_layers) {
                if (launch_norm_rows(x, nullptr, nullptr, hl[l + 1].input_norm, h, m, H, a.eps, stream, ch) !=
                    cudaSuccess)
                    return 1;
                ch = true;
            }
        }
        done += m;
        if (done == n) {
            const float *xl = x + (size_t)(m - 1) * H;
            const dim3 hg(4 * st->nsm);
            auto hk = H == 1024 ? head_kernel<1> : H == 2048 ? head_kernel<2> : head_kernel<3>;
            if (launch_k(ch, hk, hg, dim3(kHeadThreads), 0, stream, xl, a.final_norm, a.lm_head, a.V, H, a.eps,
                         a.logits, key, count, a.flags) != cudaSuccess)
                return 1;
        }
        if (cudaGetLastError() != cudaSuccess) return 1;
    }
    return 0;
}

// ------------------------------------------------------------------ batched decode

int prefill_batch_step(PrefillState *st, const DecodeArgs &a, const BatchStep &bs, cudaStream_t stream) {
    PrefillImpl *im = st->impl;
    if (!im || !st->ready || bs.B < 1 || bs.B > st->rows_max || bs.B > kBatchMax) return 1;
    const qw_config &c = im->cfg;
    const PrefillLayout &L = im->lay;
    uint8_t *buf = st->buf;
    const int H = c.hidden, Hq = c.n_heads, Hkv = c.n_kv_heads, QD = Hq * kHeadDim, KD = Hkv * kHeadDim,
              I = c.intermediate, B = bs.B;
    if (Hq != kBatchG * Hkv) return 1;
    float *x = reinterpret_cast<float *>(buf + L.x);
    __half *h = reinterpret_cast<__half *>(buf + L.h);
    __half *q16 = reinterpret_cast<__half *>(buf + L.q16);
    __half *o16 = reinterpret_cast<__half *>(buf + L.o16);
    __half *act = reinterpret_cast<__half *>(buf + L.act);
    const size_t esz = a.kv_f32 ? 4 : 2;
    const size_t plane = (size_t)Hkv * bs.max_ctx * kHeadDim;  // elements of one layer's K (or V) plane
    const DevLayer *hl = im->host_layers.data();
    const int S = batch_splits(bs.max_n);
    float *qkv_raw = reinterpret_cast<float *>(buf + L.bqkv);
    // chained launches (programmatic dependent launch) only directly after a kernel
    if (launch_batch_tokens(bs.tokens_in, bs.picks, B, bs.tokens, stream, false) != cudaSuccess) return 1;
    if (launch_norm_rows(x, bs.tokens, a.embed, hl[0].input_norm, h, B, H, a.eps, stream, true) != cudaSuccess)
        return 1;
    bool ch = true;
    if (bs.hidden) {
        cudaMemcpyAsync(bs.hidden, x, (size_t)B * H * 4, cudaMemcpyDeviceToDevice, stream);
        ch = false;
    }
    for (int l = 0; l < c.n_layers; ++l) {
        // this layer's fp16 weights (converted once by prefill_init)
        const __half *wqkv = reinterpret_cast<const __half *>(buf + L.w16) + (size_t)l * L.w_layer;
        const __half *wo = wqkv + (size_t)(QD + 2 * KD) * H, *wgu = wo + (size_t)H * QD, *wd = wgu + (size_t)2 * I * H;
        uint8_t *kc = reinterpret_cast<uint8_t *>(bs.kc) + (size_t)l * plane * esz;
        uint8_t *vc = reinterpret_cast<uint8_t *>(bs.vc) + (size_t)l * plane * esz;
        // q | k | v of the B rows, then QK-Norm, RoPE at each sequence's position, K/V rows into
        // each sequence's cache
        BatchGemv g{};
        g.B = B;
        g.W = wqkv;
        g.a = nullptr;  // RMSNorm(x) with the layer's input norm, fused into the staging
        g.x = x;
        g.norm_w = hl[l].input_norm;
        g.eps = a.eps;
        g.N = QD + 2 * KD;
        g.K = H;
        g.out = qkv_raw;
        g.ldo = QD + 2 * KD;
        if (launch_bgemv(BG_STORE, g, st->nsm, stream, ch) != cudaSuccess) return 1;
        BatchQkvPost qp{};
        qp.qkv = qkv_raw;
        qp.q_norm = hl[l].q_norm;
        qp.k_norm = hl[l].k_norm;
        qp.rope = a.rope;
        qp.row_pos = bs.row_pos;
        qp.B = B;
        qp.Hq = Hq;
        qp.Hkv = Hkv;
        qp.eps = a.eps;
        qp.q16 = q16;
        qp.q_rows = st->rows_max;
        qp.kc = kc;
        qp.vc = vc;
        qp.seq_elems = bs.seq_elems;
        qp.max_ctx = bs.max_ctx;
        if (launch_bqkv_post(qp, a.kv_f32, stream, true) != cudaSuccess) return 1;
        BatchAttn ap{};
        ap.q16 = q16;
        ap.q_rows = st->rows_max;
        ap.kc = kc;
        ap.vc = vc;
        ap.seq_elems = bs.seq_elems;
        ap.max_ctx = bs.max_ctx;
        ap.row_pos = bs.row_pos;
        ap.S = S;
        ap.Hq = Hq;
        ap.scale_log2 = kLog2e / sqrtf((float)kHeadDim);
        ap.part = bs.part;
        if (launch_batch_attn(ap, Hkv, B, a.kv_f32, stream, true) != cudaSuccess) return 1;
        if (launch_batch_merge(bs.part, S, Hq, B, o16, QD, stream, true) != cudaSuccess) return 1;
        // x += o Wo^T
        g.W = wo;
        g.a = o16;
        g.N = H;
        g.K = QD;
        g.out = x;
        g.ldo = H;
        if (launch_bgemv(BG_ADD, g, st->nsm, stream, true) != cudaSuccess) return 1;
        // a = silu(h Wg^T) * (h Wu^T), h = RMSNorm(x) with the post-attention norm (fused)
        g.W = wgu;
        g.a = nullptr;
        g.norm_w = hl[l].post_norm;
        g.N = I;
        g.K = H;
        g.act = act;
        g.ldh = I;
        if (launch_bgemv(BG_SWIGLU, g, st->nsm, stream, true) != cudaSuccess) return 1;
        // x += a Wd^T
        g.W = wd;
        g.a = act;
        g.N = H;
        g.K = I;
        g.out = x;
        g.ldo = H;
        if (launch_bgemv(BG_ADD, g, st->nsm, stream, true) != cudaSuccess) return 1;
        ch = true;
        if (bs.hidden) {
            cudaMemcpyAsync(bs.hidden + (size_t)(l + 1) * B * H, x, (size_t)B * H * 4, cudaMemcpyDeviceToDevice,
                            stream);
            ch = false;
        }
    }
    BatchHead hp{};
    hp.x = x;
    hp.final_norm = a.final_norm;
    hp.E = a.lm_head;
    hp.B = B;
    hp.V = a.V;
    hp.eps = a.eps;
    hp.logits = bs.logits;
    hp.keys = bs.keys;
    hp.picks = bs.picks;
    hp.flags = a.flags;
    if (launch_batch_head(hp, H, st->nsm, stream, ch) != cudaSuccess) return 1;
    return cudaGetLastError() != cudaSuccess;
}

// ------------------------------------------------------------------ GEMM test entry

namespace {
__device__ StepFlags g_gemm_flags;  // status of the test GEMM entry point
}

int prefill_debug_gemm(const void *a, const void *b, float *c, int M, int N, int K, int bn, cudaStream_t stream) {
    if (prefill_prepare() != cudaSuccess) return QW_CUDA_ERROR;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QW_CUDA_ERROR;
    CUtensorMap ma, mb;
    if (!make_map(&ma, a, M, K, BM) || !make_map(&mb, b, N, K, bn)) return QW_INVALID_ARGUMENT;
    StepFlags *flags = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&flags), g_gemm_flags) != cudaSuccess) return QW_CUDA_ERROR;
    if (cudaMemsetAsync(flags, 0, sizeof(StepFlags), stream) != cudaSuccess) return QW_CUDA_ERROR;
    GemmParams gp{};
    gp.M = M;
    gp.N = N;
    gp.K = K;
    gp.out = c;
    gp.ldo = N;
    gp.flags = flags;
    cudaError_t e = bn == 256 ? launch_gemm<256, EPI_STORE>(ma, mb, gp, nsm, stream)
                              : launch_gemm<128, EPI_STORE>(ma, mb, gp, nsm, stream);
    if (e != cudaSuccess) return QW_CUDA_ERROR;
    StepFlags f{};
    if (cudaMemcpyAsync(&f, flags, sizeof(f), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return QW_CUDA_ERROR;
    return f.err ? (int)f.err : QW_OK;
}

}  // namespace qw
