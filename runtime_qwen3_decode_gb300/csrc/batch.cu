// batch.cu - the CUDA-core kernels of batched decode: B independent sequences, one new token
// each per step ("Portable WebAssembly Runtime Architecture for TinyRustLM", sections "Threads,
// Scheduling" and "Prefill versus decode": every sequence runs the decode step of "Scalar-Native
// Qwen3 Reference Runtime As The Numerical Authority", section 2, on its own K/V cache).
//
// The step itself is sequenced by prefill_batch_step (prefill.cu); its kernels are here:
//   bgemv_kernel        the projections and the MLP of the B rows: every weight row read once
//                       and dotted with all B activation rows (residual add or SwiGLU fused)
//   bqkv_post_kernel    QK-Norm and RoPE of each sequence's q and k heads at its own position,
//                       q into the fp16 query rows, k and v appended to its own cache
//   batch_attn_kernel   GQA attention of each sequence's new query rows over its own cache,
//                       split over positions (one CTA per (split, KV head, sequence)), online
//                       softmax, a partial (acc, max, sum) per query head and split
//   batch_merge_kernel  the splits of each (sequence, query head) merged into the fp16 o row
//   batch_head_kernel   final RMSNorm of the B rows, the tied lm_head streamed once for all of
//                       them, logits [B][V] and one packed (logit, id) argmax key per sequence
//   batch_pick_kernel   keys -> next tokens
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "qw_batch.h"
#include "tc.cuh"

namespace qw {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kGemvWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename KT>
__device__ __forceinline__ float to_f(KT v) {
    if constexpr (sizeof(KT) == 4) return v;
    else return __bfloat162float(v);
}

// ------------------------------------------------------------------ skinny projections
//
// y[b][r] = sum_k W[r][k] a[b][k] for the B <= 8 rows of a step.  With M = B the work is a
// matrix-vector product per row: its bound is the weight bytes, each read once from HBM.
// Every CTA stages the B activation rows (fp16) in shared memory.  A unit is two weight
// rows (rows 2u, 2u + 1, or the gate and up rows of output u); a group of KS warps takes a
// unit, each warp 1/KS of K (KS = 4 from K = 2048 up, else 1, so that a warp has at least
// two chunks per row and the short rows keep one warp per unit): it issues all of its
// 16-byte weight loads before the arithmetic, accumulates f32 dot products with all B
// rows (lane l owns the 8-element chunks l + 32 c of its part) and reduces its 2 x 8 sums
// with a transposed butterfly; the group's partial sums are then added in a fixed order.  Every output element has
// one owner: no atomics, the same result every run.

// Lane l of the warp ends with sum over lanes of v[i] for i = 8 b4 + 4 b3 + 2 b2 + b1,
// b_k = bit k of l (lanes l and l ^ 1 hold the same sum): 9 shuffles for 16 sums.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int s = 16, m = 8; m >= 1; s >>= 1, m >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < m; ++i) {
            const float send = upper ? v[i] : v[i + m];
            const float keep = upper ? v[i + m] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ void half8_to_f(const uint4 &u, float (&f)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int EPI, int KC>  // KC = K / 256: 16-byte chunks per lane and row
__global__ void __launch_bounds__(kGemvWarps * 32) bgemv_kernel(const BatchGemv p) {
    constexpr int KS = KC >= 8 ? 4 : 1, NG = kGemvWarps / KS;  // warps per unit; units per pass
    static_assert(KC % KS == 0 && kGemvWarps % KS == 0, "the warps of a unit split K evenly");
    constexpr int K8 = KC * 32, KQ = KC / KS;  // row length in uint4; chunks per lane and warp
    extern __shared__ __align__(16) uint4 sa[];  // [B][K8] activation rows, 8 fp16 per entry
    __shared__ float part[NG][KS][16];            // [unit of the pass][K part][value]
    tc::chain_wait();
    tc::chain_release();
    const int B = p.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, grp = warp / KS, kq = warp % KS;
    if (p.a) {
        for (int i = threadIdx.x; i < B * K8; i += kGemvWarps * 32) sa[i] = reinterpret_cast<const uint4 *>(p.a)[i];
    } else {
        // RMSNorm of the residual rows while staging them, in the norm_rows kernel's order:
        // lane l's chunks l + 32 c summed in place, then the warp butterfly
        for (int b = warp; b < B; b += kGemvWarps) {
            const float4 *xr = reinterpret_cast<const float4 *>(p.x + (size_t)b * K8 * 8);
            float v[KC][8];
#pragma unroll
            for (int c = 0; c < KC; ++c) {
                const float4 a0 = xr[2 * (lane + 32 * c)], a1 = xr[2 * (lane + 32 * c) + 1];
                v[c][0] = a0.x, v[c][1] = a0.y, v[c][2] = a0.z, v[c][3] = a0.w;
                v[c][4] = a1.x, v[c][5] = a1.y, v[c][6] = a1.z, v[c][7] = a1.w;
            }
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < KC; ++c)
#pragma unroll
                for (int i = 0; i < 8; ++i) ss += v[c][i] * v[c][i];
#pragma unroll
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float r = rsqrtf(ss / (float)(K8 * 8) + p.eps);
            const uint4 *wr = reinterpret_cast<const uint4 *>(p.norm_w);
#pragma unroll
            for (int c = 0; c < KC; ++c) {
                const uint4 u = wr[lane + 32 * c];
                const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
                __half2 hv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(b2[i]);
                    hv[i] = __floats2half2_rn(f.x * (v[c][2 * i] * r), f.y * (v[c][2 * i + 1] * r));
                }
                sa[b * K8 + lane + 32 * c] = *reinterpret_cast<const uint4 *>(hv);
            }
        }
    }
    __syncthreads();
    const int units = EPI == BG_SWIGLU ? p.N : p.N / 2;
    for (int base = NG * blockIdx.x; base < units; base += NG * gridDim.x) {  // uniform over the CTA
        const int u = base + grp;
        // SWIGLU: gate row i of the interleaved weights is (i / 128) 256 + i % 128, up row +128
        const int r0 = EPI == BG_SWIGLU ? (u >> 7) * 256 + (u & 127) : 2 * u;
        const int r1 = EPI == BG_SWIGLU ? r0 + 128 : r0 + 1;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        if (u < units) {
            const int c0 = lane + 32 * KQ * kq;  // this warp's first chunk of the row
            const uint4 *w0 = reinterpret_cast<const uint4 *>(p.W) + (size_t)r0 * K8 + c0;
            const uint4 *w1 = reinterpret_cast<const uint4 *>(p.W) + (size_t)r1 * K8 + c0;
            uint4 x0[KQ], x1[KQ];
#pragma unroll
            for (int c = 0; c < KQ; ++c) {
                x0[c] = ld_stream(w0 + 32 * c);
                x1[c] = ld_stream(w1 + 32 * c);
            }
#pragma unroll
            for (int c = 0; c < KQ; ++c) {
                float f0[8], f1[8];
                half8_to_f(x0[c], f0);
                half8_to_f(x1[c], f1);
#pragma unroll
                for (int b = 0; b < kBatchMax; ++b) {
                    if (b < B) {
                        float av[8];
                        half8_to_f(sa[b * K8 + c0 + 32 * c], av);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            acc[b] = fmaf(f0[e], av[e], acc[b]);
                            acc[8 + b] = fmaf(f1[e], av[e], acc[8 + b]);
                        }
                    }
                }
            }
        }
        const float v = warp_sum16(acc, lane);
        if ((lane & 1) == 0) {
            const int idx = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
            part[grp][kq][idx] = v;
        }
        if (KS > 1) __syncthreads();
        else __syncwarp();
        if (u < units && kq == 0 && lane < 16) {  // value lane: row (lane < 8 ? r0 : r1), sequence lane % 8
            const int b = lane & 7;
            float y = 0.f, up = 0.f;
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                y += part[grp][k][lane];
                if (EPI == BG_SWIGLU && lane < 8) up += part[grp][k][lane + 8];
            }
            if constexpr (EPI == BG_SWIGLU) {
                if (lane < 8 && b < B) {  // g = y (gate row), up from value lane + 8
                    // SiLU(g) u as in the prefill epilogue
                    p.act[(size_t)b * p.ldh + u] = __float2half_rn(__fdividef(y, 1.0f + __expf(-y)) * up);
                }
            } else if (b < B) {
                float *o = p.out + (size_t)b * p.ldo + (lane < 8 ? r0 : r1);
                if constexpr (EPI == BG_ADD) *o += y;
                else *o = y;
            }
        }
        if (KS > 1) __syncthreads();  // part is rewritten by the next pass
        else __syncwarp();
    }
}

// One (head slot, sequence): the raw q|k|v projection of the sequence's row -> QK-Norm and
// RoPE for q and k heads at the sequence's position (the decode kernel's arithmetic:
// r = rsqrt(mean(v^2) + eps), v = w * (v * r), dims (i, i + 64) rotated), q into the fp16
// query row, k and v into the sequence's cache at that position.  Lane l holds dims l + 32 j.
template <typename KT>
__global__ void __launch_bounds__(32) bqkv_post_kernel(const BatchQkvPost p) {
    tc::chain_wait();
    tc::chain_release();
    const int slot = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
    const int QD = p.Hq * kHeadDim, W = QD + 2 * p.Hkv * kHeadDim;
    const bool is_q = slot < p.Hq, is_k = !is_q && slot < p.Hq + p.Hkv;
    const float *src = p.qkv + (size_t)b * W + (size_t)slot * kHeadDim;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = src[lane + 32 * j];
    const int pos = p.row_pos[b];
    if (is_q || is_k) {
        const __nv_bfloat16 *w = is_q ? p.q_norm : p.k_norm;
        const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
        const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __bfloat162float(w[lane + 32 * j]) * (v[j] * r);
        const float2 *cs = p.rope + (size_t)pos * (kHeadDim / 2);
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // pairs (lane + 32 j, lane + 32 j + 64)
            const float2 c = cs[lane + 32 * j];
            const float a = v[j], bb = v[j + 2];
            v[j] = a * c.x - bb * c.y;
            v[j + 2] = bb * c.x + a * c.y;
        }
    }
    if (is_q) {
        __half *dst = p.q16 + ((size_t)slot * p.q_rows + b) * kHeadDim;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = __float2half_rn(v[j]);
        return;
    }
    const int kvh = is_k ? slot - p.Hq : slot - p.Hq - p.Hkv;
    KT *dst = reinterpret_cast<KT *>(is_k ? p.kc : p.vc) + (size_t)b * p.seq_elems +
              ((size_t)kvh * p.max_ctx + pos) * kHeadDim;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (sizeof(KT) == 4) dst[lane + 32 * j] = v[j];
        else dst[lane + 32 * j] = __float2bfloat16_rn(v[j]);
    }
}

// One (split, KV head, sequence).  Warp w takes positions p0 + w, p0 + w + 8, ...; lane L holds
// dims L, L + 32, L + 64, L + 96 of the two query heads of the KV head and of each K/V row.
template <typename KT>
__global__ void __launch_bounds__(kAttnWarps * 32) batch_attn_kernel(BatchAttn p) {
    constexpr int G = kBatchG;
    __shared__ float wml[kAttnWarps][G][2];
    __shared__ float wacc[kAttnWarps][G][kHeadDim];
    tc::chain_wait();
    tc::chain_release();
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.row_pos[b] + 1;  // cached positions including this step's row
    const int per = (n + p.S - 1) / p.S;
    const int p0 = s * per, p1 = min(n, p0 + per);
    const KT *K = reinterpret_cast<const KT *>(p.kc) + (size_t)b * p.seq_elems + (size_t)h * p.max_ctx * kHeadDim;
    const KT *Vp = reinterpret_cast<const KT *>(p.vc) + (size_t)b * p.seq_elems + (size_t)h * p.max_ctx * kHeadDim;
    float q[G][4], acc[G][4], m[G], l[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __half *qr = p.q16 + ((size_t)(h * G + g) * p.q_rows + b) * kHeadDim;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[g][i] = __half2float(qr[lane + 32 * i]) * p.scale_log2;
            acc[g][i] = 0.f;
        }
        m[g] = -INFINITY;
        l[g] = 0.f;
    }
    // the next position's K and V rows load while this one's are used
    float kn[4], vn[4];
    if (p0 + warp < p1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            kn[i] = to_f(K[(size_t)(p0 + warp) * kHeadDim + lane + 32 * i]);
            vn[i] = to_f(Vp[(size_t)(p0 + warp) * kHeadDim + lane + 32 * i]);
        }
    }
    for (int j = p0 + warp; j < p1; j += kAttnWarps) {
        float k[4], v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            k[i] = kn[i];
            v[i] = vn[i];
        }
        if (j + kAttnWarps < p1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                kn[i] = to_f(K[(size_t)(j + kAttnWarps) * kHeadDim + lane + 32 * i]);
                vn[i] = to_f(Vp[(size_t)(j + kAttnWarps) * kHeadDim + lane + 32 * i]);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sc = q[g][0] * k[0] + q[g][1] * k[1] + q[g][2] * k[2] + q[g][3] * k[3];
            sc = warp_sum(sc);  // log2-domain score
            const float mn = fmaxf(m[g], sc);
            const float alpha = m[g] == -INFINITY ? 0.f : exp2f(m[g] - mn);
            const float pr = exp2f(sc - mn);
            l[g] = l[g] * alpha + pr;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[g][i] = acc[g][i] * alpha + pr * v[i];
            m[g] = mn;
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) {
            wml[warp][g][0] = m[g];
            wml[warp][g][1] = l[g];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) wacc[warp][g][lane + 32 * i] = acc[g][i];
    }
    __syncthreads();
    // combine the warps (exact rescaling to the common max) into this split's partial
    for (int t = threadIdx.x; t < G * kHeadDim; t += blockDim.x) {
        const int g = t / kHeadDim, d = t % kHeadDim;
        float mx = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) mx = fmaxf(mx, wml[w][g][0]);
        float av = 0.f, ls = 0.f;
        if (mx != -INFINITY)
            for (int w = 0; w < kAttnWarps; ++w) {
                const float mw = wml[w][g][0];
                if (mw == -INFINITY) continue;
                const float sc = exp2f(mw - mx);
                av += wacc[w][g][d] * sc;
                ls += wml[w][g][1] * sc;
            }
        float *dst = p.part + (((size_t)b * p.Hq + h * G + g) * p.S + s) * kBatchPartStride;
        dst[d] = av;
        if (d == 0) {
            dst[kHeadDim] = mx;
            dst[kHeadDim + 1] = ls;
        }
    }
}

// One (query head, sequence): o = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), splits in order.
__global__ void __launch_bounds__(kHeadDim) batch_merge_kernel(const float *part, int S, int Hq, __half *o16,
                                                                int ldo) {
    tc::chain_wait();
    tc::chain_release();
    const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const float *src = part + ((size_t)b * Hq + hq) * S * kBatchPartStride;
    float mx = -INFINITY;
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, src[(size_t)s * kBatchPartStride + kHeadDim]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < S; ++s) {
        const float ms = src[(size_t)s * kBatchPartStride + kHeadDim];
        if (ms == -INFINITY) continue;
        const float sc = exp2f(ms - mx);
        num += src[(size_t)s * kBatchPartStride + d] * sc;
        den += src[(size_t)s * kBatchPartStride + kHeadDim + 1] * sc;
    }
    o16[(size_t)b * ldo + (size_t)hq * kHeadDim + d] = __float2half_rn(num / den);
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    if (v == 0.0f) v = 0.0f;  // -0 and +0 compare equal: lowest id wins
    const uint32_t u = __float_as_uint(v);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

// Warp sums of 8 values at once: afterwards lane L holds the total of value L / 4.
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane) {
#pragma unroll
    for (int h = 4, o = 16; h >= 1; h >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h], keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    return t;
}

// Final RMSNorm of the B rows (every CTA recomputes them into shared memory), then each warp
// streams lm_head rows once and dots each with all B normalised rows.
template <int KM>
__global__ void __launch_bounds__(kBatchHeadThreads) batch_head_kernel(BatchHead p) {
    constexpr int H = 1024 * KM, NC = 4 * KM;  // 16-byte chunks of 8 bf16 per lane and row
    extern __shared__ __align__(16) float hf[];  // [B][H]
    __shared__ unsigned long long best[kBatchHeadThreads / 32][kBatchMax];
    __shared__ int bad_any;
    tc::chain_wait();
    tc::chain_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.B;
    if (threadIdx.x == 0) bad_any = 0;
    for (int b = warp; b < B; b += kBatchHeadThreads / 32) {
        const float *x = p.x + (size_t)b * H;
        float ss = 0.f;
        for (int c = lane; c < H; c += 32) ss += x[c] * x[c];
        const float r = rsqrtf(warp_sum(ss) / (float)H + p.eps);
        for (int c = lane; c < H; c += 32) hf[b * H + c] = __bfloat162float(p.final_norm[c]) * (x[c] * r);
    }
    __syncthreads();
    unsigned long long kbest = 0;  // for value lane / 4 (a sequence)
    bool bad = false;
    const int gw = blockIdx.x * (kBatchHeadThreads / 32) + warp, nw = gridDim.x * (kBatchHeadThreads / 32);
    // four rows per pass (v0 + j nw): every normalised value read from shared memory serves
    // all four (the pass is bound by those reads, not by the rows' HBM bytes), and all loads
    // of the four rows are issued before the arithmetic
    constexpr int R = 4;
    for (int v0 = gw; v0 < p.V; v0 += R * nw) {
        int vr[R];
#pragma unroll
        for (int j = 0; j < R; ++j) vr[j] = v0 + j * nw < p.V ? v0 + j * nw : v0;
        uint4 u[R][NC];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const uint4 *row = reinterpret_cast<const uint4 *>(p.E + (size_t)vr[j] * H);
#pragma unroll
            for (int i = 0; i < NC; ++i) u[j][i] = __ldg(row + lane + 32 * i);
        }
        float acc[R][8];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[j][b] = 0.f;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const int c = 8 * (lane + 32 * i);
            float w[R][8];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 t = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(&u[j][i])[e]);
                    w[j][2 * e] = t.x;
                    w[j][2 * e + 1] = t.y;
                }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (b < B) {
                    const float4 h0 = *reinterpret_cast<const float4 *>(hf + b * H + c);
                    const float4 h1 = *reinterpret_cast<const float4 *>(hf + b * H + c + 4);
                    const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                    for (int j = 0; j < R; ++j)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[j][b] = fmaf(w[j][e], hv[e], acc[j][b]);
                }
            }
        }
        const int b = lane >> 2;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float t = warp_sum8(acc[j], lane);
            const bool dup = j > 0 && vr[j] == v0;  // past the end: row v0 again, already taken
            if ((lane & 3) == 0 && b < B && !dup) {
                p.logits[(size_t)b * p.V + vr[j]] = t;
                if (!isfinite(t)) bad = true;
                const unsigned long long k = argmax_key(t, vr[j]);
                kbest = k > kbest ? k : kbest;
            }
        }
    }
    if ((lane & 3) == 0 && (lane >> 2) < kBatchMax) best[warp][lane >> 2] = kbest;
    if (bad) bad_any = 1;
    __syncthreads();
    if (threadIdx.x < B) {
        unsigned long long m = 0;
        for (int w = 0; w < kBatchHeadThreads / 32; ++w) m = best[w][threadIdx.x] > m ? best[w][threadIdx.x] : m;
        if (m) atomicMax(p.keys + threadIdx.x, m);
    }
    if (threadIdx.x == 0 && bad_any) atomicCAS(&p.flags->err, 0u, kErrNumerical);
}

__global__ void batch_pick_kernel(unsigned long long *keys, int B, int32_t *picks) {
    tc::chain_wait();
    tc::chain_release();
    const int b = threadIdx.x;
    if (b >= B) return;
    const unsigned long long k = keys[b];
    picks[b] = k ? (int)(0xffffffffu - (unsigned)(k & 0xffffffffull)) : -1;
    keys[b] = 0ull;
}

// tokens[b] = the caller's token, or (-1) this sequence's previous device-resident pick
__global__ void batch_tokens_kernel(const int32_t *in, const int32_t *picks, int B, int32_t *tokens) {
    tc::chain_wait();
    tc::chain_release();
    const int b = threadIdx.x;
    if (b < B) tokens[b] = in[b] >= 0 ? in[b] : picks[b];
}

}  // namespace

template <int EPI>
cudaError_t set_bgemv_attr() {
    const int smem = kBatchMax * 6144 * 2;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bgemv_kernel<EPI, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) ||
        (e = cudaFuncSetAttribute(bgemv_kernel<EPI, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) ||
        (e = cudaFuncSetAttribute(bgemv_kernel<EPI, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) ||
        (e = cudaFuncSetAttribute(bgemv_kernel<EPI, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) ||
        (e = cudaFuncSetAttribute(bgemv_kernel<EPI, 24>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)))
        return e;
    return cudaSuccess;
}

cudaError_t batch_prepare() {
    cudaError_t e = cudaFuncSetAttribute(batch_head_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBatchMax * 1024 * 4);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(batch_head_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBatchMax * 2048 * 4);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(batch_head_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBatchMax * 3072 * 4);
    if (e != cudaSuccess) return e;
    if ((e = set_bgemv_attr<BG_STORE>()) != cudaSuccess || (e = set_bgemv_attr<BG_ADD>()) != cudaSuccess) return e;
    return set_bgemv_attr<BG_SWIGLU>();
}

template <int EPI>
cudaError_t launch_bgemv_k(const BatchGemv &p, int nsm, cudaStream_t st, bool chained) {
    const size_t smem = (size_t)p.B * p.K * 2;
    const dim3 grid(2 * nsm), block(kGemvWarps * 32);
    switch (p.K) {
        case 1024: return launch_k(chained, bgemv_kernel<EPI, 4>, grid, block, smem, st, p);
        case 2048: return launch_k(chained, bgemv_kernel<EPI, 8>, grid, block, smem, st, p);
        case 3072: return launch_k(chained, bgemv_kernel<EPI, 12>, grid, block, smem, st, p);
        case 4096: return launch_k(chained, bgemv_kernel<EPI, 16>, grid, block, smem, st, p);
        case 6144: return launch_k(chained, bgemv_kernel<EPI, 24>, grid, block, smem, st, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bgemv(int epi, const BatchGemv &p, int nsm, cudaStream_t st, bool chained) {
    if (p.B < 1 || p.B > kBatchMax || p.N < 1 || (epi != BG_SWIGLU && (p.N & 1)) || !bgemv_supported(p.K))
        return cudaErrorInvalidValue;
    return epi == BG_STORE ? launch_bgemv_k<BG_STORE>(p, nsm, st, chained)
           : epi == BG_ADD ? launch_bgemv_k<BG_ADD>(p, nsm, st, chained)
                           : launch_bgemv_k<BG_SWIGLU>(p, nsm, st, chained);
}

cudaError_t launch_bqkv_post(const BatchQkvPost &p, int kv_f32, cudaStream_t st, bool chained) {
    const dim3 grid(p.Hq + 2 * p.Hkv, p.B), block(32);
    return kv_f32 ? launch_k(chained, bqkv_post_kernel<float>, grid, block, 0, st, p)
                  : launch_k(chained, bqkv_post_kernel<__nv_bfloat16>, grid, block, 0, st, p);
}

cudaError_t launch_batch_tokens(const int32_t *in, const int32_t *picks, int B, int32_t *tokens, cudaStream_t st,
                                bool chained) {
    return launch_k(chained, batch_tokens_kernel, dim3(1), dim3(32), 0, st, in, picks, B, tokens);
}

cudaError_t launch_batch_attn(const BatchAttn &p, int Hkv, int B, int kv_f32, cudaStream_t st, bool chained) {
    const dim3 grid(p.S, Hkv, B), block(kAttnWarps * 32);
    return kv_f32 ? launch_k(chained, batch_attn_kernel<float>, grid, block, 0, st, p)
                  : launch_k(chained, batch_attn_kernel<__nv_bfloat16>, grid, block, 0, st, p);
}

cudaError_t launch_batch_merge(const float *part, int S, int Hq, int B, __half *o16, int ldo, cudaStream_t st,
                               bool chained) {
    return launch_k(chained, batch_merge_kernel, dim3(Hq, B), dim3(kHeadDim), 0, st, part, S, Hq, o16, ldo);
}

cudaError_t launch_batch_head(const BatchHead &p, int H, int nsm, cudaStream_t st, bool chained) {
    const size_t smem = (size_t)p.B * H * 4;
    auto k = H >> 10 == 1 ? batch_head_kernel<1> : H >> 10 == 2 ? batch_head_kernel<2> : batch_head_kernel<3>;
    cudaError_t e = launch_k(chained, k, dim3(4 * nsm), dim3(kBatchHeadThreads), smem, st, p);
    if (e != cudaSuccess) return e;
    return launch_k(true, batch_pick_kernel, dim3(1), dim3(32), 0, st, p.keys, p.B, p.picks);
}

}  // namespace qw
