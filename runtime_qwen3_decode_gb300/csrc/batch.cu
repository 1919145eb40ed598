// batch.cu - the CUDA-core kernels of batched decode: B independent sequences, one new token
// each per step ("Portable WebAssembly Runtime Architecture for TinyRustLM", sections "Threads,
// Scheduling" and "Prefill versus decode": every sequence runs the decode step of "Scalar-Native
// Qwen3 Reference Runtime As The Numerical Authority", section 2, on its own K/V cache).
//
// The projections and the MLP of the B rows run as tensor-core GEMMs with M = B (prefill.cu,
// prefill_batch_step); here are the parts that differ per sequence:
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
    for (int j = p0 + warp; j < p1; j += kAttnWarps) {
        float k[4], v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            k[i] = to_f(K[(size_t)j * kHeadDim + lane + 32 * i]);
            v[i] = to_f(Vp[(size_t)j * kHeadDim + lane + 32 * i]);
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
    for (int vr = gw; vr < p.V; vr += nw) {
        const uint4 *row = reinterpret_cast<const uint4 *>(p.E + (size_t)vr * H);
        uint4 u[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) u[i] = __ldg(row + lane + 32 * i);
        float acc[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[b] = 0.f;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const int c = 8 * (lane + 32 * i);
            const __nv_bfloat162 *w2 = reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
            float2 w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = __bfloat1622float2(w2[e]);
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (b < B) {
                    const float4 h0 = *reinterpret_cast<const float4 *>(hf + b * H + c);
                    const float4 h1 = *reinterpret_cast<const float4 *>(hf + b * H + c + 4);
                    acc[b] += w[0].x * h0.x + w[0].y * h0.y + w[1].x * h0.z + w[1].y * h0.w + w[2].x * h1.x +
                              w[2].y * h1.y + w[3].x * h1.z + w[3].y * h1.w;
                }
            }
        }
        const float t = warp_sum8(acc, lane);
        const int b = lane >> 2;
        if ((lane & 3) == 0 && b < B) {
            p.logits[(size_t)b * p.V + vr] = t;
            if (!isfinite(t)) bad = true;
            const unsigned long long k = argmax_key(t, vr);
            kbest = k > kbest ? k : kbest;
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

cudaError_t batch_prepare() {
    cudaError_t e = cudaFuncSetAttribute(batch_head_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBatchMax * 1024 * 4);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(batch_head_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBatchMax * 2048 * 4);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(batch_head_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kBatchMax * 3072 * 4);
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
