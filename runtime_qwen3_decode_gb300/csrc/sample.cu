// sample.cu - on-device sampling of the next token from f32 logits.
//
// The order of "Portable WebAssembly Runtime Architecture for TinyRustLM", section
// "Sampling order", with the PCG32 of its "Deterministic sampling contract" and the
// repetition penalty of "Scalar-Native Qwen3 Reference Runtime ...", section 7:
//   repetition penalty (each token of the history once: positive / penalty,
//   negative * penalty) -> NaN to -inf, -0 to +0 -> temperature 0: the greatest
//   logit, lowest id on ties, no draw -> otherwise divide by the temperature ->
//   top-k (descending value, ascending id) -> max-shifted probabilities over the
//   survivors -> the minimal prefix whose cumulative probability reaches top_p ->
//   renormalise -> one PCG32 word u = (w >> 8) 2^-24 -> the first candidate whose
//   cumulative probability exceeds u (the last one if rounding leaves none).
//
// Three launches: mark the history in a token bitmap; per block of 1024 tokens apply
// the transforms and keep the block's best kSampleMaxTopK by a bitonic sort of packed
// (value, id) keys; one CTA sorts the candidates of every block and runs the
// probability, nucleus and draw steps in candidate order on one thread (binary32, the
// same sequence of operations as the sequential definition).
#include "qw_sample.h"

namespace qw {
namespace {

constexpr int kBlockTokens = 1024;
constexpr int kSelectThreads = 256;
constexpr int kFinalThreads = 1024;

__device__ __forceinline__ uint32_t ord_bits(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_value(uint32_t e) {
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7fffffffu) : ~e);
}
// Larger key = larger value, then smaller id; 0 is below every real key.
__device__ __forceinline__ unsigned long long cand_key(float v, int id) {
    return ((unsigned long long)ord_bits(v) << 32) | (0xffffffffu - (uint32_t)id);
}

// Descending bitonic sort of n (a power of two) keys in shared memory by the block.
__device__ void bitonic_desc(unsigned long long *k, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long a = k[lo], b = k[hi];
                if ((a < b) == desc) {
                    k[lo] = b;
                    k[hi] = a;
                }
            }
        }
    }
    __syncthreads();
}

__global__ void sample_mark_kernel(const int32_t *hist, int n, int V, uint32_t *bitmap, uint32_t *status) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int t = hist[i];
        if (t < 0 || t >= V) {
            atomicOr(status, 1u);
            continue;
        }
        atomicOr(bitmap + (t >> 5), 1u << (t & 31));
    }
}

__global__ void __launch_bounds__(kSelectThreads) sample_select_kernel(const float *logits, int V,
                                                                       const uint32_t *bitmap, float penalty,
                                                                       float temperature,
                                                                       unsigned long long *cand) {
    __shared__ unsigned long long k[kBlockTokens];
    const int base = blockIdx.x * kBlockTokens;
    for (int j = threadIdx.x; j < kBlockTokens; j += kSelectThreads) {
        const int i = base + j;
        unsigned long long key = 0ull;
        if (i < V) {
            float x = logits[i];
            if ((bitmap[i >> 5] >> (i & 31)) & 1u) {
                if (x > 0.0f)
                    x = x / penalty;
                else if (x < 0.0f)
                    x = x * penalty;
            }
            if (isnan(x)) x = -INFINITY;
            if (x == 0.0f) x = 0.0f;
            if (temperature > 0.0f) x = x / temperature;
            key = cand_key(x, i);
        }
        k[j] = key;
    }
    bitonic_desc(k, kBlockTokens);
    for (int j = threadIdx.x; j < kSampleMaxTopK; j += kSelectThreads)
        cand[(size_t)blockIdx.x * kSampleMaxTopK + j] = k[j];
}

__device__ __forceinline__ uint32_t pcg32_next(uint64_t &state, uint64_t inc) {
    const uint64_t old = state;
    state = old * 6364136223846793005ull + inc;
    const uint32_t xorshifted = (uint32_t)(((old >> 18) ^ old) >> 27);
    const uint32_t rot = (uint32_t)(old >> 59);
    return (xorshifted >> rot) | (xorshifted << ((32u - rot) & 31u));
}

__global__ void __launch_bounds__(kFinalThreads) sample_final_kernel(const unsigned long long *cand, int ncand,
                                                                     int npow, float temperature, int top_k,
                                                                     float top_p, uint64_t *rng, int32_t *token,
                                                                     int32_t *next_tok, unsigned *err,
                                                                     const uint32_t *status) {
    extern __shared__ unsigned long long k[];
    for (int j = threadIdx.x; j < npow; j += kFinalThreads) k[j] = j < ncand ? cand[j] : 0ull;
    bitonic_desc(k, npow);
    if (threadIdx.x != 0) return;
    int32_t tok = -1;
    unsigned code = 0;
    const float top = ord_value((uint32_t)(k[0] >> 32));
    if (*status) {
        code = kErrInvalidArgument;  // a history id outside [0, vocab)
    } else if (top == -INFINITY) {
        code = kErrNumerical;  // every logit masked: nothing can be drawn
    } else if (temperature == 0.0f) {
        tok = (int32_t)(0xffffffffu - (uint32_t)(k[0] & 0xffffffffull));
    } else {
        float p[kSampleMaxTopK];
        const int n_k = top_k;
        const float m = top;
        float s = 0.0f;
        for (int j = 0; j < n_k; ++j) {
            p[j] = expf(ord_value((uint32_t)(k[j] >> 32)) - m);
            s = s + p[j];
        }
        for (int j = 0; j < n_k; ++j) p[j] = p[j] / s;
        int n = n_k;
        if (top_p < 1.0f) {
            float c = 0.0f;
            for (int j = 0; j < n_k; ++j) {
                c = c + p[j];
                if (c >= top_p) {
                    n = j + 1;
                    break;
                }
            }
        }
        float z = 0.0f;
        for (int j = 0; j < n; ++j) z = z + p[j];
        uint64_t st = rng[0];
        const uint32_t w = pcg32_next(st, rng[1]);
        rng[0] = st;
        const float u = (float)(w >> 8) * (1.0f / 16777216.0f);
        int pick = n - 1;
        float c = 0.0f;
        for (int j = 0; j < n; ++j) {
            c = c + p[j] / z;
            if (c > u) {
                pick = j;
                break;
            }
        }
        tok = (int32_t)(0xffffffffu - (uint32_t)(k[pick] & 0xffffffffull));
    }
    if (token) *token = tok;
    if (next_tok && tok >= 0) *next_tok = tok;
    if (err && code) atomicCAS(err, 0u, code);
}

int select_blocks(int V) { return (V + kBlockTokens - 1) / kBlockTokens; }

int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

size_t sample_scratch_bytes(int V) {
    const size_t bitmap = (size_t)(V + 31) / 32 * 4;
    const size_t cand = (size_t)select_blocks(V) * kSampleMaxTopK * 8;
    return 256 + (bitmap + 255) / 256 * 256 + cand;
}

cudaError_t launch_sample(const float *logits, int V, const int32_t *hist, int n_hist, float temperature,
                          int top_k, float top_p, float penalty, uint64_t *rng, int32_t *token, int32_t *next_tok,
                          unsigned *err, void *scratch, cudaStream_t stream) {
    uint8_t *s = reinterpret_cast<uint8_t *>(scratch);
    uint32_t *status = reinterpret_cast<uint32_t *>(s);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(s + 256);
    const size_t bitmap_bytes = (size_t)(V + 31) / 32 * 4;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(s + 256 + (bitmap_bytes + 255) / 256 * 256);
    const int nb = select_blocks(V);
    const int ncand = nb * kSampleMaxTopK;
    const int npow = pow2_at_least(ncand);
    const size_t smem = (size_t)npow * 8;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(s, 0, 256 + bitmap_bytes, stream);
    if (e != cudaSuccess) return e;
    if (n_hist > 0 && penalty != 1.0f) {
        sample_mark_kernel<<<(n_hist + 255) / 256, 256, 0, stream>>>(hist, n_hist, V, bitmap, status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    sample_select_kernel<<<nb, kSelectThreads, 0, stream>>>(logits, V, bitmap, penalty, temperature, cand);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(sample_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    sample_final_kernel<<<1, kFinalThreads, smem, stream>>>(cand, ncand, npow, temperature, top_k, top_p, rng, token,
                                                           next_tok, err, status);
    return cudaGetLastError();
}

}  // namespace qw
