// decode.cu - host glue of the persistent decode kernel (decode_kernel.cuh): kernel selection,
// launch attributes, the cooperative launch, and the bf16 -> f32 K/V widening used by imports.
#include "qw_internal.h"

namespace qw {

const void *decode_fn_d1(int fmt, int kv_f32);
const void *decode_fn_d2(int fmt, int kv_f32);
size_t decode_smem_bytes_impl();

namespace {

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// The kernel instantiation for (SM groups, weight format, cache element type).
const void *decode_fn(int D, int fmt, int kv_f32) {
    return D == 1 ? decode_fn_d1(fmt, kv_f32) : decode_fn_d2(fmt, kv_f32);
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

size_t decode_smem_bytes() { return decode_smem_bytes_impl(); }  // the same Smem layout for every instantiation

cudaError_t decode_prepare(int *blocks_per_sm) {
    const int bytes = (int)decode_smem_bytes();
    *blocks_per_sm = 1 << 30;
    for (int D = 1; D <= 2; ++D)
    for (int fmt = 0; fmt < 3; ++fmt)
        for (int kv = 0; kv < 2; ++kv) {
            const void *fn = decode_fn(D, fmt, kv);
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kDecodeThreads, bytes);
            if (e != cudaSuccess) return e;
            if (n < *blocks_per_sm) *blocks_per_sm = n;
        }
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &a, int ncta, cudaStream_t stream) {
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
    return cudaLaunchKernelExC(&cfg, decode_fn(a.D, a.fmt, a.kv_f32), args);
}

}  // namespace qw
