// mma_rate.cu - standalone measurement of the tcgen05 tensor-core rate (not part of libqw).
//
// One thread per CTA issues R back-to-back tcgen05.mma.cta_group::1.kind::f16 (M = 128,
// K = 16, accumulate into one TMEM tile) on zero operands, commits once and waits for the
// commit; clock64 around the issue loop and the wait gives cycles per MMA.  Operand A comes
// from shared memory (SS) or from TMEM (TS); N is 64, 128 or 256; "alt" alternates two
// accumulators.  The grid is one CTA, then 148 (one per SM: 120 KB of shared memory each).
// Every access stays inside the CTA's operand tiles and its 512 TMEM columns, and the one
// wait is bounded.
//
// Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I runtime_qwen3_decode_gb300/csrc \
//        -o mma_rate runtime_qwen3_decode_gb300/csrc/probes/mma_rate.cu && ./mma_rate
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "tc.cuh"
using namespace qw::tc;

template <int N, bool TS, bool ALT>
__global__ void __launch_bounds__(128, 1) mma_rate(int R, long long *out, int *err) {
    extern __shared__ __align__(1024) uint8_t raw[];
    uint8_t *base = raw + ((1024u - (su32(raw) & 1023u)) & 1023u);
    uint8_t *sA = base;
    uint8_t *sB = base + 16384;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + N * 128);
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar + 1);
    for (int i = threadIdx.x; i < (16384 + N * 128) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(base)[i] = make_uint4(0, 0, 0, 0);
    fence_async_shared();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    const int warp = threadIdx.x >> 5;
    if (warp == 0) tmem_alloc(slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;
    if (threadIdx.x == 32) {
        constexpr uint32_t idesc = idesc_f16_f32(128, N);
        const uint32_t a = su32(sA), b = su32(sB);
        const long long t0 = clock64();
        for (int i = 0; i < R; ++i) {
            const int k = i & 3;
            const uint64_t bd = desc_sw128(b) + 2u * k;
            const uint32_t d = tm + (ALT ? (uint32_t)((i & 1) * N) : 0u);
            if (TS)
                mma_f16_ts(d, tm + 256u + 8u * k, bd, idesc, i > 1);
            else
                mma_f16(d, desc_sw128(a) + 2u * k, bd, idesc, i > 1);
        }
        const long long t1 = clock64();
        mma_commit(bar);
        const bool ok = mbar_wait(bar, 0, nullptr, false, 1000000000ull);
        const long long t2 = clock64();
        out[2 * blockIdx.x] = t1 - t0;
        out[2 * blockIdx.x + 1] = t2 - t0;
        if (!ok) atomicExch(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

template <int N, bool TS, bool ALT>
void run(const char *name, int grid) {
    const int R = 1024;
    long long *d;
    int *e;
    cudaMalloc(&d, 2 * 256 * sizeof(long long));
    cudaMalloc(&e, 4);
    cudaMemset(e, 0, 4);
    const int smem = 120 * 1024;
    cudaFuncSetAttribute(mma_rate<N, TS, ALT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    for (int rep = 0; rep < 2; ++rep) mma_rate<N, TS, ALT><<<grid, 128, smem>>>(R, d, e);
    cudaError_t st = cudaDeviceSynchronize();
    long long h[512];
    int he = 0;
    cudaMemcpy(h, d, 2 * grid * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaMemcpy(&he, e, 4, cudaMemcpyDeviceToHost);
    double iss = 0, done = 0;
    for (int i = 0; i < grid; ++i) {
        iss += h[2 * i];
        done += h[2 * i + 1];
    }
    iss /= grid;
    done /= grid;
    const double cyc = done / R;
    printf("%-10s N=%3d grid=%3d  issue %6.1f cyc/mma  complete %6.1f cyc/mma  -> %6.0f flop/clk/SM (%s%s)\n", name, N,
           grid, iss / R, cyc, 2.0 * 128 * N * 16 / cyc, cudaGetErrorString(st), he ? " WAIT-TIMEOUT" : "");
    cudaFree(d);
    cudaFree(e);
}

int main() {
    for (int grid : {1, 148}) {
        run<64, false, false>("SS", grid);
        run<128, false, false>("SS", grid);
        run<256, false, false>("SS", grid);
        run<64, true, false>("TS", grid);
        run<128, true, false>("TS", grid);
        run<256, true, false>("TS", grid);
        run<128, false, true>("SS-alt", grid);
        run<128, true, true>("TS-alt", grid);
    }
    return 0;
}
