// Dense tensor-core rate of one SM, measured with this library's own
// tcgen05 MMA wrappers: every CTA (one per SM) issues a long straight-line
// stream of 128 x 256 MMAs (both operands in shared memory, fp32 accumulate)
// and times it with clock64 from the first issue to the commit of the last.
// FLOP per clock per SM = 2 * 128 * 256 * K * count / cycles.  bf16
// (kind::f16, K = 16) and e4m3 (kind::f8f6f4, K = 32).
//
// Standalone measurement program, built and run by `bench.py --spec-peak`
// (not part of the attention library):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I. -o mma_peak mma_peak.cu   (from the repository root)
//   ./mma_peak      -> one JSON line
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <vector>

#include "exact_attention_71_gb300/csrc/sm103_ptx.cuh"

using namespace attn;

template <bool FP8>
__global__ void __launch_bounds__(128, 1) mma_stream(int outer, unsigned long long* cycles) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm) + 1023) & ~uintptr_t(1023));
    // Finite operands (the rate does not depend on the values).
    for (int i = threadIdx.x; i < 96 * 1024 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(base)[i] = make_uint4(0x3c003c00u, 0x3c003c00u, 0x38383838u, 0x38383838u);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(&tbase, 256);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    constexpr uint32_t idesc = make_idesc(FP8 ? 0u : 1u, 128, 256, 0);
    if (threadIdx.x < 32) {
        const uint64_t ad = sdesc_sw128(smem_u32(base), 16, 1024);
        const uint64_t bd = sdesc_sw128(smem_u32(base + 32768), 16, 1024);
        const long long t0 = clock64();
        for (int o = 0; o < outer; ++o) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint64_t k = (j & 3) * 2;
                if (elect_one()) {
                    if (FP8) mma_f8_ss(tm, ad + k, bd + k, idesc, 1);
                    else mma_f16_ss(tm, ad + k, bd + k, idesc, 1);
                }
                __syncwarp();
            }
        }
        if (elect_one()) {
            mma_commit(&bar);
            const long long tw = clock64();
            bool done = false;
            while (!(done = mbar_try_wait(&bar, 0)) && clock64() - tw < 4000000000ll) {
            }
            cycles[blockIdx.x] = done ? static_cast<unsigned long long>(clock64() - t0) : 0ull;
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tm, 256);
    }
}

template <bool FP8>
double flop_per_clk_per_sm(int sms, unsigned long long* d) {
    // 120 KB of shared memory: one CTA per SM, so no two streams share a tensor core.
    const int smem = 120 * 1024, outer = 256, count = outer * 16;
    cudaFuncSetAttribute(mma_stream<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    mma_stream<FP8><<<sms, 128, smem>>>(outer, d);
    if (cudaDeviceSynchronize() != cudaSuccess) return -1.0;
    std::vector<unsigned long long> h(sms);
    cudaMemcpy(h.data(), d, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
    double worst = 0.0;
    for (auto c : h) {
        if (c == 0) return -1.0;
        worst = c > worst ? static_cast<double>(c) : worst;
    }
    const double k = FP8 ? 32.0 : 16.0;
    return 2.0 * 128.0 * 256.0 * k * count / worst;
}

int main() {
    int dev = 0, sms = 0, clock_khz = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev);
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, sizeof(unsigned long long) * sms) != cudaSuccess) return 1;
    const double bf16 = flop_per_clk_per_sm<false>(sms, d);
    const double fp8 = flop_per_clk_per_sm<true>(sms, d);
    cudaFree(d);
    if (bf16 <= 0 || fp8 <= 0) {
        std::printf("{\"error\": \"MMA stream did not complete\"}\n");
        return 1;
    }
    std::printf("{\"sms\": %d, \"max_sm_mhz\": %.0f, \"bf16_flop_per_clk_per_sm\": %.1f, "
                "\"e4m3_flop_per_clk_per_sm\": %.1f}\n",
                sms, clock_khz / 1000.0, bf16, fp8);
    return 0;
}
