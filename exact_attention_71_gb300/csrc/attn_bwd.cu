// Attention backward, host side and the two memory-bound kernels around the
// fused one:
//   bwd_prep_kernel     D_i = dO_i . O_i and LSE_i * log2(e) per query row
//                       (pad rows: D = 0, LSE = +inf, so they contribute
//                       nothing), and zeroes the float32 dQ accumulator;
//   attn_bwd_kernel     dK, dV (stored) and dQ (added into the accumulator);
//   bwd_dq_kernel       dQ = bf16(scale * accumulator).
// FlashAttention-3 deep-reading report §3.4 (the backward recomputes the
// softmax from the forward's statistics, as FA2 does).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_bwd.cuh"
#include "attn_bwd_kernel.cuh"

namespace attn {
namespace {

template <int E> struct Bf16Vec;
template <> struct Bf16Vec<2> { using T = uint32_t; };
template <> struct Bf16Vec<4> { using T = uint2; };

// One warp per row of (B, H, N_pad); lane l holds elements [E l, E l + E), E = D / 32.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ lse2,
                                                       float* __restrict__ dvec, float* __restrict__ dq_acc, int B,
                                                       int H, int N, int N_pad) {
    constexpr int E = D / 32;
    using V = typename Bf16Vec<E>::T;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= static_cast<long long>(B) * H * N_pad) return;
    const int n = static_cast<int>(row % N_pad);
    const long long bh = row / N_pad;
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    if constexpr (E == 4) {
        reinterpret_cast<float4*>(dq_acc + row * D)[lane] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    } else {
        reinterpret_cast<float2*>(dq_acc + row * D)[lane] = make_float2(0.0f, 0.0f);
    }
    if (n >= N) {
        if (lane == 0) {
            dvec[row] = 0.0f;
            lse2[row] = __int_as_float(0x7f800000);   // +inf: P = 0 for pad rows
        }
        return;
    }
    const size_t off = ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E;
    const V ov = __ldg(reinterpret_cast<const V*>(o + off));
    const V dv = __ldg(reinterpret_cast<const V*>(dout + off));
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        const float2 a = __bfloat1622float2(o2[k]);
        const float2 c = __bfloat1622float2(d2[k]);
        acc = fmaf(a.x, c.x, acc);
        acc = fmaf(a.y, c.y, acc);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) {
        dvec[row] = acc;
        lse2[row] = lse[bh * N + n] * 1.4426950408889634f;
    }
}

// One warp per query row: dq (B, N, H, D) bf16 = scale * dq_acc (B, H, N_pad, D).
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                                                     int B, int H, int N, int N_pad, float scale) {
    constexpr int E = D / 32;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= static_cast<long long>(B) * N * H) return;
    const int h = static_cast<int>(row % H);
    const long long bn = row / H;
    const int n = static_cast<int>(bn % N), b = static_cast<int>(bn / N);
    const float* src = dq_acc + ((static_cast<size_t>(b) * H + h) * N_pad + n) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        const float2 a = __ldg(reinterpret_cast<const float2*>(src + e));
        const __nv_bfloat162 v = __floats2bfloat162_rn(a.x * scale, a.y * scale);
        *reinterpret_cast<__nv_bfloat162*>(dq + row * D + lane * E + e) = v;
    }
}

}  // namespace

BwdWorkspace bwd_workspace(int B, int H, int N, int d) {
    BwdWorkspace ws{};
    const long long n_pad = (static_cast<long long>(N) + 127) / 128 * 128;
    auto up = [](long long x) { return (x + 255) / 256 * 256; };
    const long long rows = static_cast<long long>(B) * H * n_pad;
    ws.n_pad = static_cast<int>(n_pad);
    ws.off_lse2 = 0;
    ws.off_dvec = up(rows * 4);
    ws.off_dq = ws.off_dvec + up(rows * 4);
    ws.bytes = ws.off_dq + up(rows * d * 4);
    return ws;
}

template <int D>
cudaError_t run_bwd_impl(const BwdMaps& maps, const BwdParams& p, const void* o, const void* dout, const float* lse,
                         void* dq, cudaStream_t stream) {
    using Cfg = BwdCfg<D>;
    const long long rows_pad = static_cast<long long>(p.B) * p.H * p.N_pad;
    const long long prep_blocks = (rows_pad + 7) / 8;
    const long long dq_blocks = (static_cast<long long>(p.B) * p.N * p.H + 7) / 8;
    const long long ctas = static_cast<long long>(p.n_kblocks) * p.B * p.H_kv;
    if (prep_blocks >= (1ll << 31) || dq_blocks >= (1ll << 31) || ctas >= (1ll << 31)) return cudaErrorInvalidValue;
    bwd_prep_kernel<D><<<static_cast<unsigned>(prep_blocks), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse,
        const_cast<float*>(p.lse2), const_cast<float*>(p.dvec), p.dq_acc, p.B, p.H, p.N, p.N_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kernel = attn_bwd_kernel<Cfg>;
    if constexpr (Cfg::REG_SPLIT) {
        // The register split (setmaxnreg) assumes every thread is launched
        // with exactly LAUNCH_REGS registers; a different count could make the
        // increase wait forever, so such a build is refused.
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kernel);
        if (e != cudaSuccess) return e;
        if (attr.numRegs != Cfg::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kernel<<<static_cast<unsigned>(ctas), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(maps.q, maps.k, maps.v, maps.dout,
                                                                                   p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq_kernel<D><<<static_cast<unsigned>(dq_blocks), 256, 0, stream>>>(p.dq_acc, static_cast<__nv_bfloat16*>(dq),
                                                                           p.B, p.H, p.N, p.N_pad, p.scale);
    return cudaGetLastError();
}

cudaError_t run_bwd(int d, const BwdMaps& maps, const BwdParams& p, const void* o, const void* dout, const float* lse,
                    void* dq, cudaStream_t stream) {
    switch (d) {
        case 64: return run_bwd_impl<64>(maps, p, o, dout, lse, dq, stream);
        case 128: return run_bwd_impl<128>(maps, p, o, dout, lse, dq, stream);
        default: return cudaErrorInvalidValue;
    }
}

int bwd_query_rows(int d) { return d == 128 ? BwdCfg<128>::BM : BwdCfg<64>::BM; }

}  // namespace attn
