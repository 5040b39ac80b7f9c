// Host-side launch of one instantiation of the fused forward kernel.
#pragma once

#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

// o: the bf16 output as {d, H, N, B} with a box of {64, 1, 32, 1} and the
// 128-byte swizzle (one softmax warp's rows, one column box).
struct FwdMaps {
    CUtensorMap q, k, v, o;
    const ItemOrder* order = nullptr;   // causal work order (nullptr or n = 0: the closed form)
};

// The causal work order of attn_fwd_kernel for nmb query blocks per head, BH
// heads and a grid of G CTAs; returns false (order->n = 0) when nmb * BH
// exceeds kOrderMax.
bool causal_item_order(int nmb, int BH, int G, ItemOrder* order);

// Tile geometry an instantiation needs from the host (tensor-map boxes).
struct FwdGeometry {
    int d, bn, nq, elem_bytes, threads, smem_bytes, stages, swizzle;
};

template <class Cfg>
FwdGeometry fwd_geometry() {
    return FwdGeometry{Cfg::D, Cfg::BN, Cfg::NQ, Cfg::ES, Cfg::THREADS, Cfg::SMEM_BYTES, Cfg::NSTAGE, Cfg::SW};
}

template <class Cfg, bool ORDERED, class Order>
cudaError_t launch_fwd_kernel(const FwdMaps& maps, const FwdParams& p, const Order& order, int max_ctas,
                              cudaStream_t stream) {
    auto kernel = attn_fwd_kernel<Cfg, ORDERED>;
    // The register split inside the kernel (setmaxnreg) assumes every thread
    // is launched with exactly LAUNCH_REGS registers; a different count could
    // make the increase wait forever, so such a build is refused.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != Cfg::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    // The attribute is per function and per device; setting it is cheap and
    // idempotent, so it is set on every launch (devices may differ per call).
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // Persistent grid: at most one CTA per SM (shared memory allows one), each
    // walking the items blockIdx.x, blockIdx.x + gridDim.x, ...
    const long long units = static_cast<long long>(p.n_mblocks) * p.B * p.H;
    const long long grid = units < max_ctas ? units : max_ctas;
    kernel<<<dim3(static_cast<unsigned>(grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream>>>(
        maps.q, maps.k, maps.v, maps.o, p, order);
    return cudaGetLastError();
}

template <class Cfg>
cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, int max_ctas, cudaStream_t stream) {
    // Causal launches of the dense d = 128 kernels with a host-built order
    // take the ordered instantiation; everything else the plain one.
    if constexpr (Cfg::D == 128 && !Cfg::SPARSE) {
        if (maps.order != nullptr && maps.order->n > 0)
            return launch_fwd_kernel<Cfg, true>(maps, p, *maps.order, max_ctas, stream);
    }
    return launch_fwd_kernel<Cfg, false>(maps, p, NoOrder{0}, max_ctas, stream);
}

// Per-instantiation entry points (one translation unit each).
cudaError_t run_fwd_bf16_d64(const FwdMaps&, const FwdParams&, int, cudaStream_t);
cudaError_t run_fwd_bf16_d128(const FwdMaps&, const FwdParams&, int, cudaStream_t);
cudaError_t run_fwd_bf16_d256(const FwdMaps&, const FwdParams&, int, cudaStream_t);
cudaError_t run_fwd_fp8_d128(const FwdMaps&, const FwdParams&, int, cudaStream_t);
FwdGeometry geom_bf16_d64();
FwdGeometry geom_bf16_d128();
FwdGeometry geom_bf16_d256();
FwdGeometry geom_fp8_d128();
cudaError_t run_fwd_fp8_d256(const FwdMaps&, const FwdParams&, int, cudaStream_t);
FwdGeometry geom_fp8_d256();
cudaError_t run_fwd_fp8_d64(const FwdMaps&, const FwdParams&, int, cudaStream_t);
FwdGeometry geom_fp8_d64();
cudaError_t run_fwd_sparse_d64(const FwdMaps&, const FwdParams&, int, cudaStream_t);
cudaError_t run_fwd_sparse_d128(const FwdMaps&, const FwdParams&, int, cudaStream_t);
cudaError_t run_fwd_sparse_d256(const FwdMaps&, const FwdParams&, int, cudaStream_t);
FwdGeometry geom_sparse_d64();
FwdGeometry geom_sparse_d128();
FwdGeometry geom_sparse_d256();

}  // namespace attn
