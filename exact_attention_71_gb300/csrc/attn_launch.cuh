// Host-side launch of one instantiation of the fused forward kernel.
#pragma once

#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

// o: the bf16 output as {d, H, N, B} with a box of {64, 1, 32, 1} and the
// 128-byte swizzle (one softmax warp's rows, one column box).
struct FwdMaps {
    CUtensorMap q, k, v, o;
};

// Tile geometry an instantiation needs from the host (tensor-map boxes).
struct FwdGeometry {
    int d, bn, nq, elem_bytes, threads, smem_bytes, stages, swizzle;
};

template <class Cfg>
FwdGeometry fwd_geometry() {
    return FwdGeometry{Cfg::D, Cfg::BN, Cfg::NQ, Cfg::ES, Cfg::THREADS, Cfg::SMEM_BYTES, Cfg::NSTAGE, Cfg::SW};
}

template <class Cfg>
cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, int max_ctas, cudaStream_t stream) {
    auto kernel = attn_fwd_kernel<Cfg>;
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
    kernel<<<dim3(static_cast<unsigned>(grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream>>>(maps.q, maps.k,
                                                                                              maps.v, maps.o, p);
    return cudaGetLastError();
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
