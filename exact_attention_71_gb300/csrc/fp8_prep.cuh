// FP8 prep: incoherent processing + block quantisation (launcher).
#pragma once

#include <cuda.h>
#include <cstdint>
#include <cuda_runtime.h>

namespace attn {

// Sign c of the +-1 diagonal: bit 63 of splitmix64 output c for state
// `seed` (output c is the mixing function applied to seed + (c + 1) * gamma;
// Steele, Lea and Flood, OOPSLA 2014).
__device__ __forceinline__ float diag_sign(unsigned long long seed, int c) {
    unsigned long long z = seed + static_cast<unsigned long long>(c + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (z >> 63) ? -1.0f : 1.0f;
}

// x / s rounded to nearest for s > 0, from the correctly rounded reciprocal
// and one residual correction (Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. R&D 1990): with
// inv = RN(1/s), q0 = RN(x * inv) and the exact residual x - q0 * s (one FMA),
// q0 + residual * inv rounds to RN(x / s) for the normal-range quotients
// here (|x / s| <= 448).  The sign is copied so that -0 / s stays -0.
__device__ __forceinline__ float div_by_scale(float x, float s, float inv) {
    const float q0 = x * inv;
    const float rem = fmaf(-q0, s, x);
    return copysignf(fmaf(rem, inv, q0), x);
}

// Launch context of the prep: SM count (persistent grid), the bounded-wait
// limit and the device status word.
struct PrepLaunch {
    int num_sms;
    unsigned long long wait_limit;
    int* status;
};

// rope: 0 = none, 1 = half-split pairs (i, i + d/2), 2 = interleaved pairs
// (2i, 2i + 1); rope_cos / rope_sin are binary32 (N, d/2) tables (rope != 0).
// map: x (bf16, (B, N, H, d)) as a 4-D tensor map {d, H, N, B} with a box of
// {d, 1, 128, 1} and no swizzle.
cudaError_t run_fp8_prep(const CUtensorMap& map, void* x8, float* scales, int B, int H, int N, int d, int mode,
                         unsigned long long sign_seed, bool is_v, const float* rope_cos, const float* rope_sin,
                         int rope, const PrepLaunch& L, cudaStream_t stream);

// One tensor of a tensor-core prep launch (e4m3 codes and block scales of a
// bf16 (B, N, H, d) tensor; rotate = 1: multiplied by diag(+-1) x Hadamard).
struct PrepTensor {
    uint8_t* x8;
    float* scales;
    int H;
    int blocks;      // B * H * nblk (0: unused slot)
    int rotate;
};

struct PrepTcParams {
    PrepTensor t[3];
    int N, nblk, total_blocks;
    unsigned long long seed;
    unsigned long long wait_limit;
    int* status;
};

// Block-scaled e4m3 prep of up to three tensors in one launch, the rotation
// as a tensor-core product (d = 64 or 128).  maps[i]: tensor i as a 4-D
// tensor map {d, H, N, B} with a box of {64, 1, 128, 1} and the 128-byte
// swizzle (the attention kernel's tile map); unused slots repeat a valid map.
cudaError_t run_fp8_prep_tc(const CUtensorMap* maps, const PrepTcParams& p, int d, const PrepLaunch& L,
                            cudaStream_t stream);

}  // namespace attn
