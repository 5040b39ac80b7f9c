// FP8 prep: incoherent processing + block quantisation (launcher).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

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

}  // namespace attn
