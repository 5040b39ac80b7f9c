// FP8 prep: incoherent processing + block quantisation (launcher).
#pragma once

#include <cuda_runtime.h>

namespace attn {

// rope: 0 = none, 1 = half-split pairs (i, i + d/2), 2 = interleaved pairs
// (2i, 2i + 1); rope_cos / rope_sin are binary32 (N, d/2) tables (rope != 0).
cudaError_t run_fp8_prep(const void* x, void* x8, float* scales, int B, int H, int N, int d, int mode,
                         unsigned long long sign_seed, bool is_v, const float* rope_cos, const float* rope_sin,
                         int rope, cudaStream_t stream);

}  // namespace attn
