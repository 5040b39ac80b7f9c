// FP8 prep: incoherent processing + block quantisation (launcher).
#pragma once

#include <cuda_runtime.h>

namespace attn {

cudaError_t run_fp8_prep(const void* x, void* x8, float* scales, int B, int H, int N, int d, int mode,
                         unsigned long long sign_seed, bool is_v, cudaStream_t stream);

}  // namespace attn
