// Attention backward: workspace layout and the host entry of the three
// launches (prep, fused backward, dQ conversion).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct BwdParams;

struct BwdMaps {
    CUtensorMap q, k, v, dout;
};

// Caller-provided workspace: LSE * log2(e) and D (float32, (B, H, N_pad)
// each), then the float32 dQ accumulator (B, H, N_pad, d); N_pad = N rounded
// up to 128.  Offsets are 256-byte aligned.
struct BwdWorkspace {
    long long off_lse2, off_dvec, off_dq, bytes;
    int n_pad;
};

BwdWorkspace bwd_workspace(int B, int H, int N, int d);

// d = 64 or 128.
cudaError_t run_bwd(int d, const BwdMaps& maps, const BwdParams& p, const void* o, const void* dout, const float* lse,
                    void* dq, cudaStream_t stream);

// Query rows per step of the fused kernel (the Q / dO tensor-map box height).
int bwd_query_rows(int d);

}  // namespace attn
