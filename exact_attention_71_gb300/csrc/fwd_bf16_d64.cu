// Instantiation of the fused forward: head_dim 64, key tile 128, 2 query tile(s) per CTA, bf16 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_bf16_d64 = FwdCfg<64, 128, 2, false>;
cudaError_t run_fwd_bf16_d64(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_bf16_d64>(m, p, g, s);
}
FwdGeometry geom_bf16_d64() { return fwd_geometry<Cfg_bf16_d64>(); }
}  // namespace attn
