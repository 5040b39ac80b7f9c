// Instantiation of the fused forward: head_dim 256, key tile 64, 1 query tile(s) per CTA, bf16 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_bf16_d256 = FwdCfg<256, 64, 1, false>;
cudaError_t run_fwd_bf16_d256(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_bf16_d256>(m, p, g, s);
}
FwdGeometry geom_bf16_d256() { return fwd_geometry<Cfg_bf16_d256>(); }
}  // namespace attn
