// Instantiation of the fused forward: head_dim 256, key tile 128, 1 query tile per CTA, e4m3 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_fp8_d256 = FwdCfg<256, 128, 1, true>;
cudaError_t run_fwd_fp8_d256(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_fp8_d256>(m, p, g, s);
}
FwdGeometry geom_fp8_d256() { return fwd_geometry<Cfg_fp8_d256>(); }
}  // namespace attn
