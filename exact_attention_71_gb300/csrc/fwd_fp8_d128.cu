// Instantiation of the fused forward: head_dim 128, key tile 128, 2 query tile(s) per CTA, e4m3 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_fp8_d128 = FwdCfg<128, 128, 2, true>;
cudaError_t run_fwd_fp8_d128(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_fp8_d128>(m, p, g, s);
}
FwdGeometry geom_fp8_d128() { return fwd_geometry<Cfg_fp8_d128>(); }
}  // namespace attn
