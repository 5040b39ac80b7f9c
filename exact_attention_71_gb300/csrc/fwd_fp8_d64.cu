// Instantiation of the fused forward: head_dim 64, key tile 128, 2 query tiles per CTA, e4m3 inputs
// (64-byte rows: 64-byte swizzle).
#include "attn_launch.cuh"

namespace attn {
using Cfg_fp8_d64 = FwdCfg<64, 128, 2, true>;
cudaError_t run_fwd_fp8_d64(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_fp8_d64>(m, p, g, s);
}
FwdGeometry geom_fp8_d64() { return fwd_geometry<Cfg_fp8_d64>(); }
}  // namespace attn
