// Instantiation of the fused forward: head_dim 256, key tile 128, one query
// tile per CTA with two S buffers in tensor memory (attn_fwd_la_kernel.cuh),
// e4m3 inputs.
#include "attn_fwd_la_kernel.cuh"
#include "attn_launch.cuh"

namespace attn {
using Cfg_fp8_d256 = LaCfg<256, 128, true, 2>;
cudaError_t run_fwd_fp8_d256(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd_la<Cfg_fp8_d256>(m.q, m.k, m.v, p, g, s);
}
FwdGeometry geom_fp8_d256() { return fwd_geometry<Cfg_fp8_d256>(); }
}  // namespace attn
