// Instantiation of the fused forward with a block-sparse key mask: head_dim 256, key tile 64, 1 query tile(s) per CTA, bf16 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_sparse_d256 = FwdCfg<256, 64, 1, false, true>;
cudaError_t run_fwd_sparse_d256(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_sparse_d256>(m, p, g, s);
}
FwdGeometry geom_sparse_d256() { return fwd_geometry<Cfg_sparse_d256>(); }
}  // namespace attn
