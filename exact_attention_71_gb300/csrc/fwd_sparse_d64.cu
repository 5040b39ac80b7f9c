// Instantiation of the fused forward with a block-sparse key mask: head_dim 64, key tile 128, 2 query tile(s) per CTA, bf16 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_sparse_d64 = FwdCfg<64, 128, 2, false, true>;
cudaError_t run_fwd_sparse_d64(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_sparse_d64>(m, p, g, s);
}
FwdGeometry geom_sparse_d64() { return fwd_geometry<Cfg_sparse_d64>(); }
}  // namespace attn
