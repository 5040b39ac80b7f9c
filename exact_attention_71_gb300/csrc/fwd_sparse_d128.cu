// Instantiation of the fused forward with a block-sparse key mask: head_dim 128, key tile 128, 2 query tile(s) per CTA, bf16 inputs.
#include "attn_launch.cuh"

namespace attn {
using Cfg_sparse_d128 = FwdCfg<128, 128, 2, false, true>;
cudaError_t run_fwd_sparse_d128(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd<Cfg_sparse_d128>(m, p, g, s);
}
FwdGeometry geom_sparse_d128() { return fwd_geometry<Cfg_sparse_d128>(); }
}  // namespace attn
