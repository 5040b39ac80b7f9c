// Instantiation of the fused forward with a block-sparse key mask: head_dim
// 256, key tile 64, one query tile per CTA with three S buffers in tensor
// memory (attn_fwd_la_kernel.cuh), bf16 inputs.
#include "attn_fwd_la_kernel.cuh"
#include "attn_launch.cuh"

namespace attn {
using Cfg_sparse_d256 = LaCfg<256, 64, false, 3, true>;
cudaError_t run_fwd_sparse_d256(const FwdMaps& m, const FwdParams& p, int g, cudaStream_t s) {
    return launch_fwd_la<Cfg_sparse_d256>(m.q, m.k, m.v, p, g, s);
}
FwdGeometry geom_sparse_d256() { return fwd_geometry<Cfg_sparse_d256>(); }
}  // namespace attn
