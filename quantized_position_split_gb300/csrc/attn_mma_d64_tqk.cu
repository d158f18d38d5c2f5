// Tensor-core decode attention instances for head_dim 64 with a TurboQuant K and V of
// the same tier (TQ2, TQ3 or TQ4), single-token and causal (see attn_mma.cuh).
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d64_tqk(const AttnParams& p, cudaStream_t s) {
  return p.causal ? mma::launch_mma_d<64, true, 2>(p, s) : mma::launch_mma_d<64, false, 2>(p, s);
}
}  // namespace qps
