// Tensor-core decode attention instances for head_dim 256 with a TQ2 or TQ4 V (the 2-
// and 4-bit TurboQuant tiers), single-token and causal (see attn_mma.cuh).
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d256_tiers(const AttnParams& p, cudaStream_t s) {
  return p.causal ? mma::launch_mma_d<256, true, 1>(p, s) : mma::launch_mma_d<256, false, 1>(p, s);
}
}  // namespace qps
