// Tensor-core decode attention instances for head_dim 256 (see attn_mma.cuh); the
// causal (verify-batch) instances are in attn_mma_d256_causal.cu.
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d256_causal(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d256(const AttnParams& p, cudaStream_t s) {
  return p.causal ? launch_attn_mma_d256_causal(p, s) : mma::launch_mma_d<256, false>(p, s);
}
}  // namespace qps
