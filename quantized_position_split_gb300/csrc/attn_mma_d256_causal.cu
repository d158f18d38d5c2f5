// Tensor-core decode attention instances for head_dim 256 with the causal limit of a
// verify batch (see attn_mma.cuh).
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d256_causal(const AttnParams& p, cudaStream_t s) {
  return mma::launch_mma_d<256, true, 0>(p, s);
}
}  // namespace qps
