// Tensor-core decode attention instances for head_dim 64 with the causal limit of a
// verify batch (see attn_mma.cuh).
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d64_causal(const AttnParams& p, cudaStream_t s) {
  return mma::launch_mma_d<64, true, 0>(p, s);
}
}  // namespace qps
