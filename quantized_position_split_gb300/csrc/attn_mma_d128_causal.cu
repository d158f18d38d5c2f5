// Tensor-core decode attention instances for head_dim 128 with the causal limit of a
// verify batch (see attn_mma.cuh).
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d128_causal(const AttnParams& p, cudaStream_t s) {
  return mma::launch_mma_d<128, true, 0>(p, s);
}
}  // namespace qps
