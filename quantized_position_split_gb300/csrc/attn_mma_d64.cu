// Tensor-core decode attention instances for head_dim 64 (see attn_mma.cuh); the
// causal (verify-batch) instances are in attn_mma_d64_causal.cu, the TQ2 / TQ4 V
// instances in attn_mma_d64_tiers.cu and the TurboQuant-K ones in attn_mma_d64_tqk.cu.
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d64_causal(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d64_tiers(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d64_tqk(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d64(const AttnParams& p, cudaStream_t s) {
  if (is_tq(p.kfmt)) return launch_attn_mma_d64_tqk(p, s);
  if (p.vfmt == QPS_FMT_TQ2 || p.vfmt == QPS_FMT_TQ4) return launch_attn_mma_d64_tiers(p, s);
  return p.causal ? launch_attn_mma_d64_causal(p, s) : mma::launch_mma_d<64, false, 0>(p, s);
}
}  // namespace qps
