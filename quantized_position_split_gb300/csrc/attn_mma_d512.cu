// Tensor-core decode attention instances for head_dim 512 (see attn_mma.cuh); the
// causal (verify-batch) instances are in attn_mma_d512_causal.cu, the TQ2 / TQ4 V
// instances in attn_mma_d512_tiers.cu, the TurboQuant-K ones in attn_mma_d512_tqk.cu,
// and single-token q8_0-K / TQ3-V decode runs the warp-specialized kernel of
// attn_ws_d512.cu.
#include "attn_mma.cuh"

namespace qps {
qps_status launch_attn_mma_d512_causal(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d512_tiers(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d512_tqk(const AttnParams& p, cudaStream_t s);
bool attn_ws_takes(const AttnParams& p);
qps_status launch_attn_ws_d512(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d512(const AttnParams& p, cudaStream_t s) {
  if (attn_ws_takes(p)) return launch_attn_ws_d512(p, s);  // the warp-specialized q8_0-K / TQ3-V kernel
  if (is_tq(p.kfmt)) return launch_attn_mma_d512_tqk(p, s);
  if (p.vfmt == QPS_FMT_TQ2 || p.vfmt == QPS_FMT_TQ4) return launch_attn_mma_d512_tiers(p, s);
  return p.causal ? launch_attn_mma_d512_causal(p, s) : mma::launch_mma_d<512, false, 0>(p, s);
}
}  // namespace qps
