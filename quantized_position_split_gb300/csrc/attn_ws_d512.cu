// The warp-specialized decode attention instance: head_dim 512, q8_0 K, TQ3 V (see
// attn_ws.cuh).
#include "attn_ws.cuh"

namespace qps {
bool attn_ws_takes(const AttnParams& p) { return ws::ws_takes(p); }
qps_status launch_attn_ws_d512(const AttnParams& p, cudaStream_t s) {
  return ws::launch_ws_t<512, QPS_FMT_Q8_0, QPS_FMT_TQ3>(p, s);
}
}  // namespace qps
