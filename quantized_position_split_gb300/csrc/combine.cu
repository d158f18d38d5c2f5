// LSE combine of normalised partial outputs.
//
// "F5 M7 — Rolling KV: position-windowed KV residency", section "Implementation
// decomposition, refined (S1 -> S2 -> S3)", item S2: O = sum_t O_t exp(lse_t - M) /
// sum_t exp(lse_t - M), M = max_t lse_t, merged in f32.  Here the maximum is tracked
// online in one pass over the parts (rescaling the running sums when it grows), which
// gives the same value up to rounding.  Parts with lse = -inf weigh nothing.
//
// One warp per output row; lane L owns D / 32 consecutive elements, so each part's row
// is one coalesced read.
#include "internal.h"

namespace qps {
namespace {

template <int E>
__global__ void __launch_bounds__(256) lse_combine_kernel(const float* __restrict__ o_parts,
                                                          const float* __restrict__ lse_parts,
                                                          int n_parts, int64_t rows,
                                                          float* __restrict__ o,
                                                          float* __restrict__ lse) {
  constexpr int D = 32 * E;
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  float m = -INFINITY, den = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int t = 0; t < n_parts; ++t) {
    const float lt = lse_parts[(int64_t)t * rows + row];
    if (lt == -INFINITY) continue;
    const float* src = o_parts + ((int64_t)t * rows + row) * D + lane * E;
    if (lt > m) {
      const float c = __expf(m - lt);  // 0 when m == -inf
      den *= c;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= c;
      m = lt;
    }
    const float w = __expf(lt - m);
    den += w;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, src[e], acc[e]);
  }
  const bool empty = !(den > 0.f);
  const float inv = empty ? 0.f : 1.0f / den;
#pragma unroll
  for (int e = 0; e < E; ++e) o[row * D + lane * E + e] = acc[e] * inv;
  if (lane == 0) lse[row] = empty ? -INFINITY : m + __logf(den);
}

}  // namespace

qps_status launch_combine(const float* o_parts, const float* lse_parts, int n_parts,
                          int64_t rows, int d, float* o, float* lse, cudaStream_t s) {
  if (rows == 0) return QPS_OK;
  const int block = 256;
  const int64_t grid = (rows * 32 + block - 1) / block;
  switch (d) {
#define QPS_COMBINE_CASE(E)                                                                  \
  case 32 * E:                                                                               \
    lse_combine_kernel<E><<<(unsigned)grid, block, 0, s>>>(o_parts, lse_parts, n_parts, rows, \
                                                           o, lse);                          \
    break;
    QPS_COMBINE_CASE(1)
    QPS_COMBINE_CASE(2)
    QPS_COMBINE_CASE(4)
    QPS_COMBINE_CASE(8)
    QPS_COMBINE_CASE(16)
    QPS_COMBINE_CASE(32)
#undef QPS_COMBINE_CASE
    default:
      return fail(QPS_ERR_UNSUPPORTED, "lse_combine: head_dim must be 32, 64, 128, 256, 512 or 1024");
  }
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

}  // namespace qps
