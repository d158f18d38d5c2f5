// LSE combine of normalised partial outputs.
//
// "F5 M7 — Rolling KV: position-windowed KV residency", section "Implementation
// decomposition, refined (S1 -> S2 -> S3)", item S2: O = sum_t O_t exp(lse_t - M) /
// sum_t exp(lse_t - M), M = max_t lse_t, merged in f32.  Here each warp tracks the
// maximum online over its share of the parts (rescaling its running sums when it grows)
// and the warps' states are merged the same way, which gives the same value up to
// rounding.  Parts with lse = -inf weigh nothing.
//
// One CTA per output row; its warps stride over the parts (a row's parts are
// independent, so a step's hundreds of split partials are read in parallel); lane L of
// a warp owns D / 32 consecutive elements, so each part's row is one coalesced read.
#include "internal.h"

namespace qps {
namespace {

constexpr int kCombineWarps = 8;

template <int E>
__global__ void __launch_bounds__(kCombineWarps * 32) lse_combine_kernel(
    const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n_parts, int64_t rows,
    float* __restrict__ o, float* __restrict__ lse) {
  constexpr int D = 32 * E;
  constexpr int U = 4;  // parts in flight per warp
  __shared__ float wm[kCombineWarps], wd[kCombineWarps];
  __shared__ float wacc[kCombineWarps][D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  float m = -INFINITY, den = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int t0 = warp * U; t0 < n_parts; t0 += kCombineWarps * U) {
    float lt[U];
    float v[U][E];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u;
      lt[u] = t < n_parts ? lse_parts[(int64_t)t * rows + row] : -INFINITY;
      if (lt[u] != -INFINITY) {
        const float* src = o_parts + ((int64_t)t * rows + row) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) v[u][e] = src[e];
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) v[u][e] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (lt[u] == -INFINITY) continue;
      if (lt[u] > m) {
        const float cr = __expf(m - lt[u]);  // 0 when m == -inf
        den *= cr;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= cr;
        m = lt[u];
      }
      const float w = __expf(lt[u] - m);
      den += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
    }
  }
  if (lane == 0) {
    wm[warp] = m;
    wd[warp] = den;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) wacc[warp][lane * E + e] = acc[e];
  __syncthreads();
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) mx = fmaxf(mx, wm[w]);
  float dt = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w)
      if (wm[w] != -INFINITY) dt += wd[w] * __expf(wm[w] - mx);
  }
  const bool empty = !(dt > 0.f);
  const float inv = empty ? 0.f : 1.0f / dt;
  for (int dd = threadIdx.x; dd < D; dd += blockDim.x) {
    float s = 0.f;
    if (!empty) {
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w)
        if (wm[w] != -INFINITY) s += wacc[w][dd] * __expf(wm[w] - mx);
    }
    o[row * D + dd] = s * inv;
  }
  if (threadIdx.x == 0) lse[row] = empty ? -INFINITY : mx + __logf(dt);
}

}  // namespace

qps_status launch_combine(const float* o_parts, const float* lse_parts, int n_parts,
                          int64_t rows, int d, float* o, float* lse, cudaStream_t s) {
  if (rows == 0) return QPS_OK;
  if (rows > 0x7fffffffLL) return fail(QPS_ERR_UNSUPPORTED, "lse_combine: too many rows");
  const unsigned grid = (unsigned)rows;
  const int block = kCombineWarps * 32;
  switch (d) {
#define QPS_COMBINE_CASE(E)                                                                 \
  case 32 * E:                                                                              \
    lse_combine_kernel<E><<<grid, block, 0, s>>>(o_parts, lse_parts, n_parts, rows, o, lse); \
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
