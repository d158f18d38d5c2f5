// LSE combine of normalised partial outputs.
//
// "F5 M7 — Rolling KV: position-windowed KV residency", section "Implementation
// decomposition, refined (S1 -> S2 -> S3)", item S2: O = sum_t O_t exp(lse_t - M) /
// sum_t exp(lse_t - M), M = max_t lse_t, merged in f32.  Here each warp tracks the
// maximum online over its share of the parts (rescaling its running sums when it grows)
// and the warps' states are merged the same way, which gives the same value up to
// rounding.  Parts with lse = -inf weigh nothing.
//
// Grid: one CTA per (output row, 32-column slice), so a step's few dozen rows still
// spread over the SMs; its warps (one per U parts, at most kCombineWarps: a combine of
// few parts launches few warps) stride over the parts, U parts in flight per warp (the
// rows' parts are independent, so the loads overlap), and lane L of a warp owns column
// 32 * blockIdx.y + L, so each part's slice is one coalesced 128-byte read.  Every
// slice of a row merges the same lse values in the same order, so all of them agree on
// the row's weights.
#include <algorithm>

#include "internal.h"

namespace qps {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineU = 8;  // parts in flight per warp

__global__ void __launch_bounds__(kCombineWarps * 32) lse_combine_kernel(
    const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n_parts, int64_t rows, int d,
    float* __restrict__ o, float* __restrict__ lse, unsigned int* err) {
  constexpr int U = kCombineU;
  __shared__ float wm[kCombineWarps], wd[kCombineWarps], wacc[kCombineWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;  // warps of this launch (<= kCombineWarps)
  const int64_t row = blockIdx.x;
  const int col = blockIdx.y * 32 + lane;
  float m = -INFINITY, den = 0.f, acc = 0.f;
  for (int t0 = warp * U; t0 < n_parts; t0 += nw * U) {
    float lt[U], v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u;
      lt[u] = t < n_parts ? lse_parts[(int64_t)t * rows + row] : -INFINITY;
      v[u] = lt[u] != -INFINITY ? o_parts[((int64_t)t * rows + row) * d + col] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (lt[u] == -INFINITY) continue;
      if (lt[u] > m) {
        const float cr = __expf(m - lt[u]);  // 0 when m == -inf
        den *= cr;
        acc *= cr;
        m = lt[u];
      }
      const float w = __expf(lt[u] - m);
      den += w;
      acc = fmaf(w, v[u], acc);
    }
  }
  if (lane == 0) {
    wm[warp] = m;
    wd[warp] = den;
  }
  wacc[warp][lane] = acc;
  __syncthreads();
  if (warp != 0) return;
  float mx = -INFINITY;
  for (int w = 0; w < nw; ++w) mx = fmaxf(mx, wm[w]);
  float dt = 0.f, s = 0.f;
  if (mx != -INFINITY) {
    for (int w = 0; w < nw; ++w) {
      if (wm[w] == -INFINITY) continue;
      const float f = __expf(wm[w] - mx);
      dt += wd[w] * f;
      s += wacc[w][lane] * f;
    }
  }
  const bool empty = !(dt > 0.f);
  if (!in_bounds(row < rows && col < d, err)) return;
  o[row * d + col] = empty ? 0.f : s / dt;
  if (blockIdx.y == 0 && lane == 0) lse[row] = empty ? -INFINITY : mx + __logf(dt);
}

}  // namespace

qps_status launch_combine(const float* o_parts, const float* lse_parts, int n_parts,
                          int64_t rows, int d, float* o, float* lse, cudaStream_t s, unsigned int* err) {
  if (rows == 0) return QPS_OK;
  if (rows > 0x7fffffffLL) return fail(QPS_ERR_UNSUPPORTED, "lse_combine: too many rows");
  if (d < 32 || d > 1024 || (d & (d - 1)))
    return fail(QPS_ERR_UNSUPPORTED, "lse_combine: head_dim must be 32, 64, 128, 256, 512 or 1024");
  const dim3 grid((unsigned)rows, (unsigned)(d / 32));
  const int warps = std::min(kCombineWarps, std::max(1, (n_parts + kCombineU - 1) / kCombineU));
  lse_combine_kernel<<<grid, warps * 32, 0, s>>>(o_parts, lse_parts, n_parts, rows, d, o, lse, err);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

}  // namespace qps
