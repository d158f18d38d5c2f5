// KV encoders: q8_0 and the 2-, 3- and 4-bit TurboQuant-MSE tiers (TQ2 / TQ3 / TQ4).
//
// q8_0 follows "F5 M6 — PolyKV (shared compressed KV pool)", section "What PolyKV is
// (reference)" (keys at int8), with 32-value blocks and an fp16 absmax/127 scale.
// The TurboQuant tiers follow the same page, sections "What PolyKV is (reference)",
// "S2 — TurboQuant tier family" and "Phase-0 fork recon": L2 norm, seeded sign diagonal,
// Walsh-Hadamard rotation over head_dim, Lloyd-Max levels of 2^bits cells.  TQ3 stores a
// 2-bit magnitude plane, a 1-bit sign plane and an fp16 norm; TQ2 and TQ4 store one
// sign-magnitude field of 2 or 4 bits per element and an fp16 norm.
//
// The encoders are bit-exact contracts: every floating-point step is an explicitly
// rounded IEEE float32 operation (__fmul_rn / __fadd_rn / __fdiv_rn / __fsqrt_rn) in a
// fixed order, so that no contraction into FMA can change a code.
#include <cmath>

#include "internal.h"

namespace qps {
namespace {

// One thread handles 8 consecutive values (16 bytes); 4 neighbouring lanes form one
// 32-value block and share its absmax through two xor-shuffles.
__global__ void __launch_bounds__(256) quant_q8_0_kernel(const __half* __restrict__ x, int64_t rows,
                                                         int d, int64_t stride,
                                                         int8_t* __restrict__ codes,
                                                         __half* __restrict__ scales) {
  const int per_row = d / 8;
  const int64_t total = rows * per_row;
  const int64_t total_padded = (total + 31) & ~int64_t(31);
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_padded;
       idx += step) {
    const bool active = idx < total;
    const int64_t row = active ? idx / per_row : 0;
    const int c8 = active ? (int)(idx % per_row) : 0;
    float v[8];
    float amax = 0.f;
    if (active) {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + row * stride + c8 * 8);
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h2[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!active) continue;
    const float d32 = __fdiv_rn(amax, 127.0f);
    const __half d16 = __float2half_rn(d32);
    const float dd = __half2float(d16);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int q = 0;
      if (dd != 0.f) {
        float r = roundf(__fdiv_rn(v[i], dd));
        r = fminf(fmaxf(r, -127.f), 127.f);
        q = (int)r;
      }
      packed[i / 4] |= (uint32_t)(q & 0xff) << (8 * (i % 4));
    }
    *reinterpret_cast<uint2*>(codes + row * d + c8 * 8) = make_uint2(packed[0], packed[1]);
    if ((c8 & 3) == 0) scales[row * (d / 32) + c8 / 4] = d16;
  }
}

struct TqConsts {
  uint32_t signs[kMaxSignWords];   // s1
  uint32_t signs2[kMaxSignWords];  // s2 (all 0: none)
  float thresholds[15];
  float kappa;  // sqrtf(D / G), correctly rounded
  int hreg;     // register FWHT stages run for H < hreg (= G / 32)
};

// One warp per row.  Lane L holds elements L + 32 e, e < D / 32, so the FWHT stages
// h < 32 are lane shuffles and the stages 32 <= h < G stay inside a lane's registers
// (stage h = 32 H pairs registers e and e + H).
// BITS = 3: plane0 = magnitudes (2 bits), plane1 = signs (1 bit); BITS = 2 / 4: plane0 =
// (sign << (BITS - 1)) | magnitude fields, plane1 unused.
template <int D, int BITS>
__global__ void __launch_bounds__(256) quant_tq_kernel(const __half* __restrict__ x, int64_t rows,
                                                       int64_t stride, TqConsts c,
                                                       uint8_t* __restrict__ plane0,
                                                       uint8_t* __restrict__ plane1,
                                                       __half* __restrict__ norms) {
  constexpr int E = D / 32;
  constexpr int L = 1 << BITS, HALF = L / 2;
  constexpr int RB0 = D * (BITS == 4 ? 4 : 2) / 8;  // plane0 bytes per row
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = warp; row < rows; row += nwarps) {
    const __half* xr = x + row * stride;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = __half2float(xr[lane + 32 * e]);

    // sum of squares: squares, then the halving fold t[i] += t[i + h], h = D/2 .. 1
    float t[E];
#pragma unroll
    for (int e = 0; e < E; ++e) t[e] = __fmul_rn(v[e], v[e]);
#pragma unroll
    for (int hh = E / 2; hh >= 1; hh /= 2) {
#pragma unroll
      for (int e = 0; e < hh; ++e) t[e] = __fadd_rn(t[e], t[e + hh]);
    }
    float nsq = t[0];
#pragma unroll
    for (int h = 16; h >= 1; h /= 2) nsq = __fadd_rn(nsq, __shfl_xor_sync(0xffffffffu, nsq, h));
    const float n = __fsqrt_rn(nsq);

    // u = FWHT(s .* x): stages h = 1 .. 16 across lanes, then h = 32 .. D/2 in registers
    float u[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      // element lane + 32 e: its sign bit is bit `lane` of word e
      u[e] = ((c.signs[e] >> lane) & 1u) ? -v[e] : v[e];
    }
#pragma unroll
    for (int h = 1; h < 32; h *= 2) {
      const bool upper = (lane & h) != 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, u[e], h);
        u[e] = upper ? __fsub_rn(other, u[e]) : __fadd_rn(u[e], other);
      }
    }
#pragma unroll
    for (int H = 1; H < E; H *= 2) {
      if (H >= c.hreg) break;  // the block width ends the transform
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & H) == 0) {
          const float a = u[e], b = u[e + H];
          u[e] = __fadd_rn(a, b);
          u[e + H] = __fsub_rn(a, b);
        }
      }
    }
    // the second sign vector and the block scale (kappa = 1 for G = D: exact)
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float v2 = ((c.signs2[e] >> lane) & 1u) ? -u[e] : u[e];
      u[e] = __fmul_rn(v2, c.kappa);
    }

    // level index k (a zero row takes k = HALF - 1: sign 0, magnitude 0), then its
    // sign and magnitude
#pragma unroll
    for (int e = 0; e < E; ++e) {
      int k = HALF - 1;
      if (n != 0.f) {
        const float z = __fdiv_rn(u[e], n);
        k = 0;
#pragma unroll
        for (int m = 0; m < L - 1; ++m) k += (z >= c.thresholds[m]) ? 1 : 0;
      }
      const bool sgn = k >= HALF;
      const uint32_t mag = sgn ? (uint32_t)(k - HALF) : (uint32_t)(HALF - 1 - k);
      uint8_t* r0 = plane0 + row * RB0;
      if constexpr (BITS == 4) {
        // 2 neighbouring lanes make one byte of 4-bit fields
        const uint32_t f = (sgn ? 8u : 0u) | mag;
        const uint32_t f1 = __shfl_down_sync(0xffffffffu, f, 1);
        if ((lane & 1) == 0) r0[(32 * e + lane) / 2] = (uint8_t)(f | (f1 << 4));
      } else {
        // 4 neighbouring lanes make one byte of 2-bit fields
        const uint32_t f = BITS == 2 ? ((sgn ? 2u : 0u) | mag) : mag;
        const uint32_t f1 = __shfl_down_sync(0xffffffffu, f, 1);
        const uint32_t f2 = __shfl_down_sync(0xffffffffu, f, 2);
        const uint32_t f3 = __shfl_down_sync(0xffffffffu, f, 3);
        if ((lane & 3) == 0) r0[(32 * e + lane) / 4] = (uint8_t)(f | (f1 << 2) | (f2 << 4) | (f3 << 6));
      }
      if constexpr (BITS == 3) {
        const uint32_t sign_word = __ballot_sync(0xffffffffu, sgn);
        if (lane == 0) *reinterpret_cast<uint32_t*>(plane1 + row * (D / 8) + 4 * e) = sign_word;
      }
    }
    if (lane == 0) norms[row] = __float2half_rn(n);
  }
}

template <int BITS>
void launch_quant_tq_bits(int d, int grid, int block, cudaStream_t s, const __half* x, int64_t rows,
                          int64_t stride, const TqConsts& c, uint8_t* p0, uint8_t* p1, __half* norms) {
  switch (d) {
    case 32: quant_tq_kernel<32, BITS><<<grid, block, 0, s>>>(x, rows, stride, c, p0, p1, norms); break;
    case 64: quant_tq_kernel<64, BITS><<<grid, block, 0, s>>>(x, rows, stride, c, p0, p1, norms); break;
    case 128: quant_tq_kernel<128, BITS><<<grid, block, 0, s>>>(x, rows, stride, c, p0, p1, norms); break;
    case 256: quant_tq_kernel<256, BITS><<<grid, block, 0, s>>>(x, rows, stride, c, p0, p1, norms); break;
    default: quant_tq_kernel<512, BITS><<<grid, block, 0, s>>>(x, rows, stride, c, p0, p1, norms); break;
  }
}

int grid_for(int64_t threads_needed, int block) {
  int64_t blocks = (threads_needed + block - 1) / block;
  const int64_t cap = (int64_t)sm_count_current() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

qps_status launch_quant_q8_0(const __half* x, int64_t rows, int d, int64_t stride, int8_t* codes,
                             __half* scales, cudaStream_t s) {
  if (rows == 0) return QPS_OK;
  const int block = 256;
  quant_q8_0_kernel<<<grid_for(rows * (d / 8), block), block, 0, s>>>(x, rows, d, stride, codes,
                                                                     scales);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

qps_status launch_quant_tq(int bits, const __half* x, int64_t rows, int d, int64_t stride,
                           const uint32_t* signs, const uint32_t* signs2, int block, uint8_t* plane0,
                           uint8_t* plane1, __half* norms, cudaStream_t s) {
  if (rows == 0) return QPS_OK;
  const Codebook* cb = tq_codebook(bits);
  if (!cb) return fail(QPS_ERR_UNSUPPORTED, "kv_quant_tq: bits must be 2, 3 or 4");
  if (d != 32 && d != 64 && d != 128 && d != 256 && d != 512)
    return fail(QPS_ERR_UNSUPPORTED, "kv_quant_tq: head_dim must be 32, 64, 128, 256 or 512");
  TqConsts c{};
  for (int i = 0; i < d / 32; ++i) c.signs[i] = signs[i];
  if (signs2)
    for (int i = 0; i < d / 32; ++i) c.signs2[i] = signs2[i];
  for (int i = 0; i < cb->n - 1; ++i) c.thresholds[i] = cb->thresholds[i];
  if (block < 32 || block > d || (block & (block - 1)))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq: block must be a power of two in [32, head_dim]");
  c.kappa = std::sqrt((float)(d / block));  // IEEE square root: correctly rounded
  c.hreg = block / 32;
  const int threads = 256;
  const int grid = grid_for(rows * 32, threads);
  if (bits == 2) launch_quant_tq_bits<2>(d, grid, threads, s, x, rows, stride, c, plane0, plane1, norms);
  else if (bits == 3) launch_quant_tq_bits<3>(d, grid, threads, s, x, rows, stride, c, plane0, plane1, norms);
  else launch_quant_tq_bits<4>(d, grid, threads, s, x, rows, stride, c, plane0, plane1, norms);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

}  // namespace qps
