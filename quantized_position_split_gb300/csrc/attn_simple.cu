// Split-KV decode attention on CUDA cores (any supported format pairing).  A
// TurboQuant K (with V in the same tier) is read in the rotated domain against the
// rotated query ("F5 M6 — PolyKV", section "S2 perf-path Level B").
//
// Computes one part of the position-split decode of "F5 M7 — Rolling KV:
// position-windowed KV residency" (section "Implementation decomposition, refined
// (S1 -> S2 -> S3)", item S2): every split chunk of positions yields a normalised
// output and its log-sum-exp; the chunks are merged later by the LSE combine.  K / V
// are dequantised in registers as they are read; a TurboQuant V is accumulated in the
// rotated domain as level x norm and inverse-rotated once per output row ("F5 M6 —
// PolyKV (shared compressed KV pool)", section "S2 perf-path Level B").
//
// Layout: one CTA per (split, KV head, batch entry or shared batch); 8 warps stride
// over the chunk's tokens; lane L holds head_dim elements [L*E, L*E + E), E = D / 32.
// Query rows (the GQA group, or every batch entry's group for a shared prefix) are
// processed RC at a time.
#include "internal.h"

namespace qps {
namespace {

constexpr int kWarps = 8;

template <int E>
__device__ __forceinline__ void load_f16(const __half* p, float* out) {
  if constexpr (E == 2) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(p));
    out[0] = f.x;
    out[1] = f.y;
  } else {
#pragma unroll
    for (int c = 0; c < E / 8 + (E < 8 ? 1 : 0); ++c) {
      if constexpr (E == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 f = __half22float2(h[i]);
          out[2 * i] = f.x;
          out[2 * i + 1] = f.y;
        }
      } else {
        const uint4 raw = *reinterpret_cast<const uint4*>(p + 8 * c);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(h[i]);
          out[8 * c + 2 * i] = f.x;
          out[8 * c + 2 * i + 1] = f.y;
        }
      }
    }
  }
}

template <int E>
__device__ __forceinline__ void load_q8(const int8_t* p, float scale, float* out) {
  uint32_t w[(E + 3) / 4];
  if constexpr (E == 2) {
    w[0] = *reinterpret_cast<const uint16_t*>(p);
  } else if constexpr (E == 4) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (E == 8) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    w[0] = r.x;
    w[1] = r.y;
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    w[0] = r.x;
    w[1] = r.y;
    w[2] = r.z;
    w[3] = r.w;
  }
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int8_t c = (int8_t)((w[i / 4] >> (8 * (i % 4))) & 0xff);
    out[i] = (float)c * scale;
  }
}

// Row `row` of a KV side, lane's E elements, as float.  A TurboQuant tier gives the
// rotated-domain value norm * level (the 1/D, the Hadamard matrix and the signs come at
// the end); `levels` is its codebook, ascending and symmetric.
template <int FMT, int D>
__device__ __forceinline__ void load_row(const KvSide& s, int64_t row, int lane,
                                         const float* levels, float* out) {
  constexpr int E = D / 32;
  if constexpr (FMT == QPS_FMT_F16) {
    load_f16<E>(reinterpret_cast<const __half*>(s.data) + row * D + lane * E, out);
  } else if constexpr (FMT == QPS_FMT_Q8_0) {
    const float sc = __half2float(
        reinterpret_cast<const __half*>(s.aux)[row * (D / 32) + (lane * E) / 32]);
    load_q8<E>(reinterpret_cast<const int8_t*>(s.data) + row * D + lane * E, sc, out);
  } else if constexpr (FMT == QPS_FMT_TQ3) {
    const uint32_t* lo = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const uint8_t*>(s.data) + row * (D / 4));
    const uint32_t* hi = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const uint8_t*>(s.aux) + row * (D / 8));
    const uint32_t lw = lo[(2 * E * lane) / 32] >> ((2 * E * lane) % 32);
    const uint32_t hw = hi[(E * lane) / 32] >> ((E * lane) % 32);
    const float n = __half2float(reinterpret_cast<const __half*>(s.aux2)[row]);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float mag = levels[4 + ((lw >> (2 * e)) & 3u)];
      out[e] = ((hw >> e) & 1u) ? n * mag : -n * mag;
    }
  } else {
    // TQ2 / TQ4: fields (sign << (B - 1)) | magnitude of B bits, little-endian
    constexpr int B = FMT == QPS_FMT_TQ2 ? 2 : 4;
    constexpr int HALF = 1 << (B - 1);
    const uint8_t* f = reinterpret_cast<const uint8_t*>(s.data) + row * (D * B / 8);
    const float n = __half2float(reinterpret_cast<const __half*>(s.aux)[row]);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int bit = B * (E * lane + e);
      const uint32_t fld = (f[bit >> 3] >> (bit & 7)) & ((1u << B) - 1);
      const float mag = levels[HALF + (fld & (HALF - 1))];
      out[e] = (fld & HALF) ? n * mag : -n * mag;
    }
  }
}

template <int D, int KF, int VF, int RC>
__global__ void __launch_bounds__(kWarps * 32) attn_simple_kernel(const AttnParams p) {
  constexpr int E = D / 32;
  extern __shared__ float smem[];
  float* qs = smem;                        // [RC][D]
  float* ms = qs + RC * D;                 // [kWarps][RC]
  float* ls = ms + kWarps * RC;            // [kWarps][RC]
  float* os = ls + kWarps * RC;            // [kWarps][RC][D]

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int bz = blockIdx.z;
  const int64_t t0 = p.begin + (int64_t)split * p.chunk;
  const int64_t t1 = min(p.end, t0 + p.chunk);
  const int R = p.rows_per_cta;
  const int64_t kbase = p.shared ? 0 : (int64_t)bz * p.k.batch;
  const int64_t vbase = p.shared ? 0 : (int64_t)bz * p.v.batch;
  const int part = p.part_offset + split;
  float levels[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) levels[i] = p.tq_levels[i];

  for (int rc0 = 0; rc0 < R; rc0 += RC) {
    const int nr = min(RC, R - rc0);
    // query rows of this chunk -> shared memory (float)
    for (int idx = threadIdx.x; idx < RC * D; idx += blockDim.x) {
      const int r = idx / D, dd = idx % D;
      float val = 0.f;
      if (r < nr) {
        const int rr = rc0 + r;
        const int b = p.shared ? rr / p.group : bz;
        const int h = g * p.group + (p.shared ? rr % p.group : rr);
        const int64_t qi = (int64_t)b * p.q_bstride + (int64_t)h * D + dd;
        if (in_bounds(qi >= 0 && qi < p.q_elems, p.err)) val = __half2float(p.q[qi]);
      }
      qs[idx] = val;
    }
    __syncthreads();
    if constexpr (is_tq(KF)) {
      // a TurboQuant K is read in the rotated domain (norm x level), so the query rows
      // become R q = s2 .* blockdiag(H_G)(s1 .* q) / sqrt(G); the logits then carry the
      // decode's 1 / sqrt(D) (k_norm_scale)
      for (int idx = threadIdx.x; idx < RC * D; idx += blockDim.x) {
        const int dd = idx % D;
        if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) qs[idx] = -qs[idx];
      }
      __syncthreads();
      for (int h = 1; h < p.vblock; h *= 2) {
        for (int pid = threadIdx.x; pid < RC * (D / 2); pid += blockDim.x) {
          const int r = pid / (D / 2), j = pid % (D / 2);
          const int i = (j / h) * 2 * h + (j % h);
          const float a = qs[r * D + i], b = qs[r * D + i + h];
          qs[r * D + i] = a + b;
          qs[r * D + i + h] = a - b;
        }
        __syncthreads();
      }
      for (int idx = threadIdx.x; idx < RC * D; idx += blockDim.x) {
        const int dd = idx % D;
        const float v = qs[idx] * p.k_rot_scale;
        qs[idx] = ((p.vsigns2[dd >> 5] >> (dd & 31)) & 1u) ? -v : v;
      }
      __syncthreads();
    }
    const float logit_scale = is_tq(KF) ? p.scale * p.k_norm_scale : p.scale;

    float m[RC], l[RC], o[RC][E];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[r][e] = 0.f;
    }

    for (int64_t t = t0 + warp; t < t1; t += kWarps) {
      float kf[E], vf[E];
      const int64_t krow = kbase + t * p.k.tok + (int64_t)g * p.k.head;
      const int64_t vrow = vbase + t * p.v.tok + (int64_t)g * p.v.head;
      // (warp-uniform: a row outside its view reads as zeros in the checked build)
      if (in_bounds(krow >= 0 && krow < p.k_rows, p.err)) {
        load_row<KF, D>(p.k, krow, lane, levels, kf);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) kf[e] = 0.f;
      }
      if (in_bounds(vrow >= 0 && vrow < p.v_rows, p.err)) {
        load_row<VF, D>(p.v, vrow, lane, levels, vf);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) vf[e] = 0.f;
      }
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        const float* qr = qs + r * D + lane * E;
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(qr[e], kf[e], acc);
#pragma unroll
        for (int h = 16; h >= 1; h /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, h);
        float s = acc * logit_scale;
        if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap);
        const float mn = fmaxf(m[r], s);
        const float corr = __expf(m[r] - mn);
        const float pr = __expf(s - mn);
        l[r] = l[r] * corr + pr;
#pragma unroll
        for (int e = 0; e < E; ++e) o[r][e] = o[r][e] * corr + pr * vf[e];
        m[r] = mn;
      }
    }

    // per-warp states -> shared memory, then merge across warps
#pragma unroll
    for (int r = 0; r < RC; ++r) {
      if (lane == 0) {
        ms[warp * RC + r] = m[r];
        ls[warp * RC + r] = l[r];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) os[(warp * RC + r) * D + lane * E + e] = o[r][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nr * D; idx += blockDim.x) {
      const int r = idx / D, dd = idx % D;
      float mx = -INFINITY;
      for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, ms[w * RC + r]);
      float acc = 0.f;
      if (mx != -INFINITY) {
        for (int w = 0; w < kWarps; ++w) {
          const float mw = ms[w * RC + r];
          if (mw != -INFINITY) acc += os[(w * RC + r) * D + dd] * __expf(mw - mx);
        }
      }
      if constexpr (is_tq(VF))  // the rotation's second sign vector
        if ((p.vsigns2[dd >> 5] >> (dd & 31)) & 1u) acc = -acc;
      qs[r * D + dd] = acc;  // the query rows are no longer needed
    }
    __syncthreads();

    if constexpr (is_tq(VF)) {
      // inverse rotation of the accumulated rows: x = s1 .* blockdiag(H_G)(s2 .* y) / sqrt(D G)
      for (int h = 1; h < p.vblock; h *= 2) {
        for (int pid = threadIdx.x; pid < nr * (D / 2); pid += blockDim.x) {
          const int r = pid / (D / 2), j = pid % (D / 2);
          const int i = (j / h) * 2 * h + (j % h);
          const float a = qs[r * D + i], b = qs[r * D + i + h];
          qs[r * D + i] = a + b;
          qs[r * D + i + h] = a - b;
        }
        __syncthreads();
      }
    }

    for (int idx = threadIdx.x; idx < nr * D; idx += blockDim.x) {
      const int r = idx / D, dd = idx % D;
      float mx = -INFINITY;
      for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, ms[w * RC + r]);
      float den = 0.f;
      if (mx != -INFINITY) {
        for (int w = 0; w < kWarps; ++w) {
          const float mw = ms[w * RC + r];
          if (mw != -INFINITY) den += ls[w * RC + r] * __expf(mw - mx);
        }
      }
      float val = qs[r * D + dd];
      if constexpr (is_tq(VF)) {
        val *= p.v_out_scale;
        if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) val = -val;
      }
      const int rr = rc0 + r;
      const int b = p.shared ? rr / p.group : bz;
      const int h = g * p.group + (p.shared ? rr % p.group : rr);
      const int64_t row = (int64_t)b * p.hq + h;
      const bool empty = !(den > 0.f);
      if (!in_bounds(part < p.parts_cap && row >= 0 && row < p.rows_total, p.err)) continue;
      p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = empty ? 0.f : val / den;
      if (dd == 0) p.lse_parts[(int64_t)part * p.rows_total + row] = empty ? -INFINITY : mx + __logf(den);
    }
    __syncthreads();
  }
}

template <int D, int KF, int VF>
qps_status launch_simple_dkv(const AttnParams& p, cudaStream_t s) {
  constexpr int RC = D >= 512 ? 4 : 8;
  const size_t smem = sizeof(float) * (RC * D + 2 * kWarps * RC + kWarps * RC * D);
  auto kern = attn_simple_kernel<D, KF, VF, RC>;
  QPS_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const dim3 grid(p.n_split, p.hkv, p.shared ? 1 : p.batch);
  kern<<<grid, kWarps * 32, smem, s>>>(p);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

template <int D>
qps_status launch_simple_d(const AttnParams& p, cudaStream_t s) {
  if (is_tq(p.kfmt) && p.vfmt == p.kfmt) {
    if (p.kfmt == QPS_FMT_TQ2) return launch_simple_dkv<D, QPS_FMT_TQ2, QPS_FMT_TQ2>(p, s);
    if (p.kfmt == QPS_FMT_TQ3) return launch_simple_dkv<D, QPS_FMT_TQ3, QPS_FMT_TQ3>(p, s);
    return launch_simple_dkv<D, QPS_FMT_TQ4, QPS_FMT_TQ4>(p, s);
  }
  if (p.kfmt == QPS_FMT_F16) {
    if (p.vfmt == QPS_FMT_F16) return launch_simple_dkv<D, QPS_FMT_F16, QPS_FMT_F16>(p, s);
    if (p.vfmt == QPS_FMT_Q8_0) return launch_simple_dkv<D, QPS_FMT_F16, QPS_FMT_Q8_0>(p, s);
    if (p.vfmt == QPS_FMT_TQ3) return launch_simple_dkv<D, QPS_FMT_F16, QPS_FMT_TQ3>(p, s);
    if (p.vfmt == QPS_FMT_TQ2) return launch_simple_dkv<D, QPS_FMT_F16, QPS_FMT_TQ2>(p, s);
    if (p.vfmt == QPS_FMT_TQ4) return launch_simple_dkv<D, QPS_FMT_F16, QPS_FMT_TQ4>(p, s);
  } else if (p.kfmt == QPS_FMT_Q8_0) {
    if (p.vfmt == QPS_FMT_F16) return launch_simple_dkv<D, QPS_FMT_Q8_0, QPS_FMT_F16>(p, s);
    if (p.vfmt == QPS_FMT_Q8_0) return launch_simple_dkv<D, QPS_FMT_Q8_0, QPS_FMT_Q8_0>(p, s);
    if (p.vfmt == QPS_FMT_TQ3) return launch_simple_dkv<D, QPS_FMT_Q8_0, QPS_FMT_TQ3>(p, s);
    if (p.vfmt == QPS_FMT_TQ2) return launch_simple_dkv<D, QPS_FMT_Q8_0, QPS_FMT_TQ2>(p, s);
    if (p.vfmt == QPS_FMT_TQ4) return launch_simple_dkv<D, QPS_FMT_Q8_0, QPS_FMT_TQ4>(p, s);
  }
  return fail(QPS_ERR_UNSUPPORTED, "attention: unsupported K/V format pairing");
}

}  // namespace

qps_status launch_attn_simple(const AttnParams& p, cudaStream_t s) {
  switch (p.d) {
    case 64: return launch_simple_d<64>(p, s);
    case 128: return launch_simple_d<128>(p, s);
    case 256: return launch_simple_d<256>(p, s);
    case 512: return launch_simple_d<512>(p, s);
    default: return fail(QPS_ERR_UNSUPPORTED, "attention: head_dim must be 64, 128, 256 or 512");
  }
}

}  // namespace qps
