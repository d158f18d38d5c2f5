// Split-KV decode attention on tensor cores (mma.sync m16n8k16, f16 x f16 -> f32).
//
// One part of the position-split decode of "F5 M7 — Rolling KV: position-windowed KV
// residency" (section "Implementation decomposition, refined (S1 -> S2 -> S3)", item
// S2): every split chunk of positions yields a normalised output and its log-sum-exp.
// K / V are dequantised in registers on their way into the tensor-core operands; a TQ3
// V is read as centroid x norm in the rotated domain and the output is inverse-rotated
// once ("F5 M6 — PolyKV (shared compressed KV pool)", section "S2 perf-path Level B").
//
// Formulation (query rows on the narrow N = 8 side, so a GQA group of 5..8 rows wastes
// nothing):   S^T[t][r] = sum_d K[t][d] Q[r][d]       (A = K tile, B = Q^T)
//             O^T[d][r] = sum_t V^T[d][t] P^T[t][r]   (A = V^T tile, B = P^T)
// P leaves the S^T accumulator layout and enters the B-operand layout through one
// movmatrix transpose per 8x8 block.
//
// Exactness: q8_0 K codes are exact in f16; each 32-value block is accumulated
// separately and multiplied by its fp32 scale afterwards, so the logits carry only
// fp32 rounding.  TQ3 levels are fp16-exact by construction.  P (in [0, 1]) and a
// q8_0 V value (code x scale) are rounded once to fp16.
//
// Data movement: the KV planes of a (KV head, batch entry) must be token-contiguous
// (tok_stride == 1).  Each warp runs a private cp.async pipeline of STAGES tiles of 16
// tokens over its own share of the chunk's tiles (tiles w, w + NW, ...), staging every
// plane of the tile into shared memory with a bank-conflict-avoiding XOR swizzle; a
// tile partly outside [t0, t1) is zero-filled past t1 and masked in the softmax.
#pragma once

#include "internal.h"

namespace qps {
namespace mma {

constexpr int kTile = 16;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 4 signed int8 codes (little-endian in w) -> two half2 {c0, c1}, {c2, c3}, exactly:
// the biased byte b + 128 becomes the mantissa of 1024 + (b + 128) and 1152 is removed.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 hl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<uint32_t*>(&hl);
  hi = *reinterpret_cast<uint32_t*>(&hh);
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, __half2 s) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), s);
  return *reinterpret_cast<uint32_t*>(&r);
}

// ---- tile geometry ---------------------------------------------------------------
__host__ __device__ constexpr int r16(int x) { return (x + 15) / 16 * 16; }

template <int D, int KF, int VF>
struct Geo {
  static constexpr int K_RB = KF == QPS_FMT_F16 ? 2 * D : D;          // K data bytes / token
  static constexpr int K_ARB = KF == QPS_FMT_Q8_0 ? D / 16 : 0;       // K scales bytes / token
  static constexpr int V_RB = VF == QPS_FMT_F16 ? 2 * D : VF == QPS_FMT_Q8_0 ? D : D / 4;
  static constexpr int V_ARB = VF == QPS_FMT_Q8_0 ? D / 16 : VF == QPS_FMT_TQ3 ? D / 8 : 0;
  static constexpr int V_A2RB = VF == QPS_FMT_TQ3 ? 2 : 0;
  static constexpr int K_OFF = 0;
  static constexpr int KA_OFF = K_OFF + kTile * K_RB;
  static constexpr int V_OFF = KA_OFF + r16(kTile * K_ARB);
  static constexpr int VA_OFF = V_OFF + kTile * V_RB;
  static constexpr int VA2_OFF = VA_OFF + r16(kTile * V_ARB);
  static constexpr int STAGE = VA2_OFF + r16(kTile * V_A2RB);
  // warps per CTA: 4, or 2 when two stages of 4 warps would not fit in shared memory
  static constexpr int NW = 4 * 2 * STAGE <= 200 * 1024 ? 4 : 2;
  static constexpr int STAGES_RAW = (96 * 1024) / (NW * STAGE);
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 6 ? 6 : STAGES_RAW);
  static constexpr int PIPE = NW * STAGES * STAGE;
};

// XOR swizzles of 16-byte chunks within a token row of a staged tile.
template <int D, int FMT, bool IS_K>
__device__ __forceinline__ int swz(int row) {
  if constexpr (FMT == QPS_FMT_F16) {
    return row & 7;  // ldmatrix: 8 rows x one chunk per phase
  } else if constexpr (FMT == QPS_FMT_Q8_0) {
    if constexpr (IS_K) return D >= 128 ? ((row & 3) << 1) : ((row & 1) << 1);
    else return D >= 512 ? ((row >> 1) & 3) : (D >= 128 ? (row & 7) : 0);
  } else {
    return 0;
  }
}

// Copy one plane of a 16-token tile (token-contiguous rows of rb bytes) into shared
// memory; rows of tokens >= valid are zero-filled without reading.
template <int RB, int SWZ_D, int SWZ_FMT, bool SWZ_K, bool SWIZZLE>
__device__ __forceinline__ void stage_plane(uint8_t* dst, const uint8_t* src, int valid_tokens, int lane,
                                            const uint8_t* safe_src) {
  constexpr int BYTES = kTile * RB;
  constexpr int CHUNKS = (BYTES + 15) / 16;
  const int valid_bytes = valid_tokens * RB;
  const uint32_t base = smem_addr(dst);
#pragma unroll 4
  for (int ch = lane; ch < CHUNKS; ch += 32) {
    int dch = ch;
    if constexpr (SWIZZLE && RB >= 16) {
      constexpr int CPR = RB / 16;  // chunks per row
      const int row = ch / CPR, x = ch % CPR;
      dch = row * CPR + (x ^ swz<SWZ_D, SWZ_FMT, SWZ_K>(row));
    }
    int nb = valid_bytes - ch * 16;
    nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
    cp_async16(base + dch * 16, nb > 0 ? (const void*)(src + ch * 16) : (const void*)safe_src, nb);
  }
}

// Where the swizzled 16-byte chunk x of row `row` lives.
template <int RB, int D, int FMT, bool IS_K>
__device__ __forceinline__ int chunk_off(int row, int x) {
  return row * RB + ((x ^ swz<D, FMT, IS_K>(row)) << 4);
}

// ---- the kernel -------------------------------------------------------------------
template <int D, int KF, int VF, int NTW>
__global__ void __launch_bounds__(Geo<D, KF, VF>::NW * 32, 2) attn_mma_kernel(const AttnParams p) {
  using G = Geo<D, KF, VF>;
  constexpr int kWarps = G::NW;
  constexpr int ROWS = 8 * NTW;  // query rows per CTA
  constexpr int MT = D / 16;     // m-tiles of O^T, k-steps of S^T
  constexpr int KQ = KF == QPS_FMT_Q8_0 ? 1 : 0;
  constexpr bool VPERM = VF != QPS_FMT_F16;  // permuted output columns (see below)
  constexpr int DT = D / 8;                  // output columns per lane group (VPERM)
  constexpr float LOG2E = 1.4426950408889634f;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* pipe = smem;
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + G::PIPE);  // TQ3: 64 half2

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, head = blockIdx.y;
  const int rgroups = (p.rows_per_cta + ROWS - 1) / ROWS;
  const int rg = blockIdx.z % rgroups, bz = blockIdx.z / rgroups;
  const int row0 = rg * ROWS;
  const int nrows = min(ROWS, p.rows_per_cta - row0);
  const int64_t t0 = p.begin + (int64_t)split * p.chunk;
  const int64_t t1 = min(p.end, t0 + p.chunk);
  const int part = p.part_offset + split;

  auto out_row = [&](int rr) -> int64_t {
    const int b = p.shared ? rr / p.group : bz;
    const int h = head * p.group + (p.shared ? rr % p.group : rr);
    return (int64_t)b * p.hq + h;
  };

  if (t0 >= t1) {  // an empty chunk: O = 0, lse = -inf
    for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
      const int r = idx / D, dd = idx % D;
      const int64_t row = out_row(row0 + r);
      p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = 0.f;
      if (dd == 0) p.lse_parts[(int64_t)part * p.rows_total + row] = -INFINITY;
    }
    return;
  }

  if constexpr (VF == QPS_FMT_TQ3) {
    // index = mag_a | mag_b << 2 | sign_a << 4 | sign_b << 5 -> half2(level_a, level_b)
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
      const float ma = p.tq_levels[4 + (i & 3)], mb = p.tq_levels[4 + ((i >> 2) & 3)];
      lut[i] = pack_h2((i & 16) ? ma : -ma, (i & 32) ? mb : -mb);
    }
  }

  // ---- query fragments (B operand of S^T), one set per 8-row n-tile --------------
  uint32_t qb[NTW][MT][2];
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    const int rr = row0 + nt * 8 + g;
    const bool valid = rr < p.rows_per_cta;
    const __half* qrow = nullptr;
    if (valid) {
      const int b = p.shared ? rr / p.group : bz;
      const int h = head * p.group + (p.shared ? rr % p.group : rr);
      qrow = p.q + (int64_t)b * p.q_bstride + (int64_t)h * D;
    }
#pragma unroll
    for (int kk = 0; kk < MT; ++kk) {
      int d0, d1;
      if constexpr (KQ) {  // permuted: lane group c owns d in [32j + 8c, +8) of block j
        const int j = kk >> 1, hh = kk & 1;
        d0 = 32 * j + 8 * c + 4 * hh;
        d1 = d0 + 2;
      } else {
        d0 = 16 * kk + 2 * c;
        d1 = d0 + 8;
      }
      qb[nt][kk][0] = valid ? *reinterpret_cast<const uint32_t*>(qrow + d0) : 0u;
      qb[nt][kk][1] = valid ? *reinterpret_cast<const uint32_t*>(qrow + d1) : 0u;
    }
  }

  // ---- plane bases of this (head, batch entry) -------------------------------------
  const int64_t krow = (p.shared ? 0 : (int64_t)bz * p.k.batch) + (int64_t)head * p.k.head;
  const int64_t vrow = (p.shared ? 0 : (int64_t)bz * p.v.batch) + (int64_t)head * p.v.head;
  const uint8_t* kd = reinterpret_cast<const uint8_t*>(p.k.data) + krow * G::K_RB;
  const uint8_t* ka = KQ ? reinterpret_cast<const uint8_t*>(p.k.aux) + krow * G::K_ARB : nullptr;
  const uint8_t* vd = reinterpret_cast<const uint8_t*>(p.v.data) + vrow * G::V_RB;
  const uint8_t* va = G::V_ARB ? reinterpret_cast<const uint8_t*>(p.v.aux) + vrow * G::V_ARB : nullptr;
  const uint8_t* va2 = G::V_A2RB ? reinterpret_cast<const uint8_t*>(p.v.aux2) + vrow * G::V_A2RB : nullptr;
  const uint8_t* safe = reinterpret_cast<const uint8_t*>(p.k.data);

  const int64_t tile0 = t0 & ~(int64_t)(kTile - 1);
  const int ntiles = (int)((t1 - tile0 + kTile - 1) / kTile);
  uint8_t* wpipe = pipe + warp * G::STAGES * G::STAGE;

  auto issue = [&](int k) {  // the warp's k-th tile -> stage k % STAGES
    const int tile = warp + k * kWarps;
    if (tile < ntiles) {
      uint8_t* st = wpipe + (k % G::STAGES) * G::STAGE;
      const int64_t tb = tile0 + (int64_t)tile * kTile;
      const int valid = (int)min((int64_t)kTile, t1 - tb);
      stage_plane<G::K_RB, D, KF, true, true>(st + G::K_OFF, kd + tb * G::K_RB, valid, lane, safe);
      if constexpr (G::K_ARB > 0)
        stage_plane<G::K_ARB, D, KF, true, false>(st + G::KA_OFF, ka + tb * G::K_ARB, valid, lane, safe);
      stage_plane<G::V_RB, D, VF, false, true>(st + G::V_OFF, vd + tb * G::V_RB, valid, lane, safe);
      if constexpr (G::V_ARB > 0)
        stage_plane<G::V_ARB, D, VF, false, false>(st + G::VA_OFF, va + tb * G::V_ARB, valid, lane, safe);
      if constexpr (G::V_A2RB > 0)
        stage_plane<G::V_A2RB, D, VF, false, false>(st + G::VA2_OFF, va2 + tb * G::V_A2RB, valid, lane, safe);
    }
    cp_async_commit();
  };

  // ---- running softmax state (log2 domain) and the O^T accumulators ---------------
  float m[NTW][2], l[NTW][2];
  float o[MT][NTW][4];
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int i = 0; i < MT; ++i) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
  }
  const float qk_scale = p.scale;
  const float cap = p.softcap;

  __syncthreads();  // the LUT is ready

#pragma unroll 1
  for (int s = 0; s < G::STAGES - 1; ++s) issue(s);

#pragma unroll 1
  for (int k = 0; warp + k * kWarps < ntiles; ++k) {
    issue(k + G::STAGES - 1);
    cp_async_wait<G::STAGES - 1>();
    __syncwarp();
    const uint8_t* st = wpipe + (k % G::STAGES) * G::STAGE;
    const int64_t tb = tile0 + (int64_t)(warp + k * kWarps) * kTile;

    // ---- S^T = K Q^T ---------------------------------------------------------------
    float sacc[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    if constexpr (KF == QPS_FMT_F16) {
      const uint32_t kbase = smem_addr(st + G::K_OFF);
      const int mi = lane >> 3;
      const int trow = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, kbase + chunk_off<G::K_RB, D, KF, true>(trow, 2 * kk + (mi >> 1)));
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) mma16816(sacc[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
      }
    } else {
      const uint8_t* kc = st + G::K_OFF;
      const __half* ks = reinterpret_cast<const __half*>(st + G::KA_OFF);
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const int x = 2 * j + (c >> 1), sub = 8 * (c & 1);
        const uint2 wg = *reinterpret_cast<const uint2*>(kc + chunk_off<G::K_RB, D, KF, true>(g, x) + sub);
        const uint2 wg8 = *reinterpret_cast<const uint2*>(kc + chunk_off<G::K_RB, D, KF, true>(g + 8, x) + sub);
        uint32_t a0[4], a1[4];
        i8x4_to_h2x2(wg.x, a0[0], a0[2]);
        i8x4_to_h2x2(wg8.x, a0[1], a0[3]);
        i8x4_to_h2x2(wg.y, a1[0], a1[2]);
        i8x4_to_h2x2(wg8.y, a1[1], a1[3]);
        const float sg = __half2float(ks[g * (D / 32) + j]);
        const float sg8 = __half2float(ks[(g + 8) * (D / 32) + j]);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(acc, a0, qb[nt][2 * j][0], qb[nt][2 * j][1]);
          mma16816(acc, a1, qb[nt][2 * j + 1][0], qb[nt][2 * j + 1][1]);
          sacc[nt][0] = fmaf(sg, acc[0], sacc[nt][0]);
          sacc[nt][1] = fmaf(sg, acc[1], sacc[nt][1]);
          sacc[nt][2] = fmaf(sg8, acc[2], sacc[nt][2]);
          sacc[nt][3] = fmaf(sg8, acc[3], sacc[nt][3]);
        }
      }
    }

    // ---- logits, masking, online softmax ---------------------------------------------
    const bool in_g = (tb + g >= t0) && (tb + g < t1);
    const bool in_g8 = (tb + g + 8 >= t0) && (tb + g + 8 < t1);
    float n_g = 1.f, n_g8 = 1.f;
    if constexpr (VF == QPS_FMT_TQ3) {
      const __half* nrm = reinterpret_cast<const __half*>(st + G::VA2_OFF);
      n_g = __half2float(nrm[g]);
      n_g8 = __half2float(nrm[g + 8]);
    }
    uint32_t pb[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sacc[nt][e] * qk_scale;
        if (cap > 0.f) v = cap * tanhf(v / cap);
        x[e] = v * LOG2E;
      }
      if (!in_g) x[0] = x[1] = -INFINITY;
      if (!in_g8) x[2] = x[3] = -INFINITY;
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float cr0 = exp2f(m[nt][0] - ms0), cr1 = exp2f(m[nt][1] - ms1);
      const float p0 = exp2f(x[0] - ms0), p1 = exp2f(x[1] - ms1);
      const float p2 = exp2f(x[2] - ms0), p3 = exp2f(x[3] - ms1);
      l[nt][0] = l[nt][0] * cr0 + (p0 + p2);
      l[nt][1] = l[nt][1] * cr1 + (p1 + p3);
      m[nt][0] = mn0;
      m[nt][1] = mn1;
      if (__any_sync(0xffffffffu, cr0 != 1.f || cr1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          o[i][nt][0] *= cr0;
          o[i][nt][1] *= cr1;
          o[i][nt][2] *= cr0;
          o[i][nt][3] *= cr1;
        }
      }
      pb[nt][0] = movmatrix_t(pack_h2(p0 * n_g, p1 * n_g));
      pb[nt][1] = movmatrix_t(pack_h2(p2 * n_g8, p3 * n_g8));
    }

    // ---- O^T += V^T P^T ---------------------------------------------------------------
    if constexpr (VF == QPS_FMT_F16) {
      const uint32_t vbase = smem_addr(st + G::V_OFF);
      const int mi = lane >> 3;
      const int trow = (lane & 7) + ((mi & 2) << 2);
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        uint32_t a[4];
        ldsm_x4_t(a, vbase + chunk_off<G::V_RB, D, VF, false>(trow, 2 * i + (mi & 1)));
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[nt][0], pb[nt][1]);
      }
    } else if constexpr (VF == QPS_FMT_Q8_0) {
      // lane group g owns output columns [g*DT, g*DT + DT); tokens 2c, 2c+1, 2c+8, 2c+9
      const uint8_t* vc = st + G::V_OFF;
      const __half* vs = reinterpret_cast<const __half*>(st + G::VA_OFF);
      constexpr int CH = DT >= 16 ? 16 : DT;  // bytes per read
#pragma unroll
      for (int q0 = 0; q0 < DT; q0 += CH) {
        uint32_t w[4][CH / 4];
        const int tok[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
        const int blk = (g * DT + q0) / 32;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int byte = g * DT + q0;
          const uint8_t* src = vc + chunk_off<G::V_RB, D, VF, false>(tok[u], byte >> 4) + (byte & 15);
          if constexpr (CH == 16) {
            const uint4 r = *reinterpret_cast<const uint4*>(src);
            w[u][0] = r.x; w[u][1] = r.y; w[u][2] = r.z; w[u][3] = r.w;
          } else {
            const uint2 r = *reinterpret_cast<const uint2*>(src);
            w[u][0] = r.x; w[u][1] = r.y;
          }
        }
        __half2 sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sc[u] = __half2half2(vs[tok[u] * (D / 32) + blk]);
#pragma unroll
        for (int wi = 0; wi < CH / 4; ++wi) {
          uint32_t hv[4][2];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            i8x4_to_h2x2(w[u][wi], hv[u][0], hv[u][1]);
            hv[u][0] = hmul2_u(hv[u][0], sc[u]);
            hv[u][1] = hmul2_u(hv[u][1], sc[u]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int i = (q0 + 4 * wi) / 2 + hh;  // m-tile: output columns base + 2i, +1
            uint32_t a[4];
            a[0] = __byte_perm(hv[0][hh], hv[1][hh], 0x5410);
            a[1] = __byte_perm(hv[0][hh], hv[1][hh], 0x7632);
            a[2] = __byte_perm(hv[2][hh], hv[3][hh], 0x5410);
            a[3] = __byte_perm(hv[2][hh], hv[3][hh], 0x7632);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[nt][0], pb[nt][1]);
          }
        }
      }
    } else {  // TQ3: levels through the LUT, tokens paired (2c, 2c+1) and (2c+8, 2c+9)
      const uint8_t* lo2 = st + G::V_OFF;
      const uint8_t* hi1 = st + G::VA_OFF;
      constexpr int LB = D / 32;  // 2-bit plane bytes per lane group and token
#pragma unroll
      for (int e0 = 0; e0 < DT; e0 += 16) {  // 16 elements = one 32-bit word of lo2
        uint32_t L[4], H[4];
        const int tok[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int lb = tok[u] * (D / 4) + g * LB + e0 / 4;
          const int hb = tok[u] * (D / 8) + g * (LB / 2) + e0 / 8;
          if constexpr (DT >= 16) {
            L[u] = *reinterpret_cast<const uint32_t*>(lo2 + lb);
            H[u] = *reinterpret_cast<const uint16_t*>(hi1 + hb);
          } else {  // D = 64: 8 elements per lane group
            L[u] = *reinterpret_cast<const uint16_t*>(lo2 + lb);
            H[u] = *reinterpret_cast<const uint8_t*>(hi1 + hb);
          }
        }
        constexpr int NE = DT >= 16 ? 16 : DT;
#pragma unroll
        for (int e = 0; e < NE; e += 2) {
          const int i = (e0 + e) / 2;
          uint32_t a[4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ee = e + hh;
            const uint32_t i01 = ((L[0] >> (2 * ee)) & 3u) | (((L[1] >> (2 * ee)) & 3u) << 2) |
                                 (((H[0] >> ee) & 1u) << 4) | (((H[1] >> ee) & 1u) << 5);
            const uint32_t i89 = ((L[2] >> (2 * ee)) & 3u) | (((L[3] >> (2 * ee)) & 3u) << 2) |
                                 (((H[2] >> ee) & 1u) << 4) | (((H[3] >> ee) & 1u) << 5);
            a[hh] = lut[i01];
            a[2 + hh] = lut[i89];
          }
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[nt][0], pb[nt][1]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- merge the warps' states, then the chunk's partial ------------------------------
  float* mw = reinterpret_cast<float*>(smem);            // [kWarps][ROWS]
  float* lw = mw + kWarps * ROWS;                         // [kWarps][ROWS]
  float* ow = lw + kWarps * ROWS;                         // [kWarps][ROWS][D]
  float* fin = ow + kWarps * ROWS * D;                    // [ROWS][D]
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float lv = l[nt][hh];
      lv += __shfl_xor_sync(0xffffffffu, lv, 4);
      lv += __shfl_xor_sync(0xffffffffu, lv, 8);
      lv += __shfl_xor_sync(0xffffffffu, lv, 16);
      if (g == 0) {
        mw[warp * ROWS + nt * 8 + 2 * c + hh] = m[nt][hh];
        lw[warp * ROWS + nt * 8 + 2 * c + hh] = lv;
      }
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      int d0, d1;
      if constexpr (VPERM) {
        d0 = g * DT + 2 * i;
        d1 = d0 + 1;
      } else {
        d0 = 16 * i + g;
        d1 = d0 + 8;
      }
      float* base = ow + (warp * ROWS + nt * 8 + 2 * c) * D;
      base[d0] = o[i][nt][0];
      base[D + d0] = o[i][nt][1];
      base[d1] = o[i][nt][2];
      base[D + d1] = o[i][nt][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ROWS * D; idx += blockDim.x) {
    const int r = idx / D, dd = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, mw[w * ROWS + r]);
    float acc = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mv = mw[w * ROWS + r];
        if (mv != -INFINITY) acc += ow[(w * ROWS + r) * D + dd] * exp2f(mv - mx);
      }
    }
    fin[idx] = acc;
  }
  __syncthreads();
  if constexpr (VF == QPS_FMT_TQ3) {  // inverse rotation x = s .* (H y) / D, in place
    for (int h = 1; h < D; h <<= 1) {
      for (int pid = threadIdx.x; pid < ROWS * (D / 2); pid += blockDim.x) {
        const int r = pid / (D / 2), j = pid % (D / 2);
        const int i = (j / h) * 2 * h + (j % h);
        const float a = fin[r * D + i], b = fin[r * D + i + h];
        fin[r * D + i] = a + b;
        fin[r * D + i + h] = a - b;
      }
      __syncthreads();
    }
  }
  for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
    const int r = idx / D, dd = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, mw[w * ROWS + r]);
    float den = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mv = mw[w * ROWS + r];
        if (mv != -INFINITY) den += lw[w * ROWS + r] * exp2f(mv - mx);
      }
    }
    float val = fin[r * D + dd];
    if constexpr (VF == QPS_FMT_TQ3) {
      val *= 1.0f / (float)D;
      if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) val = -val;
    }
    const int64_t row = out_row(row0 + r);
    const bool empty = !(den > 0.f);
    p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = empty ? 0.f : val / den;
    if (dd == 0)
      p.lse_parts[(int64_t)part * p.rows_total + row] = empty ? -INFINITY : (mx + log2f(den)) * 0.6931471805599453f;
  }
}

template <int D, int KF, int VF, int NTW>
constexpr size_t smem_bytes() {
  using G = Geo<D, KF, VF>;
  constexpr size_t pipe = (size_t)G::PIPE + 256;
  constexpr int ROWS = 8 * NTW;
  constexpr size_t merge = sizeof(float) * ((size_t)2 * G::NW * ROWS + (size_t)G::NW * ROWS * D + (size_t)ROWS * D);
  return pipe > merge ? pipe : merge;
}

template <int D, int KF, int VF, int NTW>
qps_status launch_mma_t(const AttnParams& p, cudaStream_t s) {
  constexpr size_t smem = smem_bytes<D, KF, VF, NTW>();
  static_assert(smem <= 227 * 1024, "tile staging exceeds the 227 KB shared memory of one CTA");
  auto kern = attn_mma_kernel<D, KF, VF, NTW>;
  QPS_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  constexpr int ROWS = 8 * NTW;
  const int rgroups = (p.rows_per_cta + ROWS - 1) / ROWS;
  const dim3 grid(p.n_split, p.hkv, (p.shared ? 1 : p.batch) * rgroups);
  kern<<<grid, Geo<D, KF, VF>::NW * 32, smem, s>>>(p);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

template <int D>
qps_status launch_mma_d(const AttnParams& p, cudaStream_t s) {
  // two 8-row n-tiles per warp only where the accumulators still fit in registers
  const bool wide = p.rows_per_cta > 8 && D <= 128;
#define QPS_MMA_CASE(KF, VF)                                                       \
  if (p.kfmt == KF && p.vfmt == VF)                                                \
    return wide ? launch_mma_t<D, KF, VF, (D <= 128 ? 2 : 1)>(p, s) : launch_mma_t<D, KF, VF, 1>(p, s);
  QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_F16)
  QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_Q8_0)
  QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_TQ3)
  QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_F16)
  QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_Q8_0)
  QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_TQ3)
#undef QPS_MMA_CASE
  return fail(QPS_ERR_UNSUPPORTED, "attention: unsupported K/V format pairing");
}

}  // namespace mma
}  // namespace qps
