// Warp-specialized split-KV decode attention: head_dim 512, q8_0 K, TQ3 V, up to 8 query
// rows per KV head (the Gemma-like global layers, "F5 M6 — PolyKV (shared compressed KV
// pool)", section "S2 perf-path — turbo-MMA verify kernel + scalar-K/turbo-V fused
// decode": K read true-space from int8 codes, V read in the rotated domain as level x
// norm, the output inverse-rotated once).
//
// Why a second kernel for this pairing.  In the per-warp-pipeline kernel (attn_mma.cuh)
// every warp decodes both K and V of its own tiles: at head_dim 512 its O accumulators
// alone take 128 registers, so 255 registers per thread leave 8 warps per SM with two
// 12 KB stages each; the dequantisation chains then find too few other warps to hide
// behind, and too few tiles are in flight to cover the memory latency.  Here the work of
// every tile is split by role, each role over the whole chunk in order:
//   * warp 0, the producer, keeps NS = 6 stages of the CTA's tiles in flight (tensor-map
//     boxes plus the norms by cp.async), refilling a stage once its consumers are done;
//   * KQ = 4 K-warps each own a quarter of head_dim (four q8_0 blocks): they decode their
//     quarter of the tile's K codes and write the partial logits S^T = K Q^T over it;
//   * the S-warp sums the partials, applies the logit scale, softcap and mask, runs the
//     online softmax (one running maximum and sum per row) and hands P (fp16, the V
//     norms folded in) and each row's rescale factor to the V-warps;
//   * VW = 4 V-warps each own a contiguous quarter of the output columns, lane group g
//     of V-warp v the 16 columns from 128 v + 16 g (one 32-bit word of 2-bit codes and 16
//     sign bits per token, so the warp's code loads cover 32 distinct banks): they
//     rescale, decode their TQ3 codes and accumulate O^T = V^T P^T.
// Per stage four mbarriers order the roles: full (the tile's bytes landed), sready (the
// partial logits are written), pready (P is written), empty (every consumer is done; the
// producer may refill).  All waits are bounded as in attn_mma.cuh; a give-up stops the
// producer, drains the copies in flight and leaves the CTA's partial unwritten.  The
// epilogue applies the inverse rotation once and writes the partial.
#pragma once

#include "attn_mma.cuh"

namespace qps {
namespace ws {

using namespace mma;

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

template <int D, int KF, int VF>
struct WsGeo {
  using G = GeoT<D, KF, VF, 16, 2, 0>;  // the plane offsets of a 16-token stage
  static constexpr int TT = 16;
  static constexpr int KQ = 4;  // K-warps, one quarter of head_dim each
  static constexpr int KW = 1;  // softmax states (the S-warp's)
  static constexpr int VW = 4;  // V-warps
  static constexpr int NWARP = 1 + KQ + 1 + VW;
  static constexpr int S_WARP = 1 + KQ;
  static constexpr int THREADS = 32 * NWARP;
  static constexpr int NS = 6;  // stages in flight per CTA
  static constexpr int STAGE = G::STAGE;
  static constexpr int PIPE = NS * STAGE;
  // per stage: the K-warps' partial logits (KQ x 32 lanes x float4), the P fragments (32
  // lanes x {b0, b1}) and the 8 rows' rescale factors
  static constexpr int SP_OFF = PIPE;
  static constexpr int SP_BYTES = KQ * 32 * 16;
  static constexpr int PB_OFF = SP_OFF + NS * SP_BYTES;
  static constexpr int PB_BYTES = 32 * 8 + 8 * 4;
  static constexpr int BAR_OFF = align_to(PB_OFF + NS * PB_BYTES, 8);
  static constexpr int FULL_OFF = BAR_OFF, SREADY_OFF = BAR_OFF + 8 * NS, PREADY_OFF = BAR_OFF + 16 * NS,
                       EMPTY_OFF = BAR_OFF + 24 * NS;
  static constexpr int FLAG_OFF = BAR_OFF + 32 * NS;
  static constexpr int KS_OFF = align_to(FLAG_OFF + 16, 16);  // the K-warps' final (max, sum) per row
  static constexpr int END = KS_OFF + 2 * KW * 8 * 4;
  // the epilogue, over the stages once every tile is consumed: merged rows [8][FS],
  // per-row weights, maximum, denominator and output row.  Column x of a row sits at
  // x + x / 16 and rows are FS = 8 (mod 32) floats apart, so the V-warps' stores of
  // (row 2c + rp, column 16 g + x) from the 32 lanes hit 32 distinct banks.
  static constexpr int FS = D + D / 16 + 8;
  static_assert(FS % 32 == 8, "row stride 8 mod 32 banks");
  static constexpr int FIN_OFF = 0;
  static constexpr int WK_OFF = FIN_OFF + 8 * FS * 4;
  static constexpr int RMX_OFF = WK_OFF + KW * 8 * 4;
  static constexpr int RDEN_OFF = RMX_OFF + 8 * 4;
  static constexpr int OROW_OFF = align_to(RDEN_OFF + 8 * 4, 8);
  static constexpr int EPI = OROW_OFF + 8 * 8;
  static_assert(EPI <= PIPE, "the epilogue reuses the stage memory only");
  static constexpr int SMEM = END + 1024;  // + the slack of the 1024-byte base alignment
  // consumers of a stage: the K-warps, the S-warp, the V-warps
  static constexpr int EMPTY_COUNT = KQ + 1 + VW;
};

template <int D, int KF, int VF>
__global__ void __launch_bounds__(WsGeo<D, KF, VF>::THREADS, 2)
    attn_ws_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TmaSet maps) {
  static_assert(KF == QPS_FMT_Q8_0 && VF == QPS_FMT_TQ3, "the warp-specialized kernel covers q8_0 K / TQ3 V");
  using W = WsGeo<D, KF, VF>;
  using G = typename W::G;
  constexpr int TT = W::TT, MT = D / 16, NS = W::NS, KW = W::KW, VW = W::VW, KQ = W::KQ;
  constexpr int KB = D / 32 / KQ;  // q8_0 blocks per K-warp
  constexpr int MTV = MT / VW;  // m-tiles per V-warp
  static_assert(D == 128 * VW, "a V-warp owns 128 contiguous columns, 16 per lane group");
  static_assert(G::K_RB == D && G::V_RB == D / 4 && G::V_ARB == D / 8, "q8_0 K / TQ3 V planes");
  constexpr float LOG2E = 1.4426950408889634f;
  constexpr uint32_t ALL = 0xffffffffu;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);

  // programmatic dependent launch: nothing in global memory is touched before this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, head = blockIdx.y, bz = blockIdx.z;
  const int nrows = p.rows_per_cta;  // <= 8 (checked at launch)
  const int64_t t0 = p.begin + (int64_t)split * p.chunk;
  const int64_t t1 = min(p.end, t0 + p.chunk);
  const int part = p.part_offset + split;

  auto out_row = [&](int rr) -> int64_t {
    const int h = head * p.group + rr % p.group;
    if (p.shared) return (int64_t)(rr / p.group) * p.hq + h;
    return ((int64_t)bz * p.n_q + rr / p.group) * p.hq + h;
  };

  if (t0 >= t1) {  // an empty chunk: O = 0, lse = -inf
    for (int idx = threadIdx.x; idx < nrows * D; idx += W::THREADS) {
      const int r = idx / D, dd = idx % D;
      const int64_t row = out_row(r);
      if (!in_bounds(part < p.parts_cap && row >= 0 && row < p.rows_total, p.err)) continue;
      p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = 0.f;
      if (dd == 0) p.lse_parts[(int64_t)part * p.rows_total + row] = -INFINITY;
    }
    return;
  }

  const uint32_t bar_full = smem_addr(smem + W::FULL_OFF);
  const uint32_t bar_sready = smem_addr(smem + W::SREADY_OFF);
  const uint32_t bar_pready = smem_addr(smem + W::PREADY_OFF);
  const uint32_t bar_empty = smem_addr(smem + W::EMPTY_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + W::FLAG_OFF);
  float* ks_state = reinterpret_cast<float*>(smem + W::KS_OFF);  // [KW][8] max (log2), then [KW][8] sum
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, G::ARRIVALS);
      mbar_init(bar_sready + 8 * s, KQ);
      mbar_init(bar_pready + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, W::EMPTY_COUNT);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    *abort_flag = 0;
  }
  __syncthreads();

  const int64_t tile0 = t0 & ~(int64_t)(TT - 1);
  const int ntiles = (int)((t1 - tile0 + TT - 1) / TT);
  auto aborted = [&]() { return __shfl_sync(ALL, lane == 0 ? *abort_flag : 0, 0) != 0; };
  int failed = 0;  // this warp's bounded wait gave up (warp-uniform)
  // the first give-up of the launch records where it happened; every give-up stops the
  // producer through the CTA's flag
  auto give_up = [&](int t, int issued) {
    failed = 1;
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
      if (atomicAdd(p.err + 1, 1u) == 0) {
        unsigned int* r = p.err + 2;
        r[0] = blockIdx.x;
        r[1] = blockIdx.y;
        r[2] = blockIdx.z;
        r[3] = warp;
        r[4] = t;
        r[5] = issued;
        r[6] = ntiles;
        r[7] = (unsigned)(t1 - t0);
      }
    }
  };

  if (warp == 0) {
    // ---- producer: the CTA's tiles into the stage ring ----------------------------------
    const uint8_t* va2 = reinterpret_cast<const uint8_t*>(p.v.aux2) +
                         ((p.shared ? 0 : (int64_t)bz * p.v.batch) + (int64_t)head * p.v.head) * G::V_A2RB;
    const uint8_t* v_aux2 = reinterpret_cast<const uint8_t*>(p.v.aux2);
    const uint8_t* safe = reinterpret_cast<const uint8_t*>(p.k.data);
    const int bcoord = p.shared ? 0 : bz;
    int n_issued = 0;
    int s = 0;         // stage of tile t: t mod NS
    uint32_t ph = 0;   // its use: (t / NS) mod 2
    for (int t = 0; t < ntiles; ++t, s = s + 1 == NS ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
      if (t >= NS && !mbar_wait(bar_empty + 8 * s, ph ^ 1u)) {
        give_up(t, n_issued);
        break;
      }
      if (aborted()) break;
      uint8_t* st = smem + s * W::STAGE;
      const int64_t tb = tile0 + (int64_t)t * TT;
      const uint32_t bar = bar_full + 8 * s;
      if (lane == 0) mbar_expect_tx(bar, G::TX);
      __syncwarp();
      fence_proxy_async();
      // one tensor-map box per lane: K codes, V 2-bit plane, K scales, V sign plane
      constexpr int NKB = G::PK::NB, NVB = G::PV::NB;
      static_assert(G::PKA::TMA && G::PVA::TMA && NKB + NVB + 2 <= 32, "box layout of the q8_0 / TQ3 stage");
      if (lane < NKB + NVB + 2) {
        const TensorMap* mp = &maps.k;
        int dst = G::K_OFF + lane * (TT * G::PK::IB), x = lane * G::PK::IB;
        int rb = G::K_RB, ib = G::PK::IB;
        if (lane >= NKB && lane < NKB + NVB) {
          mp = &maps.v;
          dst = G::V_OFF + (lane - NKB) * (TT * G::PV::IB);
          x = (lane - NKB) * G::PV::IB;
          rb = G::V_RB;
          ib = G::PV::IB;
        } else if (lane == NKB + NVB) {
          mp = &maps.ka;
          dst = G::KA_OFF;
          x = 0;
          rb = G::K_ARB;
          ib = G::PKA::IB;
        } else if (lane == NKB + NVB + 1) {
          mp = &maps.va;
          dst = G::VA_OFF;
          x = 0;
          rb = G::V_ARB;
          ib = G::PVA::IB;
        }
        if (in_bounds(x + ib <= rb && tb >= 0 && head < p.hkv && bcoord < (p.shared ? 1 : p.batch) &&
                          dst + TT * ib <= G::STAGE && s * W::STAGE + G::STAGE <= W::PIPE,
                      p.err))
          tma_load_4d(smem_addr(st) + dst, mp, x, (int)tb, head, bcoord, bar);
        (void)rb;
        (void)ib;
      }
      // the norms (2 bytes per token) by zero-filling cp.async; rows past kv_end read as 0
      const int valid = (int)max((int64_t)0, min((int64_t)TT, p.end - tb));
      stage_flat_zfill<G::PVA2::BYTES>(st + G::VA2_OFF, va2 + tb * G::V_A2RB, valid * G::V_A2RB, lane, safe,
                                       v_aux2, v_aux2 + p.v_rows * G::V_A2RB, p.err);
      cp_async_arrive_noinc(bar);
      n_issued = t + 1;
    }
    cp_async_wait<0>();
    if (failed || aborted()) {
      // the consumers may have stopped early: wait (bounded) for the copies of the last
      // NS issued tiles, so that none lands after the CTA has left its shared memory
      for (int t = max(0, n_issued - NS); t < n_issued; ++t) mbar_wait(bar_full + 8 * (t % NS), (uint32_t)((t / NS) & 1));
    }
  } else if (warp <= KQ) {
    // ---- K-warps: partial S^T = K Q^T over this warp's quarter of head_dim ---------------
    const int kq = warp - 1;
    const int ks_lane = g * (D / 32);
    // the query fragments (B operand of S^T) of row g for this quarter, in registers, in
    // the q8_0 order: lane column c owns d in [32 j + 8 c, +8) of block j
    uint32_t qb[2 * KB][2];
    {
      bool ok = g < nrows;
      const __half* qrow = p.q;
      if (ok) {
        const int h = head * p.group + g % p.group;
        qrow = p.shared ? p.q + (int64_t)(g / p.group) * p.q_bstride + (int64_t)h * D
                        : p.q + (int64_t)bz * p.q_bstride + ((int64_t)(g / p.group) * p.hq + h) * D;
        ok = in_bounds((int64_t)(qrow - p.q) + D <= p.q_elems, p.err);
      }
#pragma unroll
      for (int kk = 0; kk < 2 * KB; ++kk) {
        const int d0 = 32 * (KB * kq + (kk >> 1)) + 8 * c + 4 * (kk & 1);
        qb[kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qrow + d0) : 0u;
        qb[kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qrow + d0 + 2) : 0u;
      }
    }
    int s = 0;
    uint32_t ph = 0;
    for (int t = 0; t < ntiles; ++t, s = s + 1 == NS ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
      if (aborted()) break;
      if (!mbar_wait(bar_full + 8 * s, ph)) {
        give_up(t, -1);
        break;
      }
      __syncwarp();
      const uint8_t* st = smem + s * W::STAGE;
      // codes -> exact f16, two MMAs per 32-value block, the block's fp32 scale applied
      // to its partial sums
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint8_t* kc = st + G::K_OFF;
      const __half* ks = reinterpret_cast<const __half*>(st + G::KA_OFF) + ks_lane;
      // this quarter's four block scales of tokens g and g + 8: one 8-byte load each
      static_assert(KB == 4, "four q8_0 blocks per K-warp");
      float sc[2][KB];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint2 s4 = *reinterpret_cast<const uint2*>(ks + u * 8 * (D / 32) + KB * kq);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&s4.x));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&s4.y));
        sc[u][0] = f01.x;
        sc[u][1] = f01.y;
        sc[u][2] = f23.x;
        sc[u][3] = f23.y;
      }
#pragma unroll
      for (int jj = 0; jj < KB; ++jj) {
        const int j = KB * kq + jj;
        const int x = 2 * j + (c >> 1), sub = 8 * (c & 1);
        const uint2 wg = *reinterpret_cast<const uint2*>(kc + soff<G::PK::IB, G::PK::SW, TT>(g, 16 * x + sub));
        const uint2 wg8 = *reinterpret_cast<const uint2*>(kc + soff<G::PK::IB, G::PK::SW, TT>(g + 8, 16 * x + sub));
        uint32_t a0[4], a1[4];
        i8x4_to_h2x2(wg.x, a0[0], a0[2]);
        i8x4_to_h2x2(wg8.x, a0[1], a0[3]);
        i8x4_to_h2x2(wg.y, a1[0], a1[2]);
        i8x4_to_h2x2(wg8.y, a1[1], a1[3]);
        const float sg = sc[0][jj], sg8 = sc[1][jj];
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(acc, a0, qb[2 * jj][0], qb[2 * jj][1]);
        mma16816(acc, a1, qb[2 * jj + 1][0], qb[2 * jj + 1][1]);
        sacc[0] = fmaf(sg, acc[0], sacc[0]);
        sacc[1] = fmaf(sg, acc[1], sacc[1]);
        sacc[2] = fmaf(sg8, acc[2], sacc[2]);
        sacc[3] = fmaf(sg8, acc[3], sacc[3]);
      }
      reinterpret_cast<float4*>(smem + W::SP_OFF + s * W::SP_BYTES)[kq * 32 + lane] =
          make_float4(sacc[0], sacc[1], sacc[2], sacc[3]);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_sready + 8 * s);
        mbar_arrive(bar_empty + 8 * s);  // done with the stage's K planes
      }
    }
  } else if (warp == W::S_WARP) {
    // ---- the S-warp: logits, online softmax, P to the V-warps ---------------------------
    const float qk_scale = p.scale;
    const float cap = p.softcap;
    const float cap_k = cap > 0.f ? 2.f * LOG2E / cap : 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows 2c, 2c + 1 (log2 domain)
    int s = 0;
    uint32_t par = 0;
    for (int t = 0; t < ntiles; ++t, s = s + 1 == NS ? 0 : s + 1, par ^= s == 0 ? 1u : 0u) {
      if (aborted()) break;
      if (!mbar_wait(bar_sready + 8 * s, par)) {
        give_up(t, -3);
        break;
      }
      mbar_wait(bar_full + 8 * s, par);  // complete already: makes the tile's norms visible here
      __syncwarp();
      const uint8_t* st = smem + s * W::STAGE;
      const int64_t tb = tile0 + (int64_t)t * TT;
      const float4* sp = reinterpret_cast<const float4*>(smem + W::SP_OFF + s * W::SP_BYTES) + lane;
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < KQ; ++q) {
        const float4 v = sp[q * 32];
        sacc[0] += v.x;
        sacc[1] += v.y;
        sacc[2] += v.z;
        sacc[3] += v.w;
      }
      // logits (scale, softcap, mask: tokens g and g + 8 of the tile), online softmax
      const int64_t tg = tb + g;
      const bool in_g = tg >= t0 && tg < t1, in_g8 = tg + 8 >= t0 && tg + 8 < t1;
      const __half* nrm = reinterpret_cast<const __half*>(st + G::NORM_OFF);
      const float ng = __half2float(nrm[g]), ng8 = __half2float(nrm[g + 8]);
      float xv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sacc[e] * qk_scale;
        if (cap > 0.f) v = softcap_tanh(v, cap, cap_k);
        xv[e] = v * LOG2E;
      }
      if (!in_g) xv[0] = xv[1] = -INFINITY;
      if (!in_g8) xv[2] = xv[3] = -INFINITY;
      float mx0 = fmaxf(xv[0], xv[2]), mx1 = fmaxf(xv[1], xv[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(ALL, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(ALL, mx1, off));
      }
      // the reference maximum is raised only when the tile's exceeds it by more than 8
      // (log2 units) while the tile's norms stay <= 255, so P x norm stays finite in
      // fp16 (else by any amount): most tiles then need no rescale of O in the V-warps
      float nmx = fmaxf(fabsf(ng), fabsf(ng8));
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) nmx = fmaxf(nmx, __shfl_xor_sync(ALL, nmx, off));
      const float lazy = nmx <= 255.f ? 8.f : 0.f;
      const float mn0 = mx0 - m0 > lazy ? mx0 : m0, mn1 = mx1 - m1 > lazy ? mx1 : m1;  // (both -inf: NaN, keeps m)
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float cr0 = exp2f(m0 - ms0), cr1 = exp2f(m1 - ms1);
      const float p0 = exp2f(xv[0] - ms0), p1 = exp2f(xv[1] - ms1);
      const float p2 = exp2f(xv[2] - ms0), p3 = exp2f(xv[3] - ms1);
      l0 = l0 * cr0 + (p0 + p2);
      l1 = l1 * cr1 + (p1 + p3);
      m0 = mn0;
      m1 = mn1;
      // P^T in the B-operand layout, each token's V norm folded in; the rows' rescale
      uint8_t* pbs = smem + W::PB_OFF + s * W::PB_BYTES;
      reinterpret_cast<uint2*>(pbs)[lane] =
          make_uint2(movmatrix_t(pack_h2(p0 * ng, p1 * ng)), movmatrix_t(pack_h2(p2 * ng8, p3 * ng8)));
      if (g == 0) {
        reinterpret_cast<float*>(pbs + 256)[2 * c] = cr0;
        reinterpret_cast<float*>(pbs + 256)[2 * c + 1] = cr1;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_pready + 8 * s);
        mbar_arrive(bar_empty + 8 * s);  // done with the stage's norms and partial logits
      }
    }
    // the state for the epilogue: the row maximum and the row sum over the tokens
    l0 += __shfl_xor_sync(ALL, l0, 4);
    l0 += __shfl_xor_sync(ALL, l0, 8);
    l0 += __shfl_xor_sync(ALL, l0, 16);
    l1 += __shfl_xor_sync(ALL, l1, 4);
    l1 += __shfl_xor_sync(ALL, l1, 8);
    l1 += __shfl_xor_sync(ALL, l1, 16);
    if (g == 0) {
      ks_state[2 * c] = m0;
      ks_state[2 * c + 1] = m1;
      ks_state[KW * 8 + 2 * c] = l0;
      ks_state[KW * 8 + 2 * c + 1] = l1;
    }
  }

  // ---- V-warps: O^T += V^T P^T over a quarter of the columns ----------------------------
  float o[KW][MTV][4];
#pragma unroll
  for (int q = 0; q < KW; ++q)
#pragma unroll
    for (int i = 0; i < MTV; ++i) o[q][i][0] = o[q][i][1] = o[q][i][2] = o[q][i][3] = 0.f;
  const int vw = warp - 1 - W::S_WARP;
  if (warp > W::S_WARP) {
    const uint32_t tq_lo = pack_h2(p.tq_levels[4], p.tq_levels[5]);
    const uint32_t tq_hi = pack_h2(p.tq_levels[6], p.tq_levels[7]);
    // stage offsets of tokens 2c, 2c + 1, 2c + 8, 2c + 9: the 2-bit codes (4 bytes) and
    // the sign bits (2 bytes) of this lane group's columns 128 vw + 16 g .. + 15
    const int col0 = 128 * vw + 16 * g;
    int off2[4], offs[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tk = 2 * c + (u & 1) + 8 * (u >> 1);
      off2[u] = G::V_OFF + soff<G::PV::IB, G::PV::SW, TT>(tk, col0 / 4);
      offs[u] = G::VA_OFF + soff<G::PVA::IB, G::PVA::SW, TT>(tk, col0 / 8);
      in_bounds(off2[u] >= G::V_OFF && off2[u] + 4 <= G::V_OFF + G::PV::BYTES && offs[u] >= G::VA_OFF &&
                    offs[u] + 2 <= G::VA_OFF + G::PVA::BYTES,
                p.err);
    }
    static_assert(KW == 1, "one softmax state");
    constexpr int q = 0;
    int s = 0;
    uint32_t par = 0;
    for (int t = 0; t < ntiles; ++t, s = s + 1 == NS ? 0 : s + 1, par ^= s == 0 ? 1u : 0u) {
      if (aborted()) break;
      if (!mbar_wait(bar_pready + 8 * s, par)) {
        give_up(t, -2);
        break;
      }
      mbar_wait(bar_full + 8 * s, par);  // complete already: makes the tile's bytes visible here
      __syncwarp();
      const uint8_t* st = smem + s * W::STAGE;
      const uint8_t* pbs = smem + W::PB_OFF + s * W::PB_BYTES;
      const uint2 pb = reinterpret_cast<const uint2*>(pbs)[lane];
      const float cr0 = reinterpret_cast<const float*>(pbs + 256)[2 * c];
      const float cr1 = reinterpret_cast<const float*>(pbs + 256)[2 * c + 1];
      if (__any_sync(ALL, cr0 != 1.f || cr1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < MTV; ++i) {
          o[q][i][0] *= cr0;
          o[q][i][1] *= cr1;
          o[q][i][2] *= cr0;
          o[q][i][3] *= cr1;
        }
      }
      uint32_t L[4], H[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        L[u] = *reinterpret_cast<const uint32_t*>(st + off2[u]);
        H[u] = *reinterpret_cast<const uint16_t*>(st + offs[u]);
      }
      const uint32_t hab[2] = {H[0] | (H[1] << 16), H[2] | (H[3] << 16)};  // token a bits 0..15, b 16..31
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t ysel = h ? 0x7362u : 0x5140u;
        const uint32_t y[2] = {__byte_perm(L[0], L[1], ysel), __byte_perm(L[2], L[3], ysel)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e0 = j + 8 * h, e1 = e0 + 4;
          uint32_t a[4];
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            const uint32_t sel = ((y[pr] >> (2 * j)) & 0x03030303u) * 0x22u + 0x10101010u;
            const uint32_t mg0 = __byte_perm(tq_lo, tq_hi, sel);
            const uint32_t mg1 = __byte_perm(tq_lo, tq_hi, sel >> 16);
            a[2 * pr] = mg0 | (~(hab[pr] << (15 - e0)) & 0x80008000u);  // a clear sign bit: negative level
            a[2 * pr + 1] = mg1 | (~(hab[pr] << (15 - e1)) & 0x80008000u);
          }
          mma16816(o[q][2 * j + h], a, pb.x, pb.y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
  }

  // every warp is past its loop; a CTA in which any wait gave up writes no partial
  if (__syncthreads_or(failed)) return;
  asm volatile("griddepcontrol.launch_dependents;" :::);

  // ---- epilogue: merge the K-warps' states, inverse rotation, the partial -------------
  constexpr int FS = W::FS;
  float* fin = reinterpret_cast<float*>(smem + W::FIN_OFF);  // [8][FS], column x at fcol(x)
  auto fcol = [](int x) { return x + (x >> 4); };
  float* wk = reinterpret_cast<float*>(smem + W::WK_OFF);    // [KW][8] state weights
  float* rmx = reinterpret_cast<float*>(smem + W::RMX_OFF);
  float* rden = reinterpret_cast<float*>(smem + W::RDEN_OFF);
  int64_t* orow = reinterpret_cast<int64_t*>(smem + W::OROW_OFF);
  if (threadIdx.x < 8) {
    const int r = threadIdx.x;
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < KW; ++q) mx = fmaxf(mx, ks_state[q * 8 + r]);
    float den = 0.f;
#pragma unroll
    for (int q = 0; q < KW; ++q) {
      const float mq = ks_state[q * 8 + r];
      const float f = (mx != -INFINITY && mq != -INFINITY) ? exp2f(mq - mx) : 0.f;
      wk[q * 8 + r] = f;
      den += ks_state[KW * 8 + q * 8 + r] * f;
    }
    rmx[r] = mx;
    rden[r] = den;
    if (r < nrows) orow[r] = out_row(r);
  }
  __syncthreads();
  // Inverse rotation x = s1 .* blockdiag(H_G)(s2 .* y) / sqrt(D G).  Lane group g of
  // V-warp v holds columns 128 v + 16 g + x (x = 0..15) of rows 2c and 2c + 1, so the
  // butterflies of span 1..8 pair values of one lane, spans 16..64 pair lane groups (lane
  // bits 2..4: shuffles) and spans 128, 256 pair V-warps (through shared memory).
  if (warp > W::S_WARP) {
    float v[2][16];  // [row parity][x]
#pragma unroll
    for (int i = 0; i < MTV; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // m-tile i = 2 j + h holds columns j + 8 h (e < 2) and j + 8 h + 4 of the lane's 16
        const int x = ((i >> 1) & 3) + 8 * (i & 1) + 4 * (e >> 1);
        const int row = 2 * c + (e & 1), col = 128 * vw + 16 * g + x;
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < KW; ++q) acc += o[q][i][e] * wk[q * 8 + row];
        if ((p.vsigns2[col >> 5] >> (col & 31)) & 1u) acc = -acc;  // the rotation's second sign vector
        v[e & 1][x] = acc;
      }
    }
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {  // spans 1..8: inside the lane
      if (h >= p.vblock) break;          // (uniform)
#pragma unroll
      for (int rp = 0; rp < 2; ++rp)
#pragma unroll
        for (int x = 0; x < 16; ++x)
          if (!(x & h)) {
            const float a = v[rp][x], b = v[rp][x + h];
            v[rp][x] = a + b;
            v[rp][x + h] = a - b;
          }
    }
#pragma unroll
    for (int h = 16; h < 128; h <<= 1) {  // spans 16..64: lane groups g ^ (h / 16)
      if (h >= p.vblock) break;
      const int mask = 4 * (h / 16);
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int rp = 0; rp < 2; ++rp)
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float other = __shfl_xor_sync(ALL, v[rp][x], mask, 32);
          v[rp][x] = upper ? other - v[rp][x] : v[rp][x] + other;
        }
    }
#pragma unroll
    for (int rp = 0; rp < 2; ++rp)
#pragma unroll
      for (int x = 0; x < 16; ++x) fin[(2 * c + rp) * FS + fcol(128 * vw + 16 * g + x)] = v[rp][x];
  }
  // spans 128 and 256: the V-warps' column blocks v ^ 1 and v ^ 2, through shared memory
  for (int h = 128; h < D; h <<= 1) {
    if (h >= p.vblock) break;  // (uniform over the CTA)
    __syncthreads();
    float nv[2][16];
    if (warp > W::S_WARP) {
      const bool upper = (vw & (h / 128)) != 0;
#pragma unroll
      for (int rp = 0; rp < 2; ++rp)
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int col = 128 * vw + 16 * g + x;
          const float mine = fin[(2 * c + rp) * FS + fcol(col)];
          const float other = fin[(2 * c + rp) * FS + fcol(col ^ h)];
          nv[rp][x] = upper ? other - mine : mine + other;
        }
    }
    __syncthreads();
    if (warp > W::S_WARP) {
#pragma unroll
      for (int rp = 0; rp < 2; ++rp)
#pragma unroll
        for (int x = 0; x < 16; ++x) fin[(2 * c + rp) * FS + fcol(128 * vw + 16 * g + x)] = nv[rp][x];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * D; idx += W::THREADS) {
    const int r = idx / D, dd = idx % D;
    const float den = rden[r];
    float val = fin[r * FS + fcol(dd)] * p.v_out_scale;
    if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) val = -val;
    const int64_t row = orow[r];
    const bool empty = !(den > 0.f);
    if (!in_bounds(part < p.parts_cap && row >= 0 && row < p.rows_total, p.err)) continue;
    p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = empty ? 0.f : val / den;
    if (dd == 0)
      p.lse_parts[(int64_t)part * p.rows_total + row] = empty ? -INFINITY : (rmx[r] + log2f(den)) * 0.6931471805599453f;
  }
}

// Whether the warp-specialized kernel takes these arguments: head_dim 512, q8_0 K, TQ3 V,
// single-token decode without the causal limit, up to 8 query rows per KV head.
inline bool ws_takes(const AttnParams& p) {
  return p.d == 512 && p.kfmt == QPS_FMT_Q8_0 && p.vfmt == QPS_FMT_TQ3 && !p.causal && p.n_q == 1 &&
         p.rows_per_cta <= 8;
}

template <int D, int KF, int VF>
qps_status launch_ws_t(const AttnParams& p, cudaStream_t s) {
  using W = WsGeo<D, KF, VF>;
  using G = typename W::G;
  constexpr size_t smem = W::SMEM;
  static_assert(2 * (smem + 1024) <= 228 * 1024, "two CTAs per SM");
  TmaSet maps;
  std::memset(&maps, 0, sizeof(maps));
  const int nb = p.shared ? 1 : p.batch;
  if (!encode_plane_map(&maps.k, p.k.data, G::K_RB, p.end, p.hkv, p.k.head, nb, p.k.batch, G::PK::IB, G::PK::SW, W::TT) ||
      !encode_plane_map(&maps.v, p.v.data, G::V_RB, p.end, p.hkv, p.v.head, nb, p.v.batch, G::PV::IB, G::PV::SW, W::TT) ||
      !encode_plane_map(&maps.ka, p.k.aux, G::K_ARB, p.end, p.hkv, p.k.head, nb, p.k.batch, G::PKA::IB, G::PKA::SW, W::TT) ||
      !encode_plane_map(&maps.va, p.v.aux, G::V_ARB, p.end, p.hkv, p.v.head, nb, p.v.batch, G::PVA::IB, G::PVA::SW, W::TT))
    return QPS_ERR_CUDA;
  auto kern = attn_ws_kernel<D, KF, VF>;
  // as the per-warp kernel: enough shared memory that a third CTA cannot join an SM
  // early under programmatic launch
  constexpr size_t kSmPerSm = 228 * 1024, kReserved = 1024;
  constexpr size_t smem_floor = kSmPerSm / 3 - kReserved + 1;
  constexpr size_t smem_launch = smem > smem_floor ? smem : smem_floor;
  static_assert(2 * (smem_launch + kReserved) <= kSmPerSm, "the padding must not cost a CTA per SM");
  QPS_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_launch));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_split, p.hkv, p.shared ? 1 : p.batch);
  cfg.blockDim = dim3(W::THREADS);
  cfg.dynamicSmemBytes = smem_launch;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  QPS_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p, maps));
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

}  // namespace ws
}  // namespace qps
