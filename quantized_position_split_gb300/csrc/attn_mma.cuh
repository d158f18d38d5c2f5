// Split-KV decode attention on tensor cores (mma.sync m16n8k16, f16 x f16 -> f32).
//
// One part of the position-split decode of "F5 M7 — Rolling KV: position-windowed KV
// residency" (section "Implementation decomposition, refined (S1 -> S2 -> S3)", item
// S2): every split chunk of positions yields a normalised output and its log-sum-exp.
// K / V are dequantised in registers on their way into the tensor-core operands; a
// TurboQuant V (TQ2 / TQ3 / TQ4) is read as centroid x norm in the rotated domain and the
// output is inverse-rotated once ("F5 M6 — PolyKV (shared compressed KV pool)", sections
// "S2 perf-path Level B" and "S2 — TurboQuant tier family").
//
// Formulation (query rows on the narrow N = 8 side, so a GQA group of 5..8 rows wastes
// nothing):   S^T[t][r] = sum_d K[t][d] Q[r][d]       (A = K tile, B = Q^T)
//             O^T[d][r] = sum_t V^T[d][t] P^T[t][r]   (A = V^T tile, B = P^T)
// P leaves the S^T accumulator layout and enters the B-operand layout through one
// movmatrix transpose per 8x8 block.
//
// Exactness: q8_0 K codes are exact in f16; each 32-value block is accumulated
// separately and multiplied by its fp32 scale afterwards, so the logits carry only
// fp32 rounding.  TurboQuant levels are fp16-exact by construction.  P (in [0, 1]) and a
// q8_0 V value (code x scale) are rounded once to fp16.
//
// Data movement: the KV planes of a (KV head, batch entry) must be token-contiguous
// (tok_stride == 1).  Each warp runs a private pipeline of STAGES tiles of 16 tokens
// over its own share of the chunk's tiles (tiles w, w + NW, ...): every plane of a tile
// arrives by tensor-map (TMA) boxes or, for planes under 16 bytes per token, by
// zero-filling cp.async, all completing on the stage's mbarrier; waits are bounded and
// report through a device error word instead of hanging.  Rows past the view's end
// arrive as zeros; tokens outside [t0, t1) are masked in the softmax.
#pragma once

#include <cstring>

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

// Register-only operations are plain asm so that the compiler may interleave them;
// shared-memory reads stay volatile behind the barrier waits.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte permute over {b, a} (bytes 0..7) with the selector's low four nibbles: bits 0..2
// of a nibble pick a source byte, bit 3 replicates that byte's top bit over the result
// byte instead of copying it.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
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

// Logit softcap c * tanh(x / c) through tanh(y) = 1 - 2 / (1 + e^(2y)), with the
// hardware base-2 exponential and reciprocal; k = 2 log2(e) / c.  Its absolute error
// is a few 1e-7 x c (the 1 - 2r cancellation near 0), and it saturates to +-c.
__device__ __forceinline__ float softcap_tanh(float x, float c, float k) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * k));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return fmaf(-2.f * c, r, c);
}

// ---- tile geometry ---------------------------------------------------------------
__host__ __device__ constexpr int align_to(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int min_i(int a, int b) { return a < b ? a : b; }

// One plane of a TT-token stage.  Planes of >= 16 bytes per token arrive as tensor-map
// boxes of [IB bytes][TT tokens] (IB = min(row bytes, 128)); the K / V value planes
// (and the TQ3 sign plane) use the hardware XOR swizzle that matches IB so that token
// rows read at the same column fall into different bank groups.  Smaller planes (fp16
// norms, q8_0 scales at head_dim <= 128) come by 16-byte cp.async.  Either way rows past
// the view's end arrive as zeros.
template <int RB, bool VALUES, int TT>
struct PlaneG {
  static constexpr bool TMA = RB >= 16;
  static constexpr int IB = min_i(RB, 128);
  static constexpr int NB = TMA ? RB / IB : 0;
  static constexpr int SW = (VALUES && TMA) ? (IB >= 128 ? 128 : IB >= 64 ? 64 : IB >= 32 ? 32 : 0) : 0;
  static constexpr int BYTES = TT * RB;
};

// Stage bytes of one CTA when CTAS CTAs share an SM's 228 KB.  Three CTAs: 228 KB / 3
// less 1 KB reserved per CTA, the 1024-byte alignment slack and up to 192 bytes of
// barriers leaves 75584 bytes for the stages and what sits beside them; 75392 keeps
// 192 more in hand.  Two CTAs: ~104 KB.
__host__ __device__ constexpr int stage_budget(int ctas) { return ctas >= 3 ? 75392 : 104 * 1024; }

// Query fragments kept in shared memory instead of registers: a TurboQuant K's rotated
// fragments (per n-tile, k-step and lane {hi b0, hi b1, lo b0, lo b1}: fp16 hi + lo = the
// fp32 value), and at head_dim 512 with a q8_0 K and a TQ3 / TQ2 V the plain fragments
// {b0, b1}: 64 registers the accumulators and the V decode use better (the q8_0-K /
// TQ3-V window 67.9 -> 66.0 us), in 8 KB that still leave two CTAs per SM (not so with
// a TQ4 V, whose two stages already fill it, or an fp16 K, which runs one CTA per SM).
template <int D, int KF, int VF>
__host__ __device__ constexpr bool q_in_smem() {
  return is_tq(KF) || (D >= 512 && KF == QPS_FMT_Q8_0 && (VF == QPS_FMT_TQ3 || VF == QPS_FMT_TQ2));
}
template <int D, int KF, int VF, int NTW>
__host__ __device__ constexpr int qf_bytes() {
  return is_tq(KF) ? NTW * (D / 16) * 32 * 16 : q_in_smem<D, KF, VF>() ? NTW * (D / 16) * 32 * 8 : 0;
}

template <int D, int KF, int VF, int TT_, int CTAS_, int RES_>
struct GeoT {
  static constexpr int CTAS = CTAS_;
  // K data: fp16 values, q8_0 codes, TQ2 / TQ3 2-bit or TQ4 4-bit fields; K aux: q8_0
  // scales, the TQ3 sign plane or the TQ2 / TQ4 norms; K aux2: the TQ3 norms
  static constexpr int K_RB = KF == QPS_FMT_F16 ? 2 * D : KF == QPS_FMT_Q8_0 ? D : KF == QPS_FMT_TQ4 ? D / 2 : D / 4;
  static constexpr int K_ARB = KF == QPS_FMT_Q8_0 ? D / 16 : KF == QPS_FMT_TQ3 ? D / 8 : is_tq(KF) ? 2 : 0;
  static constexpr int K_A2RB = KF == QPS_FMT_TQ3 ? 2 : 0;
  // V data: fp16 values, q8_0 codes, TQ2 / TQ3 2-bit fields or TQ4 4-bit fields; V aux:
  // q8_0 scales, the TQ3 sign plane or the TQ2 / TQ4 norms; V aux2: the TQ3 norms
  static constexpr int V_RB = VF == QPS_FMT_F16 ? 2 * D : VF == QPS_FMT_Q8_0 ? D : VF == QPS_FMT_TQ4 ? D / 2 : D / 4;
  static constexpr int V_ARB = VF == QPS_FMT_Q8_0 ? D / 16 : VF == QPS_FMT_TQ3 ? D / 8 : is_tq(VF) ? 2 : 0;
  static constexpr int V_A2RB = VF == QPS_FMT_TQ3 ? 2 : 0;
  static constexpr int TT = TT_;
  static constexpr int SUB = TT / 16;
  using PK = PlaneG<K_RB, true, TT>;
  using PKA = PlaneG<K_ARB, KF == QPS_FMT_TQ3, TT>;  // TQ3 sign planes are read like values
  using PKA2 = PlaneG<K_A2RB, false, TT>;
  using PV = PlaneG<V_RB, true, TT>;
  using PVA = PlaneG<V_ARB, VF == QPS_FMT_TQ3, TT>;
  using PVA2 = PlaneG<V_A2RB, false, TT>;
  // swizzled planes first (each on a 1024-byte boundary), then the others (128-byte)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = align_to(K_OFF + PK::BYTES, 1024);
  static constexpr int END_V = V_OFF + PV::BYTES;
  static constexpr int KA_SW_OFF = align_to(END_V, 1024);
  static constexpr int END_KA_SW = PKA::SW ? KA_SW_OFF + PKA::BYTES : END_V;
  static constexpr int VA_SW_OFF = align_to(END_KA_SW, 1024);
  static constexpr int END_VA_SW = PVA::SW ? VA_SW_OFF + PVA::BYTES : END_KA_SW;
  static constexpr int KA_PL_OFF = align_to(END_VA_SW, 128);
  static constexpr int END_KA_PL = PKA::SW ? KA_PL_OFF : KA_PL_OFF + PKA::BYTES;
  static constexpr int VA_PL_OFF = align_to(END_KA_PL, 128);
  static constexpr int END_VA_PL = PVA::SW ? VA_PL_OFF : VA_PL_OFF + PVA::BYTES;
  static constexpr int KA_OFF = PKA::SW ? KA_SW_OFF : KA_PL_OFF;
  static constexpr int VA_OFF = PVA::SW ? VA_SW_OFF : VA_PL_OFF;
  static constexpr int KA2_OFF = align_to(END_VA_PL, 128);
  static constexpr int VA2_OFF = align_to(KA2_OFF + PKA2::BYTES, 128);
  static constexpr int KNORM_OFF = KF == QPS_FMT_TQ3 ? KA2_OFF : KA_OFF;  // TurboQuant K norms
  static constexpr int NORM_OFF = VF == QPS_FMT_TQ3 ? VA2_OFF : VA_OFF;   // TurboQuant V norms
  static constexpr int STAGE = align_to(VA2_OFF + PVA2::BYTES, 1024);
  // bytes the tensor-map boxes of one tile deliver
  static constexpr int TX = PK::BYTES + (PKA::TMA ? PKA::BYTES : 0) + PV::BYTES + (PVA::TMA ? PVA::BYTES : 0);
  static_assert(!PKA2::TMA && !PVA2::TMA, "aux2 planes (norms) are staged by cp.async");
  static constexpr bool SMALL = (K_ARB > 0 && !PKA::TMA) || (V_ARB > 0 && !PVA::TMA) || K_A2RB > 0 || V_A2RB > 0;
  static constexpr int ARRIVALS = 1 + (SMALL ? 32 : 0);  // expect_tx + one per lane's cp.async
  // warps per CTA: 4, or 2 when two stages of 4 warps would not fit in shared memory
  static constexpr int NW = 4 * 2 * STAGE <= 200 * 1024 ? 4 : 2;
  // the stage budget of CTAS CTAs per SM, less RES_ bytes kept beside the stages
  static constexpr int STAGES_RAW = (stage_budget(CTAS) - RES_) / (NW * STAGE);
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 6 ? 6 : STAGES_RAW);
  static constexpr int PIPE = NW * STAGES * STAGE;
  static constexpr int BARS = PIPE;                   // mbarriers after the stages
  static constexpr int END = BARS + NW * STAGES * 8;  // end of the barriers
};

// Tokens per stage: two 16-token MMA sub-tiles (independent chains for latency hiding,
// one softmax update per 32 tokens) where registers allow (head_dim <= 128) and 4 warps
// x 2 stages of 32 tokens still fit the stage budget; else one.
template <int D, int KF, int VF, int CTAS, int RES>
constexpr int stage_tokens() {
  return (D <= 128 && 4 * 2 * GeoT<D, KF, VF, 32, CTAS, RES>::STAGE <= stage_budget(CTAS) - RES) ? 32 : 16;
}
template <int D, int KF, int VF, int NTW>
struct Geo : GeoT<D, KF, VF, stage_tokens<D, KF, VF, mma_ctas_per_sm(D, NTW, VF), qf_bytes<D, KF, VF, NTW>()>(),
                  mma_ctas_per_sm(D, NTW, VF), qf_bytes<D, KF, VF, NTW>()> {};

// Tensor maps of one launch, one per tensor-map plane (unused ones left empty).
struct TmaSet {
  TensorMap k, ka, v, va;
};

// Byte offset of (token row t, byte b) of a plane staged by tensor-map boxes of IB
// bytes with swizzle SW (the 16-byte chunk index XORed with row bits, as the hardware
// writes it into a 1024-byte aligned region).
template <int IB, int SW, int TT>
__device__ __forceinline__ int soff(int t, int b) {
  const int box = b / IB, w = b % IB;
  int chunk = w >> 4;
  if constexpr (SW == 128) chunk ^= (t & 7);
  else if constexpr (SW == 64) chunk ^= ((t >> 1) & 3);
  else if constexpr (SW == 32) chunk ^= ((t >> 2) & 1);
  return box * (TT * IB) + t * IB + (chunk << 4) + (w & 15);
}

// ---- asynchronous copies completing on per-stage mbarriers --------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const TensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
// One poll that suspends the warp (instead of spinning on issue slots) until the phase
// completes or a system-dependent time limit passes; waits are bounded by the global
// timer around it.  (With an explicit 1 ms suspend hint one poll returned after about
// 4 us on GB300, and the windows ran 0.3-1.2% slower than with the default limit.)
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with the given parity: false once `limit_ns` of the GPU's
// global timer have passed without it (the clock is read only after a first poll
// fails).  A tile copy lands in microseconds; the bound, one second, only has to end a
// wait that would otherwise never end.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 >= limit_ns) return false;
  }
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// A small plane's 16-token tile by 16-byte cp.async; bytes past `valid_bytes` are
// zero-filled without being read.  The checked build also tests each chunk's source
// against the plane's addressed bytes [lo, hi) and its destination against the stage
// region of BYTES bytes; a failing chunk reads nothing (zero-filled).
template <int BYTES>
__device__ __forceinline__ void stage_flat_zfill(uint8_t* dst, const uint8_t* src, int valid_bytes, int lane,
                                                 const uint8_t* safe, const uint8_t* lo, const uint8_t* hi,
                                                 unsigned int* err) {
  constexpr int CHUNKS = (BYTES + 15) / 16;
  static_assert(BYTES % 16 == 0, "small-plane stage regions are whole 16-byte chunks");
  const uint32_t base = smem_addr(dst);
  for (int ch = lane; ch < CHUNKS; ch += 32) {
    int nb = valid_bytes - ch * 16;
    nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
    if (nb > 0 && !in_bounds(src + ch * 16 >= lo && src + ch * 16 + nb <= hi, err)) nb = 0;
    cp_async16(base + ch * 16, nb > 0 ? (const void*)(src + ch * 16) : (const void*)safe, nb);
  }
  (void)lo;
  (void)hi;
}

// Output column (within a lane group's DT columns) of row g (hh = 0) or g + 8 (hh = 1)
// of the TQ2 / TQ3 PV m-tile i: word k = i / 8 covers 16 columns, its m-tile 2j + h takes
// columns j + 8h and j + 8h + 4 (DT = 8: one half-word, m-tile j takes j and j + 4).
template <int DT>
__host__ __device__ constexpr int tq_col(int i, int hh) {
  return DT >= 16 ? 16 * (i >> 3) + ((i >> 1) & 3) + 8 * (i & 1) + 4 * hh : i + 4 * hh;
}

// Head-dim index of B-operand element e (0, 1: register b0; 2, 3: b1) of lane group c at
// k-step kk for a TurboQuant K.  Lane group c decodes the quarter [c D/4, (c+1) D/4) of
// every K row, in the order its decode produces: TQ4 four consecutive dims per k-step;
// TQ2 / TQ3 per 16-dim word w = kk / 4 the dims j, j + 4, j + 8, j + 12 (j = kk % 4).
template <int D, int KF>
__host__ __device__ constexpr int tqk_dim(int c, int kk, int e) {
  return c * (D / 4) + (KF == QPS_FMT_TQ4 ? 4 * kk + e : 16 * (kk >> 2) + 4 * e + (kk & 3));
}

// The warps' partial rows are merged through shared memory in a padded layout: one
// extra float after every D/8 columns (a lane group's output columns) and a row stride
// of D + 20 floats, so that the 32 lanes' stores of one accumulator register (rows 2c,
// 2c + 1, column base g * D/8 or 16 i + g) fall into 32 different banks.
template <int D>
__host__ __device__ constexpr int ow_stride() { return D + 20; }
template <int D>
__host__ __device__ constexpr int ow_col(int col) { return col + col / (D / 8); }

// ---- the kernel -------------------------------------------------------------------
// CAUSAL: the verify batch's causal limit (a separate instance, so that single-token
// decode compiles without it).
template <int D, int KF, int VF, int NTW, bool CAUSAL>
__global__ void __launch_bounds__(Geo<D, KF, VF, NTW>::NW * 32, Geo<D, KF, VF, NTW>::CTAS)
    attn_mma_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TmaSet maps) {
  using G = Geo<D, KF, VF, NTW>;
  constexpr int kWarps = G::NW;
  constexpr int ROWS = 8 * NTW;  // query rows per CTA
  constexpr int MT = D / 16;     // m-tiles of O^T, k-steps of S^T
  constexpr int KQ = KF == QPS_FMT_Q8_0 ? 1 : 0;
  constexpr bool VPERM = VF != QPS_FMT_F16;  // permuted output columns (see below)
  constexpr int DT = D / 8;                  // output columns per lane group (VPERM)
  constexpr int SUB = G::SUB, TT = G::TT;    // 16-token sub-tiles per stage, tokens per stage
  constexpr float LOG2E = 1.4426950408889634f;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // swizzled boxes need a 1024-byte aligned base
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t* pipe = smem;

  // Programmatic dependent launch: this grid may start while the previous kernel on
  // the stream finishes (the launch sets the attribute); everything it reads or writes
  // in global memory (q, the KV cache a preceding kernel may have appended to, the
  // partial outputs) is touched only after the previous grid has completed.  The next
  // grid is released once this CTA's tiles are done (after its main loop), so that its
  // CTAs do not sit resident beside this grid's for the whole stream.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  // the row groups of one (chunk, KV head) are adjacent CTAs, so they stream the same
  // KV rows at about the same time and all but the first read come from L2
  const int rgroups = (p.rows_per_cta + ROWS - 1) / ROWS;
  const int split = blockIdx.x / rgroups, rg = blockIdx.x % rgroups;
  const int head = blockIdx.y, bz = blockIdx.z;
  const int row0 = rg * ROWS;
  const int nrows = min(ROWS, p.rows_per_cta - row0);
  const int64_t t0 = p.begin + (int64_t)split * p.chunk;
  const int64_t t1 = min(p.end, t0 + p.chunk);
  const int part = p.part_offset + split;

  // CTA row rr: (batch entry, head) in a shared tile; (query token rr / group, head)
  // of batch entry bz otherwise
  auto out_row = [&](int rr) -> int64_t {
    const int h = head * p.group + rr % p.group;
    if (p.shared) return (int64_t)(rr / p.group) * p.hq + h;
    return ((int64_t)bz * p.n_q + rr / p.group) * p.hq + h;
  };

  if (t0 >= t1) {  // an empty chunk: O = 0, lse = -inf
    for (int idx = threadIdx.x; idx < nrows * D; idx += G::NW * 32) {
      const int r = idx / D, dd = idx % D;
      const int64_t row = out_row(row0 + r);
      if (!in_bounds(part < p.parts_cap && row >= 0 && row < p.rows_total, p.err)) continue;
      p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = 0.f;
      if (dd == 0) p.lse_parts[(int64_t)part * p.rows_total + row] = -INFINITY;
    }
    return;
  }

  // TurboQuant levels as fp16 (exact).  TQ3: magnitude m (level 4 + m) in bytes 2m,
  // 2m + 1 of {tq_lo, tq_hi}.  TQ2: the level of field f = (sign << 1) | m in bytes 2f,
  // 2f + 1 (levels 1, 0, 2, 3).  TQ4: the low bytes of the magnitudes m = 0..7 (levels
  // 8 + m) in {tq_lo, tq_hi}, their high bytes in {tq_lo2, tq_hi2}.
  uint32_t tq_lo = 0u, tq_hi = 0u, tq_lo2 = 0u, tq_hi2 = 0u;
  if constexpr (VF == QPS_FMT_TQ3) {
    tq_lo = pack_h2(p.tq_levels[4], p.tq_levels[5]);
    tq_hi = pack_h2(p.tq_levels[6], p.tq_levels[7]);
  } else if constexpr (VF == QPS_FMT_TQ2) {
    tq_lo = pack_h2(p.tq_levels[1], p.tq_levels[0]);
    tq_hi = pack_h2(p.tq_levels[2], p.tq_levels[3]);
  } else if constexpr (VF == QPS_FMT_TQ4) {
    const uint32_t m01 = pack_h2(p.tq_levels[8], p.tq_levels[9]), m23 = pack_h2(p.tq_levels[10], p.tq_levels[11]);
    const uint32_t m45 = pack_h2(p.tq_levels[12], p.tq_levels[13]), m67 = pack_h2(p.tq_levels[14], p.tq_levels[15]);
    tq_lo = __byte_perm(m01, m23, 0x6420);
    tq_hi = __byte_perm(m45, m67, 0x6420);
    tq_lo2 = __byte_perm(m01, m23, 0x7531);
    tq_hi2 = __byte_perm(m45, m67, 0x7531);
  }

  // ---- query fragments (B operand of S^T), one set per 8-row n-tile --------------
  constexpr bool QS = q_in_smem<D, KF, VF>();  // fragments in shared memory (see q_in_smem)
  constexpr int QMT = QS ? 1 : MT;
  uint32_t qb[NTW][QMT][2];
  // the CTA's give-up flag sits right after the barriers, the query fragments after it
  constexpr int ABORT_OFF = G::END;
  constexpr int QF_OFF = align_to(G::END + 16, 16);
  if constexpr (!is_tq(KF)) {
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    const int rr = row0 + nt * 8 + g;
    const bool valid = rr < p.rows_per_cta;
    const __half* qrow = nullptr;
    bool valid_q = valid;
    if (valid) {
      const int h = head * p.group + rr % p.group;
      qrow = p.shared ? p.q + (int64_t)(rr / p.group) * p.q_bstride + (int64_t)h * D
                      : p.q + (int64_t)bz * p.q_bstride + ((int64_t)(rr / p.group) * p.hq + h) * D;
      valid_q = in_bounds((int64_t)(qrow - p.q) + D <= p.q_elems, p.err);
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
      const uint32_t b0 = valid_q ? *reinterpret_cast<const uint32_t*>(qrow + d0) : 0u;
      const uint32_t b1 = valid_q ? *reinterpret_cast<const uint32_t*>(qrow + d1) : 0u;
      if constexpr (QS) {  // (each lane reads back only its own slots: no barrier needed)
        reinterpret_cast<uint2*>(smem + QF_OFF)[(nt * MT + kk) * 32 + lane] = make_uint2(b0, b1);
      } else {
        qb[nt][kk][0] = b0;
        qb[nt][kk][1] = b1;
      }
    }
  }
  }
  // query fragment {b0, b1} of n-tile nt, k-step kk (F16 / Q8_0 K)
  auto qfrag = [&](int nt, int kk) -> uint2 {
    if constexpr (QS) return reinterpret_cast<const uint2*>(smem + QF_OFF)[(nt * MT + kk) * 32 + lane];
    else return make_uint2(qb[nt][kk][0], qb[nt][kk][1]);
  };
  if constexpr (is_tq(KF)) {
    // A TurboQuant K is read in the rotated domain: q . x_hat = (n / sqrt(D)) (R q) . c, so
    // the CTA's query rows are rotated once, R q = s2 .* blockdiag(H_G)(s1 .* q) / sqrt(G),
    // in the stage memory (no tile is in flight yet), then split into fp16 hi + lo
    // fragments in the lane order of the K decode.
    static_assert(ROWS * D * 4 <= G::PIPE, "query rotation scratch must fit the stages");
    float* qs = reinterpret_cast<float*>(pipe);
    for (int idx = threadIdx.x; idx < ROWS * D; idx += G::NW * 32) {
      const int r = idx / D, dd = idx % D, rr = row0 + r;
      float v = 0.f;
      if (rr < p.rows_per_cta) {
        const int h = head * p.group + rr % p.group;
        const __half* qrow = p.shared ? p.q + (int64_t)(rr / p.group) * p.q_bstride + (int64_t)h * D
                                      : p.q + (int64_t)bz * p.q_bstride + ((int64_t)(rr / p.group) * p.hq + h) * D;
        if (in_bounds((int64_t)(qrow - p.q) + dd < p.q_elems, p.err)) v = __half2float(qrow[dd]);
        if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) v = -v;
      }
      qs[idx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int lh = 0; (1 << lh) < D; ++lh) {
      const int h = 1 << lh;
      if (h >= p.vblock) break;  // (uniform over the CTA)
      for (int pid = threadIdx.x; pid < ROWS * (D / 2); pid += G::NW * 32) {
        const int r = pid / (D / 2), j = pid % (D / 2);
        const int i = ((j >> lh) << (lh + 1)) | (j & (h - 1));
        const float a = qs[r * D + i], b = qs[r * D + i + h];
        qs[r * D + i] = a + b;
        qs[r * D + i + h] = a - b;
      }
      __syncthreads();
    }
    uint4* qf = reinterpret_cast<uint4*>(smem + QF_OFF);
    for (int f = threadIdx.x; f < NTW * MT * 32; f += G::NW * 32) {
      const int ln = f & 31, kk = (f >> 5) % MT, nt = (f >> 5) / MT;
      const int row = nt * 8 + (ln >> 2), cc = ln & 3;
      uint32_t hv[2], lv[2];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float x[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int dd = tqk_dim<D, KF>(cc, kk, 2 * b + e);
          const float v = qs[row * D + dd] * p.k_rot_scale;
          x[e] = ((p.vsigns2[dd >> 5] >> (dd & 31)) & 1u) ? -v : v;
        }
        const uint32_t hi = pack_h2(x[0], x[1]);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        hv[b] = hi;
        lv[b] = pack_h2(x[0] - hf.x, x[1] - hf.y);
      }
      qf[f] = make_uint4(hv[0], hv[1], lv[0], lv[1]);
    }
    // (the __syncthreads after the barrier set-up below orders these writes before every
    // read, and the scratch before the first tile copies)
  }

  // ---- plane bases of this (head, batch entry) -------------------------------------
  const int64_t krow = (p.shared ? 0 : (int64_t)bz * p.k.batch) + (int64_t)head * p.k.head;
  const int64_t vrow = (p.shared ? 0 : (int64_t)bz * p.v.batch) + (int64_t)head * p.v.head;
  const uint8_t* ka = G::K_ARB ? reinterpret_cast<const uint8_t*>(p.k.aux) + krow * G::K_ARB : nullptr;
  const uint8_t* ka2 = G::K_A2RB ? reinterpret_cast<const uint8_t*>(p.k.aux2) + krow * G::K_A2RB : nullptr;
  const uint8_t* va = G::V_ARB ? reinterpret_cast<const uint8_t*>(p.v.aux) + vrow * G::V_ARB : nullptr;
  const uint8_t* va2 = G::V_A2RB ? reinterpret_cast<const uint8_t*>(p.v.aux2) + vrow * G::V_A2RB : nullptr;
  const uint8_t* safe = reinterpret_cast<const uint8_t*>(p.k.data);
  const int bcoord = p.shared ? 0 : bz;  // tensor-map batch coordinate

  const int64_t tile0 = t0 & ~(int64_t)(TT - 1);
  const int ntiles = (int)((t1 - tile0 + TT - 1) / TT);
  uint8_t* wpipe = pipe + warp * G::STAGES * G::STAGE;

  const uint32_t bars = smem_addr(smem + G::BARS) + warp * G::STAGES * 8;
  // Set (to 1) by the first warp whose bounded wait gives up: from then on no warp of the
  // CTA issues another tile copy.  Read by lane 0 and broadcast, so warp-uniform.
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + ABORT_OFF);
  int n_issued = 0;  // this warp's tiles whose copies were issued (warp-uniform)

  // The warp's k-th tile -> stage k % STAGES.  Lane 0 announces the tensor-map bytes; lanes issue one box each; small planes go by
  // zero-filling cp.async from every lane, each lane then arriving on the same mbarrier
  // when its copies land.
  auto issue = [&](int k) {
    const int tile = warp + k * kWarps;
    if (tile >= ntiles) return;
    if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) return;  // a warp gave up: no new copies
    n_issued = k + 1;  // (tiles are issued in order, so every earlier one was too)
    uint8_t* st = wpipe + (k % G::STAGES) * G::STAGE;
    const int64_t tb = tile0 + (int64_t)tile * TT;
    const int tok = (int)tb;
    const uint32_t bar = bars + (k % G::STAGES) * 8;
    if (lane == 0) mbar_expect_tx(bar, G::TX);
    __syncwarp();
    fence_proxy_async();
    const uint32_t sbase = smem_addr(st);
    // one box per lane: K boxes, then V boxes, then the K-scale and V-aux planes
    constexpr int NKB = G::PK::NB, NVB = G::PV::NB;
    constexpr int NBOX = NKB + NVB + (G::PKA::TMA ? 1 : 0) + (G::PVA::TMA ? 1 : 0);
    static_assert(NBOX <= 32, "one tensor-map box per lane");
    if (lane < NBOX) {
      const TensorMap* mp = &maps.k;
      int dst = G::K_OFF + lane * (TT * G::PK::IB), x = lane * G::PK::IB;
      int rb = G::K_RB, ib = G::PK::IB;  // the plane's row bytes and the box width
      if (lane >= NKB && lane < NKB + NVB) {
        mp = &maps.v;
        dst = G::V_OFF + (lane - NKB) * (TT * G::PV::IB);
        x = (lane - NKB) * G::PV::IB;
        rb = G::V_RB;
        ib = G::PV::IB;
      } else if (lane >= NKB + NVB) {
        const bool ka = G::PKA::TMA && lane == NKB + NVB;
        mp = ka ? &maps.ka : &maps.va;
        dst = ka ? G::KA_OFF : G::VA_OFF;
        x = 0;
        rb = ka ? G::K_ARB : G::V_ARB;
        ib = ka ? G::PKA::IB : G::PVA::IB;
      }
      // the box stays inside its plane's row, tensor and this warp's stage
      const int stage_off = (int)(st - pipe);
      if (in_bounds(x >= 0 && x + ib <= rb && tb >= 0 && head < p.hkv && bcoord < (p.shared ? 1 : p.batch) &&
                        dst + TT * ib <= G::STAGE && stage_off >= 0 && stage_off + G::STAGE <= G::PIPE,
                    p.err))
        tma_load_4d(sbase + dst, mp, x, tok, head, bcoord, bar);
      (void)rb;
      (void)ib;
      (void)stage_off;
    }
    if constexpr (G::SMALL) {
      // rows past the view's end (kv_end) are zero-filled, like the tensor-map boxes
      const int valid = (int)max((int64_t)0, min((int64_t)TT, p.end - tb));
      // each plane's addressed bytes: rows [0, k_rows) / [0, v_rows) of the view
      const uint8_t* k_aux = reinterpret_cast<const uint8_t*>(p.k.aux);
      const uint8_t* v_aux = reinterpret_cast<const uint8_t*>(p.v.aux);
      const uint8_t* k_aux2 = reinterpret_cast<const uint8_t*>(p.k.aux2);
      const uint8_t* v_aux2 = reinterpret_cast<const uint8_t*>(p.v.aux2);
      if constexpr (G::K_ARB > 0 && !G::PKA::TMA)
        stage_flat_zfill<G::PKA::BYTES>(st + G::KA_OFF, ka + tb * G::K_ARB, valid * G::K_ARB, lane, safe, k_aux,
                                        k_aux + p.k_rows * G::K_ARB, p.err);
      if constexpr (G::V_ARB > 0 && !G::PVA::TMA)
        stage_flat_zfill<G::PVA::BYTES>(st + G::VA_OFF, va + tb * G::V_ARB, valid * G::V_ARB, lane, safe, v_aux,
                                        v_aux + p.v_rows * G::V_ARB, p.err);
      if constexpr (G::K_A2RB > 0)
        stage_flat_zfill<G::PKA2::BYTES>(st + G::KA2_OFF, ka2 + tb * G::K_A2RB, valid * G::K_A2RB, lane, safe,
                                         k_aux2, k_aux2 + p.k_rows * G::K_A2RB, p.err);
      if constexpr (G::V_A2RB > 0)
        stage_flat_zfill<G::PVA2::BYTES>(st + G::VA2_OFF, va2 + tb * G::V_A2RB, valid * G::V_A2RB, lane, safe,
                                         v_aux2, v_aux2 + p.v_rows * G::V_A2RB, p.err);
      cp_async_arrive_noinc(bar);
    }
  };

  // Barrier address and phase parity of the warp's k-th tile (stage k % STAGES).
  auto bar_of = [&](int k) { return bars + (k % G::STAGES) * 8; };
  auto par_of = [&](int k) { return (uint32_t)((k / G::STAGES) & 1); };

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
  // (a TurboQuant K's logits also carry the 1 / sqrt(D) of its decode)
  const float qk_scale = is_tq(KF) ? p.scale * p.k_norm_scale : p.scale;
  const float cap = p.softcap;
  const float cap_k = cap > 0.f ? 2.f * 1.4426950408889634f / cap : 0.f;  // 2 log2(e) / cap

  if (lane == 0) {
    for (int s = 0; s < G::STAGES; ++s) mbar_init(bars + s * 8, G::ARRIVALS);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();  // the barriers and the flag are ready

  // ---- per-tile work ------------------------------------------------------------------

  // per-lane stage offsets that do not change from tile to tile
  const int ks_lane = g * (D / 32);                        // K scale of (row g, block 0)
  // TQ2 / TQ3 2-bit plane and TQ3 sign plane offsets of tokens 2c, 2c+1, 2c+8, 2c+9
  int tq_off2[4] = {0, 0, 0, 0}, tq_sgn[4] = {0, 0, 0, 0};
  if constexpr (VF == QPS_FMT_TQ3 || VF == QPS_FMT_TQ2) {
    const int tk0[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      tq_off2[u] = soff<G::PV::IB, G::PV::SW, TT>(tk0[u], g * (DT / 4));
      if constexpr (VF == QPS_FMT_TQ3) tq_sgn[u] = soff<G::PVA::IB, G::PVA::SW, TT>(tk0[u], g * (DT / 8));
      // the decode reads up to DT / 4 (DT / 8) bytes from here, in every sub-tile
      in_bounds(tq_off2[u] >= 0 && tq_off2[u] + 16 * (SUB - 1) * G::PV::IB + DT / 4 <= G::PV::BYTES, p.err);
      if constexpr (VF == QPS_FMT_TQ3)
        in_bounds(tq_sgn[u] >= 0 && tq_sgn[u] + 16 * (SUB - 1) * G::PVA::IB + DT / 8 <= G::PVA::BYTES,
                  p.err);
    }
  }

  // S^T = K Q^T over this warp's columns, for each 16-token sub-tile
  auto k_part = [&](const uint8_t* st, float (&sacc)[SUB][NTW][4]) {
    // ---- S^T = K Q^T for each 16-token sub-tile (independent MMA chains) ------------
#pragma unroll
    for (int sb = 0; sb < SUB; ++sb)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) sacc[sb][nt][0] = sacc[sb][nt][1] = sacc[sb][nt][2] = sacc[sb][nt][3] = 0.f;
    if constexpr (KF == QPS_FMT_F16) {
      const uint32_t kbase = smem_addr(st + G::K_OFF);
      const int mi = lane >> 3;
      const int trow = (lane & 7) + ((mi & 1) << 3);
      // per sub-tile, two accumulator chains (even / odd k-steps)
      float sodd[SUB][NTW][4];
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb)
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) sodd[sb][nt][0] = sodd[sb][nt][1] = sodd[sb][nt][2] = sodd[sb][nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
          uint32_t a[4];
          ldsm_x4(a, kbase + soff<G::PK::IB, G::PK::SW, TT>(trow + 16 * sb, (2 * kk + (mi >> 1)) << 4));
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) {
            const uint2 qv = qfrag(nt, kk);
            if (kk & 1) mma16816(sodd[sb][nt], a, qv.x, qv.y);
            else mma16816(sacc[sb][nt], a, qv.x, qv.y);
          }
        }
      }
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb)
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[sb][nt][e] += sodd[sb][nt][e];
    } else if constexpr (KF == QPS_FMT_Q8_0) {
      const uint8_t* kc = st + G::K_OFF;
      const __half* ks = reinterpret_cast<const __half*>(st + G::KA_OFF) + ks_lane;
      // at head_dim <= 128 a row's D / 32 block scales come in one 4- or 8-byte load
      constexpr bool VEC_SCALES = (D == 64 || D == 128) && NTW <= 2;  // (three n-tiles leave no registers)
      float scv[SUB][2][VEC_SCALES ? D / 32 : 1];
      if constexpr (VEC_SCALES) {
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const __half* src = ks + (16 * sb + 8 * u) * (D / 32);
            uint32_t w[2];
            if constexpr (D == 128) {
              const uint2 r = *reinterpret_cast<const uint2*>(src);
              w[0] = r.x;
              w[1] = r.y;
            } else {
              w[0] = w[1] = *reinterpret_cast<const uint32_t*>(src);
            }
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
              scv[sb][u][2 * h] = f.x;
              scv[sb][u][2 * h + 1] = f.y;
            }
          }
      }
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const int x = 2 * j + (c >> 1), sub = 8 * (c & 1);
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
          const int r0 = g + 16 * sb, r8 = r0 + 8;
          const uint2 wg = *reinterpret_cast<const uint2*>(kc + soff<G::PK::IB, G::PK::SW, TT>(r0, 16 * x + sub));
          const uint2 wg8 = *reinterpret_cast<const uint2*>(kc + soff<G::PK::IB, G::PK::SW, TT>(r8, 16 * x + sub));
          uint32_t a0[4], a1[4];
          i8x4_to_h2x2(wg.x, a0[0], a0[2]);
          i8x4_to_h2x2(wg8.x, a0[1], a0[3]);
          i8x4_to_h2x2(wg.y, a1[0], a1[2]);
          i8x4_to_h2x2(wg8.y, a1[1], a1[3]);
          float sg, sg8;
          if constexpr (VEC_SCALES) {
            sg = scv[sb][0][j];
            sg8 = scv[sb][1][j];
          } else {
            sg = __half2float(ks[16 * sb * (D / 32) + j]);
            sg8 = __half2float(ks[(16 * sb + 8) * (D / 32) + j]);
          }
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint2 qv0 = qfrag(nt, 2 * j), qv1 = qfrag(nt, 2 * j + 1);
            mma16816(acc, a0, qv0.x, qv0.y);
            mma16816(acc, a1, qv1.x, qv1.y);
            sacc[sb][nt][0] = fmaf(sg, acc[0], sacc[sb][nt][0]);
            sacc[sb][nt][1] = fmaf(sg, acc[1], sacc[sb][nt][1]);
            sacc[sb][nt][2] = fmaf(sg8, acc[2], sacc[sb][nt][2]);
            sacc[sb][nt][3] = fmaf(sg8, acc[3], sacc[sb][nt][3]);
          }
        }
      }
    } else {
      // TurboQuant K (the same tier as V): lane group c decodes the quarter [c D/4,
      // (c+1) D/4) of tokens g and g + 8 into the A operand, the rotated query comes
      // from shared memory as hi + lo fragments (two accumulator chains), and each
      // token's logit is scaled by its norm at the end.
      static_assert(is_tq(KF) && KF == VF, "a TurboQuant K pairs with V of the same tier");
      constexpr int QB = G::K_RB / 4;           // bytes of a quarter row
      constexpr int CH = QB >= 16 ? 16 : QB;    // bytes per read
      const uint4* qf = reinterpret_cast<const uint4*>(smem + QF_OFF) + lane;
      const uint8_t* kc = st + G::K_OFF;
      float slo[SUB][NTW][4];
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb)
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) slo[sb][nt][0] = slo[sb][nt][1] = slo[sb][nt][2] = slo[sb][nt][3] = 0.f;
      // one k-step: a = {token g pair 0, token g+8 pair 0, token g pair 1, token g+8 pair 1}
      auto kstep = [&](int sb, int kk, const uint32_t (&a)[4]) {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          const uint4 qv = qf[(nt * MT + kk) * 32];
          mma16816(sacc[sb][nt], a, qv.x, qv.y);
          mma16816(slo[sb][nt], a, qv.z, qv.w);
        }
      };
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
        const int r0 = g + 16 * sb, r8 = r0 + 8;
#pragma unroll
        for (int q0 = 0; q0 < QB; q0 += CH) {
          uint32_t w[2][CH / 4];  // words of tokens r0, r8
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint8_t* src = kc + soff<G::PK::IB, G::PK::SW, TT>(u ? r8 : r0, c * QB + q0);
            if constexpr (CH == 16) {
              const uint4 r = *reinterpret_cast<const uint4*>(src);
              w[u][0] = r.x; w[u][1] = r.y; w[u][2] = r.z; w[u][3] = r.w;
            } else if constexpr (CH == 8) {
              const uint2 r = *reinterpret_cast<const uint2*>(src);
              w[u][0] = r.x; w[u][1] = r.y;
            } else {
              w[u][0] = *reinterpret_cast<const uint32_t*>(src);
            }
          }
          if constexpr (KF == QPS_FMT_TQ4) {
            // a word holds 8 dims (4-bit fields): k-steps (q0 + 4 wi) / 2 and the next
#pragma unroll
            for (int wi = 0; wi < CH / 4; ++wi) {
              uint32_t mg[2], w4[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                mg[u] = w[u][wi] & 0x77777777u;
                w4[u] = w[u][wi] << 4;
              }
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                uint32_t a[4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const uint32_t sel = hf ? mg[u] >> 16 : mg[u];
                  const uint32_t lo = prmt(tq_lo, tq_hi, sel);
                  const uint32_t pos = prmt(w[u][wi], w4[u], hf ? 0xBFAEu : 0x9D8Cu);
                  const uint32_t hi = prmt(tq_lo2, tq_hi2, sel) | (~pos & 0x80808080u);
                  a[u] = __byte_perm(lo, hi, 0x5140u);      // dims 4kk, 4kk + 1 of the quarter
                  a[2 + u] = __byte_perm(lo, hi, 0x7362u);  // dims 4kk + 2, 4kk + 3
                }
                kstep(sb, (q0 + 4 * wi) / 2 + hf, a);
              }
            }
          } else {
            // a word holds 16 dims (2-bit fields); TQ3 signs: 16 bits per word, up to four
            // words (8 sign bytes) per chunk
            uint32_t sgw[2][2] = {{0u, 0u}, {0u, 0u}};
            if constexpr (KF == QPS_FMT_TQ3) {
              constexpr int SB = CH / 2;  // sign bytes of the chunk: 2, 4 or 8
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const uint8_t* src =
                    st + G::KA_OFF + soff<G::PKA::IB, G::PKA::SW, TT>(u ? r8 : r0, c * (QB / 2) + q0 / 2);
                if constexpr (SB == 8) {
                  const uint2 r = *reinterpret_cast<const uint2*>(src);
                  sgw[u][0] = r.x;
                  sgw[u][1] = r.y;
                } else if constexpr (SB == 4) {
                  sgw[u][0] = *reinterpret_cast<const uint32_t*>(src);
                } else {
                  sgw[u][0] = *reinterpret_cast<const uint16_t*>(src);
                }
              }
            }
#pragma unroll
            for (int wi = 0; wi < CH / 4; ++wi) {
              const int wq = (q0 + 4 * wi) / 4;  // word of the quarter
              uint32_t s1[2] = {0u, 0u}, s2[2] = {0u, 0u};
              if constexpr (KF == QPS_FMT_TQ3) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const uint32_t sg16 = (sgw[u][wi >> 1] >> (16 * (wi & 1))) & 0xffffu;
                  s1[u] = sg16 | (sg16 << 12);        // dims j, j + 4 at bits j, 16 + j
                  s2[u] = (sg16 >> 8) | (sg16 << 4);  // dims j + 8, j + 12 at bits j, 16 + j
                }
              }
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t a[4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  // one code per byte (dims j, j+4, j+8, j+12), then table selectors
                  const uint32_t sel = ((w[u][wi] >> (2 * j)) & 0x03030303u) * 0x22u + 0x10101010u;
                  uint32_t m0 = __byte_perm(tq_lo, tq_hi, sel);
                  uint32_t m1 = __byte_perm(tq_lo, tq_hi, sel >> 16);
                  if constexpr (KF == QPS_FMT_TQ3) {  // a clear sign bit stores a negative level
                    m0 |= ~(s1[u] << (15 - j)) & 0x80008000u;
                    m1 |= ~(s2[u] << (15 - j)) & 0x80008000u;
                  }
                  a[u] = m0;
                  a[2 + u] = m1;
                }
                kstep(sb, 4 * wq + j, a);
              }
            }
          }
        }
      }
      const __half* kn = reinterpret_cast<const __half*>(st + G::KNORM_OFF);
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
        const float n0 = __half2float(kn[16 * sb + g]), n8 = __half2float(kn[16 * sb + g + 8]);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          sacc[sb][nt][0] = (sacc[sb][nt][0] + slo[sb][nt][0]) * n0;
          sacc[sb][nt][1] = (sacc[sb][nt][1] + slo[sb][nt][1]) * n0;
          sacc[sb][nt][2] = (sacc[sb][nt][2] + slo[sb][nt][2]) * n8;
          sacc[sb][nt][3] = (sacc[sb][nt][3] + slo[sb][nt][3]) * n8;
        }
      }
    }

  };

  // logits of the stage starting at token tb, online softmax, O^T += V^T P^T
  auto attend_tile = [&](const uint8_t* st, int64_t tb, float (&sacc)[SUB][NTW][4]) {
    // ---- logits, masking, online softmax (one update per stage) ------------------------
    bool in_g[SUB], in_g8[SUB];
    float n_g[SUB], n_g8[SUB];
#pragma unroll
    for (int sb = 0; sb < SUB; ++sb) {
      const int64_t t_g = tb + 16 * sb + g;
      in_g[sb] = (t_g >= t0) && (t_g < t1);
      in_g8[sb] = (t_g + 8 >= t0) && (t_g + 8 < t1);
      n_g[sb] = n_g8[sb] = 1.f;
      if constexpr (is_tq(VF)) {
        const __half* nrm = reinterpret_cast<const __half*>(st + G::NORM_OFF);
        n_g[sb] = __half2float(nrm[16 * sb + g]);
        n_g8[sb] = __half2float(nrm[16 * sb + g + 8]);
      }
    }
    // The reference maximum of the online softmax is raised only when a tile's maximum
    // exceeds it by more than `lazy` (log2 units): P then stays <= 2^lazy, the running
    // sum and O carry the same reference, and the rescale of O (a multiply per
    // accumulator) is skipped on most tiles.  A TurboQuant V folds its norms into the
    // fp16 P, so there lazy is 8 only while the tile's norms stay <= 255 (P x norm stays
    // finite in fp16), else 0 (P <= 1, the exact maximum).  Three n-tiles keep the exact
    // maximum: there the test's registers made the kernel spill (4-token verify batch
    // 64.5 -> 66.8 us).
    float lazy = NTW >= 3 ? 0.f : 8.f;
    if constexpr (is_tq(VF) && NTW < 3) {
      float nmx = 0.f;
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) nmx = fmaxf(nmx, fmaxf(fabsf(n_g[sb]), fabsf(n_g8[sb])));
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) nmx = fmaxf(nmx, __shfl_xor_sync(0xffffffffu, nmx, off));
      lazy = nmx <= 255.f ? 8.f : 0.f;
    }
    uint32_t pb[SUB][NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      float x[SUB][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sacc[sb][nt][e] * qk_scale;
          if (cap > 0.f) v = softcap_tanh(v, cap, cap_k);
          x[sb][e] = v * LOG2E;
        }
        if (!in_g[sb]) x[sb][0] = x[sb][1] = -INFINITY;
        if (!in_g8[sb]) x[sb][2] = x[sb][3] = -INFINITY;
        if constexpr (CAUSAL) {
          // position t is visible to CTA row r (query token r / group) iff
          // t - q_pos <= r / group, i.e. (t - q_pos) * group <= r; t - q_pos is clamped
          // so the product stays in 32 bits (rows are < 1024)
          const int64_t rel64 = tb + 16 * sb + g - p.q_pos;
          const int rel = (int)max((int64_t)-2048, min((int64_t)2048, rel64)) * p.group;
          const int r0 = row0 + nt * 8 + 2 * c, r8 = rel + 8 * p.group;
          if (rel > r0) x[sb][0] = -INFINITY;
          if (rel > r0 + 1) x[sb][1] = -INFINITY;
          if (r8 > r0) x[sb][2] = -INFINITY;
          if (r8 > r0 + 1) x[sb][3] = -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(x[sb][0], x[sb][2]));
        mx1 = fmaxf(mx1, fmaxf(x[sb][1], x[sb][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      float mn0, mn1;
      if constexpr (NTW >= 3) {
        mn0 = fmaxf(m[nt][0], mx0);
        mn1 = fmaxf(m[nt][1], mx1);
      } else {
        mn0 = mx0 - m[nt][0] > lazy ? mx0 : m[nt][0];  // (NaN if both are -inf: keeps -inf)
        mn1 = mx1 - m[nt][1] > lazy ? mx1 : m[nt][1];
      }
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float cr0 = exp2f(m[nt][0] - ms0), cr1 = exp2f(m[nt][1] - ms1);
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
        const float p0 = exp2f(x[sb][0] - ms0), p1 = exp2f(x[sb][1] - ms1);
        const float p2 = exp2f(x[sb][2] - ms0), p3 = exp2f(x[sb][3] - ms1);
        sum0 += p0 + p2;
        sum1 += p1 + p3;
        pb[sb][nt][0] = movmatrix_t(pack_h2(p0 * n_g[sb], p1 * n_g[sb]));
        pb[sb][nt][1] = movmatrix_t(pack_h2(p2 * n_g8[sb], p3 * n_g8[sb]));
      }
      l[nt][0] = l[nt][0] * cr0 + sum0;
      l[nt][1] = l[nt][1] * cr1 + sum1;
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
    }

    // ---- O^T += V^T P^T ---------------------------------------------------------------
    if constexpr (VF == QPS_FMT_F16) {
      const uint32_t vbase = smem_addr(st + G::V_OFF);
      const int mi = lane >> 3;
      const int trow = (lane & 7) + ((mi & 2) << 2);
#pragma unroll
      for (int i = 0; i < MT; ++i) {
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
          uint32_t a[4];
          ldsm_x4_t(a, vbase + soff<G::PV::IB, G::PV::SW, TT>(trow + 16 * sb, (2 * i + (mi & 1)) << 4));
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[sb][nt][0], pb[sb][nt][1]);
        }
      }
    } else if constexpr (VF == QPS_FMT_Q8_0) {
      // lane group g owns output columns [g*DT, g*DT + DT); tokens 2c, 2c+1, 2c+8, 2c+9
      const uint8_t* vc = st + G::V_OFF;
      const __half* vs = reinterpret_cast<const __half*>(st + G::VA_OFF);
      constexpr int CH = DT >= 16 ? 16 : DT;  // bytes per read
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
#pragma unroll
        for (int q0 = 0; q0 < DT; q0 += CH) {
          uint32_t w[4][CH / 4];
          const int tok[4] = {16 * sb + 2 * c, 16 * sb + 2 * c + 1, 16 * sb + 2 * c + 8, 16 * sb + 2 * c + 9};
          const int blk = (g * DT + q0) / 32;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int byte = g * DT + q0;
            const uint8_t* src = vc + soff<G::PV::IB, G::PV::SW, TT>(tok[u], byte);
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
              for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[sb][nt][0], pb[sb][nt][1]);
            }
          }
        }
      }
    } else if constexpr (VF == QPS_FMT_TQ3 || VF == QPS_FMT_TQ2) {
      // TQ2 / TQ3.  Word k of a lane group's 2-bit plane holds 16 of its output columns;
      // the codes of the two tokens of a pair are interleaved byte by byte, spread to one
      // code per byte and turned into byte-permute selectors over the fp16 level table
      // (TQ3: magnitudes, the sign plane then supplying bit 15 of each half; TQ2: the four
      // signed levels in field order).  m-tile i of word k takes columns tq_col(i, 0) and
      // tq_col(i, 1) (see the epilogue).
      constexpr int LB = DT / 4;                   // 2-bit plane bytes per lane group, token
      constexpr int HB = DT / 8;                   // sign plane bytes per lane group, token
      constexpr int NWD = DT >= 16 ? DT / 16 : 1;  // 16-column words
      constexpr int NH = DT >= 16 ? 2 : 1;         // 8-column halves of a word
      const uint8_t* lo2 = st + G::V_OFF;
      const uint8_t* hi1 = st + G::VA_OFF;
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
        uint32_t L[4][NWD];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint8_t* ls = lo2 + tq_off2[u] + 16 * sb * G::PV::IB;  // swizzle repeats every 8 rows
          if constexpr (LB == 16) {
            const uint4 r = *reinterpret_cast<const uint4*>(ls);
            L[u][0] = r.x; L[u][1] = r.y; L[u][2] = r.z; L[u][3] = r.w;
          } else if constexpr (LB == 8) {
            const uint2 r = *reinterpret_cast<const uint2*>(ls);
            L[u][0] = r.x; L[u][1] = r.y;
          } else if constexpr (LB == 4) {
            L[u][0] = *reinterpret_cast<const uint32_t*>(ls);
          } else {
            L[u][0] = *reinterpret_cast<const uint16_t*>(ls);
          }
        }
        uint32_t H[4] = {0u, 0u, 0u, 0u};  // TQ3 sign bits of 32 columns (fewer at head_dim <= 128) per token
#pragma unroll
        for (int k = 0; k < NWD; ++k) {
          uint32_t hab[2] = {0u, 0u};
          if constexpr (VF == QPS_FMT_TQ3) {
            if ((k & 1) == 0) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                // (2k stays inside the lane's 16-byte chunk: HB = 8 puts its 8 bytes in one)
                const uint8_t* hs = hi1 + tq_sgn[u] + 16 * sb * G::PVA::IB + 2 * k;
                if constexpr (HB >= 4) H[u] = *reinterpret_cast<const uint32_t*>(hs);
                else if constexpr (HB == 2) H[u] = *reinterpret_cast<const uint16_t*>(hs);
                else H[u] = *hs;
              }
            }
            // sign bits of word k: token a of the pair in bits 0..15, token b in 16..31
            const uint32_t hsel = (k & 1) ? 0x7632u : 0x5410u;
            hab[0] = __byte_perm(H[0], H[1], hsel);
            hab[1] = __byte_perm(H[2], H[3], hsel);
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            // bytes: (a, b) codes of columns 8h .. 8h + 3, then of 8h + 4 .. 8h + 7
            const uint32_t ysel = h ? 0x7362u : 0x5140u;
            const uint32_t y[2] = {__byte_perm(L[0][k], L[1][k], ysel), __byte_perm(L[2][k], L[3][k], ysel)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = DT >= 16 ? 8 * k + 2 * j + h : j;  // m-tile
              const int e0 = j + 8 * h, e1 = e0 + 4;           // columns within the word
              uint32_t a[4];
#pragma unroll
              for (int pr = 0; pr < 2; ++pr) {
                // one code per byte, then the selector nibbles (2f, 2f + 1) of table entry f
                const uint32_t sel = ((y[pr] >> (2 * j)) & 0x03030303u) * 0x22u + 0x10101010u;
                const uint32_t m0 = __byte_perm(tq_lo, tq_hi, sel);
                const uint32_t m1 = __byte_perm(tq_lo, tq_hi, sel >> 16);
                if constexpr (VF == QPS_FMT_TQ3) {
                  // a clear sign bit stores a negative level
                  a[2 * pr] = m0 | (~(hab[pr] << (15 - e0)) & 0x80008000u);
                  a[2 * pr + 1] = m1 | (~(hab[pr] << (15 - e1)) & 0x80008000u);
                } else {
                  a[2 * pr] = m0;
                  a[2 * pr + 1] = m1;
                }
              }
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[sb][nt][0], pb[sb][nt][1]);
            }
          }
        }
      }
    } else {
      // TQ4.  A lane group's DT 4-bit fields (DT / 2 bytes per token) hold its columns in
      // order, 8 per 32-bit word.  The fields of a token pair are interleaved byte by
      // byte; their magnitudes (bits 0..2) select the low and the high byte of the fp16
      // magnitude from two 8-byte tables, bit 3 (set: positive) sets the high byte's top
      // bit through a sign-replicating byte permute, and the low / high bytes are then
      // interleaved into halves.  m-tile i takes columns 2i and 2i + 1, as for q8_0.
      static_assert(VF == QPS_FMT_TQ4, "unhandled V format");
      constexpr int FB = DT / 2;               // field bytes per lane group and token
      constexpr int CH = FB >= 16 ? 16 : FB;   // bytes per read
      const uint8_t* vf = st + G::V_OFF;
#pragma unroll
      for (int sb = 0; sb < SUB; ++sb) {
        const int tok[4] = {16 * sb + 2 * c, 16 * sb + 2 * c + 1, 16 * sb + 2 * c + 8, 16 * sb + 2 * c + 9};
#pragma unroll
        for (int q0 = 0; q0 < FB; q0 += CH) {
          uint32_t w[4][CH / 4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint8_t* src = vf + soff<G::PV::IB, G::PV::SW, TT>(tok[u], g * FB + q0);
            if constexpr (CH == 16) {
              const uint4 r = *reinterpret_cast<const uint4*>(src);
              w[u][0] = r.x; w[u][1] = r.y; w[u][2] = r.z; w[u][3] = r.w;
            } else if constexpr (CH == 8) {
              const uint2 r = *reinterpret_cast<const uint2*>(src);
              w[u][0] = r.x; w[u][1] = r.y;
            } else {
              w[u][0] = *reinterpret_cast<const uint32_t*>(src);
            }
          }
#pragma unroll
          for (int wi = 0; wi < CH / 4; ++wi) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // nibbles: a c0, a c1, b c0, b c1, a c2, a c3, b c2, b c3 of columns 4h ..
              const uint32_t ysel = h ? 0x7362u : 0x5140u;
              const uint32_t y[2] = {__byte_perm(w[0][wi], w[1][wi], ysel), __byte_perm(w[2][wi], w[3][wi], ysel)};
              const uint32_t mg[2] = {y[0] & 0x77777777u, y[1] & 0x77777777u};
              // each byte's low field moved up: its sign (bit 3) becomes the byte's top bit
              const uint32_t y4[2] = {y[0] << 4, y[1] << 4};
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int i = q0 + 4 * wi + 2 * h + q;  // m-tile: columns 2i, 2i + 1
                uint32_t a[4];
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                  const uint32_t sel = q ? mg[pr] >> 16 : mg[pr];
                  const uint32_t lo = prmt(tq_lo, tq_hi, sel);
                  // 0xff per value whose sign bit is set, in selector order (a even, a odd,
                  // b even, b odd): the even column's from y4, the odd one's from y
                  const uint32_t pos = prmt(y[pr], y4[pr], q ? 0xBFAEu : 0x9D8Cu);
                  // a clear sign bit stores a negative level
                  const uint32_t hi = prmt(tq_lo2, tq_hi2, sel) | (~pos & 0x80808080u);
                  a[2 * pr] = __byte_perm(lo, hi, 0x6240u);
                  a[2 * pr + 1] = __byte_perm(lo, hi, 0x7351u);
                }
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) mma16816(o[i][nt], a, pb[sb][nt][0], pb[sb][nt][1]);
              }
            }
          }
        }
      }
    }
  };

  // ---- the warp's tiles: a private pipeline, no cross-warp traffic ---------------------
  // The loop consumes exactly the tiles whose copies were issued: after a give-up in any
  // warp of the CTA no new copies start, the tiles already in flight are consumed (or,
  // in the warp that gave up, drained), and the CTA returns without an epilogue.
#pragma unroll 1
  for (int s = 0; s < G::STAGES - 1; ++s) issue(s);
  int k_fail = -1;  // the tile whose wait gave up (warp-uniform)
#pragma unroll 1
  for (int k = 0; k < n_issued; ++k) {
    issue(k + G::STAGES - 1);  // stage (k - 1) % STAGES is free
    if (!mbar_wait(bar_of(k), par_of(k))) {
      k_fail = k;
      break;
    }
    __syncwarp();
    const uint8_t* st = wpipe + (k % G::STAGES) * G::STAGE;
    float sacc[SUB][NTW][4];
    k_part(st, sacc);
    attend_tile(st, tile0 + (int64_t)(warp + k * kWarps) * TT, sacc);
    __syncwarp();
  }
  if (k_fail >= 0) {
    // Record the failure (the host reads it through qps_device_status), stop every warp's
    // further copies, then give each copy this warp still has in flight (tiles k_fail ..
    // n_issued - 1, at most STAGES, so one per stage) one more bounded wait, so that no
    // tensor-map write lands in shared memory after the CTA has exited.  Should one of
    // those also run out, the CTA exits with that copy still outstanding.
    bool first = false;
    if (lane == 0) {
      atomicOr(p.err, 1u);
      *abort_flag = 1;
      first = atomicAdd(p.err + 1, 1u) == 0;  // this CTA's record is the launch's first
      if (first) {
        unsigned int* r = p.err + 2;
        r[0] = blockIdx.x;
        r[1] = blockIdx.y;
        r[2] = blockIdx.z;
        r[3] = warp;
        r[4] = k_fail;
        r[5] = n_issued;
        r[6] = (unsigned)((ntiles - warp + kWarps - 1) / kWarps);
        r[7] = (unsigned)(t1 - t0);
      }
    }
    for (int j = k_fail; j < n_issued; ++j) {
      const uint64_t w0 = global_ns();
      const bool done = mbar_wait(bar_of(j), par_of(j));
      if (first && j == k_fail) {
        p.err[10] = (unsigned)min((uint64_t)0xffffffffu, global_ns() - w0);
        p.err[11] = done ? 1u : 0u;
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  // every warp's outstanding copies are done (or drained); a CTA in which any wait gave
  // up writes no partial (the error word marks the launch's outputs invalid)
  if (__syncthreads_or(k_fail >= 0)) return;
  asm volatile("griddepcontrol.launch_dependents;" :::);

  // ---- merge the warps' states, then the chunk's partial ------------------------------
  constexpr int OWS = ow_stride<D>();
  float* mw = reinterpret_cast<float*>(smem);  // [kWarps][ROWS]
  float* lw = mw + kWarps * ROWS;              // [kWarps][ROWS]
  float* ow = lw + kWarps * ROWS;              // [kWarps][ROWS][OWS], columns at ow_col
  float* fin = ow + kWarps * ROWS * OWS;       // [ROWS][D]
  int64_t* orow = reinterpret_cast<int64_t*>(fin + ROWS * D);  // [ROWS] output row index
  float* wgt = reinterpret_cast<float*>(orow + ROWS);             // [kWarps][ROWS] warp weights
  float* rmx = wgt + kWarps * ROWS;                                // [ROWS] row maximum (log2)
  float* rden = rmx + ROWS;                                        // [ROWS] row denominator
  if (threadIdx.x < nrows) orow[threadIdx.x] = out_row(row0 + threadIdx.x);
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
      if constexpr (VF == QPS_FMT_TQ3 || VF == QPS_FMT_TQ2) {
        d0 = g * DT + tq_col<DT>(i, 0);
        d1 = g * DT + tq_col<DT>(i, 1);
      } else if constexpr (VPERM) {
        d0 = g * DT + 2 * i;
        d1 = d0 + 1;
      } else {
        d0 = 16 * i + g;
        d1 = d0 + 8;
      }
      float* base = ow + (warp * ROWS + nt * 8 + 2 * c) * OWS;
      base[ow_col<D>(d0)] = o[i][nt][0];
      base[OWS + ow_col<D>(d0)] = o[i][nt][1];
      base[ow_col<D>(d1)] = o[i][nt][2];
      base[OWS + ow_col<D>(d1)] = o[i][nt][3];
    }
  }
  __syncthreads();
  // per row: the maximum over the warps, each warp's weight 2^(m_w - max) (0 for a warp
  // that saw nothing of the row) and the merged denominator
  if (threadIdx.x < ROWS) {
    const int r = threadIdx.x;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, mw[w * ROWS + r]);
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mv = mw[w * ROWS + r];
      const float f = (mx != -INFINITY && mv != -INFINITY) ? exp2f(mv - mx) : 0.f;
      wgt[w * ROWS + r] = f;
      den += lw[w * ROWS + r] * f;
    }
    rmx[r] = mx;
    rden[r] = den;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ROWS * D; idx += G::NW * 32) {
    const int r = idx / D, dd = idx % D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) acc += ow[(w * ROWS + r) * OWS + ow_col<D>(dd)] * wgt[w * ROWS + r];
    if constexpr (is_tq(VF))  // the rotation's second sign vector
      if ((p.vsigns2[dd >> 5] >> (dd & 31)) & 1u) acc = -acc;
    fin[idx] = acc;
  }
  __syncthreads();
  if constexpr (is_tq(VF)) {  // inverse rotation x = s1 .* blockdiag(H_G)(s2 .* y) / sqrt(D G), in place
#pragma unroll
    for (int lh = 0; (1 << lh) < D; ++lh) {  // butterflies of span h = 2^lh
      const int h = 1 << lh;
      if (h >= p.vblock) break;  // (uniform over the CTA)
#pragma unroll 4
      for (int pid = threadIdx.x; pid < ROWS * (D / 2); pid += G::NW * 32) {
        const int r = pid / (D / 2), j = pid % (D / 2);
        const int i = ((j >> lh) << (lh + 1)) | (j & (h - 1));
        const float a = fin[r * D + i], b = fin[r * D + i + h];
        fin[r * D + i] = a + b;
        fin[r * D + i + h] = a - b;
      }
      __syncthreads();
    }
  }
  for (int idx = threadIdx.x; idx < nrows * D; idx += G::NW * 32) {
    const int r = idx / D, dd = idx % D;
    const float mx = rmx[r], den = rden[r];
    float val = fin[r * D + dd];
    if constexpr (is_tq(VF)) {
      val *= p.v_out_scale;
      if ((p.vsigns[dd >> 5] >> (dd & 31)) & 1u) val = -val;
    }
    const int64_t row = orow[r];
    const bool empty = !(den > 0.f);
    if (!in_bounds(part < p.parts_cap && row >= 0 && row < p.rows_total, p.err)) continue;
    p.o_parts[((int64_t)part * p.rows_total + row) * D + dd] = empty ? 0.f : val / den;
    if (dd == 0)
      p.lse_parts[(int64_t)part * p.rows_total + row] = empty ? -INFINITY : (mx + log2f(den)) * 0.6931471805599453f;
  }
}

template <int D, int KF, int VF, int NTW>
constexpr size_t smem_bytes() {
  using G = Geo<D, KF, VF, NTW>;
  // the stages and barriers, the give-up flag, then query fragments kept in shared memory
  constexpr size_t pipe = (size_t)align_to(G::END + 16, 16) + qf_bytes<D, KF, VF, NTW>();
  constexpr int ROWS = 8 * NTW;
  constexpr size_t merge = sizeof(float) * ((size_t)2 * G::NW * ROWS + (size_t)G::NW * ROWS * ow_stride<D>() +
                                           (size_t)ROWS * D) +
                           sizeof(int64_t) * ROWS + sizeof(float) * ((size_t)G::NW * ROWS + 2 * ROWS);
  return (pipe > merge ? pipe : merge) + 1024;  // + slack for the 1024-byte base alignment
}

template <int D, int KF, int VF, int NTW, bool CAUSAL>
qps_status launch_mma_t(const AttnParams& p, cudaStream_t s) {
  using G = Geo<D, KF, VF, NTW>;
  constexpr size_t smem = smem_bytes<D, KF, VF, NTW>();
  static_assert(smem <= 227 * 1024, "tile staging exceeds the 227 KB shared memory of one CTA");
  // G::CTAS CTAs per SM (the launch bound the registers are sized for: 228 KB less 1 KB
  // reserved per CTA), unless two-CTA stages are already at their minimum of two (fp16
  // planes at head_dim >= 256, which then run one CTA per SM)
  static_assert(G::CTAS * (smem + 1024) <= 228 * 1024 || (G::CTAS == 2 && G::STAGES == 2),
                "the CTAs per SM the instance is built for no longer fit");
  static_assert(qf_bytes<D, KF, VF, NTW>() == 0 || G::CTAS * (smem + 1024) <= 228 * 1024,
                "query fragments in shared memory must not cost a CTA per SM");
  // tensor maps over each plane as [row bytes][tokens < kv_end][KV heads][batch]
  TmaSet maps;
  std::memset(&maps, 0, sizeof(maps));
  const int nb = p.shared ? 1 : p.batch;
  if (!encode_plane_map(&maps.k, p.k.data, G::K_RB, p.end, p.hkv, p.k.head, nb, p.k.batch, G::PK::IB, G::PK::SW, G::TT) ||
      !encode_plane_map(&maps.v, p.v.data, G::V_RB, p.end, p.hkv, p.v.head, nb, p.v.batch, G::PV::IB, G::PV::SW, G::TT))
    return QPS_ERR_CUDA;
  if constexpr (G::PKA::TMA)
    if (!encode_plane_map(&maps.ka, p.k.aux, G::K_ARB, p.end, p.hkv, p.k.head, nb, p.k.batch, G::PKA::IB, G::PKA::SW, G::TT))
      return QPS_ERR_CUDA;
  if constexpr (G::PVA::TMA)
    if (!encode_plane_map(&maps.va, p.v.aux, G::V_ARB, p.end, p.hkv, p.v.head, nb, p.v.batch, G::PVA::IB, G::PVA::SW, G::TT))
      return QPS_ERR_CUDA;
  auto kern = attn_mma_kernel<D, KF, VF, NTW, CAUSAL>;
  // Ask for enough shared memory that no more than G::CTAS CTAs fit on an SM: under
  // programmatic launch the next grid's CTAs would otherwise take a spare slot early
  // and pile three of them onto some SMs (the q8_0 Qwen-like window: 39.5 -> 45 us).
  constexpr size_t kSmPerSm = 228 * 1024, kReserved = 1024;
  constexpr size_t smem_floor = kSmPerSm / (G::CTAS + 1) - kReserved + 1;
  constexpr size_t smem_launch = smem > smem_floor ? smem : smem_floor;
  static_assert(G::CTAS * (smem_launch + kReserved) <= kSmPerSm || smem_launch == smem,
                "the padding must not cost a CTA per SM");
  QPS_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_launch));
  constexpr int ROWS = 8 * NTW;
  const int rgroups = (p.rows_per_cta + ROWS - 1) / ROWS;
  const dim3 grid(p.n_split * rgroups, p.hkv, p.shared ? 1 : p.batch);
  // launched with programmatic stream serialization: overlaps this grid's launch with
  // the end of the previous kernel on the stream (the kernel waits before any global
  // memory access)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(G::NW * 32);
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

// Every format pairing and n-tile count of one head_dim, with or without the causal
// limit; SET selects the pairings: 0 K F16 / Q8_0 with V F16 / Q8_0 / TQ3, 1 the same K
// with V TQ2 / TQ4, 2 a TurboQuant K with V of the same tier.  The sets live in
// separate translation units.
template <int D, bool CAUSAL, int SET>
qps_status launch_mma_d(const AttnParams& p, cudaStream_t s) {
  // 8-row n-tiles per warp: more only where the accumulators still fit in registers
  const int ntw = mma_tile_rows(D, p.rows_per_cta, p.shared != 0) / 8;
#define QPS_MMA_CASE(KF, VF)                                                       \
  if (p.kfmt == KF && p.vfmt == VF) {                                              \
    if (ntw == 3) return launch_mma_t<D, KF, VF, (D <= 128 ? 3 : 1), CAUSAL>(p, s); \
    if (ntw == 2) return launch_mma_t<D, KF, VF, (D <= 128 ? 2 : 1), CAUSAL>(p, s); \
    return launch_mma_t<D, KF, VF, 1, CAUSAL>(p, s);                                \
  }
  if constexpr (SET == 2) {
    QPS_MMA_CASE(QPS_FMT_TQ2, QPS_FMT_TQ2)
    QPS_MMA_CASE(QPS_FMT_TQ3, QPS_FMT_TQ3)
    QPS_MMA_CASE(QPS_FMT_TQ4, QPS_FMT_TQ4)
  } else if constexpr (SET == 1) {
    QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_TQ2)
    QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_TQ4)
    QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_TQ2)
    QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_TQ4)
  } else {
    QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_F16)
    QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_Q8_0)
    QPS_MMA_CASE(QPS_FMT_F16, QPS_FMT_TQ3)
    QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_F16)
    QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_Q8_0)
    QPS_MMA_CASE(QPS_FMT_Q8_0, QPS_FMT_TQ3)
  }
#undef QPS_MMA_CASE
  return fail(QPS_ERR_UNSUPPORTED, "attention: unsupported K/V format pairing");
}

}  // namespace mma
}  // namespace qps
