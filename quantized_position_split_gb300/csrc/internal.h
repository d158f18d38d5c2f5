// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "qps.h"

namespace qps {

// ---- error reporting ------------------------------------------------------------
qps_status fail(qps_status st, const std::string& msg);
qps_status cuda_fail(cudaError_t err, const char* what);
void count_launch(int n = 1);

#define QPS_CUDA_TRY(expr)                              \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return ::qps::cuda_fail(_e, #expr); \
  } while (0)

// ---- tensor memory access descriptors ----------------------------------------------
// A byte plane seen as a 4-D tensor [row bytes][tokens][heads][batch] (innermost
// first), loaded in boxes of [box_bytes][box_rows tokens][1][1].  swizzle: 0 none, 32, 64 or
// 128 (bytes).  Returns false (with the error message set) on failure.
struct alignas(64) TensorMap {
  unsigned char bytes[128];
};
bool encode_plane_map(TensorMap* map, const void* base, int row_bytes, int64_t tokens, int heads,
                      int64_t head_stride_rows, int batch, int64_t batch_stride_rows, int box_bytes,
                      int swizzle, int box_rows);

// ---- device facts -----------------------------------------------------------------
int sm_count_current();
// The current device's error word (library-owned, allocated on first use, zeroed).
// Bits: kErrTimeout, a bounded in-kernel wait gave up; kErrBounds, a bounds check of the
// checked build failed and its access was skipped.
// The word is the first of kErrWords: [1] counts bounded waits that gave up, [2..11]
// record the first of them (block x / y / z, warp, the tile k whose wait ran out, tiles
// issued, the warp's tiles, the chunk's positions, the ns the drain wait of that tile
// took, 1 if it then completed), [12] the ns of the self-test's full bounded wait.
unsigned int* device_error_word();
constexpr unsigned int kErrTimeout = 1u, kErrBounds = 2u;
constexpr int kErrWords = 16;

// ---- the checked build ----------------------------------------------------------------
// Compiled with -DQPS_CHECK_BOUNDS=1 (the library variant libqps_checked.so), the kernels
// test every staged or addressed global / shared access against the extent it must stay
// in; a failing access is skipped and sets kErrBounds in the error word passed (none if
// NULL).  In the normal build the test is the constant true and compiles away.
#ifndef QPS_CHECK_BOUNDS
#define QPS_CHECK_BOUNDS 0
#endif
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* err) {
#if QPS_CHECK_BOUNDS
  if (!ok && err) atomicOr(err, kErrBounds);
  return ok;
#else
  (void)ok;
  (void)err;
  return true;
#endif
}

// ---- TurboQuant codebooks (computed once on the host from the Gaussian density) ----
struct Codebook {
  int n;                // levels: 4, 8 or 16
  float levels[16];     // ascending, the first n used
  float thresholds[15]; // the first n - 1 used
};
// bits = 2, 3 or 4; nullptr for any other width
const Codebook* tq_codebook(int bits);

// The TurboQuant tiers (V formats only) and their bit widths.
__host__ __device__ constexpr bool is_tq(int fmt) {
  return fmt == QPS_FMT_TQ2 || fmt == QPS_FMT_TQ3 || fmt == QPS_FMT_TQ4;
}
__host__ __device__ constexpr int tq_bits(int fmt) {
  return fmt == QPS_FMT_TQ2 ? 2 : fmt == QPS_FMT_TQ3 ? 3 : fmt == QPS_FMT_TQ4 ? 4 : 0;
}

// ---- bytes per row of each storage plane ------------------------------------------
inline int64_t plane_row_bytes(int fmt, int plane, int d) {
  switch (fmt) {
    case QPS_FMT_F16: return plane == 0 ? 2 * (int64_t)d : 0;
    case QPS_FMT_Q8_0: return plane == 0 ? d : plane == 1 ? 2 * (d / 32) : 0;
    case QPS_FMT_TQ3: return plane == 0 ? d / 4 : plane == 1 ? d / 8 : plane == 2 ? 2 : 0;
    case QPS_FMT_TQ2: return plane == 0 ? d / 4 : plane == 1 ? 2 : 0;
    case QPS_FMT_TQ4: return plane == 0 ? d / 2 : plane == 1 ? 2 : 0;
    default: return 0;
  }
}
inline int plane_count(int fmt) {
  switch (fmt) {
    case QPS_FMT_F16: return 1;
    case QPS_FMT_Q8_0: case QPS_FMT_TQ2: case QPS_FMT_TQ4: return 2;
    case QPS_FMT_TQ3: return 3;
    default: return 0;
  }
}

// ---- attention kernel parameters ---------------------------------------------------
constexpr int kMaxSignWords = 16;  // head_dim <= 512

struct KvSide {
  const void* data;
  const void* aux;
  const void* aux2;
  int64_t tok, head, batch;  // strides in rows
};

struct AttnParams {
  const __half* q;
  int64_t q_bstride;
  int batch, hq, hkv, d, group;
  int kfmt, vfmt;
  KvSide k, v;
  int64_t begin, end;
  int n_split;
  int64_t chunk;       // positions per split
  float scale, softcap;
  int shared;          // 1: every batch entry reads the same KV rows
  int n_q;             // query tokens per batch entry (>= 1)
  int causal;          // 1: query token i sees only positions <= q_pos + i
  int64_t q_pos;
  int rows_per_cta;    // shared ? batch * group : n_q * group
  int64_t rows_total;  // batch * n_q * hq
  float* o_parts;
  float* lse_parts;
  int part_offset;
  // extents the checked build tests accesses against: rows a view addresses (the
  // largest row index of [0, end) x heads x batch entries, + 1), q elements, and the
  // parts the o_parts / lse_parts buffers hold
  int64_t k_rows, v_rows, q_elems;
  int64_t parts_cap;
  unsigned int* err;  // device word set non-zero when a bounded in-kernel wait gives up
  uint32_t vsigns[kMaxSignWords];   // V rotation: s1
  uint32_t vsigns2[kMaxSignWords];  // s2 (all 0: none)
  int vblock;                       // Hadamard block width G (a power of two, <= d)
  float v_out_scale;                // 1 / sqrt(d * G)
  float k_rot_scale;                // a TurboQuant K: 1 / sqrt(G) (the rotated query)
  float k_norm_scale;               // and 1 / sqrt(d) (its decode)
  float tq_levels[16];  // the V tier's codebook (ascending)
};

// Query rows one tensor-core CTA holds (8 per n-tile): at head_dim <= 128, where the
// accumulators still fit in registers, up to 2 n-tiles, or 3 for per-entry rows (a
// verify batch: each row group would dequantise the same tiles again); a shared prefix
// is cheap to re-read from L2, so its rows keep the smaller tiles and more CTAs.
inline int mma_tile_rows(int d, int rows_per_cta, bool shared) {
  if (d > 128 || rows_per_cta <= 8) return 8;
  return (rows_per_cta <= 16 || shared) ? 16 : 24;
}

// CTAs per SM a tensor-core instance is built for (its register cap and stage budget):
// three for a TurboQuant V, whose decode chains leave the kernel latency-bound with 8
// warps per SM, where the accumulators leave registers for 12 warps (head_dim 64 with
// up to two n-tiles, 128 with one); else two (more CTAs did not help the fp16 / q8_0
// kernels, which are bound by HBM).
__host__ __device__ constexpr int mma_ctas_per_sm(int d, int ntw, int vfmt) {
  return (is_tq(vfmt) && ((d <= 64 && ntw <= 2) || (d == 128 && ntw == 1))) ? 3 : 2;
}

// Validated, resolved form of qps_attn_args.
qps_status resolve_attn(const qps_attn_args* a, AttnParams* p, int* n_split, size_t* ws_bytes);
qps_status launch_attn(const AttnParams& p, cudaStream_t stream);
qps_status launch_combine(const float* o_parts, const float* lse_parts, int n_parts,
                          int64_t rows, int d, float* o, float* lse, cudaStream_t stream,
                          unsigned int* err = nullptr);
// Runs a resolved attention in whichever output mode the args ask for; parts_capacity
// (if >= 0) is the number of parts the caller's o_parts / lse_parts buffers hold.
qps_status run_attn(const qps_attn_args* a, const AttnParams& p, int n_split, cudaStream_t s,
                    int64_t parts_capacity = -1);

qps_status launch_quant_q8_0(const __half* x, int64_t rows, int d, int64_t stride,
                             int8_t* codes, __half* scales, cudaStream_t s);
// TurboQuant encode at `bits` = 2, 3 or 4 with rotation diag(s2) blockdiag(H_block)
// diag(s1) (signs2 NULL: none); plane1 is the TQ3 sign plane (unused otherwise)
qps_status launch_quant_tq(int bits, const __half* x, int64_t rows, int d, int64_t stride,
                           const uint32_t* signs, const uint32_t* signs2, int block, uint8_t* plane0,
                           uint8_t* plane1, __half* norms, cudaStream_t s);

}  // namespace qps
