// C ABI entry points: argument validation, error reporting, the TurboQuant codebooks, the
// attention plan / dispatch, the LSE combine and the native decode-step runner.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace qps {

// ---- errors ---------------------------------------------------------------------
namespace {
thread_local std::string g_last_error;
thread_local int64_t g_launches = 0;
}  // namespace

qps_status fail(qps_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

qps_status cuda_fail(cudaError_t err, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(err) + " (" + cudaGetErrorString(err) + ")";
  cudaGetLastError();  // the status carries the error: leave no non-sticky error behind
  return QPS_ERR_CUDA;
}

void count_launch(int n) { g_launches += n; }

int sm_count_current() {
  static std::atomic<int> cache[64];  // zero-initialised; any thread may fill an entry
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// ---- tensor maps (driver entry point looked up once through the runtime) -----------
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

bool encode_plane_map(TensorMap* map, const void* base, int row_bytes, int64_t tokens, int heads,
                      int64_t head_stride_rows, int batch, int64_t batch_stride_rows, int box_bytes,
                      int swizzle, int box_rows) {
  static_assert(sizeof(TensorMap) == sizeof(CUtensorMap), "tensor map size");
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) {
    fail(QPS_ERR_CUDA, "attention: cuTensorMapEncodeTiled is not available");
    return false;
  }
  const cuuint64_t dims[4] = {(cuuint64_t)row_bytes, (cuuint64_t)(tokens > 0 ? tokens : 1), (cuuint64_t)heads,
                              (cuuint64_t)batch};
  const cuuint64_t hs = (cuuint64_t)(head_stride_rows > 0 ? head_stride_rows : tokens) * row_bytes;
  const cuuint64_t bs = batch > 1 ? (cuuint64_t)batch_stride_rows * row_bytes : hs * (cuuint64_t)heads;
  const cuuint64_t strides[3] = {(cuuint64_t)row_bytes, hs > 0 ? hs : 16, bs > 0 ? bs : 16};
  const cuuint32_t box[4] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMapSwizzle sw = swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                          : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = enc(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fail(QPS_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r));
    return false;
  }
  return true;
}

unsigned int* device_error_word() {
  static std::mutex mu;
  static unsigned int* words[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!words[dev]) {
    unsigned int* w = nullptr;
    if (cudaMalloc(&w, kErrWords * sizeof(unsigned int)) != cudaSuccess) return nullptr;
    if (cudaMemset(w, 0, kErrWords * sizeof(unsigned int)) != cudaSuccess) return nullptr;
    words[dev] = w;
  }
  return words[dev];
}

// ---- TurboQuant codebooks -----------------------------------------------------------
// Lloyd iteration for the L-level MSE-optimal quantiser of N(0,1) in double precision
// (thresholds at midpoints, levels at the conditional means of their cells, starting
// from L evenly spaced levels on [-2, 2]), then each level rounded to the nearest fp16
// value, made exactly symmetric, and the thresholds set to the exact midpoints.
namespace {

double gauss_pdf(double x) { return std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI); }
double gauss_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// Nearest fp16-representable value (round half to even) of a positive normal double.
double round_to_half_grid(double x) {
  int e = 0;
  const double m = std::frexp(x, &e);  // x = m * 2^e, m in [0.5, 1)
  return std::ldexp(std::nearbyint(std::ldexp(m, 11)), e - 11);
}

Codebook make_codebook(int L) {
  double c[16], t[15], cn[16];
  for (int i = 0; i < L; ++i) c[i] = -2.0 + 4.0 * i / (L - 1);
  for (int it = 0; it < 100000; ++it) {
    for (int i = 0; i < L - 1; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    double delta = 0.0;
    for (int k = 0; k < L; ++k) {
      const double pa = k == 0 ? 0.0 : gauss_pdf(t[k - 1]);
      const double pb = k == L - 1 ? 0.0 : gauss_pdf(t[k]);
      const double fa = k == 0 ? 0.0 : gauss_cdf(t[k - 1]);
      const double fb = k == L - 1 ? 1.0 : gauss_cdf(t[k]);
      cn[k] = (pa - pb) / (fb - fa);
      delta = std::fmax(delta, std::fabs(cn[k] - c[k]));
    }
    for (int k = 0; k < L; ++k) c[k] = cn[k];
    if (delta < 1e-14) break;
  }
  Codebook cb{};
  cb.n = L;
  const int h = L / 2;
  for (int i = 0; i < h; ++i) {
    const float pos = (float)round_to_half_grid(std::fabs(c[h + i]));
    cb.levels[h + i] = pos;
    cb.levels[h - 1 - i] = -pos;
  }
  for (int i = 0; i < L - 1; ++i) cb.thresholds[i] = (cb.levels[i] + cb.levels[i + 1]) / 2.0f;
  return cb;
}

}  // namespace

const Codebook* tq_codebook(int bits) {
  static const Codebook cb2 = make_codebook(4), cb3 = make_codebook(8), cb4 = make_codebook(16);
  return bits == 2 ? &cb2 : bits == 3 ? &cb3 : bits == 4 ? &cb4 : nullptr;
}

// ---- attention argument resolution ------------------------------------------------
namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

qps_status check_view(const qps_kv_view& v, const char* name, bool allow_tq) {
  const std::string n(name);
  if (v.reserved0 != 0) return fail(QPS_ERR_INVALID_ARG, n + ": reserved0 must be 0");
  if (v.fmt != QPS_FMT_F16 && v.fmt != QPS_FMT_Q8_0 && !is_tq(v.fmt))
    return fail(QPS_ERR_INVALID_ARG, n + ": unknown format");
  if (is_tq(v.fmt) && !allow_tq)
    return fail(QPS_ERR_UNSUPPORTED, n + ": TurboQuant formats are supported for V only");
  if (!v.data) return fail(QPS_ERR_INVALID_ARG, n + ": data is NULL");
  if (!aligned(v.data, 16)) return fail(QPS_ERR_INVALID_ARG, n + ": data must be 16-byte aligned");
  if (v.fmt != QPS_FMT_F16) {
    // q8_0 scales and TQ3 sign planes: 4-byte aligned; TQ2 / TQ4 norms: fp16 aligned
    const size_t al = (v.fmt == QPS_FMT_TQ2 || v.fmt == QPS_FMT_TQ4) ? 2 : 4;
    if (!v.aux) return fail(QPS_ERR_INVALID_ARG, n + ": aux plane is NULL");
    if (!aligned(v.aux, al))
      return fail(QPS_ERR_INVALID_ARG, n + (al == 4 ? ": aux must be 4-byte aligned" : ": aux must be 2-byte aligned"));
  }
  if (v.fmt == QPS_FMT_TQ3) {
    if (!v.aux2) return fail(QPS_ERR_INVALID_ARG, n + ": aux2 (norms) is NULL");
    if (!aligned(v.aux2, 2)) return fail(QPS_ERR_INVALID_ARG, n + ": aux2 must be 2-byte aligned");
  }
  if (v.tok_stride <= 0) return fail(QPS_ERR_INVALID_ARG, n + ": tok_stride must be > 0");
  if (v.head_stride < 0 || v.batch_stride < 0)
    return fail(QPS_ERR_INVALID_ARG, n + ": strides must be >= 0");
  return QPS_OK;
}

// Split count: enough chunks for one full wave (ctas_per_sm resident CTAs on every SM),
// each chunk at least 512 positions, so each partial amortises its merge and the
// combine reads few parts, or 256 when 512-position chunks would leave SMs without a
// CTA (a short tail tile).
int auto_split(int64_t ntok, int ctas_per_split, int ctas_per_sm) {
  const int sms = sm_count_current();
  if (sms <= 0) return -1;
  const int64_t target = (int64_t)ctas_per_sm * sms;
  const int64_t by_occupancy = (target + ctas_per_split - 1) / ctas_per_split;
  int64_t n = std::min(by_occupancy, (ntok + 511) / 512);
  if (n * ctas_per_split < sms) n = std::min(by_occupancy, (ntok + 255) / 256);
  if (n < 1) n = 1;
  if (n > 65535) n = 65535;
  return (int)n;
}

}  // namespace

qps_status resolve_attn(const qps_attn_args* a, AttnParams* p, int* n_split_out, size_t* ws_bytes) {
  if (!a) return fail(QPS_ERR_INVALID_ARG, "attention: args is NULL");
  if (!a->q) return fail(QPS_ERR_INVALID_ARG, "attention: q is NULL");
  if (!aligned(a->q, 16)) return fail(QPS_ERR_INVALID_ARG, "attention: q must be 16-byte aligned");
  if (a->batch < 1 || a->hq < 1 || a->hkv < 1)
    return fail(QPS_ERR_INVALID_ARG, "attention: batch, hq, hkv must be >= 1");
  if (a->hq % a->hkv) return fail(QPS_ERR_INVALID_ARG, "attention: hq must be a multiple of hkv");
  if (a->d != 64 && a->d != 128 && a->d != 256 && a->d != 512)
    return fail(QPS_ERR_UNSUPPORTED, "attention: head_dim must be 64, 128, 256 or 512");
  if (a->n_q < 0 || a->n_q > 64) return fail(QPS_ERR_INVALID_ARG, "attention: n_q must be in [0, 64]");
  const int n_q = a->n_q < 1 ? 1 : a->n_q;
  if (a->batch > 1 && (a->q_batch_stride < (int64_t)n_q * a->hq * a->d || a->q_batch_stride % 8))
    return fail(QPS_ERR_INVALID_ARG, "attention: q_batch_stride must be >= n_q*hq*d and a multiple of 8");
  qps_status st = check_view(a->k, "attention k", true);
  if (st != QPS_OK) return st;
  st = check_view(a->v, "attention v", true);
  if (st != QPS_OK) return st;
  if (is_tq(a->k.fmt) && a->v.fmt != a->k.fmt)
    return fail(QPS_ERR_UNSUPPORTED, "attention: a TurboQuant K needs V in the same TurboQuant tier");
  if ((a->k.batch_stride == 0) != (a->v.batch_stride == 0))
    return fail(QPS_ERR_INVALID_ARG, "attention: k and v must both be shared (batch_stride 0) or both per-batch");
  if (a->kv_begin < 0 || a->kv_end < a->kv_begin)
    return fail(QPS_ERR_INVALID_ARG, "attention: need 0 <= kv_begin <= kv_end");
  // the tensor-core kernels address tiles by 32-bit token coordinates (tensor maps)
  if (a->kv_end > (int64_t)0x7fffffff - 64)
    return fail(QPS_ERR_UNSUPPORTED, "attention: kv_end must be below 2^31 - 64 positions");
  if (!std::isfinite(a->scale) || !std::isfinite(a->softcap))
    return fail(QPS_ERR_INVALID_ARG, "attention: scale and softcap must be finite");
  if (is_tq(a->v.fmt) && !a->v_signs)
    return fail(QPS_ERR_INVALID_ARG, "attention: v_signs is required for a TurboQuant V (and K)");
  if (a->reserved1 != 0) return fail(QPS_ERR_INVALID_ARG, "attention: reserved1 must be 0");
  const int vblock = a->v_block == 0 ? a->d : a->v_block;
  if (vblock < 32 || vblock > a->d || (vblock & (vblock - 1)))
    return fail(QPS_ERR_INVALID_ARG, "attention: v_block must be 0 or a power of two in [32, head_dim]");
  if (a->n_split < 0) return fail(QPS_ERR_INVALID_ARG, "attention: n_split must be >= 0");
  const bool shared = a->k.batch_stride == 0 && a->batch > 1;
  if (shared && n_q > 1)
    return fail(QPS_ERR_UNSUPPORTED, "attention: multi-query decode needs per-entry KV rows (batch_stride != 0)");
  const int group = a->hq / a->hkv;
  const int rows_per_cta = shared ? a->batch * group : n_q * group;
  if (rows_per_cta > 1024) return fail(QPS_ERR_UNSUPPORTED, "attention: more than 1024 query rows per KV head");
  const int64_t ntok = a->kv_end - a->kv_begin;
  // CTAs per chunk: one per (KV head, batch entry) and row group of the tensor-core tile
  const int tile_rows = mma_tile_rows(a->d, rows_per_cta, shared);
  const int ctas_per_split = a->hkv * (shared ? 1 : a->batch) * ((rows_per_cta + tile_rows - 1) / tile_rows);
  int n_split = a->n_split;
  if (n_split == 0) {
    n_split = auto_split(ntok, ctas_per_split, mma_ctas_per_sm(a->d, tile_rows / 8, a->v.fmt));
    if (n_split < 0) return fail(QPS_ERR_CUDA, "attention: cannot query the current device's SM count");
  }
  if (n_split > 65535) return fail(QPS_ERR_INVALID_ARG, "attention: n_split must be <= 65535");
  const int64_t rows_total = (int64_t)a->batch * n_q * a->hq;
  const size_t ws = ((size_t)n_split * rows_total * (a->d + 1) * sizeof(float) + 1024 + 255) & ~(size_t)255;
  if (n_split_out) *n_split_out = n_split;
  if (ws_bytes) *ws_bytes = ws;
  if (!p) return QPS_OK;

  std::memset(p, 0, sizeof(*p));
  p->q = reinterpret_cast<const __half*>(a->q);
  p->q_bstride = a->batch > 1 ? a->q_batch_stride : (int64_t)n_q * a->hq * a->d;
  p->batch = a->batch;
  p->hq = a->hq;
  p->hkv = a->hkv;
  p->d = a->d;
  p->group = group;
  p->kfmt = a->k.fmt;
  p->vfmt = a->v.fmt;
  p->k = KvSide{a->k.data, a->k.aux, a->k.aux2, a->k.tok_stride, a->k.head_stride, a->k.batch_stride};
  p->v = KvSide{a->v.data, a->v.aux, a->v.aux2, a->v.tok_stride, a->v.head_stride, a->v.batch_stride};
  p->begin = a->kv_begin;
  p->end = a->kv_end;
  p->n_split = n_split;
  p->chunk = ntok == 0 ? 1 : (ntok + n_split - 1) / n_split;
  p->scale = a->scale;
  p->softcap = a->softcap > 0.f ? a->softcap : 0.f;
  p->shared = shared ? 1 : 0;
  p->n_q = n_q;
  p->causal = a->causal ? 1 : 0;
  p->q_pos = a->q_pos;
  p->rows_per_cta = rows_per_cta;
  p->rows_total = rows_total;
  // the extents the checked build tests accesses against
  {
    const int nb = shared ? 1 : a->batch;
    auto view_rows = [&](const qps_kv_view& v) -> int64_t {
      if (a->kv_end == 0) return 0;
      return (int64_t)(nb - 1) * v.batch_stride + (a->kv_end - 1) * v.tok_stride +
             (int64_t)(a->hkv - 1) * v.head_stride + 1;
    };
    p->k_rows = view_rows(a->k);
    p->v_rows = view_rows(a->v);
    p->q_elems = (int64_t)(a->batch - 1) * p->q_bstride + (int64_t)n_q * a->hq * a->d;
    p->parts_cap = n_split;  // run_attn sets the real capacity
  }
  p->vblock = vblock;
  p->v_out_scale = (float)(1.0 / std::sqrt((double)a->d * (double)vblock));
  p->k_rot_scale = (float)(1.0 / std::sqrt((double)vblock));
  p->k_norm_scale = (float)(1.0 / std::sqrt((double)a->d));
  if (is_tq(a->v.fmt)) {
    for (int i = 0; i < a->d / 32; ++i) p->vsigns[i] = a->v_signs[i];
    if (a->v_signs2)
      for (int i = 0; i < a->d / 32; ++i) p->vsigns2[i] = a->v_signs2[i];
    const Codebook* cb = tq_codebook(tq_bits(a->v.fmt));
    for (int i = 0; i < cb->n; ++i) p->tq_levels[i] = cb->levels[i];
  }
  return QPS_OK;
}

qps_status launch_attn_simple(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d64(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d128(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d256(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d512(const AttnParams& p, cudaStream_t s);

namespace {

// The tensor-core kernel stages each plane of a (KV head, batch entry) as one
// token-contiguous range with 16-byte copies: it needs tok_stride == 1 and every
// plane's head / batch offsets on 16-byte boundaries.
bool side_fits_mma(const KvSide& s, int fmt, int d) {
  if (s.tok != 1) return false;
  const void* planes[3] = {s.data, s.aux, s.aux2};
  for (int i = 0; i < plane_count(fmt); ++i) {
    const int64_t rb = plane_row_bytes(fmt, i, d);
    if (((uintptr_t)planes[i] & 15) || (s.head * rb) % 16 || (s.batch * rb) % 16) return false;
  }
  return true;
}

}  // namespace

bool attn_uses_mma(const AttnParams& p) {
  return p.end <= 0x7fffffffLL && side_fits_mma(p.k, p.kfmt, p.d) && side_fits_mma(p.v, p.vfmt, p.d);
}

qps_status launch_attn(const AttnParams& p_in, cudaStream_t s) {
  AttnParams p = p_in;
  p.err = device_error_word();
  if (!p.err) return fail(QPS_ERR_CUDA, "attention: cannot allocate the device error word");
  if (!attn_uses_mma(p_in)) {
    if (p_in.n_q > 1 || p_in.causal)
      return fail(QPS_ERR_UNSUPPORTED, "attention: multi-query / causal decode needs the tensor-core path "
                                       "(token-contiguous planes, see qps_attn_path)");
    return launch_attn_simple(p, s);
  }
  switch (p.d) {
    case 64: return launch_attn_mma_d64(p, s);
    case 128: return launch_attn_mma_d128(p, s);
    case 256: return launch_attn_mma_d256(p, s);
    case 512: return launch_attn_mma_d512(p, s);
    default: return fail(QPS_ERR_UNSUPPORTED, "attention: head_dim must be 64, 128, 256 or 512");
  }
}

qps_status run_attn(const qps_attn_args* a, const AttnParams& p_in, int n_split, cudaStream_t s,
                    int64_t parts_capacity) {
  AttnParams p = p_in;
  if (a->o_parts) {
    if (!a->lse_parts) return fail(QPS_ERR_INVALID_ARG, "attention: lse_parts is NULL");
    if (a->part_offset < 0) return fail(QPS_ERR_INVALID_ARG, "attention: part_offset must be >= 0");
    p.o_parts = a->o_parts;
    p.lse_parts = a->lse_parts;
    p.part_offset = a->part_offset;
    // a caller's buffers hold at least the parts this call writes
    p.parts_cap = parts_capacity >= 0 ? parts_capacity : (int64_t)a->part_offset + n_split;
    return launch_attn(p, s);
  }
  if (!a->o || !a->lse) return fail(QPS_ERR_INVALID_ARG, "attention: o / lse are NULL and no o_parts given");
  size_t need = 0;
  resolve_attn(a, nullptr, nullptr, &need);
  if (!a->workspace || a->workspace_bytes < need)
    return fail(QPS_ERR_INVALID_ARG, "attention: workspace missing or smaller than qps_attn_plan reports");
  if (!aligned(a->workspace, 256)) return fail(QPS_ERR_INVALID_ARG, "attention: workspace must be 256-byte aligned");
  float* ws = reinterpret_cast<float*>(a->workspace);
  const int64_t rows = p.rows_total;
  p.o_parts = ws;
  p.lse_parts = ws + (size_t)n_split * rows * p.d;
  p.part_offset = 0;
  p.parts_cap = n_split;
  qps_status st = launch_attn(p, s);
  if (st != QPS_OK) return st;
  return launch_combine(p.o_parts, p.lse_parts, n_split, rows, p.d, a->o, a->lse, s, device_error_word());
}

}  // namespace qps

using namespace qps;

extern "C" {

int32_t qps_abi_version(void) { return QPS_ABI_VERSION; }

const char* qps_last_error(void) { return g_last_error.c_str(); }

const char* qps_status_name(int32_t st) {
  switch (st) {
    case QPS_OK: return "QPS_OK";
    case QPS_ERR_INVALID_ARG: return "QPS_ERR_INVALID_ARG";
    case QPS_ERR_UNSUPPORTED: return "QPS_ERR_UNSUPPORTED";
    case QPS_ERR_CUDA: return "QPS_ERR_CUDA";
    case QPS_ERR_TIMEOUT: return "QPS_ERR_TIMEOUT";
    case QPS_ERR_STATE: return "QPS_ERR_STATE";
    case QPS_ERR_INTERNAL: return "QPS_ERR_INTERNAL";
    default: return "QPS_UNKNOWN_STATUS";
  }
}

qps_status qps_device_status(int32_t reset) {
  unsigned int* w = device_error_word();
  if (!w) return fail(QPS_ERR_CUDA, "device_status: no device error word");
  unsigned int v = 0;
  QPS_CUDA_TRY(cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost));
  if (reset) QPS_CUDA_TRY(cudaMemset(w, 0, kErrWords * sizeof(unsigned int)));
  if (v & kErrBounds)
    return fail(QPS_ERR_INTERNAL, std::string("device_status: a bounds check of the checked build failed (the access "
                                              "was skipped; outputs are not valid)") +
                                      ((v & kErrTimeout) ? "; a bounded wait also gave up" : ""));
  if (v) return fail(QPS_ERR_TIMEOUT, "device_status: a kernel's bounded wait for its tile copies gave up");
  return QPS_OK;
}

qps_status qps_device_wait_record(uint32_t* words, int32_t n) {
  if (!words || n < 0) return fail(QPS_ERR_INVALID_ARG, "device_wait_record: need words and n >= 0");
  unsigned int* w = device_error_word();
  if (!w) return fail(QPS_ERR_CUDA, "device_wait_record: no device error word");
  const int m = n < kErrWords ? n : kErrWords;
  if (m > 0) QPS_CUDA_TRY(cudaMemcpy(words, w, m * sizeof(unsigned int), cudaMemcpyDeviceToHost));
  for (int i = m; i < n; ++i) words[i] = 0;
  return QPS_OK;
}

int64_t qps_launch_count(int32_t reset) {
  const int64_t n = g_launches;
  if (reset) g_launches = 0;
  return n;
}

qps_status qps_tq_codebook(int32_t bits, float* levels, float* thresholds) {
  const Codebook* cb = tq_codebook(bits);
  if (!cb) return fail(QPS_ERR_UNSUPPORTED, "tq_codebook: bits must be 2, 3 or 4");
  if (levels) std::memcpy(levels, cb->levels, sizeof(float) * cb->n);
  if (thresholds) std::memcpy(thresholds, cb->thresholds, sizeof(float) * (cb->n - 1));
  return QPS_OK;
}

qps_status qps_tq3_codebook(float* levels, float* thresholds) { return qps_tq_codebook(3, levels, thresholds); }

static qps_status check_encoder(const void* x, int64_t rows, int32_t d, int64_t stride,
                                const char* name) {
  const std::string n(name);
  if (rows < 0) return fail(QPS_ERR_INVALID_ARG, n + ": rows must be >= 0");
  if (d != 32 && d != 64 && d != 128 && d != 256 && d != 512)
    return fail(QPS_ERR_UNSUPPORTED, n + ": head_dim must be 32, 64, 128, 256 or 512");
  if (rows > 0 && !x) return fail(QPS_ERR_INVALID_ARG, n + ": x is NULL");
  if (stride < d) return fail(QPS_ERR_INVALID_ARG, n + ": x_row_stride must be >= head_dim");
  return QPS_OK;
}

qps_status qps_kv_quant_q8_0(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                             void* codes, void* scales, void* stream) {
  qps_status st = check_encoder(x, rows, d, x_row_stride, "kv_quant_q8_0");
  if (st != QPS_OK) return st;
  if (rows == 0) return QPS_OK;
  if (!codes || !scales) return fail(QPS_ERR_INVALID_ARG, "kv_quant_q8_0: codes / scales are NULL");
  if (!aligned(x, 16) || x_row_stride % 8)
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_q8_0: x must be 16-byte aligned with a row stride multiple of 8");
  if (!aligned(codes, 8) || !aligned(scales, 2))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_q8_0: codes must be 8-byte and scales 2-byte aligned");
  return launch_quant_q8_0(reinterpret_cast<const __half*>(x), rows, d, x_row_stride,
                           reinterpret_cast<int8_t*>(codes), reinterpret_cast<__half*>(scales),
                           reinterpret_cast<cudaStream_t>(stream));
}

qps_status qps_kv_quant_tq3(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* lo2, void* hi1, void* norms, void* stream) {
  qps_status st = check_encoder(x, rows, d, x_row_stride, "kv_quant_tq3");
  if (st != QPS_OK) return st;
  if (!signs) return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq3: signs is NULL");
  if (rows == 0) return QPS_OK;
  if (!lo2 || !hi1 || !norms) return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq3: an output plane is NULL");
  if (!aligned(x, 2) || !aligned(hi1, 4) || !aligned(norms, 2))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq3: x / norms must be 2-byte and hi1 4-byte aligned");
  return launch_quant_tq(3, reinterpret_cast<const __half*>(x), rows, d, x_row_stride, signs, nullptr, d,
                         reinterpret_cast<uint8_t*>(lo2), reinterpret_cast<uint8_t*>(hi1),
                         reinterpret_cast<__half*>(norms), reinterpret_cast<cudaStream_t>(stream));
}

qps_status qps_kv_quant_tq_rot(int32_t bits, const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                               const uint32_t* signs1, const uint32_t* signs2, int32_t block, void* plane0,
                               void* plane1, void* norms, void* stream) {
  if (bits < 2 || bits > 4) return fail(QPS_ERR_UNSUPPORTED, "kv_quant_tq_rot: bits must be 2, 3 or 4");
  qps_status st = check_encoder(x, rows, d, x_row_stride, "kv_quant_tq_rot");
  if (st != QPS_OK) return st;
  if (!signs1) return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq_rot: signs1 is NULL");
  const int g = block == 0 ? d : block;
  if (g < 32 || g > d || (g & (g - 1)))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq_rot: block must be 0 or a power of two in [32, head_dim]");
  if (rows == 0) return QPS_OK;
  if (!plane0 || !norms || (bits == 3 && !plane1))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq_rot: an output plane is NULL");
  if (!aligned(x, 2) || !aligned(norms, 2) || (bits == 3 && !aligned(plane1, 4)))
    return fail(QPS_ERR_INVALID_ARG, "kv_quant_tq_rot: x / norms must be 2-byte and plane1 4-byte aligned");
  return launch_quant_tq(bits, reinterpret_cast<const __half*>(x), rows, d, x_row_stride, signs1, signs2, g,
                         reinterpret_cast<uint8_t*>(plane0), bits == 3 ? reinterpret_cast<uint8_t*>(plane1) : nullptr,
                         reinterpret_cast<__half*>(norms), reinterpret_cast<cudaStream_t>(stream));
}

// TQ2 / TQ4: one plane of sign-magnitude fields and the norms
static qps_status kv_quant_tq_fields(int bits, const char* name, const void* x, int64_t rows, int32_t d,
                                     int64_t x_row_stride, const uint32_t* signs, void* codes,
                                     void* norms, void* stream) {
  const std::string n(name);
  qps_status st = check_encoder(x, rows, d, x_row_stride, name);
  if (st != QPS_OK) return st;
  if (!signs) return fail(QPS_ERR_INVALID_ARG, n + ": signs is NULL");
  if (rows == 0) return QPS_OK;
  if (!codes || !norms) return fail(QPS_ERR_INVALID_ARG, n + ": an output plane is NULL");
  if (!aligned(x, 2) || !aligned(norms, 2))
    return fail(QPS_ERR_INVALID_ARG, n + ": x / norms must be 2-byte aligned");
  return launch_quant_tq(bits, reinterpret_cast<const __half*>(x), rows, d, x_row_stride, signs, nullptr, d,
                         reinterpret_cast<uint8_t*>(codes), nullptr, reinterpret_cast<__half*>(norms),
                         reinterpret_cast<cudaStream_t>(stream));
}

qps_status qps_kv_quant_tq2(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* codes, void* norms, void* stream) {
  return kv_quant_tq_fields(2, "kv_quant_tq2", x, rows, d, x_row_stride, signs, codes, norms, stream);
}

qps_status qps_kv_quant_tq4(const void* x, int64_t rows, int32_t d, int64_t x_row_stride,
                            const uint32_t* signs, void* codes, void* norms, void* stream) {
  return kv_quant_tq_fields(4, "kv_quant_tq4", x, rows, d, x_row_stride, signs, codes, norms, stream);
}

qps_status qps_attn_plan(const qps_attn_args* a, int32_t* n_split_out, size_t* workspace_bytes_out) {
  int n = 0;
  size_t ws = 0;
  qps_status st = resolve_attn(a, nullptr, &n, &ws);
  if (st != QPS_OK) return st;
  if (n_split_out) *n_split_out = n;
  if (workspace_bytes_out) *workspace_bytes_out = a->o_parts ? 0 : ws;
  return QPS_OK;
}

int32_t qps_attn_path(const qps_attn_args* a) {
  AttnParams p;
  int n = 0;
  const qps_attn_args* probe = a;
  qps_attn_args tmp;
  if (a && a->n_split == 0) {  // the kernel choice does not depend on the split count
    tmp = *a;
    tmp.n_split = 1;
    probe = &tmp;
  }
  qps_status st = resolve_attn(probe, &p, &n, nullptr);
  if (st != QPS_OK) return -(int32_t)st;
  return attn_uses_mma(p) ? 1 : 0;
}

qps_status qps_attn_decode_window(const qps_attn_args* a, void* stream) {
  AttnParams p;
  int n = 0;
  qps_status st = resolve_attn(a, &p, &n, nullptr);
  if (st != QPS_OK) return st;
  return run_attn(a, p, n, reinterpret_cast<cudaStream_t>(stream));
}

qps_status qps_lse_combine(const float* o_parts, const float* lse_parts, int32_t n_parts,
                           int64_t rows, int32_t d, float* o, float* lse, void* stream) {
  if (n_parts < 1) return fail(QPS_ERR_INVALID_ARG, "lse_combine: n_parts must be >= 1");
  if (rows < 0) return fail(QPS_ERR_INVALID_ARG, "lse_combine: rows must be >= 0");
  if (rows == 0) return QPS_OK;
  if (!o_parts || !lse_parts || !o || !lse) return fail(QPS_ERR_INVALID_ARG, "lse_combine: NULL pointer");
  if (!aligned(o_parts, 4) || !aligned(o, 4)) return fail(QPS_ERR_INVALID_ARG, "lse_combine: misaligned pointer");
  return launch_combine(o_parts, lse_parts, n_parts, rows, d, o, lse, reinterpret_cast<cudaStream_t>(stream),
                        device_error_word());
}

}  // extern "C"
