// Decode attention with merged output that allocates no memory at all.
//
// qps_attn_decode_window in its merged-output mode needs scratch for the per-split
// partial outputs (the caller passes it as `workspace`).  Some callers cannot provide
// or allocate device memory on the call path: code running where cudaMalloc is not
// allowed or too slow (inside a memory-pool-controlled serving loop, under an external
// allocator that owns all device memory, or in code that must not trigger the
// implicit synchronisation an allocation can cause).  For them this entry point keeps
// its scratch in a fixed, file-scope device array that the library carries in every
// GPU's memory from the moment its module is loaded until the process exits.
//
// Limits and rules (also stated in include/qps.h):
//   * the scratch holds at most kScratchBytes; larger requests are rejected;
//   * every call on a device shares the same array and leaves its contents behind; the
//     partials are fully rewritten by each call, so nothing needs clearing except the
//     error word, which is zeroed at set-up;
//   * calls that overlap on one GPU (other streams, other host threads) race on the
//     array: serialise them;
//   * the first call on each device looks up the array's device address (and zeroes
//     the error word); make that first call before any stream capture;
//   * a bounded in-kernel wait that gives up sets the error word at byte 0 of the same
//     array; this entry point never reads it back (that would need a synchronising
//     copy), and the outputs of such a call are not valid.
#include <mutex>

#include "internal.h"

namespace qps {

qps_status launch_attn_simple(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d64(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d128(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d256(const AttnParams& p, cudaStream_t s);
qps_status launch_attn_mma_d512(const AttnParams& p, cudaStream_t s);
bool attn_uses_mma(const AttnParams& p);

namespace {

// 8 MiB: room for e.g. 152 splits x 16 rows x 513 floats (head_dim 512), or
// 38 splits x 40 rows x 129 floats (head_dim 128), with headroom.
constexpr size_t kScratchBytes = (size_t)8 << 20;
constexpr size_t kErrOffset = 0;       // one unsigned int: the bounded-wait error word
constexpr size_t kPartsOffset = 256;   // the split partials start here

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch on that device
};

qps_status scratch_for_current_device(unsigned char** out) {
  static std::mutex mu;
  static DeviceScratch per_dev[64];
  int dev = 0;
  QPS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(QPS_ERR_UNSUPPORTED, "attn_decode_window_noalloc: device index >= 64");
  std::lock_guard<std::mutex> lk(mu);
  if (!per_dev[dev].base) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_window_noalloc: cudaGetSymbolAddress");
    e = cudaMemset(static_cast<unsigned char*>(ptr) + kErrOffset, 0, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_window_noalloc: clearing the error word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_window_noalloc: set-up");
    per_dev[dev].base = static_cast<unsigned char*>(ptr);
  }
  *out = per_dev[dev].base;
  return QPS_OK;
}

}  // namespace
}  // namespace qps

using namespace qps;

extern "C" qps_status qps_attn_decode_window_noalloc(const qps_attn_args* a, void* stream) {
  AttnParams p;
  int n_split = 0;
  qps_status st = resolve_attn(a, &p, &n_split, nullptr);
  if (st != QPS_OK) return st;
  if (a->o_parts) return fail(QPS_ERR_INVALID_ARG, "attn_decode_window_noalloc: merged-output mode only (o_parts must be NULL)");
  if (!a->o || !a->lse) return fail(QPS_ERR_INVALID_ARG, "attn_decode_window_noalloc: o / lse are NULL");
  const size_t o_bytes = (size_t)n_split * p.rows_total * p.d * sizeof(float);
  const size_t lse_off = kPartsOffset + ((o_bytes + 255) & ~(size_t)255);
  const size_t need = lse_off + (size_t)n_split * p.rows_total * sizeof(float);
  if (need > kScratchBytes)
    return fail(QPS_ERR_INVALID_ARG, "attn_decode_window_noalloc: the split partials need " + std::to_string(need) +
                                         " bytes, more than the fixed scratch of " + std::to_string(kScratchBytes) +
                                         " bytes; pass a smaller n_split");
  unsigned char* base = nullptr;
  st = scratch_for_current_device(&base);
  if (st != QPS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  p.o_parts = reinterpret_cast<float*>(base + kPartsOffset);
  p.lse_parts = reinterpret_cast<float*>(base + lse_off);
  p.part_offset = 0;
  p.parts_cap = n_split;
  p.err = reinterpret_cast<unsigned int*>(base + kErrOffset);
  if (!attn_uses_mma(p)) {
    // the CUDA-core kernel decodes one query token per row and has no causal limit:
    // refuse what it cannot compute, exactly as qps_attn_decode_window does
    if (p.n_q > 1 || p.causal)
      return fail(QPS_ERR_UNSUPPORTED, "attn_decode_window_noalloc: multi-query / causal decode needs the "
                                       "tensor-core path (token-contiguous planes, see qps_attn_path)");
    st = launch_attn_simple(p, s);
  } else {
    switch (p.d) {
      case 64: st = launch_attn_mma_d64(p, s); break;
      case 128: st = launch_attn_mma_d128(p, s); break;
      case 256: st = launch_attn_mma_d256(p, s); break;
      case 512: st = launch_attn_mma_d512(p, s); break;
      default: st = fail(QPS_ERR_UNSUPPORTED, "attn_decode_window_noalloc: head_dim");
    }
  }
  if (st != QPS_OK) return st;
  return launch_combine(p.o_parts, p.lse_parts, n_split, p.rows_total, p.d, a->o, a->lse, s, p.err);
}
