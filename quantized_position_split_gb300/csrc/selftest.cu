// Self-test of the kernels' bounded waits.
//
// The decode-attention kernels wait for their own asynchronous tile copies on
// shared-memory mbarriers, and every such wait is bounded: after 256 polls of at most
// about a millisecond each the wait gives up, the kernel sets the library's device
// error word and returns with invalid outputs instead of hanging the GPU.  That give-up
// path never runs in a healthy launch.  This entry point runs the same wait
// (mma::mbar_wait) on an mbarrier that nothing ever arrives on, so the path can be
// exercised on a GPU without a fault of any kind: one warp of one CTA waits well under
// a second, records the timeout in the error word and exits; qps_device_status then
// reports QPS_ERR_TIMEOUT, and the context stays usable.
#include "attn_mma.cuh"

namespace qps {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = mma::smem_addr(&bar);
  if (threadIdx.x == 0) {
    mma::mbar_init(b, 1);  // one arrival expected; none ever comes
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  const bool done = mma::mbar_wait(b, 0);
  __syncwarp();
  if (threadIdx.x == 0) {
    if (!done) atomicOr(err, 1u);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(b) : "memory");
  }
}

}  // namespace
}  // namespace qps

using namespace qps;

extern "C" qps_status qps_selftest_bounded_wait(void* stream) {
  unsigned int* err = device_error_word();
  if (!err) return fail(QPS_ERR_CUDA, "selftest_bounded_wait: no device error word");
  bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}
