// Self-test of the kernels' bounded waits.
//
// The decode-attention kernels wait for their own asynchronous tile copies on
// shared-memory mbarriers, and every such wait is bounded: once one second of the GPU's
// global timer has passed without the phase completing, the wait gives up, the kernel
// sets the library's device error word and returns with invalid outputs instead of
// hanging the GPU.  That give-up path never runs in a healthy launch.  This entry point
// runs the same wait (mma::mbar_wait) on an mbarrier that nothing ever arrives on, so
// the path can be exercised on a GPU without a fault of any kind: one warp of one CTA
// waits one second, records the timeout (and how long the wait took) in the error word
// and exits; qps_device_status then reports QPS_ERR_TIMEOUT, and the context stays
// usable.
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
  const uint64_t t0 = mma::global_ns();
  const bool done = mma::mbar_wait(b, 0);
  const uint64_t t1 = mma::global_ns();
  __syncwarp();
  if (threadIdx.x == 0) {
    err[12] = (unsigned)min((uint64_t)0xffffffffu, t1 - t0);  // how long the full bounded wait took
    if (!done) atomicOr(err, 1u);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(b) : "memory");
  }
}

// The bounds checker's own test: one thread computes an index one past a 4-word
// shared array and guards the access with the same check the kernels use.  In the
// checked build the check fails, records kErrBounds and the store is skipped; the
// index is also clamped, so that no build of this kernel can write outside the array.
__global__ void __launch_bounds__(32) bounds_check_selftest_kernel(unsigned int* err, int n) {
  __shared__ int arr[4];
  if (threadIdx.x == 0) {
    const int i = n;  // n = 4: one past the end
    if (in_bounds(i >= 0 && i < 4, err)) arr[i < 4 ? i : 3] = 1;
    __syncwarp(1u);
  }
}

}  // namespace
}  // namespace qps

using namespace qps;

extern "C" int32_t qps_build_checked(void) { return QPS_CHECK_BOUNDS ? 1 : 0; }

extern "C" qps_status qps_selftest_bounds_check(void* stream) {
  if (!QPS_CHECK_BOUNDS)
    return fail(QPS_ERR_UNSUPPORTED, "selftest_bounds_check: this library was built without bounds checks "
                                     "(build variant \"checked\")");
  unsigned int* err = device_error_word();
  if (!err) return fail(QPS_ERR_CUDA, "selftest_bounds_check: no device error word");
  bounds_check_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, 4);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}

extern "C" qps_status qps_selftest_bounded_wait(void* stream) {
  unsigned int* err = device_error_word();
  if (!err) return fail(QPS_ERR_CUDA, "selftest_bounded_wait: no device error word");
  bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  count_launch();
  QPS_CUDA_TRY(cudaGetLastError());
  return QPS_OK;
}
