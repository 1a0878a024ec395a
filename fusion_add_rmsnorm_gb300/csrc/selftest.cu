// Self-test of the device-side failure path: one thread waits, through the
// same bounded wait the pipelined kernels use, on an mbarrier that nothing
// ever arrives at.  The wait gives up after its budget (about one second),
// raises DEV_ERR_MBAR_TIMEOUT in the error word and the kernel returns
// normally, so the context stays usable and gbf_device_status() reports
// GBF_ETIMEOUT.  No fault, trap or unbounded spin is involved.
#include "kernels.h"
#include "tma.cuh"

namespace gbf {
namespace {

__global__ void bounded_wait_selftest_kernel(unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);                 // one arrival expected, none will come
  abort = 0;
  mbar_fence_init();
  mbar_wait(&bar, 0, &abort, err);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(unsigned int* err, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace gbf
