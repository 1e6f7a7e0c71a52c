// Self-check of the failure path every pipelined kernel relies on: a barrier
// wait that nothing ever satisfies must give up after its limit, record
// POETX_ERR_TIMEOUT in the device status word and let the kernel return, so
// the context stays usable.  No fault, trap or endless loop is involved.
#include "internal.h"
#include "poetx.h"
#include "ptx.cuh"

namespace poetx {
namespace {

__global__ void wait_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that no thread ever makes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns))
    atomicCAS(status, 0, static_cast<int>(POETX_ERR_TIMEOUT));
}

}  // namespace
}  // namespace poetx

extern "C" poetx_status poetx_selftest_wait_timeout(unsigned int limit_us, poetx_stream stream) {
  if (limit_us == 0 || limit_us > 1000000u) return POETX_ERR_INVALID_ARG;
  int* status = poetx::device_status_ptr();
  if (status == nullptr) return POETX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  poetx::prof_begin("selftest", s);
  poetx::wait_timeout_kernel<<<1, 32, 0, s>>>(status, 1000ull * limit_us);
  poetx::prof_end("selftest", s);
  return cudaGetLastError() == cudaSuccess ? POETX_OK : POETX_ERR_CUDA;
}
