// Self-test of the failure path that every kernel of the library shares: a
// wait on an mbarrier gives up after a time limit, records PKV_DEV_TIMEOUT in
// the device status word and lets the kernel return, so that a protocol error
// becomes a status the host reads instead of a hung GPU. The pages this
// library follows have no counterpart; the entry point exists so that tests
// can make such a wait run out on purpose (a barrier that nothing completes)
// and check the status, without faulting or hanging anything.
#include <cuda_runtime.h>

#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
namespace {

__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  sm100::mbar_init(&bar, 1);
  sm100::fence_mbar_init();
  // nothing arrives on `bar`: its first phase never completes, and the same
  // bounded wait the kernels use gives up after limit_ns
  if (!sm100::mbar_wait(&bar, 0, limit_ns)) atomicOr(dev_status, PKV_DEV_TIMEOUT);
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int32_t limit_us, pkv_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return PKV_E_SHAPE;
  int32_t* status = pkv::device_status_ptr();
  if (!status) return PKV_E_CUDA;
  pkv::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}
