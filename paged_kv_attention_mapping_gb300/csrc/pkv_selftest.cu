// Self-test of the failure path that every kernel of the library shares. The
// pipeline waits of the decode and prefill kernels all go through
// sm100::wait_or_abort / warp_wait_or_abort: a wait gives up after a time
// limit, raises the CTA's abort flag, records PKV_DEV_TIMEOUT in the call's
// error word and in the device status word, and every other waiting warp of
// the CTA sees the flag, leaves its loop and returns. A protocol error thus
// becomes a status the host reads instead of a hung GPU. The pages this library
// follows have no counterpart; the entry point exists so that tests can make
// such a wait run out on purpose (barriers that nothing completes) and check
// the status, without faulting or hanging anything.
#include <cuda_runtime.h>

#include "pagedkv.h"
#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
namespace {

constexpr int SELFTEST_WARPS = 10;   // the prefill kernel's CTA: producer, MMA issuer, 8 softmax warps

// One CTA laid out like the prefill kernel's. Nothing ever arrives on any of
// the three barriers. Warp 0 (the producer's role) waits with the caller's
// short limit and gives up first; warp 1's elected thread (the MMA issuer's
// role, a single-thread wait) and warps 2-9 (the softmax warps, warp-voted
// waits) wait with the kernels' own limit and must leave through the abort
// flag long before it. Each warp that returns counts itself in result[1].
__global__ void __launch_bounds__(SELFTEST_WARPS * 32)
    selftest_wait_kernel(uint64_t limit_ns, int32_t* dev_status, int32_t* result) {
  __shared__ __align__(8) uint64_t bar_empty, bar_full, bar_sfull;
  __shared__ volatile int s_abort;
  __shared__ int32_t s_err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar_empty, 1);
    sm100::mbar_init(&bar_full, 1);
    sm100::mbar_init(&bar_sfull, 1);
    sm100::fence_mbar_init();
    s_abort = 0;
    s_err = 0;
  }
  __syncthreads();
  bool ok;
  if (warp == 0) {
    ok = sm100::warp_wait_or_abort(&bar_empty, 0, &s_abort, &s_err, dev_status, limit_ns);
  } else if (warp == 1) {
    ok = true;
    if (lane == 0) ok = sm100::wait_or_abort(&bar_full, 0, &s_abort, &s_err, dev_status);
    ok = __shfl_sync(0xffffffffu, ok, 0);
  } else {
    ok = sm100::warp_wait_or_abort(&bar_sfull, 0, &s_abort, &s_err, dev_status);
  }
  if (result != nullptr && lane == 0 && !ok) atomicAdd(&result[1], 1);
  __syncthreads();
  if (result != nullptr && threadIdx.x == 0) result[0] = s_err;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int32_t limit_us, int32_t* result, pkv_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return PKV_E_SHAPE;
  if (((uintptr_t)result & 3u) != 0) return PKV_E_ALIGN;
  int32_t* status = pkv::device_status_ptr();
  if (!status) return PKV_E_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (result != nullptr && cudaMemsetAsync(result, 0, 2 * sizeof(int32_t), s) != cudaSuccess)
    return pkv::cuda_fail(cudaGetLastError(), "selftest memset");
  pkv::selftest_wait_kernel<<<1, pkv::SELFTEST_WARPS * 32, 0, s>>>((uint64_t)limit_us * 1000ull, status, result);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "selftest");
}
