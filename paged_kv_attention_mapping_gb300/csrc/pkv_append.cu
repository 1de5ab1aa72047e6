// kv_append: copy each new token's K and V rows into its slot of the page pool.
//
// Helios blog, "Prefill vs Decode" (decode writes the new token's slot) and
// Helios README, "Paged attention" (prefill and decode store K/V into their
// pages before attending). In the [pages, page_size, kv_heads, head_dim]
// layout one token's K row for all KV heads is Hkv * head_dim contiguous
// elements, so the append is a gather-free row copy: 16-byte vectors, one
// thread per vector, consecutive threads on consecutive vectors of one row
// (fully coalesced reads and writes). It is HBM-bound and bit-exact.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slots, int32_t T,
                                                        int32_t row_vecs, int64_t pool_slots,
                                                        uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                        int32_t* dev_status) {
  const int64_t per_token = 2 * (int64_t)row_vecs;
  const int64_t total = (int64_t)T * per_token;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t r = i - t * per_token;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (r == 0) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const bool is_v = r >= row_vecs;
    const int64_t c = is_v ? r - row_vecs : r;
    const uint4 x = __ldg((is_v ? v : k) + t * row_vecs + c);
    (is_v ? vc : kc)[slot * row_vecs + c] = x;
  }
}

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int32_t T, void* kc, void* vc,
                          const pkv_cache_desc& c, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int elt = c.dtype == PKV_F32 ? 4 : 2;
  const int32_t row_vecs = (int32_t)((int64_t)c.num_kv_heads * c.head_dim * elt / 16);
  const int64_t total = (int64_t)T * 2 * row_vecs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  KernelTimer timer("kv_append", s);
  kv_append_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      (const uint4*)k, (const uint4*)v, slots, T, row_vecs, (int64_t)c.num_pages * c.page_size, (uint4*)kc,
      (uint4*)vc, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace pkv
