// kv_append: copy each new token's K and V rows into its slot of the page pool.
//
// Helios blog, "Prefill vs Decode" (decode writes the new token's slot) and
// Helios README, "Paged attention" (prefill and decode store K/V into their
// pages before attending). In the [pages, page_size, kv_heads, head_dim]
// layout one token's K row for all KV heads is Hkv * head_dim contiguous
// elements, so the append is a gather-free row copy: 16-byte vectors, one
// thread per vector, consecutive threads on consecutive vectors of one row
// (fully coalesced reads and writes). It is HBM-bound and bit-exact.
#include <cuda_fp8.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slots, int32_t T,
                                                        int32_t row_vecs, int64_t pool_slots,
                                                        uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                        int32_t* dev_status) {
  pdl_trigger();   // the attention call's plan does not read what this kernel writes
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

// Quantising append for an e4m3 cache. mini-vLLM, "Quantization": weights kept
// in 8 bits and widened before every matmul saved memory but slowed decode,
// and a fused low-precision kernel was the missing piece. The same idea on the
// KV cache: one byte per element halves what each decode step reads, and the
// attention kernel widens the codes in registers. The code of element x of KV head h
// is e4m3(x / scale[h]): the quotient in IEEE float32, then the nearest e4m3
// value with ties to even, saturating at +-448. A thread writes 16 codes (one
// 16-byte store) from 16 source elements of one head (head_dim is a multiple
// of 16), consecutive threads on consecutive vectors of a row.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_quant_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                              const int64_t* __restrict__ slots, int32_t T_,
                                                              int32_t row_vecs, int32_t head_vecs, int64_t pool_slots,
                                                              const float* __restrict__ k_scale,
                                                              const float* __restrict__ v_scale,
                                                              uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                              int32_t* dev_status) {
  pdl_trigger();   // the attention call's plan does not read what this kernel writes
  const int64_t per_token = 2 * (int64_t)row_vecs;
  const int64_t total = (int64_t)T_ * per_token;
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
    const float sc = __ldg((is_v ? v_scale : k_scale) + c / head_vecs);
    const T* src = (is_v ? v : k) + (t * row_vecs + c) * 16;
    constexpr int PER = 16 / sizeof(T);  // elements per 16-byte load
    float x[16];
#pragma unroll
    for (int j = 0; j < 16 / PER; ++j) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + j);
      const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
      for (int u = 0; u < PER; ++u) x[j * PER + u] = to_f32(e[u]);
    }
    uint32_t packed[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * j + 0], sc), __fdiv_rn(x[4 * j + 1], sc)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * j + 2], sc), __fdiv_rn(x[4 * j + 3], sc)), __NV_SATFINITE, __NV_E4M3);
      packed[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    (is_v ? vc : kc)[slot * row_vecs + c] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

cudaError_t launch_append_quant(const void* k, const void* v, int src_dtype, const int64_t* slots, int32_t T,
                                void* kc, void* vc, const pkv_cache_desc& c, const float* k_scale,
                                const float* v_scale, int32_t* dev_status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int32_t row_vecs = (int32_t)((int64_t)c.num_kv_heads * c.head_dim / 16);
  const int32_t head_vecs = c.head_dim / 16;
  const int64_t total = (int64_t)T * 2 * row_vecs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const int64_t pool_slots = (int64_t)c.num_pages * c.page_size;
  KernelTimer timer("kv_append_quant", s);
  switch (src_dtype) {
    case PKV_F32:
      kv_append_quant_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
          (const float*)k, (const float*)v, slots, T, row_vecs, head_vecs, pool_slots, k_scale, v_scale, (uint4*)kc,
          (uint4*)vc, dev_status);
      break;
    case PKV_F16:
      kv_append_quant_kernel<__half><<<(unsigned)blocks, 256, 0, s>>>(
          (const __half*)k, (const __half*)v, slots, T, row_vecs, head_vecs, pool_slots, k_scale, v_scale,
          (uint4*)kc, (uint4*)vc, dev_status);
      break;
    default:
      kv_append_quant_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
          (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, slots, T, row_vecs, head_vecs, pool_slots, k_scale,
          v_scale, (uint4*)kc, (uint4*)vc, dev_status);
  }
  return cudaGetLastError();
}

}  // namespace pkv
