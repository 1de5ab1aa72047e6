// kv_append: copy each new token's K and V rows into its slot of the page pool.
//
// Helios blog, "Prefill vs Decode" (decode writes the new token's slot) and
// Helios README, "Paged attention" (prefill and decode store K/V into their
// pages before attending). In the [pages, page_size, kv_heads, head_dim]
// layout one token's K row for all KV heads is Hkv * head_dim contiguous
// elements, so the append is a gather-free row copy of 16-byte vectors,
// consecutive threads on consecutive vectors of one row (fully coalesced reads
// and writes), with a block per few tokens (TokenSpan). It is HBM-bound and
// bit-exact.
#include <cuda_fp8.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_U = 4;   // items a thread loads before it stores any

// Item j of this block's span: its token t (t >= T: past the tick) and its
// index c among the token's items.
__device__ __forceinline__ void span_item(const TokenSpan& sp, int j, int64_t* t, int* c) {
  const int tl = j / sp.per_token;
  *c = j - tl * sp.per_token;
  *t = (int64_t)blockIdx.x * sp.tpb + tl;
}

// K items first, then V items, of each token. Every thread issues the loads of
// up to APPEND_U items before its stores, so a block keeps 16 KB of reads in
// flight; a token's source rows are read whatever its slot (the address does
// not depend on it), the slot only decides the store.
__global__ void __launch_bounds__(APPEND_THREADS) kv_append_kernel(const uint4* __restrict__ k,
                                                                   const uint4* __restrict__ v,
                                                                   const int64_t* __restrict__ slots, TokenSpan sp,
                                                                   int32_t row_vecs, int64_t pool_slots,
                                                                   uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                                   int32_t* dev_status) {
  pdl_trigger();   // the attention call's plan does not read what this kernel writes
  const int span = sp.tpb * sp.per_token;
  for (int base = 0; base < span; base += APPEND_THREADS * APPEND_U) {
    uint4 x[APPEND_U];
    int64_t dst[APPEND_U];
    bool is_v[APPEND_U];
#pragma unroll
    for (int u = 0; u < APPEND_U; ++u) {
      const int j = base + u * APPEND_THREADS + (int)threadIdx.x;
      dst[u] = -1;
      is_v[u] = false;
      if (j >= span) continue;
      int64_t t;
      int c;
      span_item(sp, j, &t, &c);
      if (t >= sp.T) continue;
      is_v[u] = c >= row_vecs;
      const int cc = is_v[u] ? c - row_vecs : c;
      x[u] = __ldg((is_v[u] ? v : k) + t * row_vecs + cc);
      const int64_t slot = __ldg(slots + t);
      if (slot >= pool_slots) {
        if (c == 0) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
      } else if (slot >= 0) {
        dst[u] = slot * row_vecs + cc;
      }
    }
#pragma unroll
    for (int u = 0; u < APPEND_U; ++u)
      if (dst[u] >= 0) (is_v[u] ? vc : kc)[dst[u]] = x[u];
  }
}

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int32_t T, void* kc, void* vc,
                          const pkv_cache_desc& c, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int elt = c.dtype == PKV_F32 ? 4 : 2;
  const int32_t row_vecs = (int32_t)((int64_t)c.num_kv_heads * c.head_dim * elt / 16);
  const TokenSpan sp = token_span(T, 2 * row_vecs, num_sms, APPEND_U, 3);
  static const cudaError_t carve = prefer_max_shared(kv_append_kernel);
  if (carve != cudaSuccess) return carve;
  KernelTimer timer("kv_append", s);
  kv_append_kernel<<<(unsigned)sp.blocks(), APPEND_THREADS, 0, s>>>(
      (const uint4*)k, (const uint4*)v, slots, sp, row_vecs, (int64_t)c.num_pages * c.page_size, (uint4*)kc,
      (uint4*)vc, device_status_ptr());
  return cudaGetLastError();
}

// Quantising append for an e4m3 cache. mini-vLLM, "Quantization": weights kept
// in 8 bits and widened before every matmul saved memory but slowed decode,
// and a fused low-precision kernel was the missing piece. The same idea on the
// KV cache: one byte per element halves what each decode step reads, and the
// attention kernel widens the codes in registers. The code of element x of KV head h
// is e4m3(x / scale[h]): the quotient in IEEE float32, then the nearest e4m3
// value with ties to even, saturating at +-448. An item writes 16 codes (one
// 16-byte store) from 16 source elements of one head (head_dim is a multiple
// of 16), consecutive threads on consecutive vectors of a row.
template <typename T>
__global__ void __launch_bounds__(APPEND_THREADS) kv_append_quant_kernel(
    const T* __restrict__ k, const T* __restrict__ v, const int64_t* __restrict__ slots, TokenSpan sp,
    int32_t row_vecs, int32_t head_vecs, int64_t pool_slots, const float* __restrict__ k_scale,
    const float* __restrict__ v_scale, uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* dev_status) {
  pdl_trigger();   // the attention call's plan does not read what this kernel writes
  const int span = sp.tpb * sp.per_token;
  for (int j = threadIdx.x; j < span; j += APPEND_THREADS) {
    int64_t t;
    int c;
    span_item(sp, j, &t, &c);
    if (t >= sp.T) break;   // items of later tokens follow
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (c == 0) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const bool is_v = c >= row_vecs;
    const int cc = is_v ? c - row_vecs : c;
    const float sc = __ldg((is_v ? v_scale : k_scale) + cc / head_vecs);
    const T* src = (is_v ? v : k) + (t * row_vecs + cc) * 16;
    constexpr int PER = 16 / sizeof(T);  // elements per 16-byte load
    float x[16];
#pragma unroll
    for (int q = 0; q < 16 / PER; ++q) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + q);
      const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
      for (int u = 0; u < PER; ++u) x[q * PER + u] = to_f32(e[u]);
    }
    uint32_t packed[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * q + 0], sc), __fdiv_rn(x[4 * q + 1], sc)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * q + 2], sc), __fdiv_rn(x[4 * q + 3], sc)), __NV_SATFINITE, __NV_E4M3);
      packed[q] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    (is_v ? vc : kc)[slot * row_vecs + cc] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

cudaError_t launch_append_quant(const void* k, const void* v, int src_dtype, const int64_t* slots, int32_t T,
                                void* kc, void* vc, const pkv_cache_desc& c, const float* k_scale,
                                const float* v_scale, int32_t* dev_status, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int32_t row_vecs = (int32_t)((int64_t)c.num_kv_heads * c.head_dim / 16);
  const int32_t head_vecs = c.head_dim / 16;
  const TokenSpan sp = token_span(T, 2 * row_vecs, num_sms, 2);
  const unsigned blocks = (unsigned)sp.blocks();
  const int64_t pool_slots = (int64_t)c.num_pages * c.page_size;
  static const cudaError_t carve = [] {
    cudaError_t e = prefer_max_shared(kv_append_quant_kernel<float>);
    if (e == cudaSuccess) e = prefer_max_shared(kv_append_quant_kernel<__half>);
    if (e == cudaSuccess) e = prefer_max_shared(kv_append_quant_kernel<__nv_bfloat16>);
    return e;
  }();
  if (carve != cudaSuccess) return carve;
  KernelTimer timer("kv_append_quant", s);
  switch (src_dtype) {
    case PKV_F32:
      kv_append_quant_kernel<float><<<blocks, APPEND_THREADS, 0, s>>>(
          (const float*)k, (const float*)v, slots, sp, row_vecs, head_vecs, pool_slots, k_scale, v_scale, (uint4*)kc,
          (uint4*)vc, dev_status);
      break;
    case PKV_F16:
      kv_append_quant_kernel<__half><<<blocks, APPEND_THREADS, 0, s>>>(
          (const __half*)k, (const __half*)v, slots, sp, row_vecs, head_vecs, pool_slots, k_scale, v_scale,
          (uint4*)kc, (uint4*)vc, dev_status);
      break;
    default:
      kv_append_quant_kernel<__nv_bfloat16><<<blocks, APPEND_THREADS, 0, s>>>(
          (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, slots, sp, row_vecs, head_vecs, pool_slots, k_scale,
          v_scale, (uint4*)kc, (uint4*)vc, dev_status);
  }
  return cudaGetLastError();
}

}  // namespace pkv
