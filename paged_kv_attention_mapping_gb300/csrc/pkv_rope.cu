// Rotary position embedding fused into the slot-mapping append.
//
// Helios blog, "torch.sdpa and Flash Attention": Q and K are projected, RoPE
// is applied to both, then attention runs; llm-serving-engine README,
// component table "RoPE from scratch": rotary embeddings with cached sin/cos
// tables. The pages do not fix the variant; this is the half-split form: for
// pair i < d/2 of a head, x_i and x_{i+d/2} rotate by the angle
// pos * base^(-2i/d). One pass over the new tokens rotates each K row, writes
// it to its slot, copies V to its slot, and rotates the tick's Q rows, so the
// new tokens are read once instead of once for RoPE and again for the append.
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

// Work items are 16-byte vectors: a Q/K item covers E = 16 / sizeof(T)
// rotation pairs (E elements from each half of the row, with their E cos/sin
// pairs); a V item is E elements copied. A block takes a few whole tokens
// (TokenSpan) and consecutive threads take consecutive vectors of a row, so
// every access is a full, coalesced 16-byte one.
template <typename T>
__device__ __forceinline__ void rotate_vec(const T* __restrict__ src, T* __restrict__ dst, int a, int half,
                                           const float2* __restrict__ cs) {
  constexpr int E = 16 / sizeof(T);
  uint4 r1 = __ldg(reinterpret_cast<const uint4*>(src + a));
  uint4 r2 = __ldg(reinterpret_cast<const uint4*>(src + a + half));
  const T* x1 = reinterpret_cast<const T*>(&r1);
  const T* x2 = reinterpret_cast<const T*>(&r2);
  uint4 o1, o2;
  T* y1 = reinterpret_cast<T*>(&o1);
  T* y2 = reinterpret_cast<T*>(&o2);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float2 c = __ldg(cs + a + e);
    const float u = to_f32(x1[e]), w = to_f32(x2[e]);
    y1[e] = from_f32<T>(u * c.x - w * c.y);
    y2[e] = from_f32<T>(w * c.x + u * c.y);
  }
  *reinterpret_cast<uint4*>(dst + a) = o1;
  *reinterpret_cast<uint4*>(dst + a + half) = o2;
}

template <typename T>
__global__ void __launch_bounds__(256) rope_append_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                          const T* __restrict__ v, const int32_t* __restrict__ pos,
                                                          const float2* __restrict__ cs, int32_t max_pos,
                                                          const int64_t* __restrict__ slots, TokenSpan sp,
                                                          int32_t Hq, int32_t Hkv, int32_t D, int64_t pool_slots,
                                                          T* __restrict__ kc, T* __restrict__ vc, T* __restrict__ q_out,
                                                          int32_t* dev_status) {
  pdl_trigger();   // the attention call's plan does not read what this kernel writes
  constexpr int E = 16 / sizeof(T);
  const int half = D / 2;
  const int rv = half / E;                       // rotation vectors per Q/K row
  const int cv = D / E;                          // copy vectors per V row
  const int span = sp.tpb * sp.per_token;
  for (int j = threadIdx.x; j < span; j += blockDim.x) {
    const int tl = j / sp.per_token;
    int r = j - tl * sp.per_token;
    const int64_t t = (int64_t)blockIdx.x * sp.tpb + tl;
    if (t >= sp.T) break;   // items of later tokens follow
    const int p = __ldg(pos + t);
    const int64_t slot = __ldg(slots + t);
    if (r < (Hq + Hkv) * rv) {
      const int h = r / rv;
      const int a = (r - h * rv) * E;
      if (p < 0 || p >= max_pos) {
        if (a == 0) atomicOr(dev_status, PKV_DEV_BAD_POSITION);
        continue;
      }
      const float2* c = cs + (int64_t)p * half;
      if (h < Hq) {
        rotate_vec<T>(q + (t * Hq + h) * D, q_out + (t * Hq + h) * D, a, half, c);
      } else {
        if (slot < 0) continue;
        if (slot >= pool_slots) {
          if (a == 0 && h == Hq) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
          continue;
        }
        const int kh = h - Hq;
        rotate_vec<T>(k + (t * Hkv + kh) * D, kc + (slot * Hkv + kh) * D, a, half, c);
      }
    } else {
      r -= (Hq + Hkv) * rv;
      if (slot < 0 || slot >= pool_slots) continue;
      const int vh = r / cv;
      const int a = (r - vh * cv) * E;
      *reinterpret_cast<uint4*>(vc + (slot * Hkv + vh) * D + a) =
          __ldg(reinterpret_cast<const uint4*>(v + (t * Hkv + vh) * D + a));
    }
  }
}

cudaError_t launch_rope_append(const void* q, const void* k, const void* v, const int32_t* positions,
                               const float* cos_sin, int32_t max_pos, const int64_t* slots, int32_t T,
                               int32_t Hq, void* kc, void* vc, void* q_out, const pkv_cache_desc& c,
                               int32_t* dev_status, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int E = c.dtype == PKV_F32 ? 4 : 8;
  const int32_t per_token = (Hq + c.num_kv_heads) * (c.head_dim / 2 / E) + c.num_kv_heads * (c.head_dim / E);
  const TokenSpan sp = token_span(T, per_token, num_sms, 2);
  const unsigned blocks = (unsigned)sp.blocks();
  const int64_t pool_slots = (int64_t)c.num_pages * c.page_size;
  static const cudaError_t carve = [] {
    cudaError_t e = prefer_max_shared(rope_append_kernel<float>);
    if (e == cudaSuccess) e = prefer_max_shared(rope_append_kernel<__half>);
    if (e == cudaSuccess) e = prefer_max_shared(rope_append_kernel<__nv_bfloat16>);
    return e;
  }();
  if (carve != cudaSuccess) return carve;
  KernelTimer timer("rope_append", s);
  switch (c.dtype) {
    case PKV_F32:
      rope_append_kernel<float><<<blocks, 256, 0, s>>>(
          (const float*)q, (const float*)k, (const float*)v, positions, (const float2*)cos_sin, max_pos, slots, sp,
          Hq, c.num_kv_heads, c.head_dim, pool_slots, (float*)kc, (float*)vc, (float*)q_out, dev_status);
      break;
    case PKV_F16:
      rope_append_kernel<__half><<<blocks, 256, 0, s>>>(
          (const __half*)q, (const __half*)k, (const __half*)v, positions, (const float2*)cos_sin, max_pos, slots,
          sp, Hq, c.num_kv_heads, c.head_dim, pool_slots, (__half*)kc, (__half*)vc, (__half*)q_out, dev_status);
      break;
    default:
      rope_append_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
          (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, positions,
          (const float2*)cos_sin, max_pos, slots, sp, Hq, c.num_kv_heads, c.head_dim, pool_slots,
          (__nv_bfloat16*)kc, (__nv_bfloat16*)vc, (__nv_bfloat16*)q_out, dev_status);
  }
  return cudaGetLastError();
}

}  // namespace pkv

// cos/sin table: entry (p, i) = (cos(p * base^(-2i/d)), sin(...)), computed in
// double and stored as float pairs, [max_pos][d/2][2].
extern "C" int pkv_rope_table(double base, int32_t head_dim, int32_t max_pos, float* cos_sin) {
  if (!cos_sin) return PKV_E_NULL;
  if (!(base > 1.0) || head_dim < 2 || head_dim % 2 != 0 || max_pos < 1) return PKV_E_SHAPE;
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = pow(base, -2.0 * i / head_dim);
    for (int32_t p = 0; p < max_pos; ++p) {
      const double a = (double)p * inv_freq;
      cos_sin[((int64_t)p * half + i) * 2 + 0] = (float)cos(a);
      cos_sin[((int64_t)p * half + i) * 2 + 1] = (float)sin(a);
    }
  }
  return PKV_OK;
}
