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

// one warp per (token, head) row of Q, K or V; lanes walk the d/2 rotation pairs
template <typename T>
__global__ void __launch_bounds__(256) rope_append_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                          const T* __restrict__ v, const int32_t* __restrict__ pos,
                                                          const float2* __restrict__ cs, int32_t max_pos,
                                                          const int64_t* __restrict__ slots, int32_t T_,
                                                          int32_t Hq, int32_t Hkv, int32_t D, int64_t pool_slots,
                                                          T* __restrict__ kc, T* __restrict__ vc, T* __restrict__ q_out,
                                                          int32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)T_ * (Hq + 2 * Hkv);
  const int half = D / 2;
  for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < rows;
       row += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t t = row / (Hq + 2 * Hkv);
    const int h = (int)(row - t * (Hq + 2 * Hkv));
    const int p = __ldg(pos + t);
    if (h < Hq + Hkv && (p < 0 || p >= max_pos)) {
      if (lane == 0) atomicOr(dev_status, PKV_DEV_BAD_POSITION);
      continue;
    }
    if (h < Hq) {  // a query row: rotate into q_out
      const T* src = q + (t * Hq + h) * D;
      T* dst = q_out + (t * Hq + h) * D;
      for (int i = lane; i < half; i += 32) {
        const float2 c = __ldg(cs + (int64_t)p * half + i);
        const float x1 = to_f32(src[i]), x2 = to_f32(src[i + half]);
        dst[i] = from_f32<T>(x1 * c.x - x2 * c.y);
        dst[i + half] = from_f32<T>(x2 * c.x + x1 * c.y);
      }
      continue;
    }
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (lane == 0) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
      continue;
    }
    if (h < Hq + Hkv) {  // a key row: rotate into its slot
      const int kh = h - Hq;
      const T* src = k + (t * Hkv + kh) * D;
      T* dst = kc + (slot * Hkv + kh) * D;
      for (int i = lane; i < half; i += 32) {
        const float2 c = __ldg(cs + (int64_t)p * half + i);
        const float x1 = to_f32(src[i]), x2 = to_f32(src[i + half]);
        dst[i] = from_f32<T>(x1 * c.x - x2 * c.y);
        dst[i + half] = from_f32<T>(x2 * c.x + x1 * c.y);
      }
    } else {  // a value row: copied as is
      const int vh = h - Hq - Hkv;
      const T* src = v + (t * Hkv + vh) * D;
      T* dst = vc + (slot * Hkv + vh) * D;
      for (int i = lane; i < D; i += 32) dst[i] = src[i];
    }
  }
}

cudaError_t launch_rope_append(const void* q, const void* k, const void* v, const int32_t* positions,
                               const float* cos_sin, int32_t max_pos, const int64_t* slots, int32_t T,
                               int32_t Hq, void* kc, void* vc, void* q_out, const pkv_cache_desc& c,
                               int32_t* dev_status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t rows = (int64_t)T * (Hq + 2 * c.num_kv_heads);
  int64_t blocks = (rows * 32 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const int64_t pool_slots = (int64_t)c.num_pages * c.page_size;
  KernelTimer timer("rope_append", s);
  switch (c.dtype) {
    case PKV_F32:
      rope_append_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
          (const float*)q, (const float*)k, (const float*)v, positions, (const float2*)cos_sin, max_pos, slots, T,
          Hq, c.num_kv_heads, c.head_dim, pool_slots, (float*)kc, (float*)vc, (float*)q_out, dev_status);
      break;
    case PKV_F16:
      rope_append_kernel<__half><<<(unsigned)blocks, 256, 0, s>>>(
          (const __half*)q, (const __half*)k, (const __half*)v, positions, (const float2*)cos_sin, max_pos, slots,
          T, Hq, c.num_kv_heads, c.head_dim, pool_slots, (__half*)kc, (__half*)vc, (__half*)q_out, dev_status);
      break;
    default:
      rope_append_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
          (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, positions,
          (const float2*)cos_sin, max_pos, slots, T, Hq, c.num_kv_heads, c.head_dim, pool_slots,
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
