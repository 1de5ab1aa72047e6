// Row path: attention of single query rows (decode tokens, and rows of short
// chunks) over their sequence's pages, on CUDA cores, plus the split-KV merge.
//
// Helios blog, "torch.sdpa and Flash Attention": softmax(Q K^T / sqrt(d)) V,
// with the query heads of one GQA group sharing one KV head. A work item is
// (row, KV head, split): one warp streams that KV head's keys of the split
// once, page by page through the page table, and serves all g query heads of
// the group from each loaded key (online softmax in the exp2 domain with fp32
// state, warp-shuffle reductions). Keys past the row's visible length are never
// loaded, so stale or NaN slots cannot leak in. Items of rows whose keys were
// split write a normalised partial (o, lse) into the workspace; the combine
// kernel merges them: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
#include <cuda_runtime.h>

#include <type_traits>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int ROWS_WARPS = 4;
constexpr int ROWS_BLOCKS_PER_SM = 8;

int rows_kernel_workers(int num_sms) { return num_sms * ROWS_BLOCKS_PER_SM * ROWS_WARPS; }

__device__ __forceinline__ int upper_bound_dev(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// U keys per step: loads of all U keys are issued before the math.
template <typename T, int D, int G, int U>
__global__ void __launch_bounds__(ROWS_WARPS * 32) rows_kernel(AttnArgs a) {
  constexpr int DPL = D / 32;  // dims per lane
  const int lane = threadIdx.x & 31;
  int32_t* ctrl = (int32_t*)(a.ws + a.lay.ctrl);
  const int32_t* rp_row = (const int32_t*)(a.ws + a.lay.rp_row);
  const int32_t* rp_seq = (const int32_t*)(a.ws + a.lay.rp_seq);
  const int32_t* rp_keys = (const int32_t*)(a.ws + a.lay.rp_keys);
  const int32_t* rp_item_begin = (const int32_t*)(a.ws + a.lay.rp_item_begin);
  const int32_t* rp_part_begin = (const int32_t*)(a.ws + a.lay.rp_part_begin);
  float* part_o = (float*)(a.ws + a.lay.part_o);
  float* part_lse = (float*)(a.ws + a.lay.part_lse);
  const int n_items = *(volatile int32_t*)&ctrl[CTRL_N_ITEMS];
  const int n_rp = *(volatile int32_t*)&ctrl[CTRL_N_RP];
  const int C = *(volatile int32_t*)&ctrl[CTRL_CHUNK];
  const T* __restrict__ kc = (const T*)a.k_cache;
  const T* __restrict__ vc = (const T*)a.v_cache;
  const T* __restrict__ qp = (const T*)a.q;
  const int64_t kstride = (int64_t)a.Hkv * D;  // elements between consecutive slots
  const float qscale = a.scale * LOG2E;

  for (;;) {
    int item = 0;
    if (lane == 0) item = atomicAdd(&ctrl[CTRL_ITEM_NEXT], 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= n_items) break;
    // the item's row-path row; its items run split by split, KV heads adjacent
    const int rj = upper_bound_dev(rp_item_begin, n_rp + 1, item) - 1;
    const int jj = item - __ldg(rp_item_begin + rj);
    const int limit = __ldg(rp_keys + rj);   // keys the row sees
    const int part0 = __ldg(rp_part_begin + rj);
    const int r = __ldg(rp_row + rj);
    const int b = __ldg(rp_seq + rj);
    const int sp = jj / a.Hkv;
    const int kvh = jj - sp * a.Hkv;
    const int nsplit = (limit + C - 1) / C;
    const int local = kvh * nsplit + sp;      // partial slot within the row
    const int k0 = sp * C;
    const int k1 = min(limit, k0 + C);

    float qr[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      load_as_f32<T, DPL>(qp + ((int64_t)r * a.Hq + kvh * G + h) * D + lane * DPL, qr[h]);
#pragma unroll
      for (int c = 0; c < DPL; ++c) qr[h][c] *= qscale;
    }
    float m[G], l[G], o[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int c = 0; c < DPL; ++c) o[h][c] = 0.f;
    }

    const int32_t* pt = a.page_tables + (int64_t)b * a.max_pages;
    bool bad_page = false;
    int j = k0;
    while (j < k1) {
      const int pidx = j / a.P;
      const int off = j - pidx * a.P;
      const int page = __ldg(pt + pidx);
      if (page < 0 || page >= a.num_pages) {
        bad_page = true;
        break;
      }
      const int n = min(a.P - off, k1 - j);
      const int64_t base = ((int64_t)page * a.P + off) * kstride + (int64_t)kvh * D + lane * DPL;
      for (int t = 0; t < n; t += U) {
        float kf[U][DPL], vf[U][DPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (t + u < n) {
            load_as_f32<T, DPL>(kc + base + (int64_t)(t + u) * kstride, kf[u]);
            load_as_f32<T, DPL>(vc + base + (int64_t)(t + u) * kstride, vf[u]);
          } else {
#pragma unroll
            for (int c = 0; c < DPL; ++c) kf[u][c] = vf[u][c] = 0.f;
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float s[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < DPL; ++c) acc = fmaf(qr[h][c], kf[u][c], acc);
            s[u] = warp_sum(acc);
            if (t + u >= n) s[u] = -INFINITY;
          }
          float mx = m[h];
#pragma unroll
          for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u]);
          const float alpha = exp2f(m[h] - mx);
          m[h] = mx;
          float lsum = l[h] * alpha;
#pragma unroll
          for (int c = 0; c < DPL; ++c) o[h][c] *= alpha;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const float p = exp2f(s[u] - mx);
            lsum += p;
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[h][c] = fmaf(p, vf[u][c], o[h][c]);
          }
          l[h] = lsum;
        }
      }
      j += n;
    }
    if (bad_page) {
      if (lane == 0) set_status(&ctrl[CTRL_ERR], a.dev_status, PKV_DEV_BAD_PAGE);
      continue;
    }

    if (nsplit == 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float inv = 1.f / l[h];
        T* dst = (T*)a.out + ((int64_t)r * a.Hq + kvh * G + h) * D + lane * DPL;
#pragma unroll
        for (int c = 0; c < DPL; ++c) dst[c] = from_f32<T>(o[h][c] * inv);
        if (a.lse != nullptr && lane == 0) a.lse[(int64_t)r * a.Hq + kvh * G + h] = (m[h] + __log2f(l[h])) * LN2;
      }
    } else {
      const int p = part0 + local;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float inv = 1.f / l[h];
        float* dst = part_o + ((int64_t)p * G + h) * D + lane * DPL;
#pragma unroll
        for (int c = 0; c < DPL; ++c) dst[c] = o[h][c] * inv;
        if (lane == 0) part_lse[(int64_t)p * G + h] = (m[h] + __log2f(l[h])) * LN2;
      }
    }
  }
}

// One warp per (split row, q head). The split weights exp(lse_s - lse) are
// computed one split per lane; the weighted sum then walks the splits with
// each lane holding D/32 consecutive dims (one vector load per split),
// unrolled so several splits' loads are in flight at once.
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(AttnArgs a) {
  constexpr int DPL = D / 32;                       // 2, 4 or 8 dims per lane
  using V = typename std::conditional<DPL == 2, float2, float4>::type;
  constexpr int NV = DPL == 2 ? 1 : DPL / 4;        // vector loads per split and lane
  const int lane = threadIdx.x & 31;
  pdl_wait();   // launched to overlap the end of the decode kernel, whose partials it reads
  const int32_t* ctrl = (const int32_t*)(a.ws + a.lay.ctrl);
  const int32_t* rp_row = (const int32_t*)(a.ws + a.lay.rp_row);
  const int32_t* rp_keys = (const int32_t*)(a.ws + a.lay.rp_keys);
  const int32_t* rp_part_begin = (const int32_t*)(a.ws + a.lay.rp_part_begin);
  const int32_t* split_rows = (const int32_t*)(a.ws + a.lay.split_rows);
  const int C = ctrl[CTRL_CHUNK];
  const float* part_o = (const float*)(a.ws + a.lay.part_o);
  const float* part_lse = (const float*)(a.ws + a.lay.part_lse);
  const int n_rows = ctrl[CTRL_N_SPLIT_ROWS];
  const int G = a.Hq / a.Hkv;
  const int64_t total = (int64_t)n_rows * a.Hq;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t w = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); w < total; w += warps) {
    const int rj = split_rows[w / a.Hq];   // a row-path row
    const int r = rp_row[rj];
    const int h = (int)(w % a.Hq);
    const int kvh = h / G, hh = h - kvh * G;
    const int nsplit = (rp_keys[rj] + C - 1) / C;
    const int p0 = rp_part_begin[rj] + kvh * nsplit;
    // lse over the splits: per-lane online max / sum, then one warp reduction
    float mx = -INFINITY, sm = 0.f;
    for (int s = lane; s < nsplit; s += 32) {
      const float v = part_lse[(int64_t)(p0 + s) * G + hh];
      const float m2 = fmaxf(mx, v);
      sm = sm * __expf(mx - m2) + __expf(v - m2);
      mx = m2;
    }
    const float gmx = warp_max(mx);
    sm = mx == -INFINITY ? 0.f : sm * __expf(mx - gmx);
    const float lse = gmx + __logf(warp_sum(sm));
    float av[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) av[c] = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += 32) {
      const int n = min(32, nsplit - s0);
      const float wl = lane < n ? __expf(part_lse[(int64_t)(p0 + s0 + lane) * G + hh] - lse) : 0.f;
      const V* src = reinterpret_cast<const V*>(part_o + ((int64_t)(p0 + s0) * G + hh) * D) + lane * NV;
      const int64_t stride = (int64_t)G * D * sizeof(float) / sizeof(V);   // vectors between consecutive splits
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const float wgt = __shfl_sync(0xffffffffu, wl, j);
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const V x = __ldg(src + j * stride + q);
          const float* xv = reinterpret_cast<const float*>(&x);
#pragma unroll
          for (int c = 0; c < (int)(sizeof(V) / sizeof(float)); ++c)
            av[q * (int)(sizeof(V) / sizeof(float)) + c] = fmaf(wgt, xv[c], av[q * (int)(sizeof(V) / sizeof(float)) + c]);
        }
      }
    }
    T* dst = (T*)a.out + ((int64_t)r * a.Hq + h) * D + lane * DPL;
#pragma unroll
    for (int c = 0; c < DPL; ++c) dst[c] = from_f32<T>(av[c]);
    if (a.lse != nullptr && lane == 0) a.lse[(int64_t)r * a.Hq + h] = lse;
  }
}

template <typename T, int D, int G>
static cudaError_t launch_rows_g(const AttnArgs& a, cudaStream_t s) {
  // keys per step: fewer where a lane already holds many q and o values
  constexpr int U = D >= 256 ? (G >= 4 ? 1 : 2) : (G >= 8 ? 2 : 4);
  const int blocks = a.num_sms * ROWS_BLOCKS_PER_SM;
  rows_kernel<T, D, G, U><<<blocks, ROWS_WARPS * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_rows_d(const AttnArgs& a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_rows_g<T, D, 1>(a, s);
    case 2: return launch_rows_g<T, D, 2>(a, s);
    case 3: return launch_rows_g<T, D, 3>(a, s);
    case 4: return launch_rows_g<T, D, 4>(a, s);
    case 5: return launch_rows_g<T, D, 5>(a, s);
    case 6: return launch_rows_g<T, D, 6>(a, s);
    case 7: return launch_rows_g<T, D, 7>(a, s);
    case 8: return launch_rows_g<T, D, 8>(a, s);
    case 16: return launch_rows_g<T, D, 16>(a, s);
    default: return cudaErrorNotSupported;
  }
}

template <typename T>
static cudaError_t launch_rows_t(const AttnArgs& a, cudaStream_t s) {
  switch (a.D) {
    case 64: return launch_rows_d<T, 64>(a, s);
    case 128: return launch_rows_d<T, 128>(a, s);
    case 256: return launch_rows_d<T, 256>(a, s);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_rows(const AttnArgs& a, cudaStream_t s) {
  KernelTimer timer("rows", s);
  switch (a.dtype) {
    case PKV_F32: return launch_rows_t<float>(a, s);
    case PKV_F16: return launch_rows_t<__half>(a, s);
    default: return launch_rows_t<__nv_bfloat16>(a, s);
  }
}

template <typename T>
static cudaError_t launch_combine_t(const AttnArgs& a, cudaStream_t s) {
  const int blocks = a.num_sms * 2;
  static const cudaError_t carve = [] {
    cudaError_t e = prefer_max_shared(combine_kernel<T, 64>);
    if (e == cudaSuccess) e = prefer_max_shared(combine_kernel<T, 128>);
    if (e == cudaSuccess) e = prefer_max_shared(combine_kernel<T, 256>);
    return e;
  }();
  if (carve != cudaSuccess) return carve;
  // the grid may get resident once the decode kernel's CTAs have all started;
  // it waits for that grid to finish before reading the partials
  cudaError_t e = cudaErrorNotSupported;
  switch (a.D) {
    case 64: e = launch_after_trigger(combine_kernel<T, 64>, dim3(blocks), dim3(256), 0, s, a); break;
    case 128: e = launch_after_trigger(combine_kernel<T, 128>, dim3(blocks), dim3(256), 0, s, a); break;
    case 256: e = launch_after_trigger(combine_kernel<T, 256>, dim3(blocks), dim3(256), 0, s, a); break;
    default: break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s) {
  KernelTimer timer("combine", s);
  switch (a.dtype) {
    case PKV_F32: return launch_combine_t<float>(a, s);
    case PKV_F16: return launch_combine_t<__half>(a, s);
    default: return launch_combine_t<__nv_bfloat16>(a, s);
  }
}

}  // namespace pkv
