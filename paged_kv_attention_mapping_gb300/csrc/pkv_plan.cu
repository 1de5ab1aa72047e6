// Device-side work plan of one attention call.
//
// One CTA reads cu_seqlens_q and kv_lens from device memory (no host round
// trip, so a tick can be captured in a CUDA graph and replayed with new
// lengths) and writes into the caller's workspace:
//  * per packed row, the range of row-path work items (row, KV head, split)
//    and, for rows whose keys are split, the range of partial-result slots;
//  * the list of rows that need a combine;
//  * the (sequence, 128-row q tile) pairs of the tensor-core prefill kernel,
//    sorted by descending KV-tile count so that long tiles start first.
// The split size is chosen so that the row-path items number about
// `target_items` (a few per resident worker), never below `chunk_min` keys,
// and doubled until the partial results fit the workspace.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PlanLayout plan_layout(int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, int32_t /*max_kv_len*/) {
  PlanLayout L{};
  size_t off = 0;
  L.ctrl = off;            off += align256(CTRL_WORDS * 4);
  L.row_seq = off;         off += align256((size_t)T * 4 + 4);
  L.row_item_begin = off;  off += align256(((size_t)T + 1) * 4);
  L.row_part_begin = off;  off += align256((size_t)T * 4 + 4);
  L.split_rows = off;      off += align256((size_t)T * 4 + 4);
  L.seq_pair_begin = off;  off += align256(((size_t)B + 1) * 4);
  L.pair_cap = T / TC_BM + B + 1;
  L.tc_pairs = off;        off += align256((size_t)L.pair_cap * 8);
  const int g = Hq / Hkv;
  const size_t per_part = (size_t)g * D * 4;
  size_t cap = ((size_t)64 << 20) / per_part;  // at most 64 MB of partial outputs
  if (cap > 16384) cap = 16384;
  if (cap < 256) cap = 256;
  L.partial_cap = (int32_t)cap;
  L.part_lse = off;        off += align256(cap * g * 4);
  L.part_o = off;          off += align256(cap * per_part);
  L.total = off;
  return L;
}

__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Same search over an array this kernel wrote itself: plain loads, not the
// read-only path, which is only coherent for data that is constant during the kernel.
__device__ __forceinline__ int upper_bound_written(const volatile int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Exclusive scan over the 1024 threads of the block; *total gets the sum.
__device__ int block_scan_excl(int v, int* total, int* sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sm[lane] = s;
  }
  __syncthreads();
  const int res = (w > 0 ? sm[w - 1] : 0) + x - v;
  *total = sm[31];
  __syncthreads();
  return res;
}

constexpr int HIST = 2048;

struct SeqInfo {
  int q, L;
  bool bad, tc;
};

__device__ __forceinline__ SeqInfo seq_info(const PlanArgs& a, int b) {
  SeqInfo s;
  const int c0 = __ldg(a.cu + b), c1 = __ldg(a.cu + b + 1);
  s.q = c1 - c0;
  s.L = __ldg(a.kv_lens + b);
  s.bad = s.q < 0 || c0 < 0 || c1 > a.T ||
          (s.q > 0 && (s.L < s.q || s.L > a.max_kv_len || s.L > a.table_cap));
  s.tc = !s.bad && a.tc_min_q > 0 && s.q >= a.tc_min_q;
  return s;
}

// splits of row r for split size C (0 when the row has no row-path work)
__device__ __forceinline__ int row_splits(const PlanArgs& a, int r, int C, int* seq_out) {
  const int b = upper_bound_i32(a.cu, a.B + 1, r) - 1;
  *seq_out = -1;
  if (b < 0 || b >= a.B) return 0;
  const SeqInfo s = seq_info(a, b);
  const int c0 = __ldg(a.cu + b);
  if (s.bad || s.tc || r < c0 || r >= c0 + s.q) return 0;
  *seq_out = b;
  const int limit = s.L - s.q + (r - c0) + 1;
  return (limit + C - 1) / C;
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanArgs a, int32_t* dev_status) {
  int32_t* ctrl = (int32_t*)(a.ws + a.lay.ctrl);
  int32_t* row_seq = (int32_t*)(a.ws + a.lay.row_seq);
  int32_t* item_begin = (int32_t*)(a.ws + a.lay.row_item_begin);
  int32_t* part_begin = (int32_t*)(a.ws + a.lay.row_part_begin);
  int32_t* split_rows = (int32_t*)(a.ws + a.lay.split_rows);
  int32_t* pair_begin = (int32_t*)(a.ws + a.lay.seq_pair_begin);
  int2* pairs = (int2*)(a.ws + a.lay.tc_pairs);

  __shared__ unsigned long long s_keys;
  __shared__ int s_err, s_cnt;
  __shared__ int sm[32];
  __shared__ int hist[HIST];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_keys = 0;
    s_err = 0;
    s_cnt = 0;
    if (__ldg(a.cu) != 0 || __ldg(a.cu + a.B) != a.T) s_err = PKV_DEV_BAD_LENGTHS;
  }
  __syncthreads();

  // pass 1: check every sequence; count the keys the row path will visit
  unsigned long long my_keys = 0;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const SeqInfo s = seq_info(a, b);
    if (s.bad) atomicOr(&s_err, PKV_DEV_BAD_LENGTHS);
    if (!s.bad && !s.tc && s.q > 0)
      my_keys += (unsigned long long)s.q * (unsigned long long)(s.L - s.q) +
                 (unsigned long long)s.q * (s.q + 1) / 2;
  }
  atomicAdd(&s_keys, my_keys);
  __syncthreads();

  // split size: about target_items items, at least chunk_min keys, multiple of 64
  const long long work = (long long)s_keys * a.Hkv;
  long long C = (work + a.target_items - 1) / a.target_items;
  if (C < a.chunk_min) C = a.chunk_min;
  C = (C + 63) / 64 * 64;
  const long long c_max = ((long long)a.max_kv_len + 63) / 64 * 64;
  if (C > c_max) C = c_max < 64 ? 64 : c_max;

  // grow C until the partial results fit the workspace
  for (int guard = 0; guard < 40; ++guard) {
    int parts = 0;
    for (int r = tid; r < a.T; r += blockDim.x) {
      int b;
      const int n = row_splits(a, r, (int)C, &b);
      if (n > 1) parts += n * a.Hkv;
    }
    atomicAdd(&s_cnt, parts);
    __syncthreads();
    const int total = s_cnt;
    __syncthreads();
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    if (total <= a.lay.partial_cap || C >= c_max) break;
    C = C * 2 < c_max ? C * 2 : c_max;
  }

  // pass 2: per-row item and partial ranges, and the list of split rows
  int carry_items = 0, carry_parts = 0, carry_split = 0;
  for (int base = 0; base < a.T; base += blockDim.x) {
    const int r = base + tid;
    int n = 0, b = -1;
    if (r < a.T) n = row_splits(a, r, (int)C, &b);
    int t_items, t_parts, t_split;
    const int e_items = block_scan_excl(n * a.Hkv, &t_items, sm);
    const int e_parts = block_scan_excl(n > 1 ? n * a.Hkv : 0, &t_parts, sm);
    const int e_split = block_scan_excl(n > 1 ? 1 : 0, &t_split, sm);
    if (r < a.T) {
      row_seq[r] = b;
      item_begin[r] = carry_items + e_items;
      part_begin[r] = n > 1 ? carry_parts + e_parts : -1;
      if (n > 1) split_rows[carry_split + e_split] = r;
    }
    carry_items += t_items;
    carry_parts += t_parts;
    carry_split += t_split;
  }
  if (tid == 0) item_begin[a.T] = carry_items;

  // pass 3: (sequence, q tile) pairs of the prefill kernel, longest first
  int carry_pairs = 0;
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + tid;
    int n = 0;
    if (b < a.B) {
      const SeqInfo s = seq_info(a, b);
      if (s.tc) n = (s.q + TC_BM - 1) / TC_BM;
    }
    int t;
    const int e = block_scan_excl(n, &t, sm);
    if (b < a.B) pair_begin[b] = carry_pairs + e;
    carry_pairs += t;
  }
  if (tid == 0) pair_begin[a.B] = carry_pairs;
  const int n_pairs = carry_pairs;
  for (int i = tid; i < HIST; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  auto pair_work = [&](int p, int* b_out, int* qt_out) {
    const int b = upper_bound_written(pair_begin, a.B + 1, p) - 1;
    const int qt = p - pair_begin[b];
    const SeqInfo s = seq_info(a, b);
    const int q1 = min(s.q, (qt + 1) * TC_BM);
    const int keys = s.L - s.q + q1;  // keys the tile's last row sees
    int w = (keys + TC_BN - 1) / TC_BN;
    *b_out = b;
    *qt_out = qt;
    return min(w, HIST - 1);
  };
  for (int p = tid; p < n_pairs; p += blockDim.x) {
    int b, qt;
    atomicAdd(&hist[pair_work(p, &b, &qt)], 1);
  }
  __syncthreads();
  // descending exclusive offsets: hist[w] <- number of pairs with work > w
  {
    constexpr int PER = HIST / 1024;
    int vals[PER], sum = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      vals[k] = hist[HIST - 1 - (tid * PER + k)];
      sum += vals[k];
    }
    int t;
    int run = block_scan_excl(sum, &t, sm);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      hist[HIST - 1 - (tid * PER + k)] = run;
      run += vals[k];
    }
  }
  __syncthreads();
  for (int p = tid; p < n_pairs; p += blockDim.x) {
    int b, qt;
    const int w = pair_work(p, &b, &qt);
    const int pos = atomicAdd(&hist[w], 1);
    pairs[pos] = make_int2(b, qt);
  }
  __syncthreads();
  if (tid == 0) {
    ctrl[CTRL_ERR] = s_err;
    ctrl[CTRL_N_ITEMS] = carry_items;
    ctrl[CTRL_ITEM_NEXT] = 0;
    ctrl[CTRL_N_PAIRS] = n_pairs;
    ctrl[CTRL_N_TILES] = n_pairs * a.Hq;
    ctrl[CTRL_TILE_NEXT] = 0;
    ctrl[CTRL_CHUNK] = (int)C;
    ctrl[CTRL_N_SPLIT_ROWS] = carry_split;
    ctrl[CTRL_N_PARTIALS] = carry_parts;
    if (s_err) atomicOr(dev_status, s_err);
  }
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
  KernelTimer timer("plan", s);
  plan_kernel<<<1, 1024, 0, s>>>(a, a.dev_status);
  return cudaGetLastError();
}

}  // namespace pkv
