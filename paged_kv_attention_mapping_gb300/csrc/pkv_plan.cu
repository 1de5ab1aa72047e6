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
// The split size is `chunk_min` keys (a power of two that depends only on
// head_dim, so a row's result does not depend on the batch it is packed in),
// doubled until the partial results fit the workspace, and at most the
// smallest power of two that holds max_kv_len (one split a row). Being a power
// of two, the closed forms below divide by it with shifts.
#include <cuda_runtime.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Per-sequence offsets of the plan (exclusive prefix sums over sequences):
// row-path rows, work items, partial slots, split rows.
constexpr int SEQ_OFFS = 4;

PlanLayout plan_layout(int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t D, int32_t /*max_kv_len*/) {
  PlanLayout L{};
  size_t off = 0;
  L.ctrl = off;            off += align256(CTRL_WORDS * 4);
  L.rp_row = off;          off += align256((size_t)T * 4 + 4);
  L.rp_seq = off;          off += align256((size_t)T * 4 + 4);
  L.rp_keys = off;         off += align256((size_t)T * 4 + 4);
  L.rp_item_begin = off;   off += align256(((size_t)T + 1) * 4);
  L.rp_part_begin = off;   off += align256((size_t)T * 4 + 4);
  L.split_rows = off;      off += align256((size_t)T * 4 + 4);
  L.seq_pair_begin = off;  off += align256(((size_t)B + 1) * 4);
  L.seq_offs = off;        off += align256((size_t)SEQ_OFFS * B * 4 + 4);
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

// binary search over a copy in shared memory (or the input itself when it is too big)
__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
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

// Threads of the plan's one CTA. 512 (~33K registers) lets it start on an SM
// beside the append kernel's blocks (at most three per SM, ~31K), which it may
// overlap; 1024 needed an SM with no append block left and started ~5 us later
// on the mixed tick.
constexpr int PLAN_THREADS = 512;
constexpr int PLAN_WARPS = PLAN_THREADS / 32;

// Exclusive scan over the threads of the block; *total gets the sum.
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
    int s = lane < PLAN_WARPS ? sm[lane] : 0;   // the lanes past the last warp hold the total
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

// Exclusive scan of N values at once over the threads of the block.
template <int N>
__device__ void block_scan_n(const int (&v)[N], int (&ex)[N], int (&tot)[N], int (*sm)[32]) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x[N];
#pragma unroll
  for (int k = 0; k < N; ++k) x[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < N; ++k) sm[k][w] = x[k];
  }
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      int s = lane < PLAN_WARPS ? sm[k][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      sm[k][lane] = s;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    ex[k] = (w > 0 ? sm[k][w - 1] : 0) + x[k] - v[k];
    tot[k] = sm[k][31];
  }
  __syncthreads();
}

constexpr int HIST = 2048;
constexpr int RANK_SORT_MAX = 256;   // up to this many prefill pairs are ranked directly

struct SeqInfo {
  int c0, q, L;
  bool bad, tc;
};

// `partition_bad`: cu_seqlens_q does not cut [0, T) into consecutive ranges,
// so no row can be given to a sequence and every sequence counts as bad.
__device__ __forceinline__ SeqInfo seq_info(const PlanArgs& a, int b, bool partition_bad) {
  SeqInfo s;
  s.c0 = a.cu[b];
  const int c1 = a.cu[b + 1];
  s.q = c1 - s.c0;
  s.L = a.kv_lens[b];
  s.bad = partition_bad || s.q < 0 || s.c0 < 0 || c1 > a.T ||
          (s.q > 0 && (s.L < s.q || s.L > a.max_kv_len || s.L > a.table_cap));
  s.tc = !s.bad && a.tc_min_q > 0 && s.q >= a.tc_min_q;
  return s;
}

// Sum of ceil(k / C) over k = 1 .. K (K >= 0) for C = 2^s: with K = m C + r,
// the first m C terms give C (1 + .. + m) and the last r terms m + 1 each.
__device__ __forceinline__ long long ceil_div_prefix(unsigned K, int s) {
  const unsigned m = K >> s, r = K & ((1u << s) - 1u);
  return ((long long)m * (m + 1) / 2 << s) + (long long)r * (m + 1);
}

// How many SMs the prefill kernel keeps when the decode kernel can start on
// the others at once. The decode kernel streams from HBM at a rate per SM set
// by the bytes it keeps in flight there (its TMA stage ring, a property of its
// configuration) over the loaded memory latency, up to the HBM limit; the
// prefill kernel's work is its KV steps and work tiles in SM cycles at the SM
// clock. For each candidate x the model takes the time until both kernels are
// done: the prefill on x SMs, the decode on the other N - x until the prefill
// ends and on all N afterwards, and keeps the x with the shortest time. The
// decode constants were measured on GB300 (the decode kernel's rate with 16 to
// 48 SMs). The prefill constants start from the kernel's measured cycles per
// KV step (about 3250 at head_dim 128 in long launches, ~3500 in the mixed
// tick's chunks) and were then fitted so that the chosen x lands on the
// measured best split (x swept in steps of 2) of five mixes: the Qwen3-shaped
// mixed tick with 16-bit and e4m3 caches, 32 decode rows beside four 512-row
// chunks, 192 and 256 decode rows beside two chunks (head_dim 128 and 64).
// The device facts (SM count and clock, HBM rate) come from the driver. The
// split only moves time between the two kernels: every tile and item is still
// done once.
constexpr float PF_STEP_CYCLES_D128 = 3300.f;   // two 128-row query tiles x 128 keys, head_dim 128, 16-bit
constexpr float PF_STEP_CYCLES_D64 = 2700.f;    // the same at head_dim 64
constexpr float PF_STEP_CYCLES_FP8 = 3300.f;    // head_dim 128 over an e4m3 cache (tiles widened first)
constexpr float PF_TILE_CYCLES = 1700.f;        // start and end of a work tile beyond its steps
constexpr float DECODE_LATENCY_S = 2.3e-6f;     // loaded HBM latency of the decode kernel's TMA stream
constexpr float HBM_STREAM_EFF = 0.83f;         // streamable fraction of the HBM pin rate (measured copy)

// Evaluated by the 32 lanes of one warp (candidates strided over the lanes,
// then a warp argmin); every lane returns the same x.
__device__ int prefill_ctas(const PlanArgs& a, int n_pairs, unsigned long long steps, unsigned long long row_keys,
                            int lane) {
  const int N = a.num_sms;
  if (!a.share_sms || n_pairs == 0 || row_keys == 0 || N < 3) return N;
  // fp32: this part's fp64 rate is far below its fp32 rate, and a split
  // estimate needs no more than fp32 precision
  const float step_cycles = a.kv8 ? PF_STEP_CYCLES_FP8 : (a.D >= 128 ? PF_STEP_CYCLES_D128 : PF_STEP_CYCLES_D64);
  const int g = a.Hq / a.Hkv;
  const float hp = (float)(a.Hkv * ((g + 1) / 2));   // head pairs (an odd group's last head runs solo)
  const float pf = hp * ((float)steps * step_cycles + (float)n_pairs * PF_TILE_CYCLES) / a.sm_hz;   // SM-seconds
  const float dec = (float)row_keys * (float)(a.Hkv * a.D * a.kv_elt) * 2.f;                        // bytes
  const float bw_sm = a.dec_inflight_bytes / DECODE_LATENCY_S;
  const float hbm = a.hbm_bps * HBM_STREAM_EFF;
  const float r_all = fminf((float)N * bw_sm, hbm);
  // the divisions are an estimate's: __fdividef is enough (and short)
  int best = N;
  float best_t = __fdividef(pf, (float)N) + __fdividef(dec, r_all);   // one after the other on every SM
  // Below about a third of the SMs the prefill kernel's steps run well over
  // their cycle count beside a decode kernel that saturates HBM (its operand
  // loads queue behind the decode stream; measured on ticks of 192 and 256
  // decode rows beside two chunks: 563 and 164 us with 40 prefill SMs against
  // 538 and 153 us with 52), so the search starts there.
  for (int x = (N + 2) / 3 + lane; x < N; x += 32) {
    const float t_pf = __fdividef(pf, (float)x);
    const float r = fminf((float)(N - x) * bw_sm, hbm);
    const float t = dec <= t_pf * r ? t_pf : t_pf + __fdividef(dec - t_pf * r, r_all);
    if (t < best_t) {
      best_t = t;
      best = x;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
    const int ox = __shfl_xor_sync(0xffffffffu, best, o);
    if (ot < best_t || (ot == best_t && ox < best)) {
      best_t = ot;
      best = ox;
    }
  }
  return best;
}

// sequences whose lengths and offsets are staged in shared memory:
// cu (B + 1), kv_lens (B), pair offsets (B + 1) and SEQ_OFFS offsets per sequence
constexpr int PLAN_SMEM_SEQS = 6144;
constexpr int PLAN_SMEM_WORDS = (3 + SEQ_OFFS) * PLAN_SMEM_SEQS + 2;

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(PlanArgs a_in, int32_t* dev_status) {
  // stage cu_seqlens_q and kv_lens in shared memory: every row below searches them
  extern __shared__ int32_t s_seq[];
  // A decode kernel launched next may get resident now (it waits for this
  // grid). A prefill kernel launched next is let in only once the append before
  // this kernel is done (below): its CTAs would take the registers the append
  // still needs.
  if (a_in.trigger_early) pdl_trigger();
  PlanArgs a = a_in;
  const bool staged = a_in.B <= PLAN_SMEM_SEQS;
  if (staged) {
    for (int i = threadIdx.x; i <= a_in.B; i += blockDim.x) s_seq[i] = __ldg(a_in.cu + i);
    for (int i = threadIdx.x; i < a_in.B; i += blockDim.x) s_seq[a_in.B + 1 + i] = __ldg(a_in.kv_lens + i);
    a.cu = s_seq;
    a.kv_lens = s_seq + a_in.B + 1;
    __syncthreads();
  }
  int32_t* ctrl = (int32_t*)(a.ws + a.lay.ctrl);
  int32_t* rp_row = (int32_t*)(a.ws + a.lay.rp_row);
  int32_t* rp_seq = (int32_t*)(a.ws + a.lay.rp_seq);
  int32_t* rp_keys = (int32_t*)(a.ws + a.lay.rp_keys);
  int32_t* rp_item_begin = (int32_t*)(a.ws + a.lay.rp_item_begin);
  int32_t* rp_part_begin = (int32_t*)(a.ws + a.lay.rp_part_begin);
  int32_t* split_rows = (int32_t*)(a.ws + a.lay.split_rows);
  int32_t* pair_begin_g = (int32_t*)(a.ws + a.lay.seq_pair_begin);
  int32_t* pair_begin = staged ? s_seq + 2 * a_in.B + 1 : pair_begin_g;
  // per sequence: the SEQ_OFFS offsets (row-path rows, items, partial slots,
  // split rows)
  volatile int32_t* seq_off = staged ? s_seq + 3 * a_in.B + 2 : (int32_t*)(a.ws + a.lay.seq_offs);
  int2* pairs = (int2*)(a.ws + a.lay.tc_pairs);

  // per-warp partial sums (64-bit atomics on shared memory serialise badly)
  __shared__ unsigned long long s_wkeys[32], s_wsteps[32];
  __shared__ int s_err;
  __shared__ int sm[32];
  __shared__ int smn[SEQ_OFFS][32];
  __shared__ int hist[HIST];
  const int tid = threadIdx.x;
  const int B = a.B, Hkv = a.Hkv;

  // pass 1: check every sequence; count the keys the row path will visit
  const bool ends_bad = a.cu[0] != 0 || a.cu[B] != a.T;
  int my_desc = 0;
  for (int b = tid; b < B; b += blockDim.x) my_desc |= a.cu[b + 1] < a.cu[b] ? 1 : 0;
  const bool partition_bad = __syncthreads_or(my_desc) != 0 || ends_bad;
  if (tid == 0) {
    s_err = partition_bad ? PKV_DEV_BAD_LENGTHS : 0;
  }
  __syncthreads();
  unsigned long long my_keys = 0;
  int my_err = 0, my_tc = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    const SeqInfo s = seq_info(a, b, partition_bad);
    if (s.bad) my_err = PKV_DEV_BAD_LENGTHS;
    my_tc |= s.tc ? 1 : 0;
    if (!s.bad && !s.tc && s.q > 0)
      my_keys += (unsigned long long)s.q * (unsigned long long)(s.L - s.q) +
                 (unsigned long long)s.q * (s.q + 1) / 2;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    my_keys += __shfl_xor_sync(0xffffffffu, my_keys, o);
    my_err |= __shfl_xor_sync(0xffffffffu, my_err, o);
  }
  if ((tid & 31) == 0) {
    s_wkeys[tid >> 5] = my_keys;
    s_wsteps[tid >> 5] = 0;
    if (my_err) atomicOr(&s_err, my_err);
  }
  const bool any_tc = __syncthreads_or(my_tc) != 0;   // no prefill-kernel sequence: skip pass 3
  unsigned long long s_keys = (tid & 31) < PLAN_WARPS ? s_wkeys[tid & 31] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s_keys += __shfl_xor_sync(0xffffffffu, s_keys, o);
  // split size C = 2^c_shift keys: chunk_min (a power of two), at most the
  // smallest power of two >= max_kv_len (any C from there on gives one split a
  // row)
  int c_max_shift = 6;
  while (c_max_shift < 31 && (1u << c_max_shift) < (unsigned)a.max_kv_len) ++c_max_shift;
  int c_shift = 31 - __clz(a.chunk_min);
  if (c_shift > c_max_shift) c_shift = c_max_shift;

  // pass 2a: per sequence, in closed form, its row-path rows, items and
  // partial slots, turned into offsets by a block scan. Row i of a row-path
  // sequence sees k = L - q + 1 + i keys and makes ceil(k / C) items per KV
  // head; it is split, with partial slots, when k > C.
  int carry[SEQ_OFFS];
  for (int guard = 0; guard < 40; ++guard) {
#pragma unroll
    for (int k = 0; k < SEQ_OFFS; ++k) carry[k] = 0;
    const unsigned Cu = 1u << c_shift;
    for (int base = 0; base < B; base += blockDim.x) {
      const int b = base + tid;
      int cnt[SEQ_OFFS] = {0, 0, 0, 0}, ex[SEQ_OFFS], tot[SEQ_OFFS];
      if (b < B) {
        const SeqInfo s = seq_info(a, b, partition_bad);
        if (!s.bad && !s.tc && s.q > 0) {
          if (guard == 0 && a.page_tables) {
            // the decode kernel reads these entries at the start of each item
            const char* t0 = (const char*)(a.page_tables + (int64_t)b * a.max_pages);
            const int bytes = ((s.L + a.P - 1) / a.P) * 4;
            for (int off = 0; off < bytes; off += 128) prefetch_l2(t0 + off);
          }
          const unsigned k_lo = (unsigned)(s.L - s.q + 1), k_hi = (unsigned)s.L;
          const long long f_hi = ceil_div_prefix(k_hi, c_shift);
          cnt[0] = s.q;
          cnt[1] = (int)(f_hi - ceil_div_prefix(k_lo - 1, c_shift)) * Hkv;
          const unsigned k_s = k_lo > Cu + 1 ? k_lo : Cu + 1;   // first split row's key count
          if (k_hi >= k_s) {
            cnt[2] = (int)(f_hi - ceil_div_prefix(k_s - 1, c_shift)) * Hkv;
            cnt[3] = (int)(k_hi - k_s + 1);
          }
        }
      }
      block_scan_n<SEQ_OFFS>(cnt, ex, tot, smn);
      if (b < B) {
#pragma unroll
        for (int k = 0; k < SEQ_OFFS; ++k) seq_off[SEQ_OFFS * b + k] = carry[k] + ex[k];
      }
#pragma unroll
      for (int k = 0; k < SEQ_OFFS; ++k) carry[k] += tot[k];
    }
    if (carry[2] <= a.lay.partial_cap || c_shift >= c_max_shift) break;
    ++c_shift;   // grow the split until the partials fit
  }
  __syncthreads();   // seq_off complete
  const int n_rp = carry[0], n_items = carry[1], carry_parts = carry[2], carry_split = carry[3];

  // pass 2b: per row-path row j (consecutive rows on consecutive threads), its
  // sequence by binary search over the sequences' first row-path rows (zero-row
  // sequences share their successor's offset, so the last sequence whose offset
  // is <= j owns j), then its arrays from the same closed forms
  {
    const unsigned Cu = 1u << c_shift;
    for (int j = tid; j < n_rp; j += blockDim.x) {
      int lo = 0, hi = B;   // first b with seq_off[SEQ_OFFS * b] > j
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (seq_off[SEQ_OFFS * mid] <= j) lo = mid + 1; else hi = mid;
      }
      const int b = lo - 1;
      const SeqInfo s = seq_info(a, b, false);
      const int i = j - seq_off[SEQ_OFFS * b];
      const unsigned k_lo = (unsigned)(s.L - s.q + 1), k = k_lo + (unsigned)i;
      rp_row[j] = s.c0 + i;
      rp_seq[j] = b;
      rp_keys[j] = (int)k;
      rp_item_begin[j] = seq_off[SEQ_OFFS * b + 1] +
                         (int)(ceil_div_prefix(k - 1, c_shift) - ceil_div_prefix(k_lo - 1, c_shift)) * Hkv;
      int pb = -1;
      if (k > Cu) {
        const unsigned k_s = k_lo > Cu + 1 ? k_lo : Cu + 1;
        pb = seq_off[SEQ_OFFS * b + 2] + (int)(ceil_div_prefix(k - 1, c_shift) - ceil_div_prefix(k_s - 1, c_shift)) * Hkv;
        split_rows[seq_off[SEQ_OFFS * b + 3] + (int)(k - k_s)] = j;
      }
      rp_part_begin[j] = pb;
    }
  }
  if (tid == 0) rp_item_begin[n_rp] = n_items;

  // pass 3: (sequence, q tile) pairs of the prefill kernel, longest first
  int carry_pairs = 0;
  for (int base = 0; any_tc && base < a.B; base += blockDim.x) {
    const int b = base + tid;
    int n = 0;
    if (b < a.B) {
      const SeqInfo s = seq_info(a, b, partition_bad);
      if (s.tc) n = (s.q + TC_BM - 1) / TC_BM;
    }
    int t;
    const int e = block_scan_excl(n, &t, sm);
    if (b < a.B) pair_begin[b] = carry_pairs + e;
    carry_pairs += t;
  }
  if (tid == 0) pair_begin[a.B] = carry_pairs;
  __syncthreads();
  const int n_pairs = carry_pairs;
  auto pair_work = [&](int p, int* b_out, int* qt_out) {
    const int b = upper_bound_written(pair_begin, a.B + 1, p) - 1;   // shared memory when B fits
    const int qt = p - pair_begin[b];
    const SeqInfo s = seq_info(a, b, false);
    const int q1 = min(s.q, (qt + 1) * TC_BM);
    const int keys = s.L - s.q + q1;  // keys the tile's last row sees
    *b_out = b;
    *qt_out = qt;
    return (keys + TC_BN - 1) / TC_BN;
  };
  if (n_pairs > 0 && n_pairs <= RANK_SORT_MAX) {   // block-uniform
    // few pairs: thread p ranks pair p against all others (longer first, then
    // lower index), two block barriers instead of the histogram's passes
    int b = 0, qt = 0, w = 0;
    if (tid < n_pairs) {
      w = pair_work(tid, &b, &qt);
      hist[tid] = w;
    }
    unsigned long long my_steps = (unsigned long long)w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_steps += __shfl_xor_sync(0xffffffffu, my_steps, o);
    if ((tid & 31) == 0) s_wsteps[tid >> 5] = my_steps;
    __syncthreads();
    if (tid < n_pairs) {
      int rank = 0;
      for (int q = 0; q < n_pairs; ++q) {
        const int wq = hist[q];
        rank += (wq > w || (wq == w && q < tid)) ? 1 : 0;
      }
      pairs[rank] = make_int2(b, qt);
    }
    __syncthreads();
  } else if (n_pairs > 0) {   // block-uniform
    for (int i = tid; i < HIST; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    unsigned long long my_steps = 0;
    for (int p = tid; p < n_pairs; p += blockDim.x) {
      int b, qt;
      const int w = pair_work(p, &b, &qt);
      my_steps += (unsigned long long)w;
      atomicAdd(&hist[min(w, HIST - 1)], 1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_steps += __shfl_xor_sync(0xffffffffu, my_steps, o);
    if ((tid & 31) == 0) s_wsteps[tid >> 5] = my_steps;
    __syncthreads();
    // descending exclusive offsets: hist[w] <- number of pairs with work > w
    {
      constexpr int PER = HIST / PLAN_THREADS;
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
      const int w = min(pair_work(p, &b, &qt), HIST - 1);
      const int pos = atomicAdd(&hist[w], 1);
      pairs[pos] = make_int2(b, qt);
    }
    __syncthreads();
  }
  int pf_ctas = a.num_sms;
  if (tid < 32) {
    unsigned long long steps = tid < PLAN_WARPS ? s_wsteps[tid] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) steps += __shfl_xor_sync(0xffffffffu, steps, o);
    pf_ctas = prefill_ctas(a, n_pairs, steps, s_keys, tid);
  }
  if (tid == 0) {
    ctrl[CTRL_PF_CTAS] = pf_ctas;
    ctrl[CTRL_ERR] = s_err;
    ctrl[CTRL_N_ITEMS] = n_items;
    ctrl[CTRL_N_RP] = n_rp;
    ctrl[CTRL_ITEM_NEXT] = 0;
    ctrl[CTRL_N_PAIRS] = n_pairs;
    ctrl[CTRL_N_TILES] = n_pairs * a.Hq;
    ctrl[CTRL_TILE_NEXT] = 0;
    ctrl[CTRL_CHUNK] = (int)(1u << c_shift);
    ctrl[CTRL_N_SPLIT_ROWS] = carry_split;
    ctrl[CTRL_N_PARTIALS] = carry_parts;
    if (s_err) atomicOr(dev_status, s_err);
  }
  // This kernel may have started while the preceding kernel (the append) still
  // ran; finishing only after it makes every later launch see the appended K/V.
  pdl_wait();
  pdl_trigger();
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 PLAN_SMEM_WORDS * 4);
  if (attr != cudaSuccess) return attr;
  static const cudaError_t carve = prefer_max_shared(plan_kernel);
  if (carve != cudaSuccess) return carve;
  const size_t smem = a.B <= PLAN_SMEM_SEQS ? (size_t)((3 + SEQ_OFFS) * a.B + 2) * 4 : 0;
  KernelTimer timer("plan", s);
  // may overlap the preceding append, which it does not read (see pdl_wait above)
  cudaError_t e = launch_after_trigger(plan_kernel, dim3(1), dim3(PLAN_THREADS), smem, s, a, a.dev_status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
