// C-ABI entry points of libpagedkv: host-side checks, the work plan, launches
// on the caller's stream, the device status word and kernel timing.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// per-device facts and the device status word

__device__ int32_t g_device_status;

struct DeviceFacts {
  bool ready = false;
  int ok = 0;  // 1 = sm_103
  int num_sms = 0;
  float sm_hz = 2.07e9f;    // driver figures below; these stand in if a query fails
  float hbm_bps = 8.18e12f;
  int32_t* status = nullptr;
};
static std::mutex g_dev_mu;
static DeviceFacts g_dev[64];

static const DeviceFacts* device_facts() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceFacts& f = g_dev[dev];
  if (!f.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&f.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    int clk = 0, mclk = 0, bus = 0;
    if (cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev) == cudaSuccess && clk > 0) f.sm_hz = clk * 1e3f;
    if (cudaDeviceGetAttribute(&mclk, cudaDevAttrMemoryClockRate, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&bus, cudaDevAttrGlobalMemoryBusWidth, dev) == cudaSuccess && mclk > 0 && bus > 0)
      f.hbm_bps = 2.f * (mclk * 1e3f) * (bus / 8.f);   // double data rate
    cudaGetLastError();   // a refused query leaves no sticky error behind
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    f.status = (int32_t*)p;
    f.ok = (major == 10 && minor == 3) ? 1 : 0;
    f.ready = true;
  }
  return &f;
}

int32_t* device_status_ptr() {
  const DeviceFacts* f = device_facts();
  return f ? f->status : nullptr;
}

// ---------------------------------------------------------------------------
// kernel timing

struct TimingRec {
  const char* name;
  cudaEvent_t a, b;
};
static std::mutex g_t_mu;
static bool g_timing = false;
static std::vector<TimingRec> g_recs;
static std::vector<cudaEvent_t> g_free_events;

static cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

bool kernel_timing_enabled() {
  std::lock_guard<std::mutex> lk(g_t_mu);
  return g_timing;
}

KernelTimer::KernelTimer(const char* name, cudaStream_t s) : name_(name), s_(s), slot_(-1) {
  std::lock_guard<std::mutex> lk(g_t_mu);
  if (!g_timing) return;
  TimingRec r{name, take_event(), take_event()};
  if (!r.a || !r.b) return;
  cudaEventRecord(r.a, s);
  g_recs.push_back(r);
  slot_ = (int)g_recs.size() - 1;
}

KernelTimer::~KernelTimer() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lk(g_t_mu);
  if (slot_ < (int)g_recs.size()) cudaEventRecord(g_recs[slot_].b, s_);
}

static thread_local char g_last_error[256] = "no error";

// Record the text of a failed CUDA call; returns PKV_E_CUDA.
int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return PKV_E_CUDA;
}

}  // namespace pkv

using namespace pkv;

extern "C" const char* pkv_last_error(void) { return g_last_error; }

// ---------------------------------------------------------------------------
// C ABI

extern "C" const char* pkv_version(void) { return "pagedkv 0.1 (sm_103a)"; }

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_E_NULL: return "a required pointer is NULL";
    case PKV_E_DTYPE: return "unknown dtype, or one this entry point does not take";
    case PKV_E_SHAPE: return "unsupported or inconsistent sizes";
    case PKV_E_LENGTHS: return "q/kv lengths break 0 <= q_len <= kv_len";
    case PKV_E_PAGES: return "page id outside the pool or too few pages";
    case PKV_E_WORKSPACE: return "workspace too small or misaligned";
    case PKV_E_ALIGN: return "pointer not 16-byte aligned";
    case PKV_E_CUDA: return "CUDA runtime error";
    case PKV_E_DEVICE: return "current device is not an sm_103 GPU";
    case PKV_E_CAPACITY: return "output buffer too small";
    default: return "unknown status";
  }
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static int elt_bytes(int dtype) { return dtype == PKV_F32 ? 4 : dtype == PKV_FP8_E4M3 ? 1 : 2; }

static int check_cache(const pkv_cache_desc* c) {
  if (!c) return PKV_E_NULL;
  if (c->dtype < PKV_F32 || c->dtype > PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (c->num_pages < 1 || c->page_size < 1 || c->num_kv_heads < 1 || c->head_dim < 1) return PKV_E_SHAPE;
  const int elt = elt_bytes(c->dtype);
  if (((int64_t)c->num_kv_heads * c->head_dim * elt) % 16 != 0) return PKV_E_SHAPE;
  if ((int64_t)c->num_pages * c->page_size > INT32_MAX) return PKV_E_SHAPE;
  return PKV_OK;
}

extern "C" int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                             void* k_cache, void* v_cache, const pkv_cache_desc* cache, pkv_stream_t stream) {
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;  // pkv_kv_append_quant writes fp8 caches
  if (num_tokens < 0) return PKV_E_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_E_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || ((uintptr_t)slot_mapping & 7u))
    return PKV_E_ALIGN;
  const DeviceFacts* f = device_facts();
  if (!f) return PKV_E_CUDA;
  if (!f->ok) return PKV_E_DEVICE;
  cudaError_t e = launch_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, *cache, f->num_sms,
                                (cudaStream_t)stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_append");
}

extern "C" int pkv_rope_kv_append(const void* q, const void* k, const void* v, const int32_t* positions,
                                  const float* cos_sin, int32_t max_pos, const int64_t* slot_mapping,
                                  int32_t num_tokens, int32_t num_q_heads, void* k_cache, void* v_cache,
                                  const pkv_cache_desc* cache, void* q_out, pkv_stream_t stream) {
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (num_tokens < 0 || num_q_heads < 1 || cache->head_dim % 2 != 0 || max_pos < 1) return PKV_E_SHAPE;
  // rotation works on 16-byte vectors of each half row
  if ((cache->head_dim / 2 * (cache->dtype == PKV_F32 ? 4 : 2)) % 16 != 0) return PKV_E_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!q || !k || !v || !positions || !cos_sin || !slot_mapping || !k_cache || !v_cache || !q_out)
    return PKV_E_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(q_out) || ((uintptr_t)cos_sin & 7u))
    return PKV_E_ALIGN;
  const DeviceFacts* f = device_facts();
  if (!f) return PKV_E_CUDA;
  if (!f->ok) return PKV_E_DEVICE;
  cudaError_t e = launch_rope_append(q, k, v, positions, cos_sin, max_pos, slot_mapping, num_tokens, num_q_heads,
                                     k_cache, v_cache, q_out, *cache, f->status, f->num_sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "rope_append");
}

// head_dim 64 and 128 run on the TMA decode and tcgen05 prefill kernels; 256
// runs every row on the CUDA-core rows kernel
static bool head_dim_supported(int d) { return d == 64 || d == 128 || d == 256; }
// q heads per KV head the kernels are built for (1 to 8, and 16)
static bool group_supported(int g) { return (g >= 1 && g <= 8) || g == 16; }

extern "C" size_t pkv_paged_attention_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                                     const pkv_cache_desc* cache, int32_t max_kv_len) {
  if (check_cache(cache) != PKV_OK || num_seqs < 0 || total_q < 0 || num_q_heads < 1 || max_kv_len < 0) return 0;
  if (num_q_heads % cache->num_kv_heads != 0) return 0;
  return plan_layout(num_seqs, total_q, num_q_heads, cache->num_kv_heads, cache->head_dim, max_kv_len).total;
}

// Sequences whose chunk has at least this many rows run on the tensor-core
// prefill kernel (when the shape has one); shorter ones go row by row.
static constexpr int TC_MIN_Q = 64;

// Shrink the partial-result room of `lay` so that the whole layout fits
// `bytes` (the plan's per-row arrays keep their sizes). The planner then widens
// the split until the partials fit, which changes only how keys are split, not
// what is computed. Returns false when not even one partial fits.
static bool fit_partials(PlanLayout* lay, int32_t g, int32_t head_dim, size_t bytes) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t per_part = (size_t)g * 4 + (size_t)g * head_dim * 4;   // lse + o of one partial
  const size_t base = lay->part_lse;
  if (base + 1024 > bytes) return false;
  size_t cap = (bytes - base - 512) / per_part;
  if (cap > (size_t)lay->partial_cap) cap = (size_t)lay->partial_cap;
  if (cap < 1) return false;
  lay->partial_cap = (int32_t)cap;
  lay->part_o = base + al(cap * (size_t)g * 4);
  lay->total = lay->part_o + al(cap * (size_t)g * head_dim * 4);
  return lay->total <= bytes;
}

// Shared body of the attention entry points: host checks, the device plan,
// then the kernels on `stream`. q_dtype is the q/out element type; an fp8
// cache (cache->dtype == PKV_FP8_E4M3) comes with its per-KV-head scales.
// With `scratch` the workspace is the fixed-size area that scratch() returns
// (looked up only after the host checks pass), and its partial-result room is
// fitted to workspace_bytes (fit_partials) instead of the area having to hold
// the standard layout.
int pkv::attention_impl(const void* q, int q_dtype, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                        const int32_t* page_tables, int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                        int32_t max_pages_per_seq, int32_t max_kv_len, const void* k_cache, const void* v_cache,
                        const pkv_cache_desc* cache, const float* k_scale, const float* v_scale, float scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, ScratchFn scratch,
                        pkv_stream_t stream) {
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (num_seqs < 0 || total_q < 0 || num_q_heads < 1 || max_kv_len < 0) return PKV_E_SHAPE;
  if (num_q_heads % cache->num_kv_heads != 0) return PKV_E_SHAPE;
  if (!head_dim_supported(cache->head_dim) || !group_supported(num_q_heads / cache->num_kv_heads))
    return PKV_E_SHAPE;
  if (fp8 && !decode_supported(PKV_FP8_E4M3, cache->head_dim, cache->page_size)) return PKV_E_SHAPE;
  if (total_q > 0 && max_pages_per_seq < 1) return PKV_E_SHAPE;
  if ((int64_t)max_pages_per_seq * cache->page_size > INT32_MAX) return PKV_E_SHAPE;
  if (total_q == 0) return PKV_OK;
  if (!q || !cu_seqlens_q || !kv_lens || !page_tables || !k_cache || !v_cache || !out || (!workspace && !scratch))
    return PKV_E_NULL;
  if (fp8 && (!k_scale || !v_scale)) return PKV_E_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) || ((uintptr_t)lse & 3u))
    return PKV_E_ALIGN;
  if (((uintptr_t)workspace & 255u) != 0) return PKV_E_WORKSPACE;
  PlanLayout lay = plan_layout(num_seqs, total_q, num_q_heads, cache->num_kv_heads, cache->head_dim, max_kv_len);
  if (scratch && !fit_partials(&lay, num_q_heads / cache->num_kv_heads, cache->head_dim, workspace_bytes))
    return PKV_E_WORKSPACE;
  if (workspace_bytes < lay.total) return PKV_E_WORKSPACE;
  const DeviceFacts* f = device_facts();
  if (!f) return PKV_E_CUDA;
  if (!f->ok) return PKV_E_DEVICE;
  if (scratch) {
    workspace = scratch();
    if (!workspace) return cuda_fail(cudaGetLastError(), "scratch address");
    if (((uintptr_t)workspace & 255u) != 0) return PKV_E_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;

  // Chunks of TC_MIN_Q rows or more run on a tensor-core prefill kernel when
  // the shape has one (fp8 caches: the two-query-tile kernel with K/V widened
  // to fp16; other shapes take the row path). A tick with no more rows than
  // sequences is decode-only but for ticks where all rows sit in one sequence
  // and every other sequence is idle: it skips the prefill kernel, so the
  // decode kernel gets resident while the plan runs instead of queueing behind
  // an empty prefill grid (any chunk of such a tick takes the row path).
  const bool tc_shape =
      fp8 ? prefill_tc2_fp8_supported(q_dtype, cache->head_dim, cache->page_size, num_q_heads,
                                      cache->num_kv_heads, scale)
          : prefill_tc_supported(cache->dtype, cache->head_dim, cache->page_size);
  const bool tc = tc_shape && total_q >= TC_MIN_Q && total_q > num_seqs;

  PlanArgs pa{};
  pa.cu = cu_seqlens_q;
  pa.kv_lens = kv_lens;
  pa.B = num_seqs;
  pa.T = total_q;
  pa.Hq = num_q_heads;
  pa.Hkv = cache->num_kv_heads;
  pa.max_kv_len = max_kv_len;
  pa.table_cap = max_pages_per_seq * cache->page_size;
  // Split size depends only on the element size and head_dim, never on the
  // other rows of the tick, so a row's result does not change with the batch
  // it is packed into. It only grows when the partial results would overflow
  // the workspace.
  pa.chunk_min = split_chunk_keys(cache->head_dim, elt_bytes(cache->dtype));
  pa.tc_min_q = tc ? TC_MIN_Q : 0;
  pa.num_sms = f->num_sms;
  pa.sm_hz = f->sm_hz;
  pa.hbm_bps = f->hbm_bps;
  pa.dec_inflight_bytes = (float)decode_inflight_bytes(cache->dtype, cache->head_dim, num_q_heads / cache->num_kv_heads);
  pa.kv8 = fp8 ? 1 : 0;
  pa.trigger_early = tc ? 0 : 1;
  pa.D = cache->head_dim;
  pa.kv_elt = elt_bytes(cache->dtype);
  pa.share_sms = tc && decode_supported(cache->dtype, cache->head_dim, cache->page_size) && !kernel_timing_enabled();
  pa.page_tables = page_tables;
  pa.max_pages = max_pages_per_seq;
  pa.P = cache->page_size;
  pa.ws = (char*)workspace;
  pa.lay = lay;
  pa.dev_status = f->status;
  cudaError_t e = launch_plan(pa, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan");

  AttnArgs aa{};
  aa.q = q;
  aa.cu = cu_seqlens_q;
  aa.kv_lens = kv_lens;
  aa.page_tables = page_tables;
  aa.B = num_seqs;
  aa.T = total_q;
  aa.Hq = num_q_heads;
  aa.Hkv = cache->num_kv_heads;
  aa.D = cache->head_dim;
  aa.P = cache->page_size;
  aa.num_pages = cache->num_pages;
  aa.max_pages = max_pages_per_seq;
  aa.k_cache = k_cache;
  aa.v_cache = v_cache;
  aa.scale = scale;
  aa.out = out;
  aa.lse = lse;
  aa.ws = (char*)workspace;
  aa.lay = lay;
  aa.dtype = q_dtype;
  aa.kv_dtype = cache->dtype;
  aa.k_scale = k_scale;
  aa.v_scale = v_scale;
  aa.after_prefill = tc;
  aa.num_sms = f->num_sms;
  aa.dev_status = f->status;
  if (tc) {
    e = launch_prefill_tc(aa, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill_tc");
  }
  e = decode_supported(aa.kv_dtype, aa.D, aa.P) ? launch_decode(aa, s) : launch_rows(aa, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode");
  e = launch_combine(aa, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine");
  return PKV_OK;
}

extern "C" int pkv_paged_attention(const void* q, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                   const int32_t* page_tables, int32_t num_seqs, int32_t total_q,
                                   int32_t num_q_heads, int32_t max_pages_per_seq, int32_t max_kv_len,
                                   const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                   float scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                   pkv_stream_t stream) {
  if (cache && cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;  // fp8 caches: pkv_paged_attention_fp8
  return attention_impl(q, cache ? cache->dtype : 0, cu_seqlens_q, kv_lens, page_tables, num_seqs, total_q,
                        num_q_heads, max_pages_per_seq, max_kv_len, k_cache, v_cache, cache, nullptr, nullptr, scale,
                        out, lse, workspace, workspace_bytes, nullptr, stream);
}

extern "C" int pkv_paged_attention_fp8(const void* q, int32_t q_dtype, const int32_t* cu_seqlens_q,
                                       const int32_t* kv_lens, const int32_t* page_tables, int32_t num_seqs,
                                       int32_t total_q, int32_t num_q_heads, int32_t max_pages_per_seq,
                                       int32_t max_kv_len, const void* k_cache, const void* v_cache,
                                       const pkv_cache_desc* cache, const float* k_scale, const float* v_scale,
                                       float scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                       pkv_stream_t stream) {
  if (!cache) return PKV_E_NULL;
  if (cache->dtype != PKV_FP8_E4M3 || (q_dtype != PKV_BF16 && q_dtype != PKV_F16)) return PKV_E_DTYPE;
  return attention_impl(q, q_dtype, cu_seqlens_q, kv_lens, page_tables, num_seqs, total_q, num_q_heads,
                        max_pages_per_seq, max_kv_len, k_cache, v_cache, cache, k_scale, v_scale, scale, out, lse,
                        workspace, workspace_bytes, nullptr, stream);
}

extern "C" int pkv_kv_append_quant(const void* k, const void* v, int32_t src_dtype, const int64_t* slot_mapping,
                                   int32_t num_tokens, void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                   const float* k_scale, const float* v_scale, pkv_stream_t stream) {
  int st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (cache->dtype != PKV_FP8_E4M3 || src_dtype < PKV_F32 || src_dtype > PKV_BF16) return PKV_E_DTYPE;
  if (num_tokens < 0 || cache->head_dim % 16 != 0) return PKV_E_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale) return PKV_E_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || ((uintptr_t)slot_mapping & 7u))
    return PKV_E_ALIGN;
  const DeviceFacts* f = device_facts();
  if (!f) return PKV_E_CUDA;
  if (!f->ok) return PKV_E_DEVICE;
  cudaError_t e = launch_append_quant(k, v, src_dtype, slot_mapping, num_tokens, k_cache, v_cache, *cache, k_scale,
                                      v_scale, f->status, f->num_sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_append_quant");
}

extern "C" int pkv_get_device_status(int32_t* code, pkv_stream_t stream) {
  if (!code) return PKV_E_NULL;
  const DeviceFacts* f = device_facts();
  if (!f) return PKV_E_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return PKV_E_CUDA;
  int32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess) return PKV_E_CUDA;
  const int32_t zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess) return PKV_E_CUDA;
  *code = v;
  return PKV_OK;
}

extern "C" int pkv_set_kernel_timing(int enable) {
  std::lock_guard<std::mutex> lk(g_t_mu);
  g_timing = enable != 0;
  return PKV_OK;
}

extern "C" int pkv_kernel_times(const char** names, int32_t* launches, double* total_ms, int32_t max) {
  std::lock_guard<std::mutex> lk(g_t_mu);
  int n = 0;
  int status = PKV_OK;
  for (TimingRec& r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      status = PKV_E_CUDA;
    int k = 0;
    while (k < n && strcmp(names[k], r.name) != 0) ++k;
    if (k == n) {
      if (n >= max) continue;
      names[n] = r.name;
      launches[n] = 0;
      total_ms[n] = 0.0;
      ++n;
    }
    launches[k] += 1;
    total_ms[k] += ms;
  }
  for (TimingRec& r : g_recs) {
    g_free_events.push_back(r.a);
    g_free_events.push_back(r.b);
  }
  g_recs.clear();
  return status == PKV_OK ? n : status;
}
