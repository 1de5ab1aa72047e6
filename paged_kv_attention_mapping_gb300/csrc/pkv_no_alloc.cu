// pkv_paged_attention_no_alloc: the attention call for callers that cannot
// allocate device memory.
//
// pkv_paged_attention takes a caller-allocated workspace (the device work plan
// and the split-KV partial results). Some callers cannot provide one: code that
// runs where cudaMalloc is off limits (inside a custom allocator or a memory
// pool's own callbacks, in a runtime that has handed all device memory to an
// arena it does not expose, or in a plug-in that is given only the tensors it
// reads and writes). This variant uses a fixed scratch array that lives in the
// library's own device image instead: a file-scope __device__ array of
// PKV_NO_ALLOC_SCRATCH_BYTES, which every GPU that loads the library holds until
// the process exits. It calls no cudaMalloc, cudaFree or allocating library.
//
// The launch sequence is the same as pkv_paged_attention's (plan, prefill
// kernel when the shape has one, row kernel, combine); only the workspace and
// its partial-result capacity differ.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

struct ScratchSetup {
  bool ready = false;
  int ok = 0;
  int num_sms = 0;
  char* scratch = nullptr;  // device address of g_no_alloc_scratch on this device
};
std::mutex g_mu;
ScratchSetup g_setup[64];

// Once per device, with that device current: the device address of the
// scratch array (in host code its name is only a host-side stand-in).
const ScratchSetup* scratch_setup() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchSetup& s = g_setup[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    s.scratch = (char*)p;
    s.num_sms = sms;
    s.ok = (major == 10 && minor == 3) ? 1 : 0;
    s.ready = true;
  }
  return &s;
}

constexpr int kTcMinQ = 64;  // same threshold as pkv_paged_attention

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_paged_attention_no_alloc(const void* q, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                            const int32_t* page_tables, int32_t num_seqs, int32_t total_q,
                                            int32_t num_q_heads, int32_t max_pages_per_seq, int32_t max_kv_len,
                                            const void* k_cache, const void* v_cache, const pkv_cache_desc* c,
                                            float scale, void* out, float* lse, pkv_stream_t stream) {
  if (!c) return PKV_E_NULL;
  if (c->dtype < PKV_F32 || c->dtype > PKV_BF16) return PKV_E_DTYPE;   // fp8 caches: pkv_paged_attention_fp8
  if (c->num_pages < 1 || c->page_size < 1 || c->num_kv_heads < 1 || c->head_dim < 1) return PKV_E_SHAPE;
  const int elt = c->dtype == PKV_F32 ? 4 : 2;
  if (((int64_t)c->num_kv_heads * c->head_dim * elt) % 16 != 0) return PKV_E_SHAPE;
  if ((int64_t)c->num_pages * c->page_size > INT32_MAX) return PKV_E_SHAPE;
  if (num_seqs < 0 || total_q < 0 || num_q_heads < 1 || max_kv_len < 0) return PKV_E_SHAPE;
  if (num_q_heads % c->num_kv_heads != 0) return PKV_E_SHAPE;
  const int g = num_q_heads / c->num_kv_heads;
  if (!(c->head_dim == 64 || c->head_dim == 128) || !(g == 1 || g == 2 || g == 4 || g == 8 || g == 16))
    return PKV_E_SHAPE;
  if (total_q > 0 && max_pages_per_seq < 1) return PKV_E_SHAPE;
  if ((int64_t)max_pages_per_seq * c->page_size > INT32_MAX) return PKV_E_SHAPE;
  if (total_q == 0) return PKV_OK;
  if (!q || !cu_seqlens_q || !kv_lens || !page_tables || !k_cache || !v_cache || !out) return PKV_E_NULL;
  auto a16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!a16(q) || !a16(out) || !a16(k_cache) || !a16(v_cache) || ((uintptr_t)lse & 3u)) return PKV_E_ALIGN;

  // The plan's per-row arrays use the standard layout; the partial results get
  // whatever room is left in the scratch array. The planner widens the split
  // size until the partials fit, so a smaller capacity changes only how keys
  // are split, not what is computed.
  PlanLayout lay = plan_layout(num_seqs, total_q, num_q_heads, c->num_kv_heads, c->head_dim, max_kv_len);
  const size_t per_part = (size_t)g * 4 + (size_t)g * c->head_dim * 4;
  const size_t base = lay.part_lse;
  if (base + 1024 > PKV_NO_ALLOC_SCRATCH_BYTES) return PKV_E_WORKSPACE;
  size_t cap = (PKV_NO_ALLOC_SCRATCH_BYTES - base - 512) / per_part;
  if (cap > (size_t)lay.partial_cap) cap = (size_t)lay.partial_cap;
  if (cap < 1) return PKV_E_WORKSPACE;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  lay.partial_cap = (int32_t)cap;
  lay.part_o = base + al(cap * (size_t)g * 4);
  lay.total = lay.part_o + al(cap * (size_t)g * c->head_dim * 4);
  if (lay.total > PKV_NO_ALLOC_SCRATCH_BYTES) return PKV_E_WORKSPACE;

  const ScratchSetup* su = scratch_setup();
  if (!su) return PKV_E_CUDA;
  if (!su->ok) return PKV_E_DEVICE;
  int32_t* status = device_status_ptr();
  if (!status) return PKV_E_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = su->scratch;

  // as in the workspace entry point: a tick with no more rows than sequences
  // skips the tensor-core prefill kernel
  const bool tc = prefill_tc_supported(c->dtype, c->head_dim, c->page_size) && total_q >= kTcMinQ &&
                  total_q > num_seqs;
  PlanArgs pa{};
  pa.cu = cu_seqlens_q;
  pa.kv_lens = kv_lens;
  pa.B = num_seqs;
  pa.T = total_q;
  pa.Hq = num_q_heads;
  pa.Hkv = c->num_kv_heads;
  pa.max_kv_len = max_kv_len;
  pa.table_cap = max_pages_per_seq * c->page_size;
  pa.chunk_min = split_chunk_keys(c->head_dim, elt);
  pa.target_items = 1 << 30;
  pa.tc_min_q = tc ? kTcMinQ : 0;
  pa.num_sms = su->num_sms;
  pa.D = c->head_dim;
  pa.kv_elt = elt;
  pa.share_sms = tc && decode_supported(c->dtype, c->head_dim, c->page_size) && !kernel_timing_enabled();
  pa.page_tables = page_tables;
  pa.max_pages = max_pages_per_seq;
  pa.P = c->page_size;
  pa.ws = ws;
  pa.lay = lay;
  pa.dev_status = status;
  // the plan kernel rewrites every control word and counter the kernels read,
  // so nothing left in the array by an earlier call is used
  if (launch_plan(pa, s) != cudaSuccess) return PKV_E_CUDA;

  AttnArgs aa{};
  aa.q = q;
  aa.cu = cu_seqlens_q;
  aa.kv_lens = kv_lens;
  aa.page_tables = page_tables;
  aa.B = num_seqs;
  aa.T = total_q;
  aa.Hq = num_q_heads;
  aa.Hkv = c->num_kv_heads;
  aa.D = c->head_dim;
  aa.P = c->page_size;
  aa.num_pages = c->num_pages;
  aa.max_pages = max_pages_per_seq;
  aa.k_cache = k_cache;
  aa.v_cache = v_cache;
  aa.scale = scale;
  aa.out = out;
  aa.lse = lse;
  aa.ws = ws;
  aa.lay = lay;
  aa.dtype = c->dtype;
  aa.kv_dtype = c->dtype;
  aa.after_prefill = tc;
  aa.num_sms = su->num_sms;
  aa.dev_status = status;
  if (tc && launch_prefill_tc(aa, s) != cudaSuccess) return PKV_E_CUDA;
  if ((decode_supported(aa.kv_dtype, aa.D, aa.P) ? launch_decode(aa, s) : launch_rows(aa, s)) != cudaSuccess)
    return PKV_E_CUDA;
  if (launch_combine(aa, s) != cudaSuccess) return PKV_E_CUDA;
  return PKV_OK;
}
