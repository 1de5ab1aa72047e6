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
// Checks, plan and launches are pkv_paged_attention's own (attention_impl);
// only the workspace differs: the scratch array, with the partial-result room
// fitted to what the per-row plan leaves of it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

// Device address of g_no_alloc_scratch on each device, looked up once per
// device with that device current (in host code the array's name is only a
// host-side stand-in, not a device address).
struct ScratchSetup {
  bool ready = false;
  char* scratch = nullptr;
};
std::mutex g_mu;
ScratchSetup g_setup[64];

char* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchSetup& s = g_setup[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    s.scratch = (char*)p;
    s.ready = true;
  }
  return s.scratch;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_attention_no_alloc(const void* q, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                            const int32_t* page_tables, int32_t num_seqs, int32_t total_q,
                                            int32_t num_q_heads, int32_t max_pages_per_seq, int32_t max_kv_len,
                                            const void* k_cache, const void* v_cache, const pkv_cache_desc* c,
                                            float scale, void* out, float* lse, pkv_stream_t stream) {
  if (!c) return PKV_E_NULL;
  if (c->dtype < PKV_F32 || c->dtype > PKV_BF16) return PKV_E_DTYPE;   // fp8 caches: pkv_paged_attention_fp8
  // the plan kernel rewrites every control word and counter the kernels read,
  // so nothing an earlier call left in the array is used
  return pkv::attention_impl(q, c->dtype, cu_seqlens_q, kv_lens, page_tables, num_seqs, total_q, num_q_heads,
                             max_pages_per_seq, max_kv_len, k_cache, v_cache, c, nullptr, nullptr, scale, out, lse,
                             nullptr, PKV_NO_ALLOC_SCRATCH_BYTES, pkv::scratch_address, stream);
}
