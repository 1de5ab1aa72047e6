// Internal declarations shared by the translation units of libpagedkv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// ---------------------------------------------------------------------------
// device status word (one per device, in pkv_api.cu)
int32_t* device_status_ptr();  // device address of the status word on the current device
int cuda_fail(cudaError_t e, const char* where);  // records the error text, returns PKV_E_CUDA

// ---------------------------------------------------------------------------
// kernel timing hooks (pkv_api.cu). A KernelTimer brackets one launch with
// CUDA events on its stream when timing is enabled.
// True while per-kernel timing is on: events then sit between the launches,
// so kernels of one call never overlap.
bool kernel_timing_enabled();

struct KernelTimer {
  KernelTimer(const char* name, cudaStream_t s);
  ~KernelTimer();
  const char* name_;
  cudaStream_t s_;
  int slot_;
};

// ---------------------------------------------------------------------------
// work plan held in the caller's workspace

// Control words at the start of the workspace.
enum Ctrl : int {
  CTRL_ERR = 0,          // PKV_DEV_* bits seen by this call
  CTRL_N_ITEMS = 1,      // row-path work items (row, kv head, split)
  CTRL_ITEM_NEXT = 2,    // atomic work counter of the row kernel
  CTRL_N_TILES = 3,      // tensor-core prefill tiles (seq, q tile, q head)
  CTRL_TILE_NEXT = 4,    // atomic work counter of the prefill kernel
  CTRL_CHUNK = 5,        // keys per split of a row-path (row, kv head)
  CTRL_N_SPLIT_ROWS = 6, // rows whose keys were split
  CTRL_N_PARTIALS = 7,   // partial results written
  CTRL_N_PAIRS = 8,      // (seq, q tile) pairs of the prefill kernel
  CTRL_PF_CTAS = 9,      // prefill-kernel CTAs that take tiles; the SMs of the others run decode CTAs
  CTRL_N_RP = 10,        // row-path rows
  CTRL_WORDS = 64
};

// Row-path work. The rows that run on the decode / rows kernels ("row-path
// rows": every row of a sequence that is not on the tensor-core prefill
// kernel, in packed order) are numbered j = 0 .. n_rp - 1. Row j is packed
// row rp_row[j] of sequence rp_seq[j] and sees rp_keys[j] keys, split every C
// keys (CTRL_CHUNK) into nsplit = ceil(keys / C) splits; a split times a KV
// head is one work item. Row j's items are rp_item_begin[j] ..
// rp_item_begin[j + 1] - 1, split by split with the KV heads of a split
// adjacent (item = rp_item_begin[j] + split * Hkv + kvh). A split row (more
// than one split) writes its partial results to slots rp_part_begin[j] +
// kvh * nsplit + split; split_rows lists those rows (j).
struct PlanLayout {
  size_t ctrl, rp_row, rp_seq, rp_keys, rp_item_begin, rp_part_begin, split_rows, seq_pair_begin, seq_offs,
      tc_pairs, part_lse, part_o, total;
  int32_t partial_cap;  // partial results the workspace can hold
  int32_t pair_cap;     // (seq, q tile) pairs the workspace can hold
};

// Workspace layout for the given sizes (all offsets 256-byte aligned).
PlanLayout plan_layout(int32_t num_seqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t max_kv_len);

// Rows of a tensor-core prefill tile and keys of a KV tile.
constexpr int TC_BM = 128;
constexpr int TC_BN = 128;

struct PlanArgs {
  const int32_t* cu;       // [B + 1]
  const int32_t* kv_lens;  // [B]
  int32_t B, T, Hq, Hkv;
  int32_t max_kv_len, table_cap;  // table_cap = max_pages_per_seq * page_size
  int32_t chunk_min;              // split, keys (a power of two >= 64; doubled only when partials overflow)
  int32_t tc_min_q;               // sequences with q_len >= this use the prefill kernel; 0 = never
  int32_t num_sms;                // SMs of the device
  float sm_hz, hbm_bps;           // SM clock and HBM pin rate of the device (bytes / s)
  float dec_inflight_bytes;       // bytes the decode kernel keeps in flight per SM (its stage ring)
  int32_t kv8;                    // e4m3 cache
  int32_t trigger_early;          // the next launch is the decode kernel: let it get resident at once
  int32_t D, kv_elt;              // head_dim and cache element bytes (decode traffic per key)
  int32_t share_sms;              // 1: the decode kernel can start beside the prefill kernel, so give
                                  //    the prefill kernel only its share of the SMs (CTRL_PF_CTAS)
  const int32_t* page_tables;     // [B, max_pages]: the row-path sequences' entries are prefetched into L2
  int32_t max_pages, P;
  char* ws;
  PlanLayout lay;
  int32_t* dev_status;
};

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s);

// Prefer the largest shared-memory carveout for a kernel that itself needs
// little or none (the appends, the plan, the combine). Their blocks then leave
// the SM configured as the kernels launched next need it: a CTA that needs more
// shared memory than an SM's current carveout gives waits until that SM has
// drained, which kept the plan kernel (12 KB) from starting beside the append
// blocks. Called once per kernel (a function-local static at its launch site).
template <typename K>
cudaError_t prefer_max_shared(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// Launch with programmatic stream serialization: the kernel may start as soon
// as the preceding kernel of the stream calls pdl_trigger() (or completes).
template <typename... KArgs, typename... Args>
cudaError_t launch_after_trigger(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Keys per split of a row-path (row, KV head). It depends only on head_dim,
// so a row's result never depends on the batch it is packed with: 2048 keys at
// head_dim 128 (1 MB of bf16 K+V, 512 KB of fp8) and 512 at 64, where ticks of
// short contexts otherwise leave most SMs idle behind the longest rows
// (measured on the TinyLlama- and Qwen3-shaped decode ticks, 16-bit and fp8).
// Powers of two: the plan divides by the split size with shifts.
inline int32_t split_chunk_keys(int head_dim, int /*elt*/) { return head_dim >= 128 ? 2048 : 512; }

// ---------------------------------------------------------------------------
// kernels' host-side launchers

struct AttnArgs {
  const void* q;
  const int32_t* cu;
  const int32_t* kv_lens;
  const int32_t* page_tables;
  int32_t B, T, Hq, Hkv, D, P, num_pages, max_pages;
  const void* k_cache;
  const void* v_cache;
  float scale;
  void* out;
  float* lse;
  char* ws;
  PlanLayout lay;
  int dtype;     // q / out element type
  int num_sms;
  int32_t* dev_status;
  int kv_dtype = -1;               // cache element type (the q type unless an fp8 cache)
  const float* k_scale = nullptr;  // fp8 caches: per-KV-head scales (device)
  const float* v_scale = nullptr;
  bool after_prefill = false;      // the prefill kernel was launched just before (decode may overlap it)
};

// The append kernels' work split: token t has per_token 16-byte items; block b
// takes tokens [b * tpb, (b + 1) * tpb) and its 256 threads take the items of
// that span in order, so consecutive threads touch consecutive 16-byte vectors
// of one token's rows (coalesced reads and writes). tpb is chosen so that a
// thread has about items_per_thread items a pass and the grid has at least two
// blocks per SM when the tick has enough tokens. With max_per_sm > 0 the grid
// also holds at most that many blocks per SM (the blocks then loop over their
// span): the plain append uses three, so that the attention call's plan kernel,
// launched next, finds room beside them (with six append blocks on every SM it
// waited for the first SM to drain, ~5 us on the mixed tick). The quantising and
// RoPE appends take one item per thread per iteration, load then store, so more
// iterations would serialise their latency; they keep the one-pass grid.
struct TokenSpan {
  int32_t T, per_token, tpb;
  int64_t blocks() const { return ((int64_t)T + tpb - 1) / tpb; }
};
inline TokenSpan token_span(int32_t T, int32_t per_token, int num_sms, int items_per_thread, int max_per_sm = 0) {
  const int n = num_sms > 0 ? num_sms : 1;
  int32_t tpb = (256 * items_per_thread) / per_token;
  if (tpb < 1) tpb = 1;
  const int32_t for_grid = T / (2 * n);   // tokens per block with 2 blocks per SM
  if (for_grid < tpb) tpb = for_grid < 1 ? 1 : for_grid;
  if (max_per_sm > 0) {
    const int64_t cap = (int64_t)max_per_sm * n;
    const int32_t min_tpb = (int32_t)(((int64_t)T + cap - 1) / cap);
    if (tpb < min_tpb) tpb = min_tpb;
  }
  return TokenSpan{T, per_token, tpb};
}

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int32_t T, void* kc, void* vc,
                          const pkv_cache_desc& c, int num_sms, cudaStream_t s);
// e4m3 cache: codes of x / scale[kv head], sources of type src_dtype (f32/f16/bf16).
cudaError_t launch_append_quant(const void* k, const void* v, int src_dtype, const int64_t* slots, int32_t T,
                                void* kc, void* vc, const pkv_cache_desc& c, const float* k_scale,
                                const float* v_scale, int32_t* dev_status, int num_sms, cudaStream_t s);
cudaError_t launch_rope_append(const void* q, const void* k, const void* v, const int32_t* positions,
                               const float* cos_sin, int32_t max_pos, const int64_t* slots, int32_t T,
                               int32_t Hq, void* kc, void* vc, void* q_out, const pkv_cache_desc& c,
                               int32_t* dev_status, int num_sms, cudaStream_t s);
cudaError_t launch_rows(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s);
// Returns cudaErrorNotSupported when the shape has no tensor-core path.
cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t s);
bool prefill_tc_supported(int dtype, int D, int P);
// Two query tiles (two q heads of one GQA group; an odd group's last head runs
// solo) per CTA; needs a group size of at least 2 and scale > 0.
bool prefill_tc2_supported(int dtype, int D, int P, int Hq, int Hkv, float scale);
// The same kernel over an fp8 e4m3 cache (K/V codes widened to fp16 in shared
// memory; head_dim 128, any group size, q bf16 or f16).
bool prefill_tc2_fp8_supported(int q_dtype, int D, int P, int Hq, int Hkv, float scale);
// Two-query-tile kernel (16-bit caches, and fp8 caches when kv_dtype is e4m3).
cudaError_t launch_prefill_tc2(const AttnArgs& a, cudaStream_t s);
// TMA-staged decode kernel for single rows (cudaErrorNotSupported if the shape has none).
cudaError_t launch_decode(const AttnArgs& a, cudaStream_t s);
bool decode_supported(int dtype, int D, int P);
// Bytes the decode kernel keeps in flight per SM for this configuration (CTAs
// per SM x ring stages x stage bytes); 0 when it has none.
int decode_inflight_bytes(int kv_dtype, int D, int group);

// TMA tensor map of a contiguous [rows, heads, D] tensor, 128-byte swizzled boxes.
bool make_map_boxed(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elt, int D, int heads,
                    int64_t rows, int box_cols, int box_rows);

// workers of the row kernel (for the split policy)
int rows_kernel_workers(int num_sms);

// The one body behind every attention entry point (pkv_api.cu): host checks,
// the device plan and the kernel launches on `stream`. q_dtype is the q/out
// element type; an fp8 cache comes with its per-KV-head scales. With a
// `scratch` function the workspace argument is ignored: after the host checks
// pass, scratch() gives a fixed area of workspace_bytes (nullptr on a CUDA
// error), whose partial-result room is fitted to that size (the split then
// grows until the partials fit). Without it the workspace must hold the
// standard layout of pkv_paged_attention_workspace_size.
using ScratchFn = char* (*)();
int attention_impl(const void* q, int q_dtype, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                   const int32_t* page_tables, int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                   int32_t max_pages_per_seq, int32_t max_kv_len, const void* k_cache, const void* v_cache,
                   const pkv_cache_desc* cache, const float* k_scale, const float* v_scale, float scale, void* out,
                   float* lse, void* workspace, size_t workspace_bytes, ScratchFn scratch, pkv_stream_t stream);

}  // namespace pkv
