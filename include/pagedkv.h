/*
 * pagedkv.h — C ABI of libpagedkv: attention over a paged KV cache for one
 * packed, continuously batched tick of decode tokens and chunked-prefill
 * tokens with grouped-query heads, on an NVIDIA GB300 (sm_103a).
 *
 * The operations follow the serving pages' description of the problem:
 *  - the KV cache is a fixed pool of fixed-size pages shared by all sequences,
 *    one tensor per layer for K and one for V, each laid out
 *    [num_pages, page_size, num_kv_heads, head_dim] (llm-serving-engine README,
 *    component table "KV Cache" row and "KV cache memory layout" figure;
 *    Helios README, "Paged attention": a fixed pool of 256-token pages);
 *  - each sequence owns a page table that maps its positions to pages
 *    (mini-vLLM, "Paged KV-cache"; Helios README, "Paged attention");
 *  - new tokens' K/V are written into their slots first, then attention reads
 *    K/V through the page tables, never copying them into dense per-sequence
 *    buffers (Helios README, "Paged attention" and its closing remark on
 *    causal paged attention on NVIDIA GPUs; Helios blog, "Prefill vs Decode");
 *  - decode tokens and prefill chunks run in one packed pass with independent
 *    positions and page tables, decode tokens first (Helios README,
 *    "Continuous batching"; Helios blog, "Continuous batching").
 *
 * Conventions shared by every call:
 *  - Ownership: the caller allocates and owns every buffer, host or device,
 *    including the attention workspace. The library allocates no device memory
 *    and keeps no per-call state. It does hold, per process, a device status
 *    word (see pkv_get_device_status) and, when enabled, CUDA events for
 *    kernel timing.
 *  - Asynchrony: device calls are enqueued on `stream` (a cudaStream_t; NULL =
 *    the legacy default stream) and return before the work runs. Outputs are
 *    valid once the stream has been synchronised.
 *  - Errors: every call returns PKV_OK (0) or a negative PKV_E_* code. Host
 *    checks run before anything is enqueued; on an error nothing is launched.
 *    Data-dependent checks that only the device can make (a slot or page id
 *    outside the pool, a kv_len longer than its page table) set bits of the
 *    device status word and skip the offending row; nothing traps or aborts.
 *  - Dtypes: K, V, Q and the attention output share one dtype (PKV_F32,
 *    PKV_F16 or PKV_BF16); accumulation is fp32; lse is fp32.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* same handle as cudaStream_t */

typedef enum {
  PKV_F32 = 0,
  PKV_F16 = 1,
  PKV_BF16 = 2,
  PKV_FP8_E4M3 = 3 /* caches only, with per-KV-head scales (pkv_kv_append_quant,
                      pkv_paged_attention_fp8) */
} pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_E_NULL = -1,      /* a required pointer is NULL */
  PKV_E_DTYPE = -2,     /* unknown dtype */
  PKV_E_SHAPE = -3,     /* a size is out of range, Hq % Hkv != 0, or head_dim unsupported */
  PKV_E_LENGTHS = -4,   /* q/kv lengths break 0 <= q_len <= kv_len (host-checked calls) */
  PKV_E_PAGES = -5,     /* a page id outside the pool, or too few pages for a length */
  PKV_E_WORKSPACE = -6, /* workspace smaller than pkv_paged_attention_workspace_size */
  PKV_E_ALIGN = -7,     /* a pointer is not 16-byte aligned */
  PKV_E_CUDA = -8,      /* a CUDA runtime call or launch failed */
  PKV_E_DEVICE = -9,    /* the current device is not an sm_103 GPU */
  PKV_E_CAPACITY = -10  /* an output buffer is too small (host-checked calls) */
} pkv_status;

/* Bits of the device status word. */
#define PKV_DEV_BAD_SLOT 0x1    /* kv_append: slot >= num_pages * page_size; that row skipped */
#define PKV_DEV_BAD_LENGTHS 0x2 /* attention: kv_len < q_len, kv_len < 1 with rows,
                                   kv_len > max_kv_len or > max_pages_per_seq * page_size:
                                   that sequence's rows are skipped; cu_seqlens_q not
                                   non-decreasing from 0 to total_q (some q_len < 0):
                                   every row of the call is skipped */
#define PKV_DEV_BAD_PAGE 0x4    /* attention: a page id needed by a row is outside the pool;
                                   that row's output is left unwritten */
#define PKV_DEV_TIMEOUT 0x8     /* a kernel's internal wait gave up (a bug, never expected);
                                   the outputs of that call are unspecified */
#define PKV_DEV_BAD_POSITION 0x10 /* rope append: a position outside [0, max_pos); that row skipped */

/* One layer's K (or V) page pool: contiguous
 * [num_pages, page_size, num_kv_heads, head_dim] of `dtype`. */
typedef struct {
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype; /* pkv_dtype */
} pkv_cache_desc;

/* ---------------------------------------------------------------------------
 * pkv_pack_tick — host-side packing of one tick (no device work).
 *
 * Puts decode sequences (q_len == 1) first and then the others, each group in
 * arrival order (Helios README, "Continuous batching": every tick first takes
 * one token per decoding request, then spends the rest of the budget on
 * prompts; both run in one packed forward), and builds the packed metadata.
 *
 * In (host pointers, num_seqs entries unless stated):
 *   q_lens[i]        tokens sequence i adds this tick (0 = idle, 1 = decode, >1 = chunk)
 *   kv_lens[i]       context length after this tick's tokens are written
 *   page_offsets     [num_seqs + 1], CSR offsets into page_ids
 *   page_ids         physical pages of sequence i in logical order:
 *                    page_ids[page_offsets[i] .. page_offsets[i+1])
 *   page_size, num_pages, max_pages_per_seq (width of the output table)
 *   slot_capacity    length of the slot_mapping buffer
 * Out (host pointers, caller-allocated):
 *   order[num_seqs]                   arrival index of the i-th packed sequence
 *   cu_seqlens_q[num_seqs + 1]        row offsets of the packed sequences
 *   kv_lens_out[num_seqs]             kv_len of the i-th packed sequence
 *   page_tables[num_seqs * max_pages_per_seq]  row-major, unused entries -1
 *   slot_mapping[total_q]             page * page_size + offset of each packed
 *                                     row's new token (its position is
 *                                     kv_len - q_len + i for chunk row i)
 *   total_q_out                       number of packed rows
 * Errors: PKV_E_NULL, PKV_E_SHAPE (num_seqs < 0, page_size < 1, num_pages < 1,
 * max_pages_per_seq < 1), PKV_E_LENGTHS (q_len < 0, kv_len < q_len, kv_len < 1
 * with q_len > 0), PKV_E_PAGES (page id outside [0, num_pages), fewer pages
 * than ceil(kv_len / page_size), more pages than max_pages_per_seq),
 * PKV_E_CAPACITY (total_q > slot_capacity). Outputs are unspecified on error.
 */
int pkv_pack_tick(int32_t num_seqs, const int32_t* q_lens, const int32_t* kv_lens,
                  const int32_t* page_offsets, const int32_t* page_ids,
                  int32_t page_size, int32_t num_pages, int32_t max_pages_per_seq,
                  int32_t slot_capacity,
                  int32_t* order, int32_t* cu_seqlens_q, int32_t* kv_lens_out,
                  int32_t* page_tables, int64_t* slot_mapping, int32_t* total_q_out);

/* pkv_tick_positions — host: position of every packed row (kv_len - q_len + i
 * for row i of a sequence), from cu_seqlens_q[num_seqs + 1] and kv_lens
 * (host pointers), into positions[capacity]. PKV_E_LENGTHS for q_len < 0,
 * kv_len < q_len or cu[0] != 0; PKV_E_CAPACITY if the rows do not fit. */
int pkv_tick_positions(int32_t num_seqs, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                       int32_t* positions, int32_t capacity);

/* ---------------------------------------------------------------------------
 * pkv_kv_append — write each new token's K and V rows into its slot
 * (Helios blog, "Prefill vs Decode": a decode step writes its new token's
 * slot; Helios README, "Paged attention": decode stores straight into the
 * shared pool; llm-serving-engine README, engine step trace: a prefill chunk
 * stores its K/V starting at the chunk's first position).
 *
 *   k, v          device, [num_tokens, num_kv_heads, head_dim], contiguous, cache dtype
 *   slot_mapping  device, int64 [num_tokens]; row t goes to page slot / page_size,
 *                 offset slot % page_size; a negative slot skips the row
 *   k_cache, v_cache  device, the pools described by `cache`
 * Bit-exact copy. Duplicate non-negative slots in one call are a caller error
 * (which row lands is unspecified). A slot >= num_pages * page_size sets
 * PKV_DEV_BAD_SLOT and skips the row. num_tokens == 0 is a no-op.
 * Errors: PKV_E_NULL, PKV_E_DTYPE, PKV_E_SHAPE, PKV_E_ALIGN (k, v, caches must
 * be 16-byte aligned), PKV_E_CUDA.
 */
int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                  void* k_cache, void* v_cache, const pkv_cache_desc* cache, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Rotary position embedding fused into the append (Helios blog, "torch.sdpa
 * and Flash Attention": RoPE is applied to Q and K before attention;
 * llm-serving-engine README, component table "RoPE from scratch": cached
 * sin/cos tables). Half-split form: for pair i < d/2 of a head row x at
 * position p, with a = p * base^(-2i/d),
 *   x'_i = x_i cos a - x_{i+d/2} sin a,   x'_{i+d/2} = x_{i+d/2} cos a + x_i sin a.
 *
 * pkv_rope_table (host): fills cos_sin[max_pos][head_dim/2][2] (float) with
 * (cos a, sin a), computed in double. PKV_E_SHAPE unless base > 1, head_dim
 * even >= 2, max_pos >= 1.
 *
 * pkv_rope_kv_append (device): for each new token t at position positions[t]
 * (int32, device), rotates its K rows and writes them to slot slot_mapping[t]
 * (as pkv_kv_append; a negative slot skips K and V), copies its V rows to the
 * slot unrotated, and writes its rotated Q rows [num_tokens, num_q_heads,
 * head_dim] to q_out (q_out may equal q: in place). cos_sin is the device copy
 * of the table above. A position outside [0, max_pos) sets
 * PKV_DEV_BAD_POSITION and skips that token's Q and K rows. Rotation in fp32,
 * results rounded to the cache dtype. Errors as pkv_kv_append, plus PKV_E_SHAPE
 * for an odd head_dim or num_q_heads < 1.
 */
int pkv_rope_table(double base, int32_t head_dim, int32_t max_pos, float* cos_sin);
int pkv_rope_kv_append(const void* q, const void* k, const void* v, const int32_t* positions,
                       const float* cos_sin, int32_t max_pos, const int64_t* slot_mapping, int32_t num_tokens,
                       int32_t num_q_heads, void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                       void* q_out, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_attention_workspace_size — bytes of device workspace that
 * pkv_paged_attention needs for these sizes (0 on invalid sizes).
 * The workspace holds the device-side work plan and the split-KV partial
 * results; its contents need no initialisation and are not preserved.
 */
size_t pkv_paged_attention_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                          const pkv_cache_desc* cache, int32_t max_kv_len);

/* ---------------------------------------------------------------------------
 * pkv_paged_attention — attention of every packed query row over its
 * sequence's pages (Helios blog, "torch.sdpa and Flash Attention":
 * softmax(Q K^T * scale) V with grouped-query heads sharing KV heads;
 * llm-serving-engine README, engine step trace: a prefill chunk after cached
 * K/V uses a rectangular causal mask, a decode row attends the full context).
 *
 *   q             device, [total_q, num_q_heads, head_dim], cache dtype, contiguous
 *   cu_seqlens_q  device, int32 [num_seqs + 1]; cu[0] = 0, non-decreasing, cu[num_seqs] = total_q
 *   kv_lens       device, int32 [num_seqs]; context length INCLUDING this tick's
 *                 tokens (append first, then attend)
 *   page_tables   device, int32 [num_seqs, max_pages_per_seq], row-major
 *   max_kv_len    host upper bound on every kv_lens entry (sizes the work plan)
 *   scale         multiplies q.k before the softmax
 *   out           device, [total_q, num_q_heads, head_dim], cache dtype
 *   lse           device, fp32 [total_q, num_q_heads], natural log of
 *                 sum_j exp(scale * q.k_j); may be NULL
 *   workspace     device, >= pkv_paged_attention_workspace_size(...) bytes, 256-byte aligned
 * Row i of sequence b (q_len = cu[b+1] - cu[b], kv_len = kv_lens[b]) attends
 * keys 0 .. kv_len - q_len + i. q head h reads KV head h / (num_q_heads /
 * num_kv_heads). Page-table entries past ceil(kv_len / page_size) and slots at
 * positions >= kv_len are never read and may hold anything (NaN, -1).
 * Rows of sequences with bad lengths or pages (see the device status bits)
 * are skipped.
 * Errors: PKV_E_NULL, PKV_E_DTYPE, PKV_E_SHAPE (num_q_heads % num_kv_heads != 0,
 * a group num_q_heads / num_kv_heads outside 1..8 and 16, head_dim not 64,
 * 128 or 256, sizes < 0), PKV_E_ALIGN, PKV_E_WORKSPACE, PKV_E_DEVICE, PKV_E_CUDA.
 * head_dim 64 and 128 run decode rows on the TMA-staged decode kernel and
 * chunks on the tensor-core prefill kernels; at head_dim 256 every row (decode
 * and chunk) runs on the TMA-staged decode kernel over 16-bit caches and on the
 * CUDA-core rows kernel over fp32 caches.
 */
int pkv_paged_attention(const void* q, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                        const int32_t* page_tables, int32_t num_seqs, int32_t total_q,
                        int32_t num_q_heads, int32_t max_pages_per_seq, int32_t max_kv_len,
                        const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                        float scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 (e4m3) KV cache. mini-vLLM, "Quantization": 8-bit weights widened
 * before every matmul saved memory but slowed decode, and the page names a
 * fused low-precision kernel as the missing step. Here the cache holds one
 * byte per element and the attention kernel widens the codes in registers, so
 * a decode step reads half the bytes of a 16-bit cache.
 *
 * Cache dtype PKV_FP8_E4M3: same [num_pages, page_size, num_kv_heads,
 * head_dim] layout, one e4m3 code per element (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; largest finite 448; no infinities). Element
 * (slot, h, i) stands for code * k_scale[h] (K) or code * v_scale[h] (V);
 * k_scale, v_scale are device float [num_kv_heads], owned by the caller,
 * finite and > 0.
 *
 * pkv_kv_append_quant: as pkv_kv_append, but k, v are [num_tokens,
 * num_kv_heads, head_dim] of src_dtype (PKV_F32/F16/BF16) and each element x
 * is stored as e4m3(x / scale[h]): the quotient in IEEE float32 (correctly
 * rounded), then the nearest e4m3 value, ties to even, saturating to +-448
 * (NaN stays NaN). Bit-exact against that definition. head_dim must be a
 * multiple of 16. Errors as pkv_kv_append; PKV_E_DTYPE unless the cache is
 * PKV_FP8_E4M3 (pkv_kv_append and pkv_rope_kv_append answer PKV_E_DTYPE for an
 * fp8 cache).
 *
 * pkv_paged_attention_fp8: as pkv_paged_attention over an fp8 cache; q and
 * out are q_dtype (PKV_BF16 or PKV_F16), lse as there. Scores are
 * (q . code) * k_scale[h] * scale and the output is (sum p_j code_j) *
 * v_scale[h] / sum p_j. q is rounded to fp16 for the products with the codes
 * (every e4m3 value is exact in fp16), so bf16 queries must lie within fp16's
 * range. head_dim must be 128; page_size as for the 16-bit decode path. Decode
 * rows and short chunks run on the TMA-staged row kernel; a chunk of 64 rows
 * or more runs on the tensor-core prefill kernel (scale > 0, page_size a
 * multiple or divisor of 128, any group size), which widens each K/V tile to fp16
 * in shared memory before its MMAs; other chunks go row by row.
 * Errors as pkv_paged_attention, plus PKV_E_DTYPE for another cache or query
 * type and PKV_E_NULL for missing scales. pkv_paged_attention answers
 * PKV_E_DTYPE for an fp8 cache. The workspace size is
 * pkv_paged_attention_workspace_size with the fp8 cache descriptor.
 */
int pkv_kv_append_quant(const void* k, const void* v, int32_t src_dtype, const int64_t* slot_mapping,
                        int32_t num_tokens, void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                        const float* k_scale, const float* v_scale, pkv_stream_t stream);
int pkv_paged_attention_fp8(const void* q, int32_t q_dtype, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                            const int32_t* page_tables, int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                            int32_t max_pages_per_seq, int32_t max_kv_len, const void* k_cache,
                            const void* v_cache, const pkv_cache_desc* cache, const float* k_scale,
                            const float* v_scale, float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host page pool and prefix cache (no device work; host memory only).
 *
 * A fixed pool of page ids with per-page reference counts, and a cache of
 * complete prompt blocks keyed by a hash chained over the blocks before them
 * (Helios README, "Paged attention": pages come from a free list and return
 * to the pool when the last request or prefix-cache entry holding them lets
 * go; Helios blog, "Prefix caching": complete page-size prompt blocks are
 * hashed with the previous block's hash, a request reuses the longest matching
 * chain's pages, partial blocks are not stored, entries have a sliding TTL and
 * eviction takes unused leaf blocks first).
 *  - pkv_pool_alloc hands out the lowest free ids first, each with count 1;
 *    PKV_E_CAPACITY (nothing taken) when fewer than n pages are free.
 *  - pkv_pool_retain / pkv_pool_release add / drop one reference per listed
 *    page (a page may be listed several times); a page whose count reaches 0
 *    is free again. PKV_E_PAGES (nothing changed) for an id outside the pool,
 *    a free page, or more releases than references.
 *  - pkv_prefix_lookup walks tokens[0 .. n_tokens) block by block (page_size
 *    tokens each) and returns the number of leading blocks found in the cache
 *    (at most max_pages); their page ids go to pages[] and each gets one more
 *    reference, now owned by the caller; their last-use time becomes `now`.
 *  - pkv_prefix_insert stores every complete block of tokens not yet cached,
 *    on the caller's page for that block (pages[b] for block b); the cache
 *    takes one reference per stored page. Returns the number of new entries.
 *  - pkv_prefix_evict drops unused leaf entries (the cache holds the only
 *    reference and no cached block continues them): first every entry unused
 *    for more than `ttl` (sliding), then, oldest last use first, until at
 *    least want_free pages are free or nothing is evictable. Returns the
 *    number of entries dropped.
 * The pool object is not thread-safe; callers serialise access.
 */
typedef struct pkv_pool pkv_pool;
int pkv_pool_create(int32_t num_pages, int32_t page_size, pkv_pool** out);
void pkv_pool_destroy(pkv_pool* pool);
int pkv_pool_alloc(pkv_pool* pool, int32_t n, int32_t* pages);
int pkv_pool_retain(pkv_pool* pool, const int32_t* pages, int32_t n);
int pkv_pool_release(pkv_pool* pool, const int32_t* pages, int32_t n);
int pkv_pool_free_count(const pkv_pool* pool);
int pkv_pool_refcount(const pkv_pool* pool, int32_t page);
int pkv_prefix_lookup(pkv_pool* pool, const int32_t* tokens, int32_t n_tokens, double now, int32_t* pages,
                      int32_t max_pages);
int pkv_prefix_insert(pkv_pool* pool, const int32_t* tokens, int32_t n_tokens, const int32_t* pages,
                      int32_t n_pages, double now);
int pkv_prefix_evict(pkv_pool* pool, double now, double ttl, int32_t want_free);
int pkv_prefix_size(const pkv_pool* pool);

/* ---------------------------------------------------------------------------
 * pkv_paged_attention_no_alloc — pkv_paged_attention without a workspace
 * argument, for callers that cannot allocate device memory (for example code
 * running inside a memory pool's or custom allocator's own callbacks, or a
 * plug-in that is handed only the tensors it reads and writes). The serving
 * pages have no counterpart of this call; it is a deployment convenience.
 *
 * Arguments, results, layouts and errors are those of pkv_paged_attention,
 * minus workspace/workspace_bytes. The scratch the call needs (its work plan
 * and split-KV partial results) lives in a fixed array of
 * PKV_NO_ALLOC_SCRATCH_BYTES inside the library's device image, which every
 * GPU that loads the library holds until the process exits. The call itself
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *  - Limit: sizes whose work plan does not fit the array (very many packed
 *    rows) return PKV_E_WORKSPACE; the split-KV partials get the room that is
 *    left, and the split size grows until they fit.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (with that device current); make that first call before any stream
 *    capture.
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's contents; each call rewrites every counter and control word it
 *    reads before using it. Calls that overlap on the GPU (for example on two
 *    streams at once) race on the array and give undefined results: serialise
 *    them.
 */
#define PKV_NO_ALLOC_SCRATCH_BYTES (16u << 20)

int pkv_paged_attention_no_alloc(const void* q, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                 const int32_t* page_tables, int32_t num_seqs, int32_t total_q,
                                 int32_t num_q_heads, int32_t max_pages_per_seq, int32_t max_kv_len,
                                 const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                 float scale, void* out, float* lse, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Status and instrumentation. */

/* Human-readable text for a pkv_status code (static storage). */
const char* pkv_status_string(int status);

/* Text of the CUDA error behind the calling thread's last PKV_E_CUDA
 * (thread-local storage, valid until that thread's next failing call). */
const char* pkv_last_error(void);

/* Waits for `stream`, then returns in *code the OR of the PKV_DEV_* bits set
 * on the current device since the last call, and clears them. */
int pkv_get_device_status(int32_t* code, pkv_stream_t stream);

/* Kernel timing: when enabled (1), every kernel the library launches is
 * bracketed by CUDA events on its launch stream; pkv_kernel_times waits for
 * the recorded work and returns, per kernel name, the number of launches and
 * the summed device time, then clears the record. Disabled (0) by default. */
int pkv_set_kernel_timing(int enable);
/* Fills up to `max` entries; returns the number of kernels recorded (>= 0) or
 * a negative pkv_status. names[i] points at static storage. */
int pkv_kernel_times(const char** names, int32_t* launches, double* total_ms, int32_t max);

/* Self-test of the failure path (the pages have no counterpart; it checks the
 * library's own error handling). Enqueues on `stream` one CTA laid out like
 * the prefill kernel's (a producer warp, an MMA-issuer thread, eight softmax
 * warps), each waiting, through the bounded pipeline wait that every decode and
 * prefill kernel of the library uses, on a barrier that nothing ever completes.
 * The producer warp waits with a limit of limit_us microseconds, gives up
 * first, raises the CTA's abort flag and records PKV_DEV_TIMEOUT in the CTA's
 * error word and in the device status word (read and cleared by
 * pkv_get_device_status); the other warps see the flag and return. The CUDA
 * context stays usable.
 *  - result: device int32[2] or NULL. [0] = the CTA's error word
 *    (PKV_DEV_TIMEOUT), [1] = warps that left their wait without the barrier
 *    (10 when every warp drained). Cleared on `stream` before the launch.
 *  - limit_us must lie in [1, 1000000], else PKV_E_SHAPE and nothing is
 *    launched; PKV_E_ALIGN if result is not 4-byte aligned; PKV_E_CUDA if the
 *    launch fails. */
int pkv_selftest_bounded_wait(int32_t limit_us, int32_t* result, pkv_stream_t stream);

/* Library version string. */
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H_ */
