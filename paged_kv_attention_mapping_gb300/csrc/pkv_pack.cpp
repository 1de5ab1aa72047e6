// Host-side packing of one tick: decode sequences first, then chunks, and the
// packed metadata the attention call reads (row offsets, page tables, slots).
//
// Helios README, "Continuous batching": each tick takes one token per decoding
// request first, then spends the remaining budget on prompts, and runs all of
// it in one packed forward with independent positions and paged KV mappings.
// mini-vLLM, "Paged KV-cache": a per-sequence block table maps positions to
// blocks of a fixed pool.
#include <stdint.h>

#include "pagedkv.h"

extern "C" int pkv_pack_tick(int32_t num_seqs, const int32_t* q_lens, const int32_t* kv_lens,
                             const int32_t* page_offsets, const int32_t* page_ids, int32_t page_size,
                             int32_t num_pages, int32_t max_pages_per_seq, int32_t slot_capacity,
                             int32_t* order, int32_t* cu_seqlens_q, int32_t* kv_lens_out,
                             int32_t* page_tables, int64_t* slot_mapping, int32_t* total_q_out) {
  if (num_seqs < 0 || page_size < 1 || num_pages < 1 || max_pages_per_seq < 1) return PKV_E_SHAPE;
  if (!cu_seqlens_q || !total_q_out) return PKV_E_NULL;
  if (num_seqs > 0 && (!q_lens || !kv_lens || !page_offsets || !page_ids || !order || !kv_lens_out ||
                       !page_tables))
    return PKV_E_NULL;

  // validate every sequence before writing anything
  int64_t total_q = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const int32_t q = q_lens[i], L = kv_lens[i];
    if (q < 0 || L < q || (q > 0 && L < 1)) return PKV_E_LENGTHS;
    const int32_t n = page_offsets[i + 1] - page_offsets[i];
    if (page_offsets[i] < 0 || n < 0) return PKV_E_PAGES;
    if (n > max_pages_per_seq) return PKV_E_PAGES;
    if ((int64_t)n * page_size < L) return PKV_E_PAGES;
    for (int32_t j = 0; j < n; ++j) {
      const int32_t p = page_ids[page_offsets[i] + j];
      if (p < 0 || p >= num_pages) return PKV_E_PAGES;
    }
    total_q += q;
  }
  if (total_q > slot_capacity || total_q > INT32_MAX) return PKV_E_CAPACITY;
  if (total_q > 0 && !slot_mapping) return PKV_E_NULL;

  // decode sequences (q_len == 1) first, then the rest; arrival order inside each group
  int32_t n_out = 0;
  for (int pass = 0; pass < 2; ++pass)
    for (int32_t i = 0; i < num_seqs; ++i)
      if ((q_lens[i] == 1) == (pass == 0)) order[n_out++] = i;

  cu_seqlens_q[0] = 0;
  int32_t row = 0;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t i = order[b];
    const int32_t q = q_lens[i], L = kv_lens[i];
    const int32_t* pg = page_ids + page_offsets[i];
    const int32_t n = page_offsets[i + 1] - page_offsets[i];
    kv_lens_out[b] = L;
    int32_t* trow = page_tables + (int64_t)b * max_pages_per_seq;
    for (int32_t j = 0; j < max_pages_per_seq; ++j) trow[j] = j < n ? pg[j] : -1;
    // the chunk's tokens occupy positions L - q .. L - 1
    for (int32_t t = 0; t < q; ++t) {
      const int32_t pos = L - q + t;
      slot_mapping[row++] = (int64_t)pg[pos / page_size] * page_size + pos % page_size;
    }
    cu_seqlens_q[b + 1] = row;
  }
  *total_q_out = row;
  return PKV_OK;
}

// Position of every packed row (the slot position of its new token):
// kv_len - q_len + i for row i of a sequence (the chunk's tokens occupy the
// last q_len positions of the context).
extern "C" int pkv_tick_positions(int32_t num_seqs, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                  int32_t* positions, int32_t capacity) {
  if (num_seqs < 0) return PKV_E_SHAPE;
  if (!cu_seqlens_q || (num_seqs > 0 && (!kv_lens || !positions))) return PKV_E_NULL;
  if (cu_seqlens_q[0] != 0) return PKV_E_LENGTHS;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t q = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    if (q < 0 || kv_lens[b] < q) return PKV_E_LENGTHS;
  }
  if (cu_seqlens_q[num_seqs] > capacity) return PKV_E_CAPACITY;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t q = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    for (int32_t i = 0; i < q; ++i) positions[cu_seqlens_q[b] + i] = kv_lens[b] - q + i;
  }
  return PKV_OK;
}
