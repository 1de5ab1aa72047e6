#pragma once
// Decode attention: single query rows over their pages, HBM-bound.
//
// Helios blog, "torch.sdpa and Flash Attention": softmax(Q K^T / sqrt(d)) V,
// with the query heads of a GQA group sharing one KV head, so one pass over a
// KV head's keys serves the whole group; Helios README, "Paged attention": K/V
// are read through the page table, never gathered into a dense copy.
//
// Work item = (row, KV head, split of the keys), from the device plan. One
// CTA = 1 producer warp + 4 compute warps, persistent, 2 CTAs per SM (3 when a
// stage is at most 16 KB, i.e. head_dim 64 at 16 bits or fp8 with groups up to 8):
//  * producer: takes items from the plan (CTA c starts with item c when the
//    whole grid starts at once, then an atomic counter) into a 2-slot item
//    queue, decoding each with warp-wide searches of the plan; bulk-copies the
//    item's q rows; holds 32 logical pages of the page table in its lanes; and
//    streams 64-key K and V tiles with 3-D TMA boxes (one per page, K or V and
//    128-byte swizzle atom, issued by that many lanes at once) into a ring of
//    3-6 stages, running ahead across item boundaries.
//  * compute warps: warp w owns keys 16w..16w+15 of every tile. 16-bit and
//    fp8 caches use mma.sync m16n8k16 with fp32 accumulators. For groups up to
//    8 the keys are the M rows: S^T = K Q^T and O^T += V^T P^T with the group's
//    heads as the 8 N columns, K and V fragments from ldmatrix (.trans for V),
//    P^T transposed in registers with movmatrix; groups of 16 put the heads on
//    the M rows instead. fp8 codes are widened to fp16 in registers, the K scale
//    folded into the score scale and the V scale into the result. fp32 caches
//    run on CUDA cores with packed fp32x2 FMAs. Online softmax in the exp2
//    domain with shuffle reductions.
//  * end of item: the 4 warps' (m, l, o) merge in shared memory (in the stage
//    of the item's last tile where a separate buffer would cost a CTA per SM);
//    the result goes to out/lse, or to the workspace as a partial when the row
//    was split.
// Keys past the item's end are masked in S and their V rows zeroed in shared
// memory, so stale or NaN slots never enter a sum. Every pipeline wait is the
// bounded sm100::wait_or_abort (PKV_DEV_TIMEOUT, then drain).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_sm100.cuh"

// GQA group sizes the decode kernel is built for (keys as MMA rows up to 8 q
// heads per KV head, heads as rows for 16).
#define PKV_DECODE_GROUPS(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(16)

namespace pkv {
using namespace sm100;

// The templates live in an unnamed namespace: every file that includes this
// header instantiates its own (one cache type each, built in parallel).
namespace {

constexpr int BT = 64;             // keys per tile
constexpr int NCW = 4;             // compute warps
constexpr int NTHREADS = (NCW + 1) * 32;
#ifndef PKV_DEC_CPS_SMALL
#define PKV_DEC_CPS_SMALL 3
#endif

struct DecParams {
  const int32_t* cu;
  const int32_t* kv_lens;
  const int32_t* page_tables;
  const void* q;
  int B, T, Hq, Hkv, P, num_pages, max_pages;
  float scale_log2;
  void* out;
  float* lse;
  int32_t* ctrl;
  // the plan's row-path rows (see PlanLayout): packed row, sequence, keys,
  // first item, first partial slot
  const int32_t* rp_row;
  const int32_t* rp_seq;
  const int32_t* rp_keys;
  const int32_t* rp_item_begin;
  const int32_t* rp_part_begin;
  float* part_o;
  float* part_lse;
  int32_t* dev_status;
  const float* k_scale;  // fp8 caches: dequantisation scale per KV head (else null)
  const float* v_scale;
  int wait_first;        // launched right after the plan kernel: wait for it before reading the plan
};

struct Item {
  int valid;
  int r, kvh, b, k0, k1, nsplit, part;   // part: the item's partial slot when its row is split
  int n_tiles;
};

template <typename T>
struct Elt {
  static constexpr int BYTES = sizeof(T);
};

// 8 bytes of T -> floats (4 bf16/f16 or 2 f32)
__device__ __forceinline__ void cvt16(const uint4& raw, float2 (&o)[4], __nv_bfloat16*) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
__device__ __forceinline__ void cvt16(const uint4& raw, float2 (&o)[4], __half*) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
}
__device__ __forceinline__ void cvt16(const uint4& raw, float2 (&o)[2], float*) {
  o[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
  o[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
}

template <typename T>
__device__ __forceinline__ float2 cvt_pair(uint32_t w);
template <>
__device__ __forceinline__ float2 cvt_pair<__nv_bfloat16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 cvt_pair<__half>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// First index i in [0, n) with a[i] > x (n if none) for a non-decreasing a,
// searched by the whole warp: each round probes 32 evenly spaced entries in
// one load, so n entries take about log32(n) dependent loads. Same result in
// every lane.
__device__ __forceinline__ int warp_upper_bound(const int32_t* a, int n, int x, int lane) {
  int lo = 0, hi = n;   // the answer lies in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(a + idx) <= x;
    const int c = __popc(__ballot_sync(0xffffffffu, le));   // probes 0 .. c-1 are <= x
    if (c == 0) return lo;
    const int nlo = lo + (c - 1) * step + 1;
    const int nhi = lo + c * step;
    lo = nlo;
    hi = nhi < hi ? nhi : hi;
  }
  const int idx = lo + lane;
  const bool le = idx < hi && __ldg(a + idx) <= x;
  return lo + __popc(__ballot_sync(0xffffffffu, le));
}

// --- mma.sync m16n8k16 helpers (16-bit A/B, fp32 accumulators) -------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// transpose of an 8x8 matrix of 16-bit values held in mma fragment layout
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
template <typename T>
__device__ __forceinline__ uint32_t pack2h(float a, float b) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// two e4m3 codes (low byte first) -> two fp16 values packed (low half first)
__device__ __forceinline__ uint32_t fp8x2_to_h2(uint32_t codes) {
  uint32_t out;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"((uint16_t)codes));
  return out;
}

template <typename TKV, int D, int G>
struct DCfg {
  static constexpr int ELT = sizeof(TKV);
  static constexpr int ROW_BYTES = D * ELT;            // one key of one KV head
  static constexpr int ATOMS = ROW_BYTES / 128;        // 128-byte swizzle atoms per key row
  static constexpr int ATOM_ELEMS = 128 / ELT;
  static constexpr int TILE_BYTES = BT * ROW_BYTES;    // K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int Q_BYTES = G * D * 4;
  static constexpr int MERGE_BYTES = NCW * G * D * 4 + NCW * G * 8;
  // Stages: enough bytes in flight to cover HBM latency. Small stages (fp8,
  // head_dim 64) get as many as fit two CTAs per SM, up to 6.
  // CTAs per SM: small stages (head_dim 64 at 16 bits, fp8) run CPS_SMALL CTAs
  // so that more producers stream at once (a CTA's TMA boxes are processed in
  // order, so each CTA's stream has a fixed rate); 64 KB stages (head_dim 256)
  // run one CTA (with three stages up to 6 q heads per KV head, two above);
  // the rest run 2.
  static constexpr int CPS = (STAGE_BYTES <= 16384 && ELT <= 2 && G <= 8) ? PKV_DEC_CPS_SMALL
                             : STAGE_BYTES > 32768                         ? 1
                                                                           : 2;
  static constexpr int BASE_NST = STAGE_BYTES <= 32768 ? 3 : 2;
  // 228 KB of shared memory per SM, 1 KB of it reserved per CTA, ~0.5 KB static
  static constexpr int nst_for(int merge_smem) {
    const int fit = (233472 / CPS - 1536 - Q_BYTES - merge_smem - 1024) / STAGE_BYTES;
    return CPS > 2 ? (fit < 6 ? fit : 6) : (fit > BASE_NST ? (fit < 6 ? fit : 6) : BASE_NST);
  }
  static constexpr int SEP_SMEM = nst_for(MERGE_BYTES) * STAGE_BYTES + Q_BYTES + MERGE_BYTES + 1024;
  // The warps' states are merged in a buffer of their own, unless that buffer
  // would keep CPS CTAs from fitting on an SM (head_dim 128 with 8 q heads per
  // KV head); then they are merged in the stage of the item's last tile, which
  // is released only after the merge. (Measured: merging in the stage where
  // the buffer fits anyway was slower.)
  static constexpr int IN_STAGE_SMEM = nst_for(0) * STAGE_BYTES + Q_BYTES + 1024;
  static constexpr bool MERGE_IN_STAGE = MERGE_BYTES <= STAGE_BYTES && CPS * (SEP_SMEM + 1536) > 233472 &&
                                         CPS * (IN_STAGE_SMEM + 1536) <= 233472;
  static constexpr int MERGE_SMEM = MERGE_IN_STAGE ? 0 : MERGE_BYTES;
  static constexpr int NST = nst_for(MERGE_SMEM);
  static constexpr int SMEM = NST * STAGE_BYTES + Q_BYTES + MERGE_SMEM + 1024;
  static constexpr int DPL = D / 32;                   // PV: dims per lane
  static_assert(ROW_BYTES % 128 == 0, "key rows must be whole swizzle atoms");
};

// address of 16-byte chunk `chunk16` (byte offset chunk16*16 in the key row) of tile row `row`
template <int ATOMS>
__device__ __forceinline__ uint32_t sw_addr(uint32_t tile_base, int row, int byte_off) {
  const int atom = byte_off >> 7;
  const int ch = (byte_off >> 4) & 7;
  return tile_base + atom * (BT * 128) + row * 128 + ((ch ^ (row & 7)) << 4) + (byte_off & 15);
}

// T: query/output element type; TKV: cache element type (T, or uint8_t for an
// fp8 e4m3 cache, dequantised to fp16 in registers for the mma.sync path).
template <typename T, typename TKV, int D, int G>
__global__ void __launch_bounds__(NTHREADS, DCfg<TKV, D, G>::CPS)
    decode_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, DecParams p) {
  using C = DCfg<TKV, D, G>;
  constexpr bool FP8 = std::is_same<TKV, uint8_t>::value;
  using TM = typename std::conditional<FP8, __half, T>::type;   // mma operand type
  constexpr bool MMA = C::ELT == 2 || FP8;
  // keys as the M rows (S^T = K Q^T, O^T = V^T P^T): one n-tile of 8 holds the
  // whole group when G <= 8, half the MMAs of heads-as-rows. The producer then
  // also copies each item's q rows (16-bit) into one of two shared slots.
  constexpr bool KM = MMA && G <= 8;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sStage = sm;
  float* sQ = (float*)(sm + C::NST * C::STAGE_BYTES);
  float* sMergeO = sQ + G * D;                   // [NCW][G][D]
  float* sMergeML = sMergeO + NCW * G * D;       // [NCW][G][2]

  __shared__ __align__(8) uint64_t bar_full[C::NST], bar_empty[C::NST], bar_ifull[2], bar_iempty[2], bar_q[2], bar_cw;
  __shared__ Item s_item[2];
  __shared__ int s_bad[2];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (p.wait_first) pdl_wait();
  pdl_trigger();   // the combine kernel may get resident now; it waits for this grid to finish
  // no item in this call (every CTA reads the same word): leave before any
  // barrier set-up
  const int n_items = *(volatile const int32_t*)&p.ctrl[CTRL_N_ITEMS];
  const int n_rp = *(volatile const int32_t*)&p.ctrl[CTRL_N_RP];
  const int Cchunk = *(volatile const int32_t*)&p.ctrl[CTRL_CHUNK];
  if (n_items == 0) {
    pdl_wait();
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], NCW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_ifull[s], 1);
      mbar_init(&bar_iempty[s], NCW);
      mbar_init(&bar_q[s], 1);
    }
    mbar_init(&bar_cw, NCW * 32);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  if (warp == NCW) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
    }
    uint32_t stage_use = 0;
    uint32_t q_loads = 0;   // q copies issued (lane 0), slots alternate from 0
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      if (!warp_wait_or_abort(&bar_iempty[slot], ((it >> 1) & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status))
        break;
      // next item, decoded by the whole warp (few dependent loads)
      // When every CTA starts at once (not beside the prefill kernel, whose SMs
      // some CTAs wait for), the first item of CTA c is item c and the counter
      // hands out the rest; otherwise the counter hands out every item.
      const int first_static = p.wait_first ? (int)gridDim.x : 0;
      int i = (int)blockIdx.x;
      if ((it > 0 || !first_static) && lane == 0)
        i = s_abort ? n_items : first_static + atomicAdd(&p.ctrl[CTRL_ITEM_NEXT], 1);
      i = __shfl_sync(0xffffffffu, i, 0);
      Item item;
      item.valid = 0;
      if (i < n_items) {
        // the item's row-path row, then the row's fields in one dependent
        // round; a row's items run split by split, the KV heads of one split
        // next to each other, so that CTAs working at the same time read the
        // same pages (the heads of a key row share its DRAM pages)
        const int rj = warp_upper_bound(p.rp_item_begin, n_rp + 1, i, lane) - 1;
        const int jj = i - __ldg(p.rp_item_begin + rj);
        const int keys = __ldg(p.rp_keys + rj);
        const int part0 = __ldg(p.rp_part_begin + rj);
        item.r = __ldg(p.rp_row + rj);
        item.b = __ldg(p.rp_seq + rj);
        const int sp = jj / p.Hkv;
        item.kvh = jj - sp * p.Hkv;
        item.nsplit = (keys + Cchunk - 1) / Cchunk;
        item.k0 = sp * Cchunk;
        item.k1 = min(keys, item.k0 + Cchunk);
        item.part = item.nsplit > 1 ? part0 + item.kvh * item.nsplit + sp : -1;
        item.n_tiles = (item.k1 - item.k0 + BT - 1) / BT;
        item.valid = 1;
      }
      if (lane == 0) {
        s_item[slot] = item;
        s_bad[slot] = 0;
        if constexpr (KM) {
          if (item.valid) {
            constexpr uint32_t QB = G * D * 2;
            mbar_arrive_expect_tx(&bar_q[slot], QB);
            bulk_load(reinterpret_cast<unsigned char*>(sQ) + slot * QB,
                      (const T*)p.q + ((int64_t)item.r * p.Hq + item.kvh * G) * D, QB, &bar_q[slot]);
            ++q_loads;
          }
        }
        mbar_arrive(&bar_ifull[slot]);
      }
      if (!item.valid) break;
      // the item's page ids, 32 logical pages per coalesced warp load; lane j
      // holds page wb + j (-1 past the item's last page)
      const int32_t* pt = p.page_tables + (int64_t)item.b * p.max_pages;
      const int lp_last = (item.k1 - 1) / p.P;
      int wb = item.k0 / p.P;
      int pg = wb + lane <= lp_last ? __ldg(pt + wb + lane) : -1;
      const int per = p.P >= BT ? 1 : BT / p.P;   // pages per tile (at most BT / 8)
      bool ok = true;
      for (int t = 0; t < item.n_tiles; ++t) {
        const int kb = item.k0 + t * BT;
        const int lp0 = kb / p.P;
        const int npg = p.P >= BT ? 1 : min(per, (item.k1 - kb + p.P - 1) / p.P);
        if (lp0 + npg - 1 >= wb + 32) {   // next window (warp-uniform)
          wb = lp0;
          pg = wb + lane <= lp_last ? __ldg(pt + wb + lane) : -1;
        }
        int page[BT / 8];
        bool bad = false;
#pragma unroll
        for (int pp = 0; pp < BT / 8; ++pp) {
          page[pp] = __shfl_sync(0xffffffffu, pg, (lp0 + pp - wb) & 31);
          if (pp < npg) bad |= page[pp] < 0 || page[pp] >= p.num_pages;
        }
        const uint32_t st = stage_use % C::NST, round = stage_use / C::NST;
        ++stage_use;
        if (!warp_wait_or_abort(&bar_empty[st], (round & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        // The copies of a tile are issued by several lanes at once, one copy
        // (page, K or V, 128-byte atom) per lane, after lane 0 has armed the
        // barrier.
        unsigned char* kdst = sStage + st * C::STAGE_BYTES;
        unsigned char* vdst = kdst + C::TILE_BYTES;
        if (bad) {
          if (lane == 0) {
            s_bad[slot] = 1;
            mbar_arrive(&bar_full[st]);
          }
        } else {
          const int n_copies = npg * 2 * C::ATOMS;
          if (lane == 0)
            mbar_arrive_expect_tx(&bar_full[st], (uint32_t)(2 * npg * C::ROW_BYTES * (p.P >= BT ? BT : p.P)));
          __syncwarp();
          constexpr int MAX_COPIES = (BT / 8) * 2 * C::ATOMS;
#pragma unroll
          for (int base = 0; base < MAX_COPIES; base += 32) {
            const int idx = base + lane;
            const int pp = idx / (2 * C::ATOMS), a = (idx >> 1) % C::ATOMS;
            const int pid = __shfl_sync(0xffffffffu, pg, (lp0 + pp - wb) & 31);   // page of logical page lp0 + pp
            if (idx < n_copies) {
              const int row = p.P >= BT ? pid * p.P + (kb - lp0 * p.P) : pid * p.P;
              const uint32_t off = a * BT * 128 + pp * p.P * 128;
              if (idx & 1) tma_load_3d(vdst + off, &mv, &bar_full[st], a * C::ATOM_ELEMS, item.kvh, row);
              else tma_load_3d(kdst + off, &mk, &bar_full[st], a * C::ATOM_ELEMS, item.kvh, row);
            }
          }
        }
      }
      if (!ok) break;
    }
    // let any copy this warp issued land before the CTA may exit
    if (lane == 0) {
      for (int s = 0; s < C::NST; ++s) {
        const uint32_t uses = stage_use / C::NST + (s < (int)(stage_use % C::NST) ? 1 : 0);
        if (uses > 0) mbar_wait(&bar_full[s], (uses - 1) & 1, 500000000ull);
      }
      for (int s = 0; s < 2; ++s) {
        const uint32_t uses = q_loads / 2 + (s < (int)(q_loads % 2) ? 1 : 0);
        if (uses > 0) mbar_wait(&bar_q[s], (uses - 1) & 1, 500000000ull);
      }
    }
    return;
  }

  // ================================================================= compute
  uint32_t stage_use = 0;
  uint32_t cw_phase = 0;
  // barrier of the 128 compute threads, bounded like every other wait
  auto cw_sync = [&]() -> bool {
    mbar_arrive(&bar_cw);
    const bool ok = wait_or_abort(&bar_cw, cw_phase & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
    ++cw_phase;
    return __all_sync(0xffffffffu, ok);
  };
  // With MERGE_IN_STAGE the merge buffers are the stage of the item's last
  // tile: wait until every warp is done reading it.
  uint32_t merge_st = 0;
  auto merge_into_last_stage = [&]() -> bool {
    if constexpr (C::MERGE_IN_STAGE) {
      merge_st = (stage_use - 1) % C::NST;
      sMergeO = reinterpret_cast<float*>(sStage + merge_st * C::STAGE_BYTES);
      sMergeML = sMergeO + NCW * G * D;
      return cw_sync();
    }
    return true;
  };
  const uint32_t stage0 = smem_u32(sStage);
  const int grp = lane >> 2, tig = lane & 3;   // mma fragment coordinates
  for (uint32_t it = 0;; ++it) {
    const int slot = it & 1;
    if (!warp_wait_or_abort(&bar_ifull[slot], (it >> 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) break;
    const Item item = s_item[slot];
    if (!item.valid) break;
    const T* qg = (const T*)p.q + ((int64_t)item.r * p.Hq + item.kvh * G) * D;
    if constexpr (!MMA) {
      // q of the group, scaled into the exp2 domain, into shared memory
      for (int e = tid; e < G * D; e += NCW * 32) sQ[e] = to_f32(qg[e]) * p.scale_log2;
    }
    // also keeps the previous item's merge reads ahead of this item's merge writes
    if (!cw_sync()) break;
    bool ok = true;
    bool bad = false;
    if constexpr (KM) {
      // ------------------------------------------------ tensor cores, keys as rows
      // Q^T as the B operand: column n = head grp (zero for grp >= G). For fp8
      // the contraction index of each 16-dim block is permuted so that k slots
      // (2tig, 2tig+1 | 2tig+8, 2tig+9) hold dims (4tig, 4tig+1 | 4tig+2, 4tig+3),
      // the four bytes one ldmatrix lane receives from a key row.
      if (!warp_wait_or_abort(&bar_q[slot], (it >> 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) break;
      const T* qs = reinterpret_cast<const T*>(reinterpret_cast<const unsigned char*>(sQ) + slot * (G * D * 2));
      uint32_t qb[D / 16][2];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int c0 = kk * 16 + (FP8 ? tig * 4 : tig * 2);
        constexpr int HI_K = FP8 ? 2 : 8;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint32_t w = 0u;
          if (grp < G) {
            w = *reinterpret_cast<const uint32_t*>(qs + grp * D + c0 + u * HI_K);
            if constexpr (FP8 && !std::is_same<T, __half>::value)
              w = pack2h<__half>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));  // bf16 -> fp16
          }
          qb[kk][u] = w;
        }
      }
      // an fp8 cache stores K / k_scale: fold the scale into the score scale
      const float qk_scale = FP8 ? p.scale_log2 * __ldg(p.k_scale + item.kvh) : p.scale_log2;
      // per lane: heads 2tig, 2tig+1; O^T tiles: rows = dims, columns = heads
      float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
      float o[D / 16][4];
#pragma unroll
      for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      for (int t = 0; t < item.n_tiles; ++t) {
        const uint32_t st = stage_use % C::NST, round = stage_use / C::NST;
        ++stage_use;
        if (!warp_wait_or_abort(&bar_full[st], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        const uint32_t kbase = stage0 + st * C::STAGE_BYTES;
        const uint32_t vbase = kbase + C::TILE_BYTES;
        const int tile_keys = min(BT, item.k1 - (item.k0 + t * BT));
        const int nvalid = min(16, tile_keys - warp * 16);   // this warp's keys in the tile (may be <= 0)
        if (nvalid > 0) {
          // keys past the end: zero their V rows so 0 * (stale or NaN) cannot reach O
          if (nvalid < 16) {
            for (int e = lane; e < (16 - nvalid) * (C::ROW_BYTES / 16); e += 32) {
              const int rr = warp * 16 + nvalid + e / (C::ROW_BYTES / 16);
              const int bo = (e % (C::ROW_BYTES / 16)) * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sw_addr<C::ATOMS>(vbase, rr, bo)),
                           "r"(0u)
                           : "memory");
            }
            __syncwarp();
          }
          // S^T = K Q^T: rows = the warp's 16 keys, columns = heads; two
          // accumulators (even / odd 16-dim blocks) halve the dependent chain
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          const int krow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          if constexpr (FP8) {
            // ldmatrix.x4: (keys 0-7 | 8-15) x (chunk 2j | 2j+1); lane gets bytes 4tig..4tig+3
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
              uint32_t r[4];
              ldsm_x4(sw_addr<C::ATOMS>(kbase, krow, (2 * j + (lane >> 4)) * 16), r[0], r[1], r[2], r[3]);
              const uint32_t a0[4] = {fp8x2_to_h2(r[0] & 0xffffu), fp8x2_to_h2(r[1] & 0xffffu),
                                      fp8x2_to_h2(r[0] >> 16), fp8x2_to_h2(r[1] >> 16)};
              const uint32_t a1[4] = {fp8x2_to_h2(r[2] & 0xffffu), fp8x2_to_h2(r[3] & 0xffffu),
                                      fp8x2_to_h2(r[2] >> 16), fp8x2_to_h2(r[3] >> 16)};
              mma16816<TM>(sa, a0, qb[2 * j][0], qb[2 * j][1]);
              mma16816<TM>(sb, a1, qb[2 * j + 1][0], qb[2 * j + 1][1]);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              uint32_t a[4];
              ldsm_x4(sw_addr<C::ATOMS>(kbase, krow, (kk * 16 + (lane >> 4) * 8) * 2), a[0], a[1], a[2], a[3]);
              mma16816<TM>((kk & 1) ? sb : sa, a, qb[kk][0], qb[kk][1]);
            }
          }
          // lane: keys grp (s[0..1]) and grp + 8 (s[2..3]), heads 2tig + e
          float pr[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v0 = grp < nvalid ? (sa[e] + sb[e]) * qk_scale : -INFINITY;
            const float v1 = grp + 8 < nvalid ? (sa[2 + e] + sb[2 + e]) * qk_scale : -INFINITY;
            float mx = fmaxf(v0, v1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[e], mx);
            const float alpha = exp2f(m_run[e] - m_new);
            m_run[e] = m_new;
            pr[e] = exp2f(v0 - m_new);
            pr[2 + e] = exp2f(v1 - m_new);
            l_part[e] = l_part[e] * alpha + pr[e] + pr[2 + e];
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              o[i][e] *= alpha;
              o[i][2 + e] *= alpha;
            }
          }
          // P^T as the B operand: transpose the (keys x heads) fragments in registers
          const uint32_t pb0 = movm_t(pack2h<TM>(pr[0], pr[1]));   // keys 0-7
          const uint32_t pb1 = movm_t(pack2h<TM>(pr[2], pr[3]));   // keys 8-15
          // O^T += V^T P^T
          if constexpr (FP8) {
            // ldmatrix.trans of 16-bit units over (keys 0-7 | 8-15) x (16 bytes | next 16):
            // lane gets dims (2grp, 2grp+1) of keys (2tig, 2tig+1); a byte permute splits
            // them, so tile 2j+h has rows grp -> dim 32j+16h+2grp, grp+8 -> that + 1
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
              uint32_t r[4];
              ldsm_x4_t(sw_addr<C::ATOMS>(vbase, krow, j * 32 + (lane >> 4) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t lo = __byte_perm(r[2 * h], 0u, 0x3120);      // keys 2tig, 2tig+1
                const uint32_t hi = __byte_perm(r[2 * h + 1], 0u, 0x3120);  // keys 2tig+8, 2tig+9
                const uint32_t a[4] = {fp8x2_to_h2(lo & 0xffffu), fp8x2_to_h2(lo >> 16), fp8x2_to_h2(hi & 0xffffu),
                                       fp8x2_to_h2(hi >> 16)};
                mma16816<TM>(o[2 * j + h], a, pb0, pb1);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              // matrices: (keys 0-7, dims +0), (keys 0-7, dims +8), (keys 8-15, +0), (keys 8-15, +8)
              const int vrow = warp * 16 + (lane >> 4) * 8 + (lane & 7);
              uint32_t a[4];
              ldsm_x4_t(sw_addr<C::ATOMS>(vbase, vrow, (i * 16 + ((lane >> 3) & 1) * 8) * 2), a[0], a[1], a[2],
                        a[3]);
              mma16816<TM>(o[i], a, pb0, pb1);
            }
          }
          if (nvalid < 16) fence_proxy_async_smem();   // our zeroing before the next TMA write
        }
        __syncwarp();
        if (lane == 0 && !(C::MERGE_IN_STAGE && t == item.n_tiles - 1)) mbar_arrive(&bar_empty[st]);
      }
      bad = s_bad[slot] != 0;                          // final once the item's last tile landed
      if (lane == 0) mbar_arrive(&bar_iempty[slot]);   // the item slot may be refilled
      if (!__all_sync(0xffffffffu, ok)) break;
      if (!merge_into_last_stage()) break;
      // this warp's state into shared memory
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = tig * 2 + e;
        float l = l_part[e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (h < G) {
          if (grp == 0) {
            sMergeML[(warp * G + h) * 2 + 0] = m_run[e];
            sMergeML[(warp * G + h) * 2 + 1] = l;
          }
          float* dst = sMergeO + (warp * G + h) * D;
#pragma unroll
          for (int i = 0; i < D / 16; ++i) {
            if constexpr (FP8) {
              const int d0 = (i >> 1) * 32 + (i & 1) * 16 + 2 * grp;
              dst[d0] = o[i][e];
              dst[d0 + 1] = o[i][2 + e];
            } else {
              dst[i * 16 + grp] = o[i][e];
              dst[i * 16 + grp + 8] = o[i][2 + e];
            }
          }
        }
      }
    } else if constexpr (MMA) {
      // ------------------------------------------------ tensor cores, heads as rows (G = 16)
      // Q (the group's G heads as the 16 rows of the A operand, rows >= G zero)
      uint32_t qa[D / 16][4];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // fp8: the contraction index of each 16-dim block is permuted so that
        // k slots (2tig, 2tig+1 | 2tig+8, 2tig+9) hold dims (4tig, 4tig+1 | 4tig+2, 4tig+3),
        // the four bytes one ldmatrix lane receives from a key row
        const int c0 = kk * 16 + (FP8 ? tig * 4 : tig * 2);
        constexpr int HI_K = FP8 ? 2 : 8;       // offset of the k slots 2tig+8, 2tig+9
        auto ld2 = [&](int row, int col) -> uint32_t {
          if (row >= G) return 0u;
          const uint32_t w = *reinterpret_cast<const uint32_t*>(qg + row * D + col);
          if constexpr (FP8 && !std::is_same<T, __half>::value) {
            return pack2h<__half>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));  // bf16 -> fp16
          } else {
            return w;
          }
        };
        qa[kk][0] = ld2(grp, c0);
        qa[kk][1] = ld2(grp + 8, c0);
        qa[kk][2] = ld2(grp, c0 + HI_K);
        qa[kk][3] = ld2(grp + 8, c0 + HI_K);
      }
      constexpr bool HI = G > 8;                 // rows grp + 8 are real heads
      // an fp8 cache stores K / k_scale: fold the scale into the score scale
      const float qk_scale = FP8 ? p.scale_log2 * __ldg(p.k_scale + item.kvh) : p.scale_log2;
      float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
      float o[D / 8][4];
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
      for (int t = 0; t < item.n_tiles; ++t) {
        const uint32_t st = stage_use % C::NST, round = stage_use / C::NST;
        ++stage_use;
        if (!warp_wait_or_abort(&bar_full[st], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        const uint32_t kbase = stage0 + st * C::STAGE_BYTES;
        const uint32_t vbase = kbase + C::TILE_BYTES;
        const int tile_keys = min(BT, item.k1 - (item.k0 + t * BT));
        const int nvalid = min(16, tile_keys - warp * 16);   // this warp's keys in the tile (may be <= 0)
        if (nvalid > 0) {
          // keys past the end: zero their V rows so 0 * (stale or NaN) cannot reach O
          if (nvalid < 16) {
            for (int e = lane; e < (16 - nvalid) * (C::ROW_BYTES / 16); e += 32) {
              const int rr = warp * 16 + nvalid + e / (C::ROW_BYTES / 16);
              const int bo = (e % (C::ROW_BYTES / 16)) * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sw_addr<C::ATOMS>(vbase, rr, bo)),
                           "r"(0u)
                           : "memory");
            }
            __syncwarp();
          }
          // S = Q K^T for the warp's 16 keys (two n-tiles of 8)
          float s[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            if constexpr (FP8) {
              // one ldmatrix.x4 = four 16-byte chunks (64 dims) of the n-tile's 8 keys;
              // lane (grp, tig) gets bytes 4tig..4tig+3 of key grp in each chunk
#pragma unroll
              for (int j = 0; j < D / 64; ++j) {
                const int krow = warp * 16 + nt * 8 + (lane & 7);
                uint32_t r[4];
                ldsm_x4(sw_addr<C::ATOMS>(kbase, krow, (j * 4 + (lane >> 3)) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                  mma16816<TM>(s[nt], qa[j * 4 + m], fp8x2_to_h2(r[m] & 0xffffu), fp8x2_to_h2(r[m] >> 16));
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; kk += 2) {
                const int mtx = lane >> 3;
                const int krow = warp * 16 + nt * 8 + (lane & 7);
                const int dim = (kk + (mtx >> 1)) * 16 + (mtx & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sw_addr<C::ATOMS>(kbase, krow, dim * 2), b0, b1, b2, b3);
                mma16816<TM>(s[nt], qa[kk], b0, b1);
                mma16816<TM>(s[nt], qa[kk + 1], b2, b3);
              }
            }
          }
          // online softmax over the warp's keys (rows: head grp, and grp + 8)
          float pv[2][4];
#pragma unroll
          for (int hr = 0; hr < (HI ? 2 : 1); ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int key = nt * 8 + tig * 2 + e;
                float v = s[nt][hr * 2 + e] * qk_scale;
                v = key < nvalid ? v : -INFINITY;
                s[nt][hr * 2 + e] = v;
                mx = fmaxf(mx, v);
              }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[hr], mx);
            const float alpha = exp2f(m_run[hr] - m_new);
            m_run[hr] = m_new;
            float ls = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float pe = exp2f(s[nt][hr * 2 + e] - m_new);
                pv[nt][hr * 2 + e] = pe;
                ls += pe;
              }
            l_part[hr] = l_part[hr] * alpha + ls;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
              o[nd][hr * 2] *= alpha;
              o[nd][hr * 2 + 1] *= alpha;
            }
          }
          if (!HI) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) pv[nt][2] = pv[nt][3] = 0.f;
          }
          // P as the A operand: keys 0-7 from n-tile 0, keys 8-15 from n-tile 1
          uint32_t pa[4];
          pa[0] = pack2h<TM>(pv[0][0], pv[0][1]);
          pa[1] = pack2h<TM>(pv[0][2], pv[0][3]);
          pa[2] = pack2h<TM>(pv[1][0], pv[1][1]);
          pa[3] = pack2h<TM>(pv[1][2], pv[1][3]);
          // O += P V over the warp's 16 keys
          if constexpr (FP8) {
            // ldmatrix.trans of 16-bit units: lane (grp, tig) gets, per 8x16-byte
            // matrix, dims (2grp, 2grp+1) of keys (2tig, 2tig+1). A byte permute
            // splits them into the even-dim and odd-dim B fragments, so n-tile
            // 4j+u covers dims 32j + 16(u>>1) + 2n + (u&1) (undone in the epilogue)
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
              const int vrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
              uint32_t r[4];
              ldsm_x4_t(sw_addr<C::ATOMS>(vbase, vrow, j * 32 + (lane >> 4) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t lo = __byte_perm(r[hh * 2], 0u, 0x3120);      // keys 2tig, 2tig+1
                const uint32_t hi = __byte_perm(r[hh * 2 + 1], 0u, 0x3120);  // keys 2tig+8, 2tig+9
                mma16816<TM>(o[4 * j + 2 * hh], pa, fp8x2_to_h2(lo & 0xffffu), fp8x2_to_h2(hi & 0xffffu));
                mma16816<TM>(o[4 * j + 2 * hh + 1], pa, fp8x2_to_h2(lo >> 16), fp8x2_to_h2(hi >> 16));
              }
            }
          } else {
#pragma unroll
            for (int nd = 0; nd < D / 8; nd += 2) {
              uint32_t b0, b1, b2, b3;
              const int mtx = lane >> 3;
              const int vrow = warp * 16 + (mtx & 1) * 8 + (lane & 7);
              const int dim = (nd + (mtx >> 1)) * 8;
              ldsm_x4_t(sw_addr<C::ATOMS>(vbase, vrow, dim * 2), b0, b1, b2, b3);
              mma16816<TM>(o[nd], pa, b0, b1);
              mma16816<TM>(o[nd + 1], pa, b2, b3);
            }
          }
          if (nvalid < 16) fence_proxy_async_smem();   // our zeroing before the next TMA write
        }
        __syncwarp();
        if (lane == 0 && !(C::MERGE_IN_STAGE && t == item.n_tiles - 1)) mbar_arrive(&bar_empty[st]);
      }
      bad = s_bad[slot] != 0;                          // final once the item's last tile landed
      if (lane == 0) mbar_arrive(&bar_iempty[slot]);   // the item slot may be refilled
      if (!__all_sync(0xffffffffu, ok)) break;
      if (!merge_into_last_stage()) break;
      // this warp's state into shared memory
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int h = grp + hr * 8;
        float l = l_part[hr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (h < G) {
          if (tig == 0) {
            sMergeML[(warp * G + h) * 2 + 0] = m_run[hr];
            sMergeML[(warp * G + h) * 2 + 1] = l;
          }
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd) {
            if constexpr (FP8) {
              // n-tile nd = 4j + u: columns 2tig, 2tig+1 are dims base, base + 2
              const int j = nd >> 2, u = nd & 3;
              float* dst = sMergeO + (warp * G + h) * D + j * 32 + (u >> 1) * 16 + tig * 4 + (u & 1);
              dst[0] = o[nd][hr * 2];
              dst[2] = o[nd][hr * 2 + 1];
            } else {
              float* dst = sMergeO + (warp * G + h) * D + nd * 8 + tig * 2;
              dst[0] = o[nd][hr * 2];
              dst[1] = o[nd][hr * 2 + 1];
            }
          }
        }
      }
    } else {
      // ------------------------------------------------ CUDA-core (fp32) path
      const int j16 = lane & 15;        // QK: key within the warp's 16
      const int half = lane >> 4;       // QK: which half of head_dim
      float m_run[G], l_part[G];
      float2 acc[G][C::DPL / 2 > 0 ? C::DPL / 2 : 1];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
#pragma unroll
        for (int c = 0; c < (C::DPL / 2 > 0 ? C::DPL / 2 : 1); ++c) acc[h][c] = make_float2(0.f, 0.f);
      }
      for (int t = 0; t < item.n_tiles; ++t) {
        const uint32_t st = stage_use % C::NST, round = stage_use / C::NST;
        ++stage_use;
        if (!warp_wait_or_abort(&bar_full[st], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        const uint32_t kbase = stage0 + st * C::STAGE_BYTES;
        const uint32_t vbase = kbase + C::TILE_BYTES;
        const int tile_keys = min(BT, item.k1 - (item.k0 + t * BT));
        const int row = warp * 16 + j16;
        const int nvalid = min(16, tile_keys - warp * 16);   // keys of this warp in the tile (may be <= 0)
        // ---- QK: lanes (j16, half) -> partial dot over half of head_dim
        float s[G];
        {
          float2 a2[G];
#pragma unroll
          for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
          constexpr int HB = C::ROW_BYTES / 2;           // bytes of half a key row
#pragma unroll
          for (int cb = 0; cb < HB; cb += 16) {
            const int boff = half * HB + cb;
            uint4 raw;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                         : "r"(sw_addr<C::ATOMS>(kbase, row, boff)));
            constexpr int NE = 16 / C::ELT;              // elements in the chunk
            float2 kf[NE / 2];
            cvt16(raw, kf, (T*)nullptr);
            const int d0 = boff / C::ELT;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float4* qv = reinterpret_cast<const float4*>(sQ + h * D + d0);
#pragma unroll
              for (int e = 0; e < NE / 4; ++e) {
                const float4 q4 = qv[e];
                a2[h] = __ffma2_rn(make_float2(q4.x, q4.y), kf[2 * e], a2[h]);
                a2[h] = __ffma2_rn(make_float2(q4.z, q4.w), kf[2 * e + 1], a2[h]);
              }
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float v = a2[h].x + a2[h].y;
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            s[h] = j16 < nvalid ? v : -INFINITY;
          }
        }
        // ---- online softmax over the warp's keys
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mx = s[h];
#pragma unroll
          for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
          const float m_new = fmaxf(m_run[h], mx);
          const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run[h] - m_new);
          m_run[h] = m_new;
          pr[h] = m_new == -INFINITY ? 0.f : exp2f(s[h] - m_new);
          l_part[h] = l_part[h] * alpha + (half == 0 ? pr[h] : 0.f);
#pragma unroll
          for (int c = 0; c < (C::DPL / 2 > 0 ? C::DPL / 2 : 1); ++c)
            acc[h][c] = __fmul2_rn(acc[h][c], make_float2(alpha, alpha));
        }
        // ---- PV: lanes own DPL dims of every head
        for (int k = 0; k < nvalid; ++k) {
          const int vrow = warp * 16 + k;
          float pk[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pk[h] = __shfl_sync(0xffffffffu, pr[h], k);
          if constexpr (C::DPL * C::ELT == 8) {  // 2 x f32 per lane
            uint2 raw;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(raw.x), "=r"(raw.y)
                         : "r"(sw_addr<C::ATOMS>(vbase, vrow, lane * 8)));
            const float2 v0 = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h][0] = __ffma2_rn(make_float2(pk[h], pk[h]), v0, acc[h][0]);
          } else {  // 4 x f32 per lane
            uint4 raw;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                         : "r"(sw_addr<C::ATOMS>(vbase, vrow, lane * 16)));
            const float2 v0 = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
            const float2 v1 = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
#pragma unroll
            for (int h = 0; h < G; ++h) {
              acc[h][0] = __ffma2_rn(make_float2(pk[h], pk[h]), v0, acc[h][0]);
              acc[h][1] = __ffma2_rn(make_float2(pk[h], pk[h]), v1, acc[h][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0 && !(C::MERGE_IN_STAGE && t == item.n_tiles - 1)) mbar_arrive(&bar_empty[st]);
      }
      bad = s_bad[slot] != 0;
      if (lane == 0) mbar_arrive(&bar_iempty[slot]);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (!merge_into_last_stage()) break;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float l = l_part[h];
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o2);
        if (lane == 0) {
          sMergeML[(warp * G + h) * 2 + 0] = m_run[h];
          sMergeML[(warp * G + h) * 2 + 1] = l;
        }
        float* dst = sMergeO + (warp * G + h) * D + lane * C::DPL;
#pragma unroll
        for (int c = 0; c < C::DPL; ++c) dst[c] = (c & 1) ? acc[h][c >> 1].y : acc[h][c >> 1].x;
      }
    }
    // ---- merge the 4 warps' states
    if (!cw_sync()) break;
    if (!bad) {
      for (int e = tid; e < G * D; e += NCW * 32) {
        const int h = e / D;
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) m = fmaxf(m, sMergeML[(w * G + h) * 2]);
        float l = 0.f, ov = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float mw = sMergeML[(w * G + h) * 2];
          const float sc = mw == -INFINITY ? 0.f : exp2f(mw - m);
          l += sMergeML[(w * G + h) * 2 + 1] * sc;
          ov += sMergeO[(w * G + h) * D + (e - h * D)] * sc;
        }
        ov /= l;
        if constexpr (FP8) ov *= __ldg(p.v_scale + item.kvh);   // the cache stores V / v_scale
        const float lse_n = (m + __log2f(l)) * LN2;
        if (item.nsplit == 1) {
          ((T*)p.out)[((int64_t)item.r * p.Hq + item.kvh * G) * D + e] = from_f32<T>(ov);
          if (p.lse && (e - h * D) == 0) p.lse[(int64_t)item.r * p.Hq + item.kvh * G + h] = lse_n;
        } else {
          const int pidx = item.part;
          p.part_o[((int64_t)pidx * G) * D + e] = ov;
          if ((e - h * D) == 0) p.part_lse[(int64_t)pidx * G + h] = lse_n;
        }
      }
    } else if (tid == 0) {
      atomicOr(&p.ctrl[CTRL_ERR], PKV_DEV_BAD_PAGE);
      atomicOr(p.dev_status, PKV_DEV_BAD_PAGE);
    }
    if constexpr (C::MERGE_IN_STAGE) {
      // this warp is done with the merge buffers: hand the stage back (the
      // fence orders our generic writes before the next TMA write into it)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_empty[merge_st]);
    }
  }
  // When launched to overlap the prefill kernel, finish only after it, so that
  // whatever follows this kernel also follows the prefill.
  pdl_wait();
}

template <typename T, typename TKV, int D, int G>
cudaError_t launch_dec(const AttnArgs& a, cudaStream_t s) {
  using C = DCfg<TKV, D, G>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel<T, TKV, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const CUtensorMapDataType dt = std::is_same<TKV, float>::value    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : std::is_same<TKV, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : std::is_same<TKV, uint8_t>::value ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int box_rows = a.P >= BT ? BT : a.P;
  CUtensorMap mk, mv;
  if (!make_map_boxed(&mk, a.k_cache, dt, C::ELT, D, a.Hkv, (int64_t)a.num_pages * a.P, C::ATOM_ELEMS, box_rows) ||
      !make_map_boxed(&mv, a.v_cache, dt, C::ELT, D, a.Hkv, (int64_t)a.num_pages * a.P, C::ATOM_ELEMS, box_rows))
    return cudaErrorInvalidValue;
  DecParams p;
  p.cu = a.cu;
  p.kv_lens = a.kv_lens;
  p.page_tables = a.page_tables;
  p.q = a.q;
  p.B = a.B;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.P = a.P;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  p.scale_log2 = a.scale * LOG2E;
  p.out = a.out;
  p.lse = a.lse;
  p.ctrl = (int32_t*)(a.ws + a.lay.ctrl);
  p.rp_row = (const int32_t*)(a.ws + a.lay.rp_row);
  p.rp_seq = (const int32_t*)(a.ws + a.lay.rp_seq);
  p.rp_keys = (const int32_t*)(a.ws + a.lay.rp_keys);
  p.rp_item_begin = (const int32_t*)(a.ws + a.lay.rp_item_begin);
  p.rp_part_begin = (const int32_t*)(a.ws + a.lay.rp_part_begin);
  p.part_o = (float*)(a.ws + a.lay.part_o);
  p.part_lse = (float*)(a.ws + a.lay.part_lse);
  p.dev_status = a.dev_status;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  // After the prefill kernel: rows of the decode path and tiles of the prefill
  // kernel are disjoint, and the plan both read finished before the prefill
  // kernel started, so this grid may start as soon as the prefill kernel has
  // (its CTAs take the SMs the prefill kernel leaves) and waits for it only
  // before it exits. Right after the plan kernel (which triggers at its
  // start): the CTAs get resident during the plan and wait for it first.
  p.wait_first = a.after_prefill ? 0 : 1;
  const cudaError_t e = launch_after_trigger(decode_kernel<T, TKV, D, G>, dim3(a.num_sms * C::CPS),
                                             dim3(NTHREADS), C::SMEM, s, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, typename TKV, int D>
cudaError_t launch_dec_g(const AttnArgs& a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
#define PKV_DEC_CASE(g) \
  case g:               \
    return launch_dec<T, TKV, D, g>(a, s);
    PKV_DECODE_GROUPS(PKV_DEC_CASE)
#undef PKV_DEC_CASE
    default: return cudaErrorNotSupported;
  }
}

template <typename T>
cudaError_t launch_dec_d(const AttnArgs& a, cudaStream_t s) {
  if constexpr (sizeof(T) == 2) {
    if (a.D == 256) return launch_dec_g<T, T, 256>(a, s);   // 16-bit caches only: 64 KB stages
  }
  return a.D == 64 ? launch_dec_g<T, T, 64>(a, s) : launch_dec_g<T, T, 128>(a, s);
}

}  // namespace
}  // namespace pkv
