// Prefill-chunk attention on tcgen05, two query tiles per CTA.
//
// Same problem as pkv_prefill_tc.cu (a chunk of new tokens after a cached
// prefix: whole prefix visible, causal inside the chunk; llm-serving-engine
// README, engine step trace "_step_prefill"; Helios README, "Paged attention"),
// arranged so that the tensor core always has the other tile's work while one
// tile is in its softmax. A work tile is (sequence, 128 query rows, two q heads
// of the same GQA group): both query tiles read the same K/V tiles and have the
// same causal mask, so every K/V tile fetched by TMA feeds four MMAs.
//
//   warp 0      TMA producer: Q of both heads, then K_j, V_j into a ring of
//               5 (head_dim 128) or 8 (head_dim 64) shared-memory slots
//               (V rows past kv_len zeroed in the last tile)
//   warp 1      TMEM owner (512 columns) and MMA issuer, per KV tile j and
//               query tile w: O_w += P_w V_{j-1} (A operand read from TMEM),
//               then S_w = Q_w K_j^T into the same TMEM columns; the MMA pipe
//               runs in issue order, so S_w is only overwritten after the PV
//               that reads P_w, and S_w complete implies that PV complete
//   warps 2-5   softmax of query tile 0, one thread per row
//   warps 6-9   softmax of query tile 1
// The softmax reads its S row from TMEM, takes the row max (causal mask only on
// tiles that cross the diagonal), and writes P = exp2(scale * S - m) in
// bf16/fp16 back over S with tcgen05.st (packed pairs: the TMEM layout of a
// 16-bit A operand). O is rescaled in TMEM only when a row's max grows by more
// than 2^8. P never goes through shared memory, which leaves room for a deep
// K/V ring.
// Work tiles follow one another without a block-wide barrier: the producer
// claims the next tile into a 2-entry ring while the current one runs and
// reloads Q once the current tile's last QK MMA is done; the MMA thread starts
// the next tile's first QK while the softmax warps still write the previous
// tile's output.
// fp8 (e4m3) caches use the same kernel with fp16 MMAs: the TMA lands each
// K/V tile as codes in the upper half of its ring slot, two more warps
// (10 and 11) widen the codes to fp16 in the slot's MMA layout (and narrow a
// bf16 Q tile to fp16), and only then release the slot to the MMA thread; the
// K scale is folded into the softmax scale and the V scale into the output
// (mini-vLLM, "Quantization": a fused low-precision kernel instead of
// dequantising before every matmul).
// Every mbarrier wait is bounded (PKV_DEV_TIMEOUT); TMEM accesses are
// warp-uniform.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
using namespace sm100;

namespace {

constexpr int BM = TC_BM;
constexpr int BN = TC_BN;
constexpr int NWG = 2;
constexpr int NTHREADS = (2 + 4 * NWG) * 32;
// fp8 caches: two more warps widen the K/V codes (and narrow a bf16 Q) for
// the MMA; 12 warps still get the 168 registers a softmax thread needs
constexpr int NCONV = 2;
constexpr int NTHREADS_KV8 = NTHREADS + NCONV * 32;

// What the fp8 widening warps need to know about one K/V load of the ring
// (written by the producer before it issues the load).
struct LoadDesc {
  int zero_from;   // rows from here are written as zeros (BN: none)
  int vfix_e;      // >= 0: the last V tile of the work tile in entry vfix_e
  int q_first;     // narrow this work tile's Q (bf16 queries) before the tile
  int q_par;       // parity of that Q load
  int stop;        // no more loads: the widening warps leave
};
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.f;

struct Params2 {
  const int32_t* cu;
  const int32_t* kv_lens;
  const int32_t* page_tables;
  int B, T, Hq, Hkv, P, num_pages, max_pages;
  float scale_log2;  // > 0
  void* out;
  float* lse;
  int32_t* ctrl;
  const int2* pairs;
  int32_t* dev_status;
  const float* k_scale;  // fp8 caches: per-KV-head dequantisation scales (> 0), else null
  const float* v_scale;
};

// A work tile: query tile w attends q head h + w, unless solo: then the GQA
// group has an odd size, h is its last head and query tile 1 repeats head h
// (its MMAs and softmax run, its output is not stored).
struct Tile2 {
  int valid;
  int b, h, kvh, solo, row0, nr, L, p_first, n_kv, j_mask, zero_from;
};

template <int D>
struct Cfg2 {
  static constexpr int HALVES = D / 64;
  static constexpr int NSLOT = D == 128 ? 5 : 8;
  static constexpr uint32_t Q_BYTES = BM * D * 2;       // one query tile
  static constexpr uint32_t SLOT_BYTES = BN * D * 2;
  static constexpr uint32_t SMEM = NWG * Q_BYTES + NSLOT * SLOT_BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory");
};

// tcgen05.mma .kind::f16 with the A operand (M x K, 16-bit, packed in pairs per
// 32-bit column, one row per lane) in TMEM and B in shared memory.
// D[tmem] (+)= A[tmem] * B[smem], the warp-wide form of mma_f16_ss_warp.
__device__ __forceinline__ void mma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (sm_100 family); exact, like two fmaxf.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

template <typename T>
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Two e4m3 codes (the low 16 bits, first element in the low byte) -> two fp16
// values packed (first in the low half). Exact: every e4m3 value, NaN included,
// is an fp16 value. (Measured against an integer-and-multiply widening on the
// mixed tick over an fp8 cache: 255 vs 370 us for the attention call.)
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t codes) {
  uint32_t out;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"((uint16_t)codes));
  return out;
}

// fp8 caches: widen one K or V tile of e4m3 codes into the slot's 16-bit
// layout. The codes arrive by TMA in the upper half of the slot as BN rows of
// 128 codes (head_dim 128), 128-byte swizzled; the fp16 tile is the layout a
// 16-bit TMA load would have made: two 64-column halves of BN 128-byte rows,
// 128-byte swizzled (16-byte chunk c of row r at chunk c ^ (r & 7)). A lane
// reads all 128 codes of its row before writing it, so row r of the upper half
// (its own codes) is overwritten only after it was read. Rows >= zero_from are
// written as zeros (the V rows past the sequence's end: 0 * (NaN code) must not
// reach O), decided once per row: a select per converted pair instead made the
// widening warps, which share SM sub-partitions with the softmax warps, cost the
// chunks of the mixed tick 177 us against 155 us.
__device__ __forceinline__ void widen_rows(unsigned char* slot, int r0, int r1, int lane, int zero_from) {
  const unsigned char* stg = slot + BN * 128;
  for (int r = r0 + lane; r < r1; r += 32) {
    const int sw = r & 7;
    if (r >= zero_from) {
      // a V row past the sequence's end (only in the last tile): zeros
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        unsigned char* row = slot + (k >> 2) * BN * 128 + r * 128;
        *reinterpret_cast<uint4*>(row + (((k & 3) * 2) ^ sw) * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(row + ((((k & 3) * 2 + 1) ^ sw) * 16)) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    uint4 c[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = *reinterpret_cast<const uint4*>(stg + r * 128 + ((k ^ sw) << 4));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        h[2 * q] = e4m3x2_to_h2(w[q]);
        h[2 * q + 1] = e4m3x2_to_h2(w[q] >> 16);
      }
      unsigned char* row = slot + (k >> 2) * BN * 128 + r * 128;   // dims 16k..16k+15: half k / 4
      const int ch = (k & 3) * 2;
      *reinterpret_cast<uint4*>(row + ((ch ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(row + (((ch + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// fp8 caches with bf16 queries: the tcgen05 f16 MMA takes both operands in one
// type, so the Q tiles are narrowed to fp16 in place (same layout, element by
// element, round to nearest).
__device__ __forceinline__ void q_bf16_to_half(unsigned char* q, uint32_t bytes, int lane) {
  uint4* v = reinterpret_cast<uint4*>(q);
  for (uint32_t i = lane; i < bytes / 16; i += 32) {
    uint4 x = v[i];
    uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    v[i] = x;
  }
}

// TQ: query/output element type. KV8: the cache holds e4m3 codes (head_dim 128);
// the MMAs then run in fp16 on widened K/V tiles, the K scale folded into the
// score scale and the V scale into the output.
template <int D, typename TQ, bool KV8>
__global__ void __launch_bounds__(KV8 ? NTHREADS_KV8 : NTHREADS, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, Params2 p) {
  using C = Cfg2<D>;
  using T = typename std::conditional<KV8, __half, TQ>::type;   // MMA operand type
  constexpr bool QCONV = KV8 && std::is_same<TQ, __nv_bfloat16>::value;
  static_assert(!KV8 || D == 128, "fp8 tiles are one 128-code swizzle atom wide");
  constexpr int NS = C::NSLOT;
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sQ = sm;                                   // [NWG][Q tile]
  unsigned char* sRing = sQ + NWG * C::Q_BYTES;             // [NS][slot]

  // Work tiles pass through a 2-entry ring (tile t in entry t & 1): the producer
  // claims tile t + 1 and loads its Q while tile t finishes, so no role waits
  // for a block-wide barrier between tiles.
  __shared__ __align__(8) uint64_t bar_q, bar_full[NS], bar_empty[NS], bar_sfull[NWG], bar_pfull[NWG],
      bar_odone[NWG], bar_qempty, bar_tfull[2], bar_tempty[2], bar_vfix[2], bar_drain;
  // fp8 caches: the TMA lands codes (bar_tma) and Q (bar_qtma); the widening
  // warps convert them and only then arrive on bar_full / bar_q / bar_vfix
  __shared__ __align__(8) uint64_t bar_tma[KV8 ? NS : 1], bar_qtma;
  __shared__ LoadDesc s_ld[KV8 ? NS : 1];
  __shared__ uint32_t s_tmem;
  __shared__ Tile2 s_tile[2];
  __shared__ volatile int s_abort;
  __shared__ int s_bad[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched to get resident while the plan kernel runs: wait for the plan,
  // then let the decode kernel that follows start (it reads the plan too, and
  // nothing this kernel writes).
  pdl_wait();
  pdl_trigger();
  // no tile in this call (every CTA reads the same word): leave before any
  // barrier or tensor-memory set-up
  if (*(volatile const int32_t*)&p.ctrl[CTRL_N_TILES] == 0) return;
  // CTAs past the prefill share leave their SMs to the decode kernel, which
  // may start as soon as every CTA here has passed pdl_trigger
  if ((int)blockIdx.x >= *(volatile const int32_t*)&p.ctrl[CTRL_PF_CTAS]) return;
  if (tid == 0) {
    mbar_init(&bar_q, QCONV ? NCONV : 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], KV8 ? NCONV : 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int w = 0; w < NWG; ++w) {
      mbar_init(&bar_sfull[w], 1);
      mbar_init(&bar_pfull[w], 128);
      mbar_init(&bar_odone[w], 1);
    }
    mbar_init(&bar_qempty, 1);
    for (int e = 0; e < 2; ++e) {
      mbar_init(&bar_tfull[e], 1);
      mbar_init(&bar_tempty[e], 1 + 4 * NWG);   // the MMA thread and every softmax warp
      mbar_init(&bar_vfix[e], KV8 ? NCONV : 1);
    }
    mbar_init(&bar_drain, 1);
    if constexpr (KV8) {
      for (int s = 0; s < NS; ++s) mbar_init(&bar_tma[s], 1);
      mbar_init(&bar_qtma, 1);
    }
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
  }
  if (warp == 1) tmem_alloc(&s_tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int g = p.Hq / p.Hkv;
  const int gpairs = (g + 1) / 2;        // head pairs per GQA group (the last one solo when g is odd)
  const int hpairs = p.Hkv * gpairs;
  const int n_tiles = *(volatile int32_t*)&p.ctrl[CTRL_N_PAIRS] * hpairs;

  uint32_t ring = 0;                   // producer / MMA: K/V loads before the current tile

  if (warp == 0) {
    // --------------------------------------------------------------- producer
    uint32_t fills[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) fills[s] = 0;
    bool ok = true;
    for (uint32_t t = 0; ok; ++t) {
      const uint32_t e = t & 1;
      // entry e is free again once every consumer is done with tile t - 2
      if (t >= 2 &&
          !warp_wait_or_abort(&bar_tempty[e], ((t >> 1) - 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        Tile2 ti;
        ti.valid = 0;
        const int tt = s_abort ? n_tiles : atomicAdd(&p.ctrl[CTRL_TILE_NEXT], 1);
        if (tt < n_tiles) {
          const int2 pr = p.pairs[tt / hpairs];
          ti.b = pr.x;
          const int hp = tt % hpairs;
          ti.kvh = hp / gpairs;
          const int k2 = 2 * (hp - ti.kvh * gpairs);   // first head of the pair within its group
          ti.h = ti.kvh * g + k2;
          ti.solo = k2 + 1 < g ? 0 : 1;
          const int c0 = p.cu[ti.b];
          const int qlen = p.cu[ti.b + 1] - c0;
          ti.L = p.kv_lens[ti.b];
          const int q0 = pr.y * BM;
          ti.row0 = c0 + q0;
          ti.nr = min(BM, qlen - q0);
          ti.p_first = ti.L - qlen + q0;
          const int p_last = ti.p_first + ti.nr - 1;
          ti.n_kv = (p_last + 1 + BN - 1) / BN;
          ti.j_mask = (ti.p_first + 1) / BN;
          ti.zero_from = min(BN, ti.L - (ti.n_kv - 1) * BN);
          ti.valid = 1;
        }
        s_tile[e] = ti;
        s_bad[e] = 0;
        mbar_arrive(&bar_tfull[e]);   // releases the entry's fields to its waiters
      }
      __syncwarp();
      const Tile2 ti = s_tile[e];
      if (!ti.valid) break;
      const int32_t* pt = p.page_tables + (int64_t)ti.b * p.max_pages;
      // Q of this tile replaces the previous tile's once its last QK MMA is done
      if (t >= 1 && !warp_wait_or_abort(&bar_qempty, (t - 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        // fp8 caches with bf16 queries: Q lands on bar_qtma and the widening
        // warps narrow it to fp16 before bar_q releases it to the MMA thread
        uint64_t* qbar = QCONV ? &bar_qtma : &bar_q;
        mbar_arrive_expect_tx(qbar, NWG * C::Q_BYTES);
#pragma unroll
        for (int w = 0; w < NWG; ++w)
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_load_3d(sQ + w * C::Q_BYTES + hf * BM * 128, &mq, qbar, hf * 64, ti.h + (ti.solo ? 0 : w), ti.row0);
      }
      const int n_pages_seq = (ti.L + p.P - 1) / p.P;
      for (int j = 0; j < ti.n_kv && ok; ++j) {
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const uint32_t slot = ring % NS, round = ring / NS;
          ++ring;
          if (!warp_wait_or_abort(&bar_empty[slot], (round & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
            ok = false;
            break;
          }
          unsigned char* dst = sRing + slot * C::SLOT_BYTES;
          const CUtensorMap* map = kv == 0 ? &mk : &mv;
          // 16-bit caches load straight into the MMA layout; fp8 codes land in
          // the upper half of the slot (one 128-code box per page run)
          uint64_t* lbar = KV8 ? &bar_tma[slot] : &bar_full[slot];
          unsigned char* ldst = KV8 ? dst + BN * 128 : dst;
          constexpr int LD_HALVES = KV8 ? 1 : C::HALVES;
          constexpr uint32_t ROW_BYTES = KV8 ? D : D * 2;
          const bool last_v = kv == 1 && j == ti.n_kv - 1;
          if (KV8 && lane == 0) {
            // read by the widening warps once this load's barrier completes
            LoadDesc d;
            d.zero_from = last_v ? ti.zero_from : BN;
            d.vfix_e = last_v ? (int)e : -1;
            d.q_first = QCONV && j == 0 && kv == 0;
            d.q_par = t & 1;
            d.stop = 0;
            s_ld[slot] = d;
          }
          if (lane == 0) {
            if (p.P >= BN) {
              const int lp = (j * BN) / p.P;
              const int off = (j * BN) - lp * p.P;
              const int page = pt[lp];
              if (page < 0 || page >= p.num_pages) {
                atomicOr(&s_bad[e], 1);
                mbar_arrive(lbar);
              } else {
                mbar_arrive_expect_tx(lbar, BN * ROW_BYTES);
#pragma unroll
                for (int hf = 0; hf < LD_HALVES; ++hf)
                  tma_load_3d(ldst + hf * BN * 128, map, lbar, hf * 64, ti.kvh, page * p.P + off);
              }
            } else {
              const int per = BN / p.P;
              const int lp0 = j * per;
              const int cnt = min(per, n_pages_seq - lp0);
              bool bad = false;
              for (int pp = 0; pp < cnt; ++pp) {
                const int page = pt[lp0 + pp];
                bad |= page < 0 || page >= p.num_pages;
              }
              if (bad) {
                atomicOr(&s_bad[e], 1);
                mbar_arrive(lbar);
              } else {
                mbar_arrive_expect_tx(lbar, (uint32_t)cnt * p.P * ROW_BYTES);
                for (int pp = 0; pp < cnt; ++pp) {
                  const int page = pt[lp0 + pp];
#pragma unroll
                  for (int hf = 0; hf < LD_HALVES; ++hf)
                    tma_load_3d(ldst + hf * BN * 128 + pp * p.P * 128, map, lbar, hf * 64, ti.kvh, page * p.P);
                }
              }
            }
          }
          fills[slot] += 1;
          if constexpr (KV8) {
            // the widening warps zero the V rows past the end and arrive on bar_vfix
          } else if (last_v) {
            if (ti.zero_from < BN) {
              if (!warp_wait_or_abort(&bar_full[slot], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
                ok = false;
                break;
              }
              for (int hf = 0; hf < C::HALVES; ++hf) {
                uint4* base = (uint4*)(dst + hf * BN * 128);
                for (int q = ti.zero_from * 8 + lane; q < BN * 8; q += 32) base[q] = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            if (lane == 0) mbar_arrive(&bar_vfix[e]);
          }
        }
      }
    }
    if constexpr (KV8) {
      // no more loads: let the widening warps leave (the slot's previous load
      // must be consumed before its descriptor is rewritten)
      const uint32_t slot = ring % NS, round = ring / NS;
      if (ok && warp_wait_or_abort(&bar_empty[slot], (round & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status) &&
          lane == 0) {
        s_ld[slot].stop = 1;
        mbar_arrive(&bar_tma[slot]);
      }
    }
    if (!ok && lane == 0) {
      // let every copy this warp issued land before the CTA may exit
      for (int s = 0; s < NS; ++s)
        if (fills[s] > 0) mbar_wait(KV8 ? &bar_tma[s] : &bar_full[s], (fills[s] - 1) & 1, 500000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs this loop: operands, ring positions and barrier
    // waits are warp-uniform, and elect.sync picks the one lane that issues
    // every MMA and commit (the same lane each time, so each commit tracks all
    // the MMAs before it). Issued from one lane's divergent code instead, the
    // MMA stream loses issue slots to the softmax warps of its SM
    // sub-partition: measured on GB300, a dense FMA stream in those warps
    // slowed back-to-back M128 N128 K16 MMAs from 64 to ~140 cycles each,
    // against ~67 with the warp-uniform loop.
    // The tensor pipe holds only a few MMAs ahead of the issue, and each
    // barrier wait or commit here costs on the order of 100 cycles, so the
    // waits for the next operands sit behind MMAs already queued: K_j after
    // PV_0 of step j, V_j (used in step j + 1) after PV_1. Ring slots and
    // parities advance incrementally; descriptors are built once per operand
    // tile and stepped by constant offsets (the start-address field is the
    // low 14 bits, and every address stays inside shared memory).
    const uint32_t id_qk = idesc_f16(BM, BN, BF16, false);
    const uint32_t id_pv = idesc_f16(BM, D, BF16, true);
    const uint32_t ring_u32 = smem_u32(sRing);
    const uint64_t qd = smem_desc(smem_u32(sQ), 16, 1024, LAYOUT_SW128);
    uint32_t p_use[NWG] = {0, 0};   // P hand-offs consumed per query tile
    auto issue_qk = [&](int w, uint32_t slot) {
      const uint64_t kd = smem_desc(ring_u32 + slot * C::SLOT_BYTES, 16, 1024, LAYOUT_SW128);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * BM * 128 + (kk % 4) * 32;
        const uint32_t offk = (kk / 4) * BN * 128 + (kk % 4) * 32;
        mma_f16_ss_warp(tmem + w * 128, qd + (uint64_t)((w * C::Q_BYTES + off) >> 4), kd + (uint64_t)(offk >> 4),
                         id_qk, kk > 0 ? 1u : 0u);
      }
      mma_commit_warp(&bar_sfull[w]);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return warp_wait_or_abort(bar, parity, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
    };
    bool ok = true;
    for (uint32_t t = 0; ok; ++t) {
      const uint32_t e = t & 1;
      if (!wait(&bar_tfull[e], (t >> 1) & 1)) break;
      const Tile2 ti = s_tile[e];
      if (!ti.valid) break;
      // K_j is the tile's load 2j and V_j load 2j + 1 of the ring
      uint32_t ks = ring % NS, kph = (ring / NS) & 1;
      uint32_t vs = ks + 1, vph = kph;
      if (vs == (uint32_t)NS) {
        vs = 0;
        vph ^= 1;
      }
      ring += 2 * ti.n_kv;
      ok = wait(&bar_q, t & 1);
      tc_fence_after();
      // step 0: S_w = Q_w K_0^T (the previous tile's last PV, issued earlier,
      // has read the P held in these columns)
      if (ok) ok = wait(&bar_full[ks], kph);
      if (ok) {
#pragma unroll
        for (int w = 0; w < NWG; ++w) issue_qk(w, ks);
        mma_commit_warp(&bar_empty[ks]);
        if (ti.n_kv == 1) mma_commit_warp(&bar_qempty);
        ks += 2;
        if (ks >= (uint32_t)NS) {
          ks -= NS;
          kph ^= 1;
        }
        ok = wait(&bar_full[vs], vph);
      }
      // step j >= 1, per query tile w: O_w (+)= P_w V_{j-1}, then S_w = Q_w K_j^T.
      // The first PV of a tile overwrites O_w: its P hand-off comes after the
      // softmax threads have read the previous tile's O_w out of TMEM.
      for (int j = 1; j <= ti.n_kv && ok; ++j) {
        const bool qk = j < ti.n_kv;
        if (j == ti.n_kv && !wait(&bar_vfix[e], (t >> 1) & 1)) {
          ok = false;
          break;
        }
        const uint64_t vd = smem_desc(ring_u32 + vs * C::SLOT_BYTES, BN * 128, 1024, LAYOUT_SW128);
        const uint32_t acc0 = j > 1 ? 1u : 0u;
        const uint32_t kslot = ks;
#pragma unroll
        for (int w = 0; w < NWG; ++w) {
          if (!wait(&bar_pfull[w], p_use[w] & 1)) {
            ok = false;
            break;
          }
          ++p_use[w];
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_f16_ts_warp(tmem + 256 + w * 128, tmem + w * 128 + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4),
                             id_pv, kk > 0 ? 1u : acc0);
          if (j == ti.n_kv) mma_commit_warp(&bar_odone[w]);
          if (w == NWG - 1) {
            // V_{j-1} has no reader left
            mma_commit_warp(&bar_empty[vs]);
            vs += 2;
            if (vs >= (uint32_t)NS) {
              vs -= NS;
              vph ^= 1;
            }
          }
          if (qk) {
            if (w == 0 && !wait(&bar_full[kslot], kph)) {
              ok = false;
              break;
            }
            if (w == NWG - 1 && !wait(&bar_full[vs], vph)) {
              ok = false;
              break;
            }
            issue_qk(w, kslot);
          }
        }
        if (!ok) break;
        if (qk) {
          mma_commit_warp(&bar_empty[kslot]);
          if (j == ti.n_kv - 1) mma_commit_warp(&bar_qempty);
          ks += 2;
          if (ks >= (uint32_t)NS) {
            ks -= NS;
            kph ^= 1;
          }
        }
      }
      if (ok && lane == 0) mbar_arrive(&bar_tempty[e]);
      __syncwarp();
    }
  } else if (KV8 && warp >= 2 + 4 * NWG) {
    // -------------------------------------------------- fp8: widening warps
    // Loads are taken in ring order; warp cw widens rows [64 cw, 64 cw + 64)
    // of every K/V tile and narrows query tile cw of each work tile.
    const int cw = warp - (2 + 4 * NWG);
    constexpr int ROWS = BN / NCONV;
    for (uint32_t n = 0;; ++n) {
      const uint32_t slot = n % NS, par = (n / NS) & 1;
      if (!warp_wait_or_abort(&bar_tma[slot], par, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) break;
      // the descriptor was written before the load's barrier completed
      const volatile LoadDesc* dv = &s_ld[slot];
      LoadDesc d;
      d.zero_from = dv->zero_from;
      d.vfix_e = dv->vfix_e;
      d.q_first = dv->q_first;
      d.q_par = dv->q_par;
      d.stop = dv->stop;
      if (d.stop) break;
      if (QCONV && d.q_first) {
        if (!warp_wait_or_abort(&bar_qtma, d.q_par, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) break;
        q_bf16_to_half(sQ + cw * C::Q_BYTES, C::Q_BYTES, lane);
        fence_proxy_async_smem();   // the MMA (async proxy) reads what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_q);
      }
      widen_rows(sRing + slot * C::SLOT_BYTES, cw * ROWS, cw * ROWS + ROWS, lane, d.zero_from);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_full[slot]);
        if (d.vfix_e >= 0) mbar_arrive(&bar_vfix[d.vfix_e]);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int w = (warp - 2) >> 2;                // query tile of this warpgroup
    const int qq = warp & 3;                      // TMEM lane quarter of this warp
    const int i = qq * 32 + lane;                 // row within the tile
    const uint32_t lrow = (uint32_t)(qq * 32) << 16;
    const uint32_t s_col = w * 128, o_col = 256 + w * 128;
    uint32_t my_s = 0;   // S hand-offs consumed by this thread
    for (uint32_t t = 0;; ++t) {
      const uint32_t e = t & 1;
      if (!warp_wait_or_abort(&bar_tfull[e], (t >> 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) break;
      const Tile2 ti = s_tile[e];
      if (!ti.valid) break;
      const int p_i = min(ti.p_first + i, ti.L - 1);
      // fp8: the MMA multiplies q by the codes, K = codes * k_scale
      const float sc = KV8 ? p.scale_log2 * __ldg(p.k_scale + ti.kvh) : p.scale_log2;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < ti.n_kv && ok; ++j) {
        // S_w complete also means every earlier MMA (the PV that read P_w) is done
        if (!warp_wait_or_abort(&bar_sfull[w], my_s & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        ++my_s;
        tc_fence_after();
        const bool masked = j >= ti.j_mask;
        const int lim = p_i - j * BN;               // keys with index <= lim are visible
        uint32_t r[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem + lrow + s_col + c * 32, r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) reg_fence(r[c]);
        // row max of the raw scores (scale > 0 keeps the order). The
        // softmax threads share their SM sub-partitions with the MMA thread,
        // whose issue slots a dense run of FMA/ALU work takes away, so the
        // arithmetic here uses as few instructions as it can: three-input
        // max, and fp32x2 FMA / add below.
        if (masked) {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e > lim) r[c][e] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx[(e >> 1) & 7] = max3(mx[(e >> 1) & 7], __uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1]));
        const float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sc;
        const bool first = j == 0;
        const bool grow = first || mt > m_run + RESCALE_LOG2;
        const float m_new = grow ? fmaxf(mt, m_run) : m_run;
        if (!first && __any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? ex2(m_run - m_new) : 1.f;
          l_run *= alpha;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_wait(tmem + lrow + o_col + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32_wait(tmem + lrow + o_col + c * 32, o);
          }
        }
        m_run = m_new;
        // P = exp2(scale * S - m) in 16-bit, packed pairs over the first 64 S
        // columns (masked keys hold -inf: exp2 gives 0 since scale > 0)
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_run, -m_run);
        float2 ls[4];   // partial row sums: ls[k] holds the keys 2k, 2k + 1 (mod 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = hf * 64 + 2 * e;
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(r[k0 >> 5][k0 & 31]), __uint_as_float(r[(k0 + 1) >> 5][(k0 + 1) & 31])),
                sc2, nm2);
            const float a = ex2(x.x), b = ex2(x.y);
            ls[e & 3] = __fadd2_rn(ls[e & 3], make_float2(a, b));
            pw[e] = pack_h2<T>(a, b);
          }
          tmem_st32(tmem + lrow + s_col + hf * 32, pw);
          tmem_wait_st();
          reg_fence(pw);
        }
        l_run += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        tc_fence_before();
        mbar_arrive(&bar_pfull[w]);
      }
      if (ok) ok = warp_wait_or_abort(&bar_odone[w], t & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
      if (ok) ok = warp_wait_or_abort(&bar_vfix[e], (t >> 1) & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
      tc_fence_after();
      if (ok) {
        const int bad = s_bad[e];
        // read here, not kept live through the KV loop (registers are tight)
        const int solo = *(volatile const int*)&s_tile[e].solo;
        const bool store = i < ti.nr && !bad && !(solo && w == 1);
        // fp8: V = codes * v_scale, applied once to the normalised output
        const float inv = (KV8 ? __ldg(p.v_scale + ti.kvh) : 1.f) / l_run;
        const int head = ti.h + (solo ? 0 : w);
        TQ* dst = (TQ*)p.out + ((int64_t)(ti.row0 + i) * p.Hq + head) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_wait(tmem + lrow + o_col + c * 32, o);
          if (!store) continue;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            pk.x = pack_h2<TQ>(__uint_as_float(o[v * 8 + 0]) * inv, __uint_as_float(o[v * 8 + 1]) * inv);
            pk.y = pack_h2<TQ>(__uint_as_float(o[v * 8 + 2]) * inv, __uint_as_float(o[v * 8 + 3]) * inv);
            pk.z = pack_h2<TQ>(__uint_as_float(o[v * 8 + 4]) * inv, __uint_as_float(o[v * 8 + 5]) * inv);
            pk.w = pack_h2<TQ>(__uint_as_float(o[v * 8 + 6]) * inv, __uint_as_float(o[v * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) = pk;
          }
        }
        if (store && p.lse) p.lse[(int64_t)(ti.row0 + i) * p.Hq + head] = (m_run + __log2f(l_run)) * LN2;
        if (i == 0 && w == 0 && bad) {
          atomicOr(&p.ctrl[CTRL_ERR], PKV_DEV_BAD_PAGE);
          atomicOr(p.dev_status, PKV_DEV_BAD_PAGE);
        }
      }
      tc_fence_before();
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tempty[e]);
    }
  }

  if (warp == 1) {
    // every MMA this warp issued is complete before TMEM is released
    mma_commit_warp(&bar_drain);
    mbar_wait(&bar_drain, 0, 500000000ull);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D, typename TQ, bool KV8>
cudaError_t launch2(const AttnArgs& a, cudaStream_t s) {
  using C = Cfg2<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tc2_kernel<D, TQ, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const CUtensorMapDataType dt =
      std::is_same<TQ, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType kdt = KV8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : dt;
  const int kelt = KV8 ? 1 : 2;
  CUtensorMap mq, mk, mv;
  const int box = a.P >= BN ? BN : a.P;
  if (!make_map_boxed(&mq, a.q, dt, 2, D, a.Hq, a.T, 64, BM) ||
      !make_map_boxed(&mk, a.k_cache, kdt, kelt, D, a.Hkv, (int64_t)a.num_pages * a.P, 128 / kelt, box) ||
      !make_map_boxed(&mv, a.v_cache, kdt, kelt, D, a.Hkv, (int64_t)a.num_pages * a.P, 128 / kelt, box))
    return cudaErrorInvalidValue;
  Params2 p;
  p.cu = a.cu;
  p.kv_lens = a.kv_lens;
  p.page_tables = a.page_tables;
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
  p.pairs = (const int2*)(a.ws + a.lay.tc_pairs);
  p.dev_status = a.dev_status;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  const cudaError_t e = launch_after_trigger(prefill_tc2_kernel<D, TQ, KV8>, dim3(a.num_sms),
                                             dim3(KV8 ? NTHREADS_KV8 : NTHREADS), C::SMEM, s, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Any group size but 1 (odd groups pair their heads and run the last one solo;
// with one q head per KV head every tile would be solo, and the one-tile
// kernel does that work without the second tile's idle MMAs).
bool prefill_tc2_supported(int dtype, int D, int P, int Hq, int Hkv, float scale) {
  if (!prefill_tc_supported(dtype, D, P)) return false;
  return Hq / Hkv >= 2 && scale > 0.f;
}

// e4m3 caches have no other tensor-core prefill kernel, so every group size
// takes this one.
bool prefill_tc2_fp8_supported(int q_dtype, int D, int P, int Hq, int Hkv, float scale) {
  // the page rows must split into whole 128-key tiles, as for 16-bit caches
  if (!prefill_tc_supported(q_dtype, D, P) || D != 128) return false;
  return scale > 0.f;
}

cudaError_t launch_prefill_tc2(const AttnArgs& a, cudaStream_t s) {
  KernelTimer timer("prefill_tc", s);
  if (a.kv_dtype == PKV_FP8_E4M3) {
    if (a.D != 128) return cudaErrorNotSupported;
    return a.dtype == PKV_BF16 ? launch2<128, __nv_bfloat16, true>(a, s) : launch2<128, __half, true>(a, s);
  }
  if (a.dtype == PKV_BF16)
    return a.D == 64 ? launch2<64, __nv_bfloat16, false>(a, s) : launch2<128, __nv_bfloat16, false>(a, s);
  return a.D == 64 ? launch2<64, __half, false>(a, s) : launch2<128, __half, false>(a, s);
}

}  // namespace pkv
