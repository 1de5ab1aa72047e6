// Prefill-chunk attention on the tcgen05 tensor cores.
//
// A chunk of new tokens that continues after cached K/V attends the whole
// prefix and, inside the chunk, only earlier positions (llm-serving-engine
// README, engine step trace, "_step_prefill": K/V written at the chunk start,
// prior K/V gathered, rectangular causal mask; Helios README, "Paged
// attention": causal paged attention that reads K/V through page tables).
// QK^T and PV are dense contractions, so they run on the tensor cores; K/V
// tiles come straight out of the page pool by TMA, through the page table,
// never gathered into a dense copy.
//
// Work tile = (sequence, 128 query rows, one q head). Persistent CTAs (one per
// SM) take tiles, longest first, from the device plan. Per CTA:
//   warp 0     TMA producer: Q tile once, then K_j, V_j (128 keys each) into a
//              ring of 4 shared-memory slots; zeroes V rows past kv_len in the
//              last tile so stale or NaN slots never reach the PV product
//   warp 1     TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into one of
//              two TMEM S buffers, O += P_{j-1} V_{j-1} into the TMEM O buffer
//   warps 2-5  softmax, one thread per query row: S row out of TMEM, scale,
//              causal mask, running max with lazy rescale of O (only when the
//              max grows by more than 2^8), P = exp2(S - m) in bf16/fp16 into
//              shared memory (128-byte swizzled K-major, the A operand of PV),
//              and the epilogue O / l, lse.
// Every mbarrier wait is bounded; a timeout sets PKV_DEV_TIMEOUT and the CTA
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
using namespace sm100;

namespace {

constexpr int BM = TC_BM;        // query rows per tile
constexpr int BN = TC_BN;        // keys per KV tile
constexpr int NSLOT = 4;         // K/V ring slots
constexpr int NTHREADS = 192;    // 6 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S = 0;   // two S buffers at columns 0 and 128
constexpr uint32_t TMEM_O = 256;
constexpr float RESCALE_LOG2 = 8.f;

struct TcParams {
  const int32_t* cu;
  const int32_t* kv_lens;
  const int32_t* page_tables;
  int B, T, Hq, Hkv, P, num_pages, max_pages;
  float scale_log2;
  void* out;
  float* lse;
  int32_t* ctrl;
  const int2* pairs;
  int32_t* dev_status;
};

struct TileInfo {
  int valid;
  int b, h, kvh;
  int row0;     // first packed row of the tile
  int nr;       // valid rows (<= BM)
  int L;        // kv_len of the sequence
  int p_first;  // position of the tile's first row
  int n_kv;     // KV tiles the tile's last row needs
  int j_mask;   // first KV tile that needs the causal mask
  int zero_from;  // rows >= zero_from of the last V tile are past kv_len (BN = none)
};

template <int D>
struct Cfg {
  static constexpr int HALVES = D / 64;                 // 64-column (128-byte) swizzle atoms per row
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t SLOT_BYTES = BN * D * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t SMEM = Q_BYTES + NSLOT * SLOT_BYTES + P_BYTES + 1024;
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D, typename T>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, TcParams p) {
  using C = Cfg<D>;
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sQ = sm;
  unsigned char* sRing = sm + C::Q_BYTES;
  unsigned char* sP = sRing + NSLOT * C::SLOT_BYTES;

  __shared__ __align__(8) uint64_t bar_q, bar_full[NSLOT], bar_empty[NSLOT], bar_sfull[2], bar_sfree[2], bar_pfull,
      bar_odone, bar_vfix, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ TileInfo s_tile;
  __shared__ volatile int s_abort;
  __shared__ int s_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched to get resident while the plan kernel runs: wait for the plan,
  // then let the decode kernel that follows start (it reads the plan too, and
  // nothing this kernel writes).
  pdl_wait();
  pdl_trigger();
  // no tile in this call (every CTA reads the same word): leave before any
  // barrier or tensor-memory set-up
  if (*(volatile const int32_t*)&p.ctrl[CTRL_N_TILES] == 0) return;
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_sfull[s], 1);
      mbar_init(&bar_sfree[s], 128);
    }
    mbar_init(&bar_pfull, 128);
    mbar_init(&bar_odone, 1);
    mbar_init(&bar_vfix, 1);
    mbar_init(&bar_drain, 1);
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
  const int n_tiles = *(volatile int32_t*)&p.ctrl[CTRL_N_TILES];
  const int g = p.Hq / p.Hkv;

  // per-role running counters (each role sees the same tile sequence)
  uint32_t ring = 0;      // producer / MMA: K,V slot uses
  uint32_t s_cnt = 0;     // MMA / softmax: S buffer uses
  uint32_t p_cnt = 0;     // MMA: P tiles consumed
  uint32_t o_cnt = 0;     // softmax: PV completions waited
  uint32_t tile_cnt = 0;  // tiles processed by this CTA
  uint32_t fills[NSLOT] = {0, 0, 0, 0};  // producer: fills issued per slot

  for (;;) {
    if (tid == 0) {
      TileInfo ti;
      ti.valid = 0;
      const int t = atomicAdd(&p.ctrl[CTRL_TILE_NEXT], 1);
      if (t < n_tiles && !s_abort) {
        const int2 pr = p.pairs[t / p.Hq];
        ti.b = pr.x;
        ti.h = t % p.Hq;
        ti.kvh = ti.h / g;
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
      s_tile = ti;
      s_bad = 0;
    }
    __syncthreads();
    const TileInfo ti = s_tile;
    if (!ti.valid) break;
    const int32_t* pt = p.page_tables + (int64_t)ti.b * p.max_pages;

    if (warp == 0) {
      // ------------------------------------------------------------- producer
      bool ok = true;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_q, C::Q_BYTES);
#pragma unroll
        for (int hf = 0; hf < C::HALVES; ++hf) tma_load_3d(sQ + hf * BM * 128, &mq, &bar_q, hf * 64, ti.h, ti.row0);
      }
      const int n_pages_seq = (ti.L + p.P - 1) / p.P;
      for (int j = 0; j < ti.n_kv && ok; ++j) {
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const uint32_t slot = ring % NSLOT, round = ring / NSLOT;
          ++ring;
          if (!warp_wait_or_abort(&bar_empty[slot], (round & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
            ok = false;
            break;
          }
          unsigned char* dst = sRing + slot * C::SLOT_BYTES;
          const CUtensorMap* map = kv == 0 ? &mk : &mv;
          if (lane == 0) {
            if (p.P >= BN) {
              const int lp = (j * BN) / p.P;
              const int off = (j * BN) - lp * p.P;
              const int page = pt[lp];
              if (page < 0 || page >= p.num_pages) {
                atomicOr(&s_bad, 1);
                mbar_arrive(&bar_full[slot]);
              } else {
                mbar_arrive_expect_tx(&bar_full[slot], C::SLOT_BYTES);
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
                  tma_load_3d(dst + hf * BN * 128, map, &bar_full[slot], hf * 64, ti.kvh, page * p.P + off);
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
                atomicOr(&s_bad, 1);
                mbar_arrive(&bar_full[slot]);
              } else {
                mbar_arrive_expect_tx(&bar_full[slot], (uint32_t)cnt * p.P * D * 2);
                for (int pp = 0; pp < cnt; ++pp) {
                  const int page = pt[lp0 + pp];
#pragma unroll
                  for (int hf = 0; hf < C::HALVES; ++hf)
                    tma_load_3d(dst + hf * BN * 128 + pp * p.P * 128, map, &bar_full[slot], hf * 64, ti.kvh,
                                page * p.P);
                }
              }
            }
          }
          fills[slot] += 1;
          if (kv == 1 && j == ti.n_kv - 1) {
            if (ti.zero_from < BN) {
              // the last V tile holds slots past kv_len: zero them before PV
              if (!warp_wait_or_abort(&bar_full[slot], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
                ok = false;
                break;
              }
              const int nbytes_row = 128;
              for (int hf = 0; hf < C::HALVES; ++hf) {
                uint4* base = (uint4*)(dst + hf * BN * 128);
                for (int e = ti.zero_from * (nbytes_row / 16) + lane; e < BN * (nbytes_row / 16); e += 32)
                  base[e] = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            if (lane == 0) mbar_arrive(&bar_vfix);
          }
        }
      }
      if (!ok && lane == 0) {
        // let the copies this warp issued land before the CTA leaves
        for (int s = 0; s < NSLOT; ++s)
          if (fills[s] > 0) mbar_wait(&bar_full[s], (fills[s] - 1) & 1, 500000000ull);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t id_qk = idesc_f16(BM, BN, BF16, false);
        const uint32_t id_pv = idesc_f16(BM, D, BF16, true);
        const uint32_t base = ring;
        bool ok = wait_or_abort(&bar_q, tile_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
        tc_fence_after();
        auto issue_pv = [&](int jj) -> bool {
          const uint32_t iv = base + 2 * jj + 1;
          const uint32_t slot = iv % NSLOT, round = iv / NSLOT;
          if (!wait_or_abort(&bar_full[slot], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) return false;
          if (jj == ti.n_kv - 1 && !wait_or_abort(&bar_vfix, tile_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status))
            return false;
          if (!wait_or_abort(&bar_pfull, p_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) return false;
          ++p_cnt;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sRing + slot * C::SLOT_BYTES);
          const uint32_t p_base = smem_u32(sP);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = smem_desc(p_base + (kk / 4) * BM * 128 + (kk % 4) * 32, 16, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(v_base + kk * 16 * 128, BN * 128, 1024, LAYOUT_SW128);
            mma_f16_ss(tmem + TMEM_O, ad, bd, id_pv, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bar_empty[slot]);
          mma_commit(&bar_odone);
          return true;
        };
        for (int j = 0; j < ti.n_kv && ok; ++j) {
          const uint32_t ik = base + 2 * j;
          const uint32_t slot = ik % NSLOT, round = ik / NSLOT;
          const uint32_t sb = s_cnt & 1, su = s_cnt >> 1;
          ok = wait_or_abort(&bar_full[slot], round & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status) &&
               wait_or_abort(&bar_sfree[sb], (su & 1) ^ 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
          if (!ok) break;
          ++s_cnt;
          tc_fence_after();
          const uint32_t q_base = smem_u32(sQ);
          const uint32_t k_base = smem_u32(sRing + slot * C::SLOT_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * BM * 128 + (kk % 4) * 32;
            const uint32_t offk = (kk / 4) * BN * 128 + (kk % 4) * 32;
            const uint64_t ad = smem_desc(q_base + off, 16, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(k_base + offk, 16, 1024, LAYOUT_SW128);
            mma_f16_ss(tmem + TMEM_S + sb * BN, ad, bd, id_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar_sfull[sb]);
          mma_commit(&bar_empty[slot]);
          if (j > 0) ok = issue_pv(j - 1);
        }
        if (ok) ok = issue_pv(ti.n_kv - 1);
      }
      ring += 2 * ti.n_kv;
    } else {
      // --------------------------------------------------------------- softmax
      const int qq = warp & 3;
      const int i = qq * 32 + lane;                 // query row within the tile
      const uint32_t lrow = (uint32_t)(qq * 32) << 16;
      const int p_i = min(ti.p_first + i, ti.L - 1);
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < ti.n_kv && ok; ++j) {
        const uint32_t sb = s_cnt & 1, su = s_cnt >> 1;
        ++s_cnt;
        // tcgen05.ld/st are warp-collective: every decision before one is warp-uniform
        if (!warp_wait_or_abort(&bar_sfull[sb], su & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_wait(tmem + lrow + TMEM_S + sb * BN + c * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
        }
        tc_fence_before();
        mbar_arrive(&bar_sfree[sb]);
        float mt = -INFINITY;
        if (j >= ti.j_mask) {
          const int lim = p_i - j * BN;   // keys with index <= lim are visible
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            s[c] = c <= lim ? s[c] * p.scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            s[c] *= p.scale_log2;
            mt = fmaxf(mt, s[c]);
          }
        }
        const bool first = (j == 0);
        const bool grow = first || mt > m_run + RESCALE_LOG2;
        const float m_new = grow ? fmaxf(mt, m_run) : m_run;
        if (j > 0) {
          // PV_{j-1} must be finished before P is overwritten or O rescaled
          if (!warp_wait_or_abort(&bar_odone, o_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status)) {
            ok = false;
            break;
          }
          ++o_cnt;
          tc_fence_after();
        }
        // rows decide on their own whether the max grew; the warp rescales its
        // 32 rows of O together (alpha = 1 for the rows that keep their max)
        if (!first && __any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? exp2f(m_run - m_new) : 1.f;
          l_run *= alpha;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32_wait(tmem + lrow + TMEM_O + c * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32_wait(tmem + lrow + TMEM_O + c * 32, r);
          }
        }
        m_run = m_new;
        float lsum = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = exp2f(s[hf * 64 + ch * 8 + 2 * e] - m_run);
              const float b = exp2f(s[hf * 64 + ch * 8 + 2 * e + 1] - m_run);
              lsum += a + b;
              w[e] = pack2<T>(a, b);
            }
            unsigned char* dst = sP + hf * BM * 128 + i * 128 + ((ch ^ (i & 7)) * 16);
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        l_run += lsum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_pfull);
      }
      if (ok) ok = warp_wait_or_abort(&bar_odone, o_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
      ++o_cnt;
      if (ok) ok = warp_wait_or_abort(&bar_vfix, tile_cnt & 1, &s_abort, &p.ctrl[CTRL_ERR], p.dev_status);
      tc_fence_after();
      if (ok) {
        // the whole warp reads O; only rows of the chunk are stored
        const bool store = i < ti.nr && !s_bad;
        const float inv = 1.f / l_run;
        T* dst = (T*)p.out + ((int64_t)(ti.row0 + i) * p.Hq + ti.h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_wait(tmem + lrow + TMEM_O + c * 32, r);
          if (!store) continue;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            pk.x = pack2<T>(__uint_as_float(r[v * 8 + 0]) * inv, __uint_as_float(r[v * 8 + 1]) * inv);
            pk.y = pack2<T>(__uint_as_float(r[v * 8 + 2]) * inv, __uint_as_float(r[v * 8 + 3]) * inv);
            pk.z = pack2<T>(__uint_as_float(r[v * 8 + 4]) * inv, __uint_as_float(r[v * 8 + 5]) * inv);
            pk.w = pack2<T>(__uint_as_float(r[v * 8 + 6]) * inv, __uint_as_float(r[v * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) = pk;
          }
        }
        if (store && p.lse) p.lse[(int64_t)(ti.row0 + i) * p.Hq + ti.h] = (m_run + __log2f(l_run)) * LN2;
      }
      if (ok && i == 0 && s_bad) {
        atomicOr(&p.ctrl[CTRL_ERR], PKV_DEV_BAD_PAGE);
        atomicOr(p.dev_status, PKV_DEV_BAD_PAGE);
      }
      tc_fence_before();
    }
    ++tile_cnt;
    __syncthreads();
    if (s_abort) break;
  }

  // drain: every MMA this CTA issued completes before TMEM is released
  if (warp == 1) {
    if (lane == 0) {
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, 500000000ull);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// --------------------------------------------------------------------------- host

template <int D, typename T>
cudaError_t launch_tc(const AttnArgs& a, cudaStream_t s) {
  using C = Cfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tc_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const CUtensorMapDataType dt =
      std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv;
  const int box = a.P >= BN ? BN : a.P;
  if (!make_map_boxed(&mq, a.q, dt, 2, D, a.Hq, a.T, 64, BM) ||
      !make_map_boxed(&mk, a.k_cache, dt, 2, D, a.Hkv, (int64_t)a.num_pages * a.P, 64, box) ||
      !make_map_boxed(&mv, a.v_cache, dt, 2, D, a.Hkv, (int64_t)a.num_pages * a.P, 64, box))
    return cudaErrorInvalidValue;
  TcParams p;
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
  const cudaError_t e =
      launch_after_trigger(prefill_tc_kernel<D, T>, dim3(a.num_sms), dim3(NTHREADS), C::SMEM, s, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int dtype, int D, int P) {
  if (dtype != PKV_BF16 && dtype != PKV_F16) return false;
  if (D != 64 && D != 128) return false;
  if (P % BN == 0) return true;
  return P >= 8 && P % 8 == 0 && BN % P == 0;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t s) {
  if (a.kv_dtype == PKV_FP8_E4M3) {
    if (!prefill_tc2_fp8_supported(a.dtype, a.D, a.P, a.Hq, a.Hkv, a.scale)) return cudaErrorNotSupported;
    return launch_prefill_tc2(a, s);
  }
  if (!prefill_tc_supported(a.dtype, a.D, a.P)) return cudaErrorNotSupported;
  if (prefill_tc2_supported(a.dtype, a.D, a.P, a.Hq, a.Hkv, a.scale)) return launch_prefill_tc2(a, s);
  KernelTimer timer("prefill_tc", s);
  if (a.dtype == PKV_BF16) return a.D == 64 ? launch_tc<64, __nv_bfloat16>(a, s) : launch_tc<128, __nv_bfloat16>(a, s);
  return a.D == 64 ? launch_tc<64, __half>(a, s) : launch_tc<128, __half>(a, s);
}

}  // namespace pkv
