// Decode attention: host-side dispatch of the decode kernel (pkv_decode.cuh)
// to the files that build it for one cache type each, and the kernel's
// configuration facts the planner uses.
#include "pkv_decode.cuh"

namespace pkv {

// defined in pkv_decode_{bf16,f16,f32,fp8}.cu
cudaError_t launch_decode_bf16(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_decode_f16(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_decode_f32(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_decode_fp8(const AttnArgs& a, cudaStream_t s);

namespace {
template <typename TKV, int D>
int inflight_g(int group) {
  switch (group) {
#define PKV_INFLIGHT_CASE(g) \
  case g:                    \
    return DCfg<TKV, D, g>::CPS * DCfg<TKV, D, g>::NST * DCfg<TKV, D, g>::STAGE_BYTES;
    PKV_DECODE_GROUPS(PKV_INFLIGHT_CASE)
#undef PKV_INFLIGHT_CASE
    default: return 0;
  }
}
}  // namespace

int decode_inflight_bytes(int kv_dtype, int D, int group) {
  if (kv_dtype == PKV_FP8_E4M3) return D == 128 ? inflight_g<uint8_t, 128>(group) : 0;
  if (kv_dtype == PKV_F32) return D == 64 ? inflight_g<float, 64>(group) : inflight_g<float, 128>(group);
  if (D == 256) return inflight_g<__half, 256>(group);
  return D == 64 ? inflight_g<__half, 64>(group) : inflight_g<__half, 128>(group);
}

bool decode_supported(int dtype, int D, int P) {
  if (D != 64 && D != 128 && !(D == 256 && (dtype == PKV_F16 || dtype == PKV_BF16))) return false;
  if (dtype == PKV_FP8_E4M3 && D != 128) return false;   // fp8 rows must fill a 128-byte swizzle atom
  if (P % BT == 0) return true;
  return P >= 8 && P % 8 == 0 && BT % P == 0;
}

cudaError_t launch_decode(const AttnArgs& a, cudaStream_t s) {
  if (!decode_supported(a.kv_dtype, a.D, a.P)) return cudaErrorNotSupported;
  KernelTimer timer("decode", s);
  if (a.kv_dtype == PKV_FP8_E4M3) return launch_decode_fp8(a, s);
  switch (a.dtype) {
    case PKV_F32: return launch_decode_f32(a, s);
    case PKV_F16: return launch_decode_f16(a, s);
    default: return launch_decode_bf16(a, s);
  }
}

}  // namespace pkv
