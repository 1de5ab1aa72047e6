// The decode kernel (pkv_decode.cuh) built for e4m3 caches (bf16 or fp16 queries).
#include "pkv_decode.cuh"

namespace pkv {

cudaError_t launch_decode_fp8(const AttnArgs& a, cudaStream_t s) {
  return a.dtype == PKV_F16 ? launch_dec_g<__half, uint8_t, 128>(a, s)
                            : launch_dec_g<__nv_bfloat16, uint8_t, 128>(a, s);
}

}  // namespace pkv
