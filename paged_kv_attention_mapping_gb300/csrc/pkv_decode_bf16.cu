// The decode kernel (pkv_decode.cuh) built for bf16 caches.
#include "pkv_decode.cuh"

namespace pkv {

cudaError_t launch_decode_bf16(const AttnArgs& a, cudaStream_t s) {
  return launch_dec_d<__nv_bfloat16>(a, s);
}

}  // namespace pkv
