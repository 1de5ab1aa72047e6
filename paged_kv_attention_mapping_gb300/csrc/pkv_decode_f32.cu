// The decode kernel (pkv_decode.cuh) built for fp32 caches.
#include "pkv_decode.cuh"

namespace pkv {

cudaError_t launch_decode_f32(const AttnArgs& a, cudaStream_t s) {
  return launch_dec_d<float>(a, s);
}

}  // namespace pkv
