// The decode kernel (pkv_decode.cuh) built for fp16 caches.
#include "pkv_decode.cuh"

namespace pkv {

cudaError_t launch_decode_f16(const AttnArgs& a, cudaStream_t s) {
  return launch_dec_d<__half>(a, s);
}

}  // namespace pkv
