// kvq_decode_generic_b2.cu -- the CUDA-core decode kernel for 2-bit codes
// (kvq_decode_generic.cuh), all head_dims and query-block sizes.
#include "kvq_decode_generic.cuh"

namespace kvq {

cudaError_t launch_decode_generic_b2(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                     cudaStream_t st) {
  return generic_detail::launch_width<2>(s, p, a, st);
}

}  // namespace kvq
