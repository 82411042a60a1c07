// kvq_decode_generic.cu -- dispatch of the CUDA-core decode kernel
// (kvq_decode_generic.cuh) on the code width.
#include "kvq_decode_generic.cuh"

namespace kvq {

cudaError_t launch_decode_generic(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                  cudaStream_t st) {
  if (s.bits == 4) return launch_decode_generic_b4(s, p, a, st);
  if (s.bits == 3) return launch_decode_generic_b3(s, p, a, st);
  return launch_decode_generic_b2(s, p, a, st);
}

}  // namespace kvq
