// kvq_testing.cu -- exhaustive checks of the quantizer's fast arithmetic
// against the IEEE operations it stands in for (testing hook, see kvq.h).
//
//  * div_by_const<K> (Markstein's corrected product by the reciprocal) against
//    __fdiv_rn(d, K) for every non-negative finite float d, K = 15, 7, 3;
//    mismatches are counted separately for the quantizer's domain (0, and the
//    differences of fp16 values: 2^-24 .. 131008).
//  * rcp_approx against the exact reciprocal for every positive finite fp16
//    value (the scales): the largest relative error.
#include <string.h>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

template <int K>
__global__ void check_div_kernel(unsigned long long* all, unsigned long long* domain) {
  const uint64_t n = 0x7f800000ull;  // every non-negative finite float
  unsigned long long bad = 0, bad_dom = 0;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const float d = __uint_as_float((uint32_t)i);
    if (__float_as_uint(div_by_const<K>(d)) != __float_as_uint(__fdiv_rn(d, (float)K))) {
      ++bad;
      if (i >= 0x33800000u && i <= 0x47FFE000u) ++bad_dom;
    }
  }
  if (bad) atomicAdd(all, bad);
  if (bad_dom) atomicAdd(domain, bad_dom);
}

__global__ void check_rcp_kernel(unsigned long long* worst_bits) {
  const unsigned h = blockIdx.x * blockDim.x + threadIdx.x;  // fp16 bit pattern
  if (h == 0 || h >= 0x7c00u) return;
  const float s = __half2float(__ushort_as_half((unsigned short)h));
  const double exact = 1.0 / (double)s;
  const double rel = fabs((double)rcp_approx(s) - exact) / exact;
  // non-negative doubles order as their bit patterns
  atomicMax(worst_bits, (unsigned long long)__double_as_longlong(rel));
}

// The counts (a static device array: the check allocates nothing).
__device__ unsigned long long g_check_counts[7];

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_testing_check_arithmetic(uint64_t* div_mismatches, double* rcp_worst_rel) {
  if (!div_mismatches || !rcp_worst_rel) return KVQ_ERR_INVALID_ARG;
  unsigned long long* d = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d), kvq::g_check_counts) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  cudaError_t e = cudaMemset(d, 0, 7 * sizeof(unsigned long long));
  const dim3 grid(1024), block(256);
  if (e == cudaSuccess) {
    kvq::check_div_kernel<15><<<grid, block>>>(d + 0, d + 1);
    kvq::check_div_kernel<7><<<grid, block>>>(d + 2, d + 3);
    kvq::check_div_kernel<3><<<grid, block>>>(d + 4, d + 5);
    kvq::check_rcp_kernel<<<0x7c00 / 256, 256>>>(d + 6);
    e = cudaGetLastError();
  }
  unsigned long long h[7] = {0};
  if (e == cudaSuccess) e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  for (int i = 0; i < 6; ++i) div_mismatches[i] = h[i];
  memcpy(rcp_worst_rel, &h[6], sizeof(double));
  return KVQ_OK;
}
