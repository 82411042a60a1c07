// kvq_testing.cu -- exhaustive checks of the quantizer's fast arithmetic
// against the IEEE operations it stands in for, and a measurement of how the
// tensor cores' f16 -> f32 MMA rounds (testing hooks, see kvq.h).
//
//  * div_by_const<K> (Markstein's corrected product by the reciprocal) against
//    __fdiv_rn(d, K) for every non-negative finite float d, K = 15, 7, 3;
//    mismatches are counted separately for the quantizer's domain (0, and the
//    differences of fp16 values: 2^-24 .. 131008).
//  * rcp_approx against the exact reciprocal for every positive finite fp16
//    value (the scales): the largest relative error.
#include <string.h>

#include "kvq_internal.cuh"
#include "kvq_ptx.cuh"

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

// One mma.sync m16n8k16 (f16 operands, f32 accumulate) per case: C = c0 plus
// products k = 0 -> big, k = 1..15 -> small (as 2^-12 * (small * 2^12), all
// fp16-exact).  Every row and column of the result is the same; lane 0 writes
// element (0, 0).
constexpr int kMmaCases = 8;
__device__ float g_mma_out[kMmaCases];
__constant__ float kMmaSmall[kMmaCases] = {0.5f, 0.25f, 0.125f, 0.0625f, 0.5f, 0.25f, -0.5f, -0.25f};
__constant__ float kMmaC0[kMmaCases] = {0.f, 0.f, 0.f, 0.f, 1.f, 1.f, 0.f, 0.f};
__constant__ float kMmaBig[kMmaCases] = {1.f, 1.f, 1.f, 1.f, 0.f, 0.f, 1.f, 1.f};

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void mma_rounding_kernel() {
  const int t = threadIdx.x & 3;
  const float ulp1 = 1.f / 8388608.f;  // 2^-23, the spacing of floats at 1
  for (int cs = 0; cs < kMmaCases; ++cs) {
    float av[16], bv[16];
    for (int k = 0; k < 16; ++k) {
      av[k] = 1.f / 4096.f;
      bv[k] = kMmaSmall[cs] * ulp1 * 4096.f;
    }
    av[0] = 1.f;
    bv[0] = kMmaBig[cs];
    // A fragment (row g; k 2t, 2t+1 | 2t+8, 2t+9), the same for rows g + 8;
    // B fragment (k 2t, 2t+1 | 2t+8, 2t+9; column g)
    const uint32_t a0 = pack_f16x2(av[2 * t], av[2 * t + 1]);
    const uint32_t a2 = pack_f16x2(av[2 * t + 8], av[2 * t + 9]);
    const uint32_t b0 = pack_f16x2(bv[2 * t], bv[2 * t + 1]);
    const uint32_t b1 = pack_f16x2(bv[2 * t + 8], bv[2 * t + 9]);
    float c[4] = {kMmaC0[cs], kMmaC0[cs], kMmaC0[cs], kMmaC0[cs]};
    ptx::mma_16816(c, a0, a0, a2, a2, b0, b1);
    if (threadIdx.x == 0) g_mma_out[cs] = c[0];
  }
}

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

extern "C" kvq_status kvq_testing_mma_rounding(float* out, int32_t n) {
  if (!out || n < 0 || n > kvq::kMmaCases) return KVQ_ERR_INVALID_ARG;
  kvq::mma_rounding_kernel<<<1, 32>>>();
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(out, kvq::g_mma_out, n * sizeof(float));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
