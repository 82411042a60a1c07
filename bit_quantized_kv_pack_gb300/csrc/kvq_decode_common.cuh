// kvq_decode_common.cuh -- arguments and helpers shared by the decode kernels.
#pragma once

#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

// Everything a split kernel needs; the partial layout is
//   o_part [B][Hkv][nqb][S][qb][d] fp32 (unnormalised, relative to m)
//   ml_part[B][Hkv][nqb][S][qb] float2 {m, l}, m in log2 units (scores * log2(e)/sqrt(d))
struct DecodeArgs {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const uint32_t* k_params;
  const uint32_t* v_params;
  const __half* k_res;
  const __half* v_res;
  const int32_t* packed_len;
  const int32_t* res_len;
  const int32_t* res_head;
  uint32_t* err_word;
  const __half* q;  // [B][Hq][d]
  __half* out;      // [B][Hq][d]
  float* o_part;
  float2* ml_part;
  int Hkv, Hq, gq, qb, nqb, S, cap, Nr, d;
  float qk_scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ float half_lo(uint32_t hh) {
  return __half2float(__ushort_as_half((unsigned short)(hh & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t hh) {
  return __half2float(__ushort_as_half((unsigned short)(hh >> 16)));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int64_t ceil_div64(int64_t x, int64_t y) { return (x + y - 1) / y; }

// Token range of split s of S over Lp packed tokens (cost cp bytes each) followed
// by Lr residual tokens (cost cr each): the tokens whose byte offset in that
// concatenation falls in [s*U/S, (s+1)*U/S), U the total.  Packed tokens
// [i0, i1), residual tokens [j0, j1) (in age order).
__device__ __forceinline__ void split_range(int Lp, int Lr, int s, int S, int64_t cp, int64_t cr,
                                            int& i0, int& i1, int& j0, int& j1) {
  const int64_t P = (int64_t)Lp * cp;
  const int64_t U = P + (int64_t)Lr * cr;
  const int64_t lo = U * s / S;
  const int64_t hi = U * (s + 1) / S;
  i0 = (int)min(ceil_div64(lo, cp), (int64_t)Lp);
  i1 = (int)min(ceil_div64(hi, cp), (int64_t)Lp);
  j0 = (int)min(ceil_div64(max(lo - P, (int64_t)0), cr), (int64_t)Lr);
  j1 = (int)min(ceil_div64(max(hi - P, (int64_t)0), cr), (int64_t)Lr);
}

cudaError_t launch_decode_generic(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                  cudaStream_t st);
cudaError_t launch_combine(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                           cudaStream_t st);

}  // namespace kvq
