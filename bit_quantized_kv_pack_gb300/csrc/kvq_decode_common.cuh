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
  uint32_t* counters;  // [B][Hkv][nqb] arrival tickets, zero between calls
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

// Tensor-core kernel: head_dim 128, 1 <= gq <= 4 (kvq_decode_tc.cu).
bool tc_supported(const kvq_cache_desc& D, int gq);
int tc_threads();
cudaError_t launch_decode_tc(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                             cudaStream_t st);

// ------------------------------------------------ last-CTA combine ---------
//
// Each split CTA writes its partial (o, m, l), then takes a ticket on its
// (sequence, KV head, query block) counter; the CTA that draws the last ticket
// merges the S partials by log-sum-exp and writes the fp16 output:
//   M = max_s m_s,  O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// atomicInc wraps the counter back to zero, so it is ready for the next call.
// `scratch` holds at least S * qb + 2 * qb floats of shared memory.
template <int NT>
__device__ __forceinline__ bool take_last_ticket(const DecodeArgs& a, int64_t unit, int* flag) {
  __threadfence();  // this CTA's partial is visible before its ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicInc(&a.counters[unit], (unsigned)(a.S - 1));
    *flag = (old == (unsigned)(a.S - 1));
  }
  __syncthreads();
  const bool last = *flag != 0;
  if (last) __threadfence();  // the other CTAs' partials are visible after it
  return last;
}

template <int NT, int D>
__device__ __forceinline__ void combine_unit(const DecodeArgs& a, int b, int h, int qbi,
                                             float* scratch) {
  const int S = a.S, qb = a.qb;
  const int64_t unit = ((int64_t)b * a.Hkv + h) * a.nqb + qbi;
  const int64_t base = unit * S;
  float* w = scratch;              // [S][qb]: m_s, then the weights 2^(m_s - M)
  float* Mq = scratch + S * qb;    // [qb]
  float* Lq = Mq + qb;             // [qb]
  for (int idx = threadIdx.x; idx < S * qb; idx += NT) w[idx] = __ldcg(&a.ml_part[base * qb + idx].x);
  __syncthreads();
  if (threadIdx.x < qb) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, w[s * qb + threadIdx.x]);
    Mq[threadIdx.x] = M;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < S * qb; idx += NT) {
    const float M = Mq[idx % qb];
    w[idx] = M > -INFINITY ? exp2f(w[idx] - M) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < qb) {
    float L = 0.f;
    for (int s = 0; s < S; ++s) L = fmaf(w[s * qb + threadIdx.x], __ldcg(&a.ml_part[(base + s) * qb + threadIdx.x].y), L);
    Lq[threadIdx.x] = L;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < qb * D; idx += NT) {
    const int i = idx / D, e = idx % D;
    const int qi = qbi * qb + i;
    if (qi >= a.gq) continue;
    const float* op = a.o_part + (base * qb + i) * D + e;
    const int64_t stride = (int64_t)qb * D;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= S; s += 4) {  // four independent loads in flight
      const float o0 = __ldcg(op + (s + 0) * stride), o1 = __ldcg(op + (s + 1) * stride);
      const float o2 = __ldcg(op + (s + 2) * stride), o3 = __ldcg(op + (s + 3) * stride);
      acc0 = fmaf(w[(s + 0) * qb + i], o0, acc0);
      acc1 = fmaf(w[(s + 1) * qb + i], o1, acc1);
      acc2 = fmaf(w[(s + 2) * qb + i], o2, acc2);
      acc3 = fmaf(w[(s + 3) * qb + i], o3, acc3);
    }
    for (; s < S; ++s) acc0 = fmaf(w[s * qb + i], __ldcg(op + s * stride), acc0);
    const float L = Lq[i];
    const float o = (acc0 + acc1) + (acc2 + acc3);
    a.out[((int64_t)b * a.Hq + h * a.gq + qi) * D + e] = __float2half_rn(L > 0.f ? o / L : 0.f);
  }
}

cudaError_t launch_decode_generic(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                  cudaStream_t st);

}  // namespace kvq
