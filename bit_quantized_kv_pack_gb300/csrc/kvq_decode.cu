// kvq_decode.cu -- decode planning, the log-sum-exp combine of split partials,
// and the dispatch between decode kernels.
//
// Combine: with per-split maxima m_s, sums l_s and unnormalised outputs o_s,
//   M = max_s m_s,  O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
// (m in log2 units), written as fp16; a head with no tokens gets zeros.
#include <math.h>

#include "kvq_decode_common.cuh"

namespace kvq {
namespace {

__global__ void combine_kernel(DecodeArgs a) {
  const int bhq = blockIdx.x;
  const int b = bhq / a.Hq;
  const int hq = bhq % a.Hq;
  const int h = hq / a.gq;
  const int qi = hq % a.gq;
  const int qbi = qi / a.qb;
  const int i = qi % a.qb;
  const int64_t base = (((int64_t)b * a.Hkv + h) * a.nqb + qbi) * a.S;
  float M = -INFINITY;
  for (int s = 0; s < a.S; ++s) M = fmaxf(M, a.ml_part[(base + s) * a.qb + i].x);
  for (int e = threadIdx.x; e < a.d; e += blockDim.x) {
    float osum = 0.f, lsum = 0.f;
    if (M > -INFINITY) {
      for (int s = 0; s < a.S; ++s) {
        const float2 ml = a.ml_part[(base + s) * a.qb + i];
        const float f = exp2f(ml.x - M);
        lsum = fmaf(ml.y, f, lsum);
        osum = fmaf(a.o_part[((base + s) * a.qb + i) * a.d + e], f, osum);
      }
    }
    a.out[(int64_t)bhq * a.d + e] = __float2half_rn(lsum > 0.f ? osum / lsum : 0.f);
  }
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear a no-device error so it does not leak into later calls
    return 152;
  }
  return n;
}

DecodePlan plan_decode(const kvq_cache_desc& D, int num_q_heads, int sm_count) {
  DecodePlan p;
  p.kernel = 0;
  p.gq = num_q_heads / D.num_kv_heads;
  p.qb = next_pow2(p.gq < 8 ? p.gq : 8);
  p.nqb = (p.gq + p.qb - 1) / p.qb;
  p.threads = 128;
  const int64_t units = (int64_t)D.batch * D.num_kv_heads * p.nqb;
  const int64_t tokens_max = (int64_t)D.capacity + D.residual;
  const int64_t target = (int64_t)sm_count * 4;
  int64_t S = (target + units - 1) / units;
  const int64_t by_len = (tokens_max + 255) / 256;
  if (S > by_len) S = by_len;
  if (S < 1) S = 1;
  if (S > 1024) S = 1024;
  p.splits = (int)S;
  const int64_t nparts = units * S * p.qb;
  p.ws_partials = (size_t)nparts * D.head_dim * sizeof(float);
  const size_t ml_off = (p.ws_partials + 255) & ~(size_t)255;
  p.ws_total = ml_off + (size_t)nparts * sizeof(float2);
  return p;
}

cudaError_t launch_combine(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                           cudaStream_t st) {
  const int threads = s.d < 128 ? s.d : 128;
  combine_kernel<<<(unsigned)(s.B * a.Hq), threads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Dims& s, const DecodePlan& p, const kvq_cache_view& v,
                          const __half* q, int Hq, __half* out, void* workspace,
                          cudaStream_t st) {
  DecodeArgs a;
  a.k_codes = v.k_codes;
  a.v_codes = v.v_codes;
  a.k_params = v.k_params;
  a.v_params = v.v_params;
  a.k_res = reinterpret_cast<const __half*>(v.k_res);
  a.v_res = reinterpret_cast<const __half*>(v.v_res);
  a.packed_len = v.packed_len;
  a.res_len = v.res_len;
  a.res_head = v.res_head;
  a.err_word = v.err_word;
  a.q = q;
  a.out = out;
  a.o_part = reinterpret_cast<float*>(workspace);
  a.ml_part = reinterpret_cast<float2*>(reinterpret_cast<char*>(workspace) +
                                        ((p.ws_partials + 255) & ~(size_t)255));
  a.Hkv = s.Hkv;
  a.Hq = Hq;
  a.gq = p.gq;
  a.qb = p.qb;
  a.nqb = p.nqb;
  a.S = p.splits;
  a.cap = s.cap;
  a.Nr = s.Nr;
  a.d = s.d;
  a.qk_scale_log2 = (float)(1.4426950408889634 / sqrt((double)s.d));
  cudaError_t e = launch_decode_generic(s, p, a, st);
  if (e != cudaSuccess) return e;
  return launch_combine(s, p, a, st);
}

}  // namespace kvq
