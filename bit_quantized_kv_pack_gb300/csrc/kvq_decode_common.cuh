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
  RowMap rm;  // packed token -> row of the codes / params / mode arrays
  const __half* k_sink;  // [B][Hkv][Ns][d] (attention-sink window)
  const __half* v_sink;
  const int32_t* sink_len;
  const __half* q;  // [B][Hq][d]
  void* out;        // [B][Hq][d], fp16 or (out_f32) fp32
  int out_f32;
  float* o_part;
  float2* ml_part;
  uint32_t* counters;     // [B][Hkv][nqb] arrival tickets, zero between calls
  uint32_t* seq_tickets;  // [B] fused step: units of the sequence done, zero between calls
  // tensor-core kernel: shared-reference accumulation of the split results
  // (zero between calls; layout at DecodePlan)
  uint32_t* ref_max;
  uint32_t* fb_flag;
  float* o_acc;
  float* l_acc;
  // fused step (append, then attend): the new token and the cache as writable
  const __half* k_new;  // [B][Hkv][d]
  const __half* v_new;
  uint8_t* w_codes[2];
  uint32_t* w_params[2];
  __half* w_res[2];
  uint8_t* w_modes[2];  // mode bytes of a hybrid cache
  int32_t* w_packed_len;
  int32_t* w_res_len;
  int32_t* w_res_head;
  int Hkv, Hq, gq, qb, nqb, S, cap, Nr, d, row_bytes;
  int Ns;  // sink rows per (sequence, KV head) in the layout (0: no sink)
  int hybrid;  // the fused step quantizes by the hybrid rule
  int early;  // fused step: counters and first tiles may be read before griddepcontrol.wait
  int Sp;  // tensor-core kernel: splits s < Sp take packed tokens, s >= Sp fp16 ones
  uint32_t wait_limit_us;  // bounded waits give up after this long (1 s unless a test set it)
  uint32_t fault_tx;       // testing hook: extra bytes one tile's barrier expects (0: off)
  int fold;                // tensor-core kernel: the last packed split also takes the fp16 rows
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

// Four consecutive output values starting at element `idx` of out (a multiple of
// four), rounded once to the output type.
__device__ __forceinline__ void store_out4(const DecodeArgs& a, int64_t idx, float4 o) {
  if (a.out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + idx) = o;
  } else {
    __half2* dst = reinterpret_cast<__half2*>(static_cast<__half*>(a.out) + idx);
    dst[0] = __floats2half2_rn(o.x, o.y);
    dst[1] = __floats2half2_rn(o.z, o.w);
  }
}

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
int tc_ctas_per_sm(bool several_waves);  // resident CTAs per SM of the variant launched
int tc_residual_rows();
// tokens per pipeline stage of the variant for packed splits of up to
// split_tokens tokens each (128, or 192 for long INT2 splits in one wave)
int tc_tile_tokens(const kvq_cache_desc& D, int cps, int64_t split_tokens);
cudaError_t launch_decode_tc(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                             cudaStream_t st, bool step);

// ------------------------------------------------ last-CTA combine ---------
//
// Each split CTA writes its partial (o, m, l), then takes a ticket on its
// (sequence, KV head, query block) counter; the CTA that draws the last ticket
// merges the S partials by log-sum-exp and writes the fp16 output:
//   M = max_s m_s,  O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// atomicInc wraps the counter back to zero, so it is ready for the next call.
template <int NT>
__device__ __forceinline__ bool take_last_ticket(const DecodeArgs& a, int64_t unit, int* flag) {
  __syncthreads();  // every thread's partial stores precede thread 0's fence
  if (threadIdx.x == 0) {
    __threadfence();  // cumulative: the CTA's partial is visible before its ticket
    const unsigned old = atomicInc(&a.counters[unit], (unsigned)(a.S - 1));
    *flag = (old == (unsigned)(a.S - 1));
    if (*flag) __threadfence();  // the other CTAs' partials are visible after it
  }
  __syncthreads();
  return *flag != 0;
}

// The same ticket with one acquire-release atomic instead of fence, atomic,
// fence: its release makes the CTA's partial and additions (ordered before it
// by the barrier) visible before the ticket, and the last CTA's acquire makes
// the others' visible to it.
template <int NT>
__device__ __forceinline__ bool take_last_ticket_acq_rel(const DecodeArgs& a, int64_t unit, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(&a.counters[unit]), "r"((unsigned)(a.S - 1))
                 : "memory");
    *flag = (old == (unsigned)(a.S - 1));
  }
  __syncthreads();
  return *flag != 0;
}

// Merge the S partials of one (sequence, KV head, query block).  The first CH
// partials of a thread's first output are loaded in one round together with the
// m/l values (all of them when S <= CH); maxima, weights and sums use warp
// reductions.  `scratch` holds at least 2 * S * qb + qb floats of shared memory.
template <int NT, int D, int CH>
__device__ __forceinline__ void combine_unit(const DecodeArgs& a, int b, int h, int qbi,
                                             float* scratch) {
  constexpr int D4 = D / 4;
  constexpr int NW = NT / 32;
  const int S = a.S, qb = a.qb;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t unit = ((int64_t)b * a.Hkv + h) * a.nqb + qbi;
  const int64_t base = unit * S;
  float* w = scratch;            // [S][qb]: m_s, then the weights 2^(m_s - M)
  float* lv = w + S * qb;        // [S][qb]: l_s
  float* Lq = lv + S * qb;       // [qb]
  const int64_t stride = (int64_t)qb * D4;  // float4 elements between splits

  // this thread's first output: one query, four consecutive head_dim values
  const int idx0 = threadIdx.x;
  const int i_0 = idx0 / D4;
  const bool has0 = idx0 < qb * D4 && (qbi * qb + i_0) < a.gq;
  const float4* op0 = reinterpret_cast<const float4*>(a.o_part + (base * qb + i_0) * D) + idx0 % D4;
  float4 v0[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k)
    v0[k] = (has0 && k < S) ? __ldcg(op0 + k * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int idx = threadIdx.x; idx < S * qb; idx += NT) {
    const float2 ml = __ldcg(&a.ml_part[base * qb + idx]);
    w[idx] = ml.x;
    lv[idx] = ml.y;
  }
  __syncthreads();
  for (int q = warp; q < qb; q += NW) {
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, w[s * qb + q]);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float wt = M > -INFINITY ? exp2f(w[s * qb + q] - M) : 0.f;
      w[s * qb + q] = wt;
      L = fmaf(wt, lv[s * qb + q], L);
    }
    L = warp_sum(L);
    if (lane == 0) Lq[q] = L;
  }
  __syncthreads();
  auto finish = [&](int i, int e4, float4 acc) {
    const float L = Lq[i];
    const float inv = L > 0.f ? 1.f / L : 0.f;
    store_out4(a, ((int64_t)b * a.Hq + h * a.gq + qbi * qb + i) * D + 4 * e4,
               make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  };
  // the first output: its first CH partials are already in registers
  if (has0) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const float wk = k < S ? w[k * qb + i_0] : 0.f;
      acc.x = fmaf(wk, v0[k].x, acc.x);
      acc.y = fmaf(wk, v0[k].y, acc.y);
      acc.z = fmaf(wk, v0[k].z, acc.z);
      acc.w = fmaf(wk, v0[k].w, acc.w);
    }
    for (int s = CH; s < S; ++s) {
      const float4 v = __ldcg(op0 + s * stride);
      const float wk = w[s * qb + i_0];
      acc.x = fmaf(wk, v.x, acc.x);
      acc.y = fmaf(wk, v.y, acc.y);
      acc.z = fmaf(wk, v.z, acc.z);
      acc.w = fmaf(wk, v.w, acc.w);
    }
    finish(i_0, idx0 % D4, acc);
  }
  // further outputs (when qb * D / 4 > NT): eight loads in flight
  for (int idx = threadIdx.x + NT; idx < qb * D4; idx += NT) {
    const int i = idx / D4, e4 = idx % D4;
    if (qbi * qb + i >= a.gq) continue;
    const float4* op = reinterpret_cast<const float4*>(a.o_part + (base * qb + i) * D) + e4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = (s0 + k < S) ? __ldcg(op + (s0 + k) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float wk = (s0 + k < S) ? w[(s0 + k) * qb + i] : 0.f;
        acc.x = fmaf(wk, v[k].x, acc.x);
        acc.y = fmaf(wk, v[k].y, acc.y);
        acc.z = fmaf(wk, v[k].z, acc.z);
        acc.w = fmaf(wk, v[k].w, acc.w);
      }
    }
    finish(i, e4, acc);
  }
}

cudaError_t launch_decode_generic(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                  cudaStream_t st);

}  // namespace kvq
