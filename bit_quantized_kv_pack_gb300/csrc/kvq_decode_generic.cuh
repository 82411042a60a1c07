// kvq_decode_generic.cuh -- split-KV decode attention on CUDA cores (any head_dim
// in {32, 64, 128, 256}, any GQA ratio).
//
// Computes O = softmax(q K^T / sqrt(d)) V for every query head over the packed
// tokens, dequantized as min + code * scale (InnerQ page, section 3.1), the
// fp16 residual window (BitDecoding page, section 2.2) and the fp16
// attention-sink rows (InnerQ page, section 2.3).  One CTA serves all query
// heads of a KV head block, so the cache is read once per block of up to 8
// query heads (the GQA regrouping of the BitDecoding page, section 2.3).
//
// The per-group scale is factored out of the dot product:
//   q . k^ = sum_g ( scale_g * sum_{e in g} c_e q_e + min_g * sum_{e in g} q_e )
// so the inner loop multiplies integer codes by q in fp32.
//
// Split-KV: each (sequence, KV head, query block) is cut into S pieces of about
// equal byte cost (a packed token costs its code and param bytes, an fp16 token
// -- sink rows first, then the window in age order -- its fp16 bytes, both for
// K and V); each CTA writes a partial (o, m, l)
// and the last one to finish merges the S partials (combine_unit).
//
// The kernel template lives here; kvq_decode_generic_b{2,3,4}.cu instantiate it
// for one code width each (separate translation units compile in parallel),
// and kvq_decode_generic.cu dispatches on the width.
#pragma once

#include <atomic>

#include <math.h>

#include "kvq_decode_common.cuh"
#include "kvq_internal.cuh"

namespace kvq {
namespace generic_detail {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

template <int D, int BITS, int QB>
__global__ void __launch_bounds__(kThreads) decode_generic_kernel(DecodeArgs a) {
  constexpr int NG = D / kGroup;
  constexpr int DPL = D / 32;  // head_dim values per lane in the PV phase
  constexpr int RB = D * BITS / 8;
  constexpr int QMAX = (1 << BITS) - 1;
  static_assert(DPL * BITS <= 32, "one 32-bit word per lane");

  __shared__ float q_s[QB][D];
  __shared__ float qsum_s[QB][NG];
  __shared__ float red_m[kWarps][QB];
  __shared__ float red_l[kWarps][QB];
  __shared__ float red_o[kWarps][QB][D];

  const int s = blockIdx.x;
  const int h = blockIdx.y / a.nqb;
  const int qbi = blockIdx.y % a.nqb;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int Lp = a.packed_len[b];
  const int Lr = a.res_len[b];
  const int rh = a.res_head[b];
  const int Ls = a.Ns > 0 ? a.sink_len[b] : 0;
  const int Lf = Ls + Lr;  // fp16 tokens: sink rows, then the window

  for (int idx = threadIdx.x; idx < QB * D; idx += kThreads) {
    const int i = idx / D, e = idx % D;
    const int qi = qbi * QB + i;
    float v = 0.f;
    if (qi < a.gq) v = __half2float(a.q[((int64_t)b * a.Hq + h * a.gq + qi) * D + e]);
    q_s[i][e] = v;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < QB * NG; idx += kThreads) {
    const int i = idx / NG, g = idx % NG;
    float sum = 0.f;
    for (int e = 0; e < kGroup; ++e) sum += q_s[i][g * kGroup + e];
    qsum_s[i][g] = sum;
  }
  __syncthreads();
  if (s == 0 && qbi == 0 && Lp + Lf == 0 && threadIdx.x == 0) set_error(a.err_word, KVQ_ERRBIT_EMPTY);

  int i0, i1, j0, j1;
  split_range(Lp, Lf, s, a.S, 2 * (RB + 4 * NG), 4 * D, i0, i1, j0, j1);

  float m[QB], l[QB], o[QB][DPL];
#pragma unroll
  for (int i = 0; i < QB; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[i][j] = 0.f;
  }
  const int64_t bh = (int64_t)b * a.Hkv + h;
  // fp16 token j: sink row j, or window token j - Ls (ring slot (rh + j - Ls) % Nr)
  auto fp16_row = [&](const __half* sink, const __half* res, int j) {
    return j < Ls ? sink + (bh * a.Ns + j) * D : res + (bh * a.Nr + (rh + j - Ls) % a.Nr) * D;
  };

  // Online softmax over one chunk of up to 32 tokens (lane = token), given the
  // lane's raw scores; returns p per query for the lane's token.
  auto softmax_chunk = [&](bool valid, const float (&sc)[QB], float (&p)[QB]) {
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      const float sv = valid ? sc[i] * a.qk_scale_log2 : -INFINITY;
      const float mnew = fmaxf(m[i], warp_max(sv));
      // a chunk with no valid token while nothing is accumulated (a page
      // outside the pool) leaves the state as it is instead of exp2(-inf + inf)
      const float alpha = mnew == -INFINITY ? 1.f : exp2f(m[i] - mnew);
      p[i] = valid ? exp2f(sv - mnew) : 0.f;
      l[i] = l[i] * alpha + warp_sum(p[i]);
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[i][j] *= alpha;
      m[i] = mnew;
    }
  };

  // ---- packed tokens
  for (int base = i0 + warp * 32; base < i1; base += kThreads) {
    const int t = base + lane;
    const int64_t row = t < i1 ? a.rm.row(b, h, t) : -1;
    if (t < i1 && row < 0) set_error(a.err_word, KVQ_ERRBIT_BADPAGE);
    const bool valid = row >= 0;  // a token on a page outside the pool is skipped
    float sc[QB];
#pragma unroll
    for (int i = 0; i < QB; ++i) sc[i] = 0.f;
    if (valid) {
      const uint8_t* krow = a.k_codes + row * RB;
      const uint32_t* kp = a.k_params + row * NG;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const uint32_t prm = kp[g];
        const float scale = half_lo(prm), mn = half_hi(prm);
        uint32_t w[BITS];  // the group's 4 * BITS code bytes
        if constexpr (BITS == 4) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(krow + g * 16);
          w[0] = v4.x;
          w[1] = v4.y;
          w[2] = v4.z;
          w[3] = v4.w;
        } else if constexpr (BITS == 3) {  // 12 bytes, 4-byte aligned
          const uint32_t* w3 = reinterpret_cast<const uint32_t*>(krow + g * 12);
          w[0] = w3[0];
          w[1] = w3[1];
          w[2] = w3[2];
        } else {
          const uint2 v2 = *reinterpret_cast<const uint2*>(krow + g * 8);
          w[0] = v2.x;
          w[1] = v2.y;
        }
        float acc[QB];
#pragma unroll
        for (int i = 0; i < QB; ++i) acc[i] = 0.f;
#pragma unroll
        for (int e = 0; e < kGroup; ++e) {
          const int bit = e * BITS;
          uint32_t cw = w[bit / 32] >> (bit % 32);
          if (bit % 32 > 32 - BITS) cw |= w[bit / 32 + 1] << (32 - bit % 32);  // 3-bit straddle
          const float cf = (float)(cw & QMAX);
#pragma unroll
          for (int i = 0; i < QB; ++i) acc[i] = fmaf(cf, q_s[i][g * kGroup + e], acc[i]);
        }
#pragma unroll
        for (int i = 0; i < QB; ++i) sc[i] += scale * acc[i] + mn * qsum_s[i][g];
      }
    }
    float p[QB];
    softmax_chunk(valid, sc, p);
    const int nvalid = min(32, i1 - base);
    const int bo = lane * DPL * BITS;  // bit offset of the lane's values in a row
    const int g_l = (lane * DPL) / kGroup;
    for (int tt = 0; tt < nvalid; ++tt) {
      const int64_t row = a.rm.row(b, h, base + tt);  // the same for every lane
      if (row < 0) continue;
      const uint32_t prm = a.v_params[row * NG + g_l];
      const float scale = half_lo(prm), mn = half_hi(prm);
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(a.v_codes + row * RB) + bo / 32;
      uint32_t w = vw[0] >> (bo % 32);
      if (BITS == 3 && bo % 32 + DPL * BITS > 32) w |= vw[1] << (32 - bo % 32);  // rows are whole words
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const float pt = __shfl_sync(0xffffffffu, p[i], tt);
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          const float v = fmaf((float)((w >> (j * BITS)) & QMAX), scale, mn);
          o[i][j] = fmaf(pt, v, o[i][j]);
        }
      }
    }
  }

  // ---- fp16 tokens (sink rows, then ring slots (res_head + j - Ls) % Nr)
  for (int base = j0 + warp * 32; base < j1; base += kThreads) {
    const int j = base + lane;
    const bool valid = j < j1;
    float sc[QB];
#pragma unroll
    for (int i = 0; i < QB; ++i) sc[i] = 0.f;
    if (valid) {
      const __half* krow = fp16_row(a.k_sink, a.k_res, j);
      for (int e0 = 0; e0 < D; e0 += 8) {
        float x[8];
        unpack8_f16(*reinterpret_cast<const uint4*>(krow + e0), x);
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int i = 0; i < QB; ++i) sc[i] = fmaf(x[e], q_s[i][e0 + e], sc[i]);
      }
    }
    float p[QB];
    softmax_chunk(valid, sc, p);
    const int nvalid = min(32, j1 - base);
    for (int tt = 0; tt < nvalid; ++tt) {
      const __half* vrow = fp16_row(a.v_sink, a.v_res, base + tt) + lane * DPL;
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const float pt = __shfl_sync(0xffffffffu, p[i], tt);
#pragma unroll
        for (int jj = 0; jj < DPL; ++jj) o[i][jj] = fmaf(pt, __half2float(vrow[jj]), o[i][jj]);
      }
    }
  }

  // ---- merge the warps and write this split's partial
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      red_m[warp][i] = m[i];
      red_l[warp][i] = l[i];
    }
  }
#pragma unroll
  for (int i = 0; i < QB; ++i)
#pragma unroll
    for (int j = 0; j < DPL; ++j) red_o[warp][i][lane * DPL + j] = o[i][j];
  __syncthreads();
  const int64_t pidx = (((int64_t)b * a.Hkv + h) * a.nqb + qbi) * a.S + s;
  for (int idx = threadIdx.x; idx < QB * D; idx += kThreads) {
    const int i = idx / D, e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][i]);
    float osum = 0.f, lsum = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(red_m[w][i] - M);
        osum = fmaf(red_o[w][i][e], f, osum);
        lsum = fmaf(red_l[w][i], f, lsum);
      }
    }
    a.o_part[(pidx * QB + i) * D + e] = osum;
    if (e == 0) a.ml_part[pidx * QB + i] = make_float2(M, lsum);
  }
  // the last split of this (KV head, query block) to finish merges all S partials
  __shared__ int s_last;
  if (take_last_ticket<kThreads>(a, ((int64_t)b * a.Hkv + h) * a.nqb + qbi, &s_last)) {
    extern __shared__ float dyn_scratch[];
    combine_unit<kThreads, D, 8>(a, b, h, qbi, dyn_scratch);
  }
}

template <int D, int BITS, int QB>
cudaError_t launch_one(dim3 grid, size_t smem, const DecodeArgs& a, cudaStream_t st) {
  // largest dynamic size opted in so far for this instance, per device (the
  // attribute is per device; a process may drive several GPUs from threads)
  constexpr int kMaxDev = 64;
  static std::atomic<size_t> smem_set[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev || smem > smem_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(decode_generic_kernel<D, BITS, QB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDev) {
      size_t cur = smem_set[dev].load(std::memory_order_relaxed);
      while (cur < smem && !smem_set[dev].compare_exchange_weak(cur, smem)) {
      }
    }
  }
  decode_generic_kernel<D, BITS, QB><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D, int BITS>
cudaError_t launch_generic_d_bits(const DecodePlan& p, dim3 grid, const DecodeArgs& a,
                                  cudaStream_t st) {
  // dynamic shared memory: the combine's weights and sums, 2 * S * qb + qb floats
  const size_t smem = (size_t)(2 * p.splits * p.qb + p.qb) * sizeof(float);
  switch (p.qb) {
    case 1: return launch_one<D, BITS, 1>(grid, smem, a, st);
    case 2: return launch_one<D, BITS, 2>(grid, smem, a, st);
    case 4: return launch_one<D, BITS, 4>(grid, smem, a, st);
    default: return launch_one<D, BITS, 8>(grid, smem, a, st);
  }
}

// All head_dims of one code width.
template <int BITS>
cudaError_t launch_width(const Dims& s, const DecodePlan& p, const DecodeArgs& a, cudaStream_t st) {
  dim3 grid((unsigned)p.splits, (unsigned)(s.Hkv * p.nqb), (unsigned)s.B);
  switch (s.d) {
    case 32: return launch_generic_d_bits<32, BITS>(p, grid, a, st);
    case 64: return launch_generic_d_bits<64, BITS>(p, grid, a, st);
    case 128: return launch_generic_d_bits<128, BITS>(p, grid, a, st);
    default: return launch_generic_d_bits<256, BITS>(p, grid, a, st);
  }
}

}  // namespace generic_detail

// One per code width, each in its own translation unit.
cudaError_t launch_decode_generic_b2(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                     cudaStream_t st);
cudaError_t launch_decode_generic_b3(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                     cudaStream_t st);
cudaError_t launch_decode_generic_b4(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                                     cudaStream_t st);

}  // namespace kvq
