// kvq_internal.cuh -- device helpers and launch plans shared by the kernels of
// libkvq.so.  Layout and semantics are those of include/kvq.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kGroup = 32;  // G: values per quantization group along head_dim

// ----------------------------------------------------------------- sizes ---

struct Dims {
  int B, Hkv, d, bits, cap, Nr;
  int Ns;        // attention-sink window length (0: none)
  int hybrid;    // 1: hybrid sym/asym groups with mode bytes
  int page;      // 0: contiguous packed rows; kPage: paged through a block table
  int npages;    // pages in the pool of a paged cache
  int Ng;        // groups per token row
  int row_bytes; // packed code bytes per token row
};

inline Dims dims_of(const kvq_cache_desc& D) {
  Dims s;
  s.B = D.batch;
  s.Hkv = D.num_kv_heads;
  s.d = D.head_dim;
  s.bits = D.bits;
  s.cap = D.capacity;
  s.Nr = D.residual;
  s.Ns = D.sink;
  s.hybrid = D.hybrid;
  s.page = D.page_size;
  s.npages = D.page_size ? D.num_pages : 0;
  s.Ng = D.head_dim / kGroup;
  s.row_bytes = D.head_dim * D.bits / 8;
  return s;
}

constexpr int kPage = 32;  // tokens per page of a paged cache

// Where packed token t of (sequence b, KV head h) sits in the codes, params and
// mode arrays: row (b * Hkv + h) * cap + t of a contiguous cache, or row
// (page * Hkv + h) * 32 + t % 32 of a paged one, page = block_table[b][t / 32].
// -1 for a page outside the pool (the caller sets KVQ_ERRBIT_BADPAGE and skips).
struct RowMap {
  const int32_t* block_table;  // [B][cap / 32] (paged)
  int Hkv, cap, paged, npages;

  __device__ __forceinline__ int page_of(int b, int j) const {  // j = t / 32
    return __ldg(block_table + (int64_t)b * (cap / kPage) + j);
  }
  __device__ __forceinline__ int64_t row(int b, int h, int t) const {
    if (!paged) return ((int64_t)b * Hkv + h) * cap + t;
    const int pg = page_of(b, t / kPage);
    if (pg < 0 || pg >= npages) return -1;
    return ((int64_t)pg * Hkv + h) * kPage + (t % kPage);
  }
};

inline RowMap row_map(const Dims& s, const int32_t* block_table) {
  RowMap m;
  m.block_table = block_table;
  m.Hkv = s.Hkv;
  m.cap = s.cap;
  m.paged = s.page != 0;
  m.npages = s.npages;
  return m;
}

// ------------------------------------------------------------ error word ---

__device__ __forceinline__ void set_error(uint32_t* err_word, uint32_t bit) {
  if (err_word) atomicOr(err_word, bit);
}

// ----------------------------------------------------- group quantizer ------
//
// One group of 32 fp16 values is held by 4 consecutive lanes, 8 values each
// (lane q of the quad holds values 8q .. 8q+7 as one 16-byte word).  Steps
// Q1-Q4 with the op order fixed by the header:
//   Q1  min/max over the quad: fp16 min of the lane's values and of their
//       negations (max = -min(-x), exact), then shuffle-xor 1 and 2 of both as one
//       half2 -- min and max of fp16 values are exact in any order
//   Q2  scale_f = (mx - mn) / (2^b - 1) in fp32, correctly rounded (div_by_const)
//   Q3  scale_h = fp16_rne(scale_f); min_h = fp16(mn + 0)
//   Q4  code = clamp(rint((x - mn) / s), 0, 2^b - 1) with s = (float)scale_h and
//       the IEEE divide, or 0 when s == 0.
// How Q4 is computed (same codes as the plain divide):
//   dx = x - mn is one fp32 subtraction straight from the fp16 operand (exact
//   conversion, one rounding, as (float)x - mn).  While s is fp16-normal it is
//   within 2^-11 of scale_f, so the quotient stays below 2^b - 1 + 0.008 and
//   rounds to at most 2^b - 1 (no clamp).  q = dx * rcp(s), with the hardware
//   reciprocal (within 2^-22 relative over every fp16 value, checked by
//   kvq_testing_check_arithmetic), lies within 3
//   ulp of the IEEE quotient (so within 6e-6), so rint can only differ where q is
//   within 1e-5 of a half-integer; there, and for a subnormal s, the lane
//   recomputes its codes with the IEEE divide and the clamp.  rint itself is
//   the round-to-nearest-even fp32 addition of 1.5 * 2^23, which leaves the
//   integer in the low mantissa bits (0 <= q < 2^22), and each code is added in
//   at its bit offset with one shift-add (the constant mantissa bits of the
//   eight sums are subtracted once at the end, modulo 2^32).
// Returns the lane's 8 codes packed little-endian (8 * b bits) and the group's
// {scale, min} half2 bits.  All 32 lanes of the warp must call it (the shuffles
// use the full mask); `active` lanes only matter for the result, inactive lanes
// pass any finite values.
//
// hybrid: the group also gets the symmetric candidate (H1 of the header) and
// keeps it when it can be stored and its squared error (H2) is strictly below
// the asymmetric one's (H3, InnerQ page section 2.2); *asym_bit = 1 for the
// asymmetric result, 0 for the symmetric one.

// H2 over a quad: lane q sums e_j^2 over its values j = 8q .. 8q+7 in order,
// then (S_0 + S_1) + (S_2 + S_3) by two shuffle-xor steps (every lane of the
// quad ends with the same value).  Every operation is rounded on its own.
template <int BITS>
__device__ __forceinline__ float lane_sq_error(const float (&x)[8], uint32_t packed, float sc,
                                               float mn) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float xh = __fadd_rn(mn, __fmul_rn((float)((packed >> (BITS * j)) & kMask), sc));
    const float e = __fsub_rn(x[j], xh);
    acc = __fadd_rn(acc, __fmul_rn(e, e));
  }
  return acc;
}
template <int BITS>
__device__ __forceinline__ float quad_sq_error(const float (&x)[8], uint32_t packed, float sc,
                                               float mn) {
  float acc = lane_sq_error<BITS>(x, packed, sc, mn);
  acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
  acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
  return acc;
}

// Packed fp32 pairs (low element first) and their element-wise IEEE
// round-to-nearest-even add, subtract and multiply.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint32_t lo_bits(uint64_t v) { return (uint32_t)v; }
__device__ __forceinline__ uint32_t hi_bits(uint64_t v) { return (uint32_t)(v >> 32); }
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// d / K rounded to nearest even, for the divisors of the quantizer (K = 2^b - 1:
// 15, 7, 3) and d in its domain (0, or a difference of two fp16 values: 2^-24
// .. 131008).  Markstein's correction of the product by the reciprocal: with
// c = RN(1/K), q0 = RN(d c) and the exact residual r = d - q0 K (one fused
// multiply-add), RN(q0 + r c) is the correctly rounded quotient.  Checked
// against the IEEE divide for every d of that domain and each K (the
// library's kvq_testing_check_arithmetic).
template <int K>
__device__ __forceinline__ float div_by_const(float d) {
  if (K == 1) return d;
  constexpr float c = 1.0f / (float)K;
  const float q0 = __fmul_rn(d, c);
  const float r = __fmaf_rn(-q0, (float)K, d);
  return __fmaf_rn(r, c, q0);
}

// The hardware's approximate reciprocal (within about 1 ulp; the quantizer's
// near-tie window absorbs it).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// (float)h - f with one rounding: the fp16 operand converts exactly.
__device__ __forceinline__ float sub_f16_f32(unsigned short h, float f) {
  float d;
  asm("sub.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(h), "f"(f));
  return d;
}

// Q1 over the lane's 8 values: (min, -max) as one half2.
__device__ __forceinline__ __half2 lane_min_negmax(const uint4& raw) {
  const __half2* hv = reinterpret_cast<const __half2*>(&raw);
  const __half2 lo = __hmin2(__hmin2(hv[0], hv[1]), __hmin2(hv[2], hv[3]));
  const __half2 nhi = __hmin2(__hmin2(__hneg2(hv[0]), __hneg2(hv[1])),
                              __hmin2(__hneg2(hv[2]), __hneg2(hv[3])));
  return __halves2half2(__hmin(__low2half(lo), __high2half(lo)),
                        __hmin(__low2half(nhi), __high2half(nhi)));
}
// (min, -max) over the `lanes` lanes of a group (shuffle-xor; full mask).
template <int LANES>
__device__ __forceinline__ __half2 group_min_negmax(__half2 mm) {
#pragma unroll
  for (int o = 1; o < LANES; o <<= 1) {
    const uint32_t other = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<const uint32_t*>(&mm), o);
    mm = __hmin2(mm, *reinterpret_cast<const __half2*>(&other));
  }
  return mm;
}

// Q2 and the stored params: scale = RN((mx - mn) / (2^b - 1)) in fp32, both
// rounded to fp16; s = the fp16 scale as a float and r its reciprocal.
template <int BITS>
struct GroupScale {
  __half scale_h, min_h;
  float s, r;
  __device__ __forceinline__ GroupScale(float mn, float mx) {
    constexpr int kQmax = (1 << BITS) - 1;
    scale_h = __float2half_rn(div_by_const<kQmax>(__fsub_rn(mx, mn)));
    min_h = __float2half_rn(__fadd_rn(mn, 0.0f));
    s = __half2float(scale_h);
    r = s != 0.0f ? rcp_approx(s) : 0.0f;
  }
  __device__ __forceinline__ uint32_t params() const {
    return (uint32_t)__half_as_ushort(scale_h) | ((uint32_t)__half_as_ushort(min_h) << 16);
  }
};

// Q3 for 8 values of a group (raw), packed little-endian in 8 * b bits.  The
// pairs of values go through packed fp32x2 instructions (each element rounded
// as its scalar operation would be).  No clamp is needed while s is
// fp16-normal: s is within 2^-11 of the fp32 scale, so q <= (2^b - 1)(1 +
// 2^-11 + 2^-23) rounds to at most 2^b - 1.  A quotient within 1e-5 of a
// half-integer, or a subnormal s, sends these 8 values to the IEEE divide and
// the clamp.
template <int BITS>
__device__ __forceinline__ uint32_t codes8(const uint4& raw, float mn, const GroupScale<BITS>& gs) {
  constexpr int kQmax = (1 << BITS) - 1;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  constexpr uint32_t kMagicBits = 0x4B400000u;
  uint32_t magic_sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) magic_sum += kMagicBits << (BITS * j);
  const unsigned short* xs = reinterpret_cast<const unsigned short*>(&raw);
  const float s = gs.s;
  const uint64_t r2 = pack_f32x2(gs.r, gs.r);
  const uint64_t m2 = pack_f32x2(kMagic, kMagic);
  float dx[8];
  uint32_t acc = 0;
  bool near_tie = s != 0.0f && s < 6.103515625e-05f;  // subnormal fp16 scale (< 2^-14)
#pragma unroll
  for (int jp = 0; jp < 4; ++jp) {
    dx[2 * jp] = sub_f16_f32(xs[2 * jp], mn);
    dx[2 * jp + 1] = sub_f16_f32(xs[2 * jp + 1], mn);
    const uint64_t q2 = mul_f32x2(pack_f32x2(dx[2 * jp], dx[2 * jp + 1]), r2);
    const uint64_t t2 = add_f32x2(q2, m2);
    const uint64_t h2 = sub_f32x2(q2, sub_f32x2(t2, m2));  // q - rint(q)
    acc += lo_bits(t2) << (BITS * 2 * jp);
    acc += hi_bits(t2) << (BITS * (2 * jp + 1));
    near_tie |= fabsf(__uint_as_float(lo_bits(h2))) > 0.49999f;
    near_tie |= fabsf(__uint_as_float(hi_bits(h2))) > 0.49999f;
  }
  uint32_t packed = acc - magic_sum;
  if (near_tie) {
    packed = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = s != 0.0f ? min(max(__float2int_rn(__fdiv_rn(dx[j], s)), 0), kQmax) : 0;
      packed |= (uint32_t)c << (BITS * j);
    }
  }
  return packed;
}

__device__ __forceinline__ void unpack8_f16(const uint4& v, float (&x)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// H1, the symmetric candidate: scale = absmax / (2^(b-1) - 1), codes t +
// 2^(b-1), min = -2^(b-1) * scale (both fp16); storable unless that min
// overflows fp16.
template <int BITS>
struct SymScale {
  __half ssh, smh;
  float ss, rs;
  bool storable;
  __device__ __forceinline__ SymScale(float mn, float mx) {
    constexpr int kHalf = 1 << (BITS - 1);
    constexpr int kQs = kHalf - 1;
    const float amax = fmaxf(fabsf(mn), fabsf(mx));
    ssh = __float2half_rn(__fdiv_rn(amax, (float)kQs));
    ss = __half2float(ssh);
    smh = __float2half_rn(__fadd_rn(__fmul_rn(-(float)kHalf, ss), 0.0f));
    storable = (__half_as_ushort(smh) & 0x7c00u) != 0x7c00u;
    rs = ss != 0.0f ? __frcp_rn(ss) : 0.0f;
  }
  __device__ __forceinline__ uint32_t params() const {
    return (uint32_t)__half_as_ushort(ssh) | ((uint32_t)__half_as_ushort(smh) << 16);
  }
};

// Symmetric codes of 8 values: x / ss through the reciprocal, the IEEE divide
// near rounding boundaries (|x / ss| <= 2^(b-1), so the same 3-ulp argument as
// for the asymmetric codes holds), clamped to +-(2^(b-1) - 1).
template <int BITS>
__device__ __forceinline__ uint32_t sym_codes8(const float (&x)[8], const SymScale<BITS>& ys) {
  constexpr int kHalf = 1 << (BITS - 1);
  constexpr int kQs = kHalf - 1;
  uint32_t sp = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int t = 0;
    if (ys.ss != 0.0f) {
      float qf = __fmul_rn(x[j], ys.rs);
      if (fabsf(qf - floorf(qf) - 0.5f) < 1e-5f) qf = __fdiv_rn(x[j], ys.ss);
      t = __float2int_rn(qf);
      t = min(max(t, -kQs), kQs);
    }
    sp |= (uint32_t)(t + kHalf) << (BITS * j);
  }
  return sp;
}

template <int BITS>
__device__ __forceinline__ uint32_t quantize_quad(const uint4& raw, uint32_t& params_out,
                                                  bool hybrid = false, uint32_t* asym_bit = nullptr) {
  // Q1: (min, -max) of the lane's values, then of the quad
  const __half2 mm = group_min_negmax<4>(lane_min_negmax(raw));
  const float mn = __low2float(mm);
  const float mx = -__high2float(mm);
  const GroupScale<BITS> gs(mn, mx);
  const __half scale_h = gs.scale_h, min_h = gs.min_h;
  const float s = gs.s;
  uint32_t packed = codes8<BITS>(raw, mn, gs);
  params_out = (uint32_t)__half_as_ushort(scale_h) | ((uint32_t)__half_as_ushort(min_h) << 16);
  if (hybrid) {
    float x[8];
    unpack8_f16(raw, x);
    const SymScale<BITS> ys(mn, mx);
    const uint32_t sp = sym_codes8<BITS>(x, ys);
    // H2, H3
    const float ea = quad_sq_error<BITS>(x, packed, s, __half2float(min_h));
    const float es = quad_sq_error<BITS>(x, sp, ys.ss, __half2float(ys.smh));
    const bool sym = ys.storable && es < ea;
    if (sym) {
      packed = sp;
      params_out = ys.params();
    }
    if (asym_bit) *asym_bit = sym ? 0u : 1u;
  } else if (asym_bit) {
    *asym_bit = 1u;
  }
  return packed;
}

// One lane quantizes a whole group (its 32 values in raw[0..3]): the same
// operations as quantize_quad, with the error sums of the hybrid rule taken
// in the same order (8 values at a time, then (S0 + S1) + (S2 + S3)).  codes[k]
// holds values 8k .. 8k+7 packed little-endian (8 * b bits).
template <int BITS, bool HYB>
__device__ __forceinline__ void quantize_group32(const uint4 (&raw)[4], uint32_t (&codes)[4],
                                                 uint32_t& params_out, uint32_t& asym_bit) {
  const __half2 mm = __hmin2(__hmin2(lane_min_negmax(raw[0]), lane_min_negmax(raw[1])),
                             __hmin2(lane_min_negmax(raw[2]), lane_min_negmax(raw[3])));
  const float mn = __low2float(mm);
  const float mx = -__high2float(mm);
  const GroupScale<BITS> gs(mn, mx);
#pragma unroll
  for (int k = 0; k < 4; ++k) codes[k] = codes8<BITS>(raw[k], mn, gs);
  params_out = gs.params();
  asym_bit = 1u;
  if constexpr (HYB) {
    const SymScale<BITS> ys(mn, mx);
    const float amin = __half2float(gs.min_h), smin = __half2float(ys.smh);
    uint32_t sp[4];
    float ea[4], es[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x[8];
      unpack8_f16(raw[k], x);
      sp[k] = sym_codes8<BITS>(x, ys);
      ea[k] = lane_sq_error<BITS>(x, codes[k], gs.s, amin);
      es[k] = lane_sq_error<BITS>(x, sp[k], ys.ss, smin);
    }
    const float eat = __fadd_rn(__fadd_rn(ea[0], ea[1]), __fadd_rn(ea[2], ea[3]));
    const float est = __fadd_rn(__fadd_rn(es[0], es[1]), __fadd_rn(es[2], es[3]));
    if (ys.storable && est < eat) {
#pragma unroll
      for (int k = 0; k < 4; ++k) codes[k] = sp[k];
      params_out = ys.params();
      asym_bit = 0u;
    }
  }
}

// Store a group's 32 codes at its first byte `grp` (4 * BITS bytes; lane q of
// the quad holds codes 8q .. 8q+7 packed little-endian in 8 * BITS bits).  INT4
// and INT2: one 32- or 16-bit store per lane.  3-bit: the four 24-bit pieces
// are spliced into three 32-bit words, written by lanes 0-2.  All 32 lanes must
// call it; only `active` lanes store.
template <int BITS>
__device__ __forceinline__ void store_group_codes(uint8_t* grp, uint32_t packed, int quad,
                                                  bool active) {
  if (BITS == 3) {
    const uint32_t next = __shfl_down_sync(0xffffffffu, packed, 1);
    if (active && quad < 3)
      reinterpret_cast<uint32_t*>(grp)[quad] = (packed >> (8 * quad)) | (next << (24 - 8 * quad));
  } else if (BITS == 4) {
    if (active) reinterpret_cast<uint32_t*>(grp)[quad] = packed;
  } else {
    if (active) reinterpret_cast<uint16_t*>(grp)[quad] = (uint16_t)packed;
  }
}

// The mode byte of a token row from a ballot of (quad lane 0 && asymmetric):
// groups k0 .. k0 + ng - 1 of the warp sit at lanes 4k; bit g of the result is
// group k0 + g's.
__device__ __forceinline__ uint8_t mode_byte(uint32_t ballot, int k0, int ng) {
  uint32_t m = 0;
  for (int g = 0; g < ng; ++g) m |= ((ballot >> (4 * (k0 + g))) & 1u) << g;
  return (uint8_t)m;
}


// -------------------------------------------------------- decode planning ---

// Work split of one decode call.  Each (sequence, KV head, query block) is cut
// into `splits` pieces of roughly equal byte cost; partials (o, m, l) go to the
// workspace and the last split to finish merges them by log-sum-exp.
struct DecodePlan {
  int kernel;   // 0 = generic CUDA-core path, 1 = tensor-core path
  int gq;       // query heads per KV head
  int qb;       // query heads handled by one CTA (power of two, <= 8)
  int nqb;      // query blocks per KV head = ceil(gq / qb)
  int splits;   // S (all splits)
  int splits_packed;  // tensor-core kernel: the first splits_packed take packed tokens
  int threads;  // threads per CTA of the split kernel
  int cps;      // tensor-core kernel: resident CTAs per SM of the variant (3 or 4)
  int fold;     // tensor-core kernel: no fp16 splits; the last packed split takes those rows
  int tile;     // tensor-core kernel: tokens per pipeline stage (128 or 192)
  // Workspace layout.  The tickets sit at fixed offsets (they depend only on the
  // cache shape and head count), so a workspace shared by calls with different
  // split counts never has a partial land on a ticket.
  size_t ws_cnt_off;   // 0: per-unit arrival tickets [B][Hkv][nqb] (zero between calls)
  size_t ws_seq_off;   // per-sequence tickets [B] of the fused step (zero between calls)
  // tensor-core kernel, zero between calls: per unit and query the reference
  // max (float bits + 1, 0 = unset), a fallback flag per unit, and the fp32
  // accumulators of o [qb][d] and l [qb]
  size_t ws_ref_off;   // uint32 [units][qb]
  size_t ws_flag_off;  // uint32 [units]
  size_t ws_oacc_off;  // float [units][qb][d]
  size_t ws_lacc_off;  // float [units][qb]
  size_t ws_ml_off;    // {m, l} partials
  size_t ws_part_off;  // o partials
  size_t ws_total;     // bytes of the whole workspace
};

// step: plan for kvq_decode_step (the tensor-core kernel then always has a
// residual split per KV head, which takes the appended token).
DecodePlan plan_decode(const kvq_cache_desc& D, int num_q_heads, int sm_count, bool step = false);
int device_sm_count();
// kvq_decode_attention_noalloc: the next call on the current device clears the
// static array's counters first (called when a wait ran out).
void noalloc_forget_layout();
// kvq_testing_wait_fault: the bounded-wait limit in microseconds the decode
// calls use to make one wait run out (0: off, normal behaviour).
void set_testing_wait_fault_us(uint32_t us);
uint32_t testing_wait_fault_us();

// ------------------------------------------------------------- launchers ---

// k, vv: element (b, h, t, j) at base + b * strides[0] + h * strides[1] +
// t * strides[2] + j.
cudaError_t launch_quantize_pack(const Dims& s, const kvq_cache_view& v, const __half* k,
                                 const __half* vv, const int32_t* seq_lens, int Lmax,
                                 const int64_t strides[3], cudaStream_t st);
cudaError_t launch_append(const Dims& s, const kvq_cache_view& v, const __half* k_new,
                          const __half* v_new, cudaStream_t st);
// k_new/v_new non-null: the fused step (append, then attend).  out is fp16, or
// fp32 with KVQ_OUT_F32 in flags.
cudaError_t launch_decode(const Dims& s, const DecodePlan& p, const kvq_cache_view& v,
                          const __half* q, int Hq, void* out, void* workspace, cudaStream_t st,
                          const __half* k_new, const __half* v_new, uint32_t flags);

}  // namespace kvq
