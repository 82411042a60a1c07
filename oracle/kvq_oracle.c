/*
 * kvq_oracle.c -- plain, slow CPU oracle for the low-bit KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and the passage each step follows:
 *   Quantize (Q1-Q4): asymmetric uniform quantization of one group of 32 fp16
 *     values, scale = (max - min) / (2^b - 1), code = round((x - min) / scale)
 *     ("Tensor Core accelerated low-bit KV cache decoding" page, section 2.1),
 *     groups of 32 along head_dim (InnerQ page, section 2.1).
 *     Readings of points the pages leave open: fp32 arithmetic with an IEEE
 *     divide; the stored fp16 scale is the one that quantizes; round half to
 *     even; a zero scale gives all-zero codes; a -0 minimum is stored as +0.
 *   Pack (Q5): codes as a little-endian bit string, 32 consecutive head_dim
 *     values per group (InnerQ page, section 3.2); params as half2 {scale, min}.
 *     Bit widths 2, 4 and 3 (eight 3-bit codes per 24 bits, TurboQuant page,
 *     section 3.1, on the same asymmetric rule).
 *   Hybrid mode (H1-H3, optional): per group a symmetric candidate beside the
 *     asymmetric one, the smaller squared error wins and a 1-bit mask records
 *     the choice (InnerQ page, section 2.2).  Readings of points the page leaves
 *     open: symmetric = absmax / (2^(b-1) - 1) with codes in +-(2^(b-1) - 1),
 *     stored offset by 2^(b-1) with min = -2^(b-1) * scale (so both modes
 *     dequantize as min + code * scale); the error is the sum of squared fp32
 *     reconstruction errors in a fixed order (below), which decides an integer
 *     and so is taken in the kernel's precision; a tie keeps the asymmetric
 *     candidate; a symmetric min that is not a finite fp16 rules it out.
 *   Residual split (Q6): the last min(Nr, L) tokens stay fp16 (BitDecoding page,
 *     section 2.2); with an attention-sink window the first min(sink, L) tokens
 *     stay fp16 too, fixed after the prefill (InnerQ page, section 2.3).
 *   Append (Q7): sliding recent window, the oldest token is quantized when the
 *     window is full (InnerQ page, section 2.3).
 *   Decode (D1-D4): dequantize min + code * scale (InnerQ page, section 3.1),
 *     then softmax(q K^T / sqrt(d)) V in double precision, two passes over the
 *     scores (max, then exp-sum), query head hq reading KV head hq / gq
 *     (BitDecoding page, section 2.3).
 *
 * The fp16 <-> fp32 conversions below are written from the IEEE 754 binary16
 * definition (1 sign, 5 exponent, 10 fraction bits, bias 15, subnormals, round to
 * nearest even).
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fno-fast-math -shared -fPIC -lm.
 * The fp32 steps rely on float arithmetic being evaluated in float (SSE on x86-64,
 * plain on aarch64) without contraction into fused multiply-adds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- fp16 ---- */

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary16 -> double, exact. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* binary16 -> float, exact (every binary16 value is a float). */
float oracle_f16_to_f32(uint16_t h) { return (float)oracle_f16_to_f64(h); }

/* float -> binary16, round to nearest, ties to even, subnormals kept, overflow
 * to infinity, NaN kept quiet. */
uint16_t oracle_f32_to_f16(float f) {
  uint32_t u = f32_bits(f);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  int32_t e = (int32_t)((u >> 23) & 0xff);
  uint32_t m = u & 0x7fffffu;
  if (e == 0xff) return (uint16_t)(sign | 0x7c00u | (m ? 0x200u : 0u));
  if (e == 0 && m == 0) return sign;
  /* Value = mant * 2^exp2 with mant an integer (24 significant bits for normals). */
  uint32_t mant;
  int32_t exp2;
  if (e == 0) {
    mant = m;
    exp2 = -149;
  } else {
    mant = m | 0x800000u;
    exp2 = e - 150;
  }
  /* binary16 has quantum 2^-24 for |v| < 2^-14 and 2^(E-10) in binade [2^E, 2^(E+1)).
   * Find the binade of the value: value in [2^E, 2^(E+1)) with E = exponent of mant. */
  int32_t top = 31;
  while (!((mant >> top) & 1u)) top--;
  int32_t E = exp2 + top;
  int32_t q = (E < -14) ? -24 : E - 10; /* log2 of the binary16 quantum there */
  /* Round mant * 2^exp2 to a multiple of 2^q. */
  int32_t shift = q - exp2;
  uint64_t n; /* the result as a multiple of 2^q */
  if (shift <= 0) {
    n = (uint64_t)mant << (-shift);
  } else if (shift >= 40) {
    n = 0; /* far below half a quantum */
  } else {
    uint64_t mm = mant;
    uint64_t whole = mm >> shift;
    uint64_t rem = mm & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (whole & 1ull))) whole++;
    n = whole;
  }
  /* n * 2^q: re-encode. */
  if (n == 0) return sign;
  if (q == -24 && n < 1024) return (uint16_t)(sign | n); /* subnormal */
  /* normal: n in [1024, 2048] (2048 after rounding up means next binade) */
  int32_t ee = q + 10; /* exponent of 2^ee for n == 1024 */
  while (n >= 2048) {
    n >>= 1;
    ee++;
  }
  int32_t biased = ee + 15;
  if (biased >= 31) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | ((uint32_t)biased << 10) | (uint32_t)(n - 1024));
}

/* Vectorised helpers for the tests. */
void oracle_f32_to_f16_array(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f16_to_f64_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(in[i]);
}

/* ------------------------------------------------------------ quantize ---- */

/* Q1-Q4 on one group of 32 fp16 values.  codes[j] in [0, 2^bits - 1]. */
void oracle_quantize_group(const uint16_t* x, int bits, uint8_t* codes, uint16_t* scale_h,
                           uint16_t* min_h) {
  const int G = 32;
  const int qmax = (1 << bits) - 1;
  /* Q1: exact min and max of the fp16 values, compared as numbers. */
  float mn = oracle_f16_to_f32(x[0]);
  float mx = mn;
  for (int j = 1; j < G; ++j) {
    float v = oracle_f16_to_f32(x[j]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  /* Q2: fp32 subtract, then fp32 divide by 2^b - 1. */
  volatile float range = mx - mn;
  volatile float scale_f = range / (float)qmax;
  /* Q3: the stored scale and min. */
  *scale_h = oracle_f32_to_f16(scale_f);
  *min_h = oracle_f32_to_f16(mn + 0.0f);
  /* Q4: the codes use the stored scale. */
  float s = oracle_f16_to_f32(*scale_h);
  for (int j = 0; j < G; ++j) {
    if (s == 0.0f) {
      codes[j] = 0;
      continue;
    }
    volatile float diff = oracle_f16_to_f32(x[j]) - mn;
    volatile float ratio = diff / s;
    float r = rintf(ratio); /* default rounding mode: to nearest, ties to even */
    if (r < 0.0f) r = 0.0f;
    if (r > (float)qmax) r = (float)qmax;
    codes[j] = (uint8_t)r;
  }
}

/* H1: the symmetric candidate of one group.  a = max |x_j| (exact); scale =
 * fp16(a / (2^(b-1) - 1)) (fp32 IEEE divide); s = the stored scale; t_j =
 * clamp(rint(x_j / s), -(2^(b-1) - 1), 2^(b-1) - 1) (fp32 IEEE divide, ties to
 * even; 0 when s == 0); stored code t_j + 2^(b-1); stored min fp16(-2^(b-1) * s
 * + 0), exact when finite.  Returns 0 when that min overflows fp16 (the
 * candidate cannot be stored), else 1. */
int oracle_quantize_group_sym(const uint16_t* x, int bits, uint8_t* codes, uint16_t* scale_h,
                              uint16_t* min_h) {
  const int G = 32;
  const int half = 1 << (bits - 1);
  const int qs = half - 1;
  float a = 0.0f;
  for (int j = 0; j < G; ++j) {
    float v = fabsf(oracle_f16_to_f32(x[j]));
    if (v > a) a = v;
  }
  volatile float scale_f = a / (float)qs;
  *scale_h = oracle_f32_to_f16(scale_f);
  float s = oracle_f16_to_f32(*scale_h);
  volatile float m = -(float)half * s;
  *min_h = oracle_f32_to_f16(m + 0.0f);
  for (int j = 0; j < G; ++j) {
    float t = 0.0f;
    if (s != 0.0f) {
      volatile float ratio = oracle_f16_to_f32(x[j]) / s;
      t = rintf(ratio);
      if (t < (float)-qs) t = (float)-qs;
      if (t > (float)qs) t = (float)qs;
    }
    codes[j] = (uint8_t)((int)t + half);
  }
  return ((*min_h & 0x7c00u) != 0x7c00u) ? 1 : 0;
}

/* H2: squared reconstruction error of a group's candidate, fp32, in this order:
 * x^_j = (float)min + (float)code_j * (float)scale (multiply, then add, each
 * rounded), e_j = x_j - x^_j, and per quarter q (values 8q .. 8q+7) the running
 * sum S_q = ((e_8q^2 + e_8q+1^2) + ...) in index order; the result is
 * (S_0 + S_1) + (S_2 + S_3). */
float oracle_group_sq_error(const uint16_t* x, const uint8_t* codes, uint16_t scale_h,
                            uint16_t min_h) {
  const float sc = oracle_f16_to_f32(scale_h), mn = oracle_f16_to_f32(min_h);
  volatile float part[4];
  for (int q = 0; q < 4; ++q) {
    volatile float acc = 0.0f;
    for (int j = 8 * q; j < 8 * q + 8; ++j) {
      volatile float prod = (float)codes[j] * sc;
      volatile float xh = mn + prod;
      volatile float e = oracle_f16_to_f32(x[j]) - xh;
      volatile float e2 = e * e;
      acc = acc + e2;
    }
    part[q] = acc;
  }
  volatile float lo = part[0] + part[1];
  volatile float hi = part[2] + part[3];
  return lo + hi;
}

/* H3: hybrid quantization of one group: the symmetric candidate when it can be
 * stored and its error (H2) is strictly below the asymmetric one's, else the
 * asymmetric candidate (Q1-Q4).  Returns the mode bit: 1 asymmetric, 0 symmetric. */
int oracle_quantize_group_hybrid(const uint16_t* x, int bits, uint8_t* codes, uint16_t* scale_h,
                                 uint16_t* min_h) {
  uint8_t cs[32];
  uint16_t ss, ms;
  oracle_quantize_group(x, bits, codes, scale_h, min_h);
  if (!oracle_quantize_group_sym(x, bits, cs, &ss, &ms)) return 1;
  float ea = oracle_group_sq_error(x, codes, *scale_h, *min_h);
  float es = oracle_group_sq_error(x, cs, ss, ms);
  if (!(es < ea)) return 1;
  memcpy(codes, cs, sizeof(cs));
  *scale_h = ss;
  *min_h = ms;
  return 0;
}

/* Q5: pack d codes of one token row; returns bytes written (d * bits / 8).
 * Code e occupies bits [e*bits, e*bits + bits) of the row's little-endian bit
 * string; a 3-bit code can straddle two bytes. */
int oracle_pack_row(const uint8_t* codes, int d, int bits, uint8_t* out) {
  int nbytes = d * bits / 8;
  memset(out, 0, (size_t)nbytes);
  for (int e = 0; e < d; ++e) {
    int bit = e * bits;
    unsigned v = (unsigned)codes[e] << (bit % 8); /* up to 16 bits wide */
    out[bit / 8] |= (uint8_t)(v & 0xffu);
    if (bit % 8 + bits > 8) out[bit / 8 + 1] |= (uint8_t)(v >> 8);
  }
  return nbytes;
}

/* Inverse of Q5, for the tests. */
void oracle_unpack_row(const uint8_t* packed, int d, int bits, uint8_t* codes) {
  int mask = (1 << bits) - 1;
  for (int e = 0; e < d; ++e) {
    int bit = e * bits;
    unsigned v = packed[bit / 8];
    if (bit % 8 + bits > 8) v |= (unsigned)packed[bit / 8 + 1] << 8;
    codes[e] = (uint8_t)((v >> (bit % 8)) & (unsigned)mask);
  }
}

/* Quantize and pack one token of one head: src = d fp16 values.  With hybrid,
 * each group takes H3 and *mode_byte gets bit g = group g's mode bit. */
static void quantize_token(const uint16_t* src, int d, int bits, int hybrid, uint8_t* code_row,
                           uint32_t* param_row, uint8_t* mode_byte) {
  uint8_t codes[256];
  uint8_t mode = 0;
  for (int g = 0; g < d / 32; ++g) {
    uint16_t sh, mh;
    if (hybrid)
      mode |= (uint8_t)(oracle_quantize_group_hybrid(src + 32 * g, bits, codes + 32 * g, &sh, &mh) << g);
    else
      oracle_quantize_group(src + 32 * g, bits, codes + 32 * g, &sh, &mh);
    param_row[g] = (uint32_t)sh | ((uint32_t)mh << 16);
  }
  oracle_pack_row(codes, d, bits, code_row);
  if (hybrid) *mode_byte = mode;
}

/* Shapes of one cache, mirroring the library's description. */
typedef struct {
  int32_t batch, num_kv_heads, head_dim, bits, group, capacity, residual, sink, hybrid;
} oracle_desc;

static int desc_ok(const oracle_desc* D) {
  return D && D->batch >= 1 && D->num_kv_heads >= 1 && D->head_dim >= 32 && D->head_dim <= 256 &&
         D->head_dim % 32 == 0 && D->bits >= 2 && D->bits <= 4 && D->group == 32 &&
         D->capacity >= 0 && D->residual >= 0 && D->residual <= 1024 && D->sink >= 0 &&
         D->sink <= 256 && (D->hybrid == 0 || D->hybrid == 1);
}

/* Q1-Q6 over a whole prefill for one of K or V.
 *   x         fp16 [B][Hkv][Lmax][d]
 *   codes     [B][Hkv][cap][d*b/8]; params [B][Hkv][cap][Ng]; res [B][Hkv][Nr][d];
 *   sink_rows [B][Hkv][sink][d] (may be NULL when sink == 0)
 *   modes     [B][Hkv][cap] mode bytes (H3; may be NULL unless hybrid)
 *   packed_len, res_len, res_head, sink_len  [B] outputs.
 * With an attention-sink window (InnerQ page, section 2.3), the first
 * min(sink, L) tokens are kept verbatim in sink_rows and the rest is split as
 * without one: the last min(Nr, rest) go to the residual, the others are packed.
 * Returns a bit set: 1 = a sequence passed the capacity, 8 = a bad length. */
int oracle_quantize_pack(const oracle_desc* D, const uint16_t* x, const int32_t* seq_lens,
                         int32_t Lmax, uint8_t* codes, uint32_t* params, uint16_t* res,
                         uint16_t* sink_rows, uint8_t* modes, int32_t* packed_len,
                         int32_t* res_len, int32_t* res_head, int32_t* sink_len) {
  if (!desc_ok(D)) return -1;
  const int d = D->head_dim, Ng = d / 32, rb = d * D->bits / 8, Nr = D->residual, S = D->sink;
  const int64_t cap = D->capacity;
  int err = 0;
  for (int b = 0; b < D->batch; ++b) {
    int32_t L = seq_lens[b];
    if (L < 0 || L > Lmax) {
      err |= 8;
      continue;
    }
    int32_t ns = L < S ? L : S;
    int32_t rest = L - ns;
    int32_t nres = rest < Nr ? rest : Nr;
    int32_t npk = rest - nres;
    if (npk > cap) {
      err |= 1;
      npk = (int32_t)cap;
    }
    for (int h = 0; h < D->num_kv_heads; ++h) {
      int64_t bh = (int64_t)b * D->num_kv_heads + h;
      const uint16_t* src = x + bh * Lmax * d;
      for (int32_t j = 0; j < ns; ++j)
        memcpy(sink_rows + (bh * S + j) * d, src + (int64_t)j * d, (size_t)d * sizeof(uint16_t));
      for (int32_t t = 0; t < npk; ++t)
        quantize_token(src + (int64_t)(ns + t) * d, d, D->bits, D->hybrid,
                       codes + (bh * cap + t) * rb, params + (bh * cap + t) * Ng,
                       modes ? modes + bh * cap + t : NULL);
      for (int32_t j = 0; j < nres; ++j)
        memcpy(res + (bh * Nr + j) * d, src + (int64_t)(L - nres + j) * d,
               (size_t)d * sizeof(uint16_t));
    }
    packed_len[b] = npk;
    res_len[b] = nres;
    res_head[b] = 0;
    sink_len[b] = ns;
  }
  return err;
}

/* Q7: append one token per sequence for one of K or V.
 *   xnew fp16 [B][Hkv][d].  The counters are read from packed_len/res_len/res_head
 *   and the updated values written to the *_out arrays (so K and V can share the
 *   same inputs).  Returns 1 if a sequence hit the capacity (left unchanged). */
int oracle_append(const oracle_desc* D, const uint16_t* xnew, uint8_t* codes, uint32_t* params,
                  uint16_t* res, uint8_t* modes, const int32_t* packed_len, const int32_t* res_len,
                  const int32_t* res_head, int32_t* packed_len_out, int32_t* res_len_out,
                  int32_t* res_head_out) {
  if (!desc_ok(D)) return -1;
  const int d = D->head_dim, Ng = d / 32, rb = d * D->bits / 8, Nr = D->residual;
  const int64_t cap = D->capacity;
  int err = 0;
  for (int b = 0; b < D->batch; ++b) {
    int32_t pl = packed_len[b], rl = res_len[b], rh = res_head[b];
    int full = (rl == Nr);
    if (full && pl >= cap) {
      err |= 1;
      packed_len_out[b] = pl;
      res_len_out[b] = rl;
      res_head_out[b] = rh;
      continue;
    }
    for (int h = 0; h < D->num_kv_heads; ++h) {
      int64_t bh = (int64_t)b * D->num_kv_heads + h;
      const uint16_t* src = xnew + bh * d;
      uint8_t* mode_byte = modes ? modes + bh * cap + pl : NULL;
      if (Nr == 0) {
        quantize_token(src, d, D->bits, D->hybrid, codes + (bh * cap + pl) * rb,
                       params + (bh * cap + pl) * Ng, mode_byte);
      } else if (full) {
        uint16_t* oldest = res + (bh * Nr + rh) * d;
        quantize_token(oldest, d, D->bits, D->hybrid, codes + (bh * cap + pl) * rb,
                       params + (bh * cap + pl) * Ng, mode_byte);
        memcpy(oldest, src, (size_t)d * sizeof(uint16_t));
      } else {
        memcpy(res + (bh * Nr + (rh + rl) % Nr) * d, src, (size_t)d * sizeof(uint16_t));
      }
    }
    if (Nr == 0) {
      packed_len_out[b] = pl + 1;
      res_len_out[b] = 0;
      res_head_out[b] = 0;
    } else if (full) {
      packed_len_out[b] = pl + 1;
      res_len_out[b] = rl;
      res_head_out[b] = (rh + 1) % Nr;
    } else {
      packed_len_out[b] = pl;
      res_len_out[b] = rl + 1;
      res_head_out[b] = rh;
    }
  }
  return err;
}

/* -------------------------------------------------------------- decode ---- */

/* D1: dequantize the packed tokens of one (sequence, KV head) into out [n][d]. */
static void dequant_rows(const uint8_t* code_rows, const uint32_t* param_rows, int64_t n, int d,
                         int bits, double* out) {
  const int rb = d * bits / 8, Ng = d / 32;
  uint8_t codes[256];
  for (int64_t t = 0; t < n; ++t) {
    oracle_unpack_row(code_rows + t * rb, d, bits, codes);
    for (int e = 0; e < d; ++e) {
      uint32_t p = param_rows[t * Ng + e / 32];
      double scale = oracle_f16_to_f64((uint16_t)(p & 0xffffu));
      double mn = oracle_f16_to_f64((uint16_t)(p >> 16));
      out[t * d + e] = mn + (double)codes[e] * scale;
    }
  }
}

/* Gather the keys or values of (b, h) as doubles: the sink rows (fp16), the
 * packed tokens (dequantized), then the residual ring in age order.  Returns
 * the token count; *rows is malloc'ed. */
static int64_t gather_kv(const oracle_desc* D, const uint8_t* codes, const uint32_t* params,
                         const uint16_t* res, const uint16_t* sink_rows, int32_t sl, int32_t pl,
                         int32_t rl, int32_t rh, int b, int h, double** rows) {
  const int d = D->head_dim, Ng = d / 32, rb = d * D->bits / 8, Nr = D->residual, S = D->sink;
  const int64_t cap = D->capacity;
  int64_t n = (int64_t)sl + pl + rl;
  double* x = (double*)malloc((size_t)(n > 0 ? n : 1) * d * sizeof(double));
  int64_t bh = (int64_t)b * D->num_kv_heads + h;
  for (int32_t j = 0; j < sl; ++j) {
    const uint16_t* src = sink_rows + (bh * S + j) * d;
    for (int e = 0; e < d; ++e) x[(int64_t)j * d + e] = oracle_f16_to_f64(src[e]);
  }
  dequant_rows(codes + bh * cap * rb, params + bh * cap * Ng, pl, d, D->bits, x + (int64_t)sl * d);
  for (int32_t j = 0; j < rl; ++j) {
    const uint16_t* src = res + (bh * Nr + (rh + j) % Nr) * d;
    for (int e = 0; e < d; ++e) x[((int64_t)sl + pl + j) * d + e] = oracle_f16_to_f64(src[e]);
  }
  *rows = x;
  return n;
}

/* D2-D4 for one query vector against n keys/values: out[d] in double. */
static void attend(const double* q, const double* K, const double* V, int64_t n, int d,
                   double* out) {
  double* s = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  double smax = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int e = 0; e < d; ++e) acc += q[e] * K[t * d + e];
    s[t] = acc * inv_sqrt_d;
    if (s[t] > smax) smax = s[t];
  }
  double denom = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    s[t] = exp(s[t] - smax);
    denom += s[t];
  }
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  for (int64_t t = 0; t < n; ++t)
    for (int e = 0; e < d; ++e) out[e] += s[t] * V[t * d + e];
  for (int e = 0; e < d; ++e) out[e] = n > 0 ? out[e] / denom : 0.0;
  free(s);
}

/* Decode for a list of (b, hq) pairs (pairs[2i], pairs[2i+1]); out [npairs][d] double.
 * q is fp16 [B][Hq][d].  A sequence with no tokens gives zeros. */
int oracle_decode_pairs(const oracle_desc* D, const uint8_t* k_codes, const uint32_t* k_params,
                        const uint16_t* k_res, const uint16_t* k_sink, const uint8_t* v_codes,
                        const uint32_t* v_params, const uint16_t* v_res, const uint16_t* v_sink,
                        const int32_t* packed_len, const int32_t* res_len,
                        const int32_t* res_head, const int32_t* sink_len, const uint16_t* q,
                        int32_t num_q_heads, const int32_t* pairs, int32_t npairs, double* out) {
  if (!desc_ok(D) || num_q_heads < 1 || num_q_heads % D->num_kv_heads) return -1;
  const int d = D->head_dim;
  const int gq = num_q_heads / D->num_kv_heads;
  int cached_b = -1, cached_h = -1;
  double *K = NULL, *V = NULL;
  int64_t n = 0;
  double qd[256];
  for (int32_t i = 0; i < npairs; ++i) {
    int b = pairs[2 * i], hq = pairs[2 * i + 1];
    if (b < 0 || b >= D->batch || hq < 0 || hq >= num_q_heads) return -1;
    int h = hq / gq;
    if (b != cached_b || h != cached_h) {
      free(K);
      free(V);
      n = gather_kv(D, k_codes, k_params, k_res, k_sink, sink_len[b], packed_len[b], res_len[b],
                    res_head[b], b, h, &K);
      gather_kv(D, v_codes, v_params, v_res, v_sink, sink_len[b], packed_len[b], res_len[b],
                res_head[b], b, h, &V);
      cached_b = b;
      cached_h = h;
    }
    for (int e = 0; e < d; ++e) qd[e] = oracle_f16_to_f64(q[((int64_t)b * num_q_heads + hq) * d + e]);
    attend(qd, K, V, n, d, out + (int64_t)i * d);
  }
  free(K);
  free(V);
  return 0;
}

/* Decode for every (b, hq): out [B][Hq][d] double. */
int oracle_decode(const oracle_desc* D, const uint8_t* k_codes, const uint32_t* k_params,
                  const uint16_t* k_res, const uint16_t* k_sink, const uint8_t* v_codes,
                  const uint32_t* v_params, const uint16_t* v_res, const uint16_t* v_sink,
                  const int32_t* packed_len, const int32_t* res_len, const int32_t* res_head,
                  const int32_t* sink_len, const uint16_t* q, int32_t num_q_heads, double* out) {
  if (!desc_ok(D) || num_q_heads < 1 || num_q_heads % D->num_kv_heads) return -1;
  int32_t np = D->batch * num_q_heads;
  int32_t* pairs = (int32_t*)malloc((size_t)np * 2 * sizeof(int32_t));
  for (int b = 0; b < D->batch; ++b)
    for (int hq = 0; hq < num_q_heads; ++hq) {
      pairs[2 * (b * num_q_heads + hq)] = b;
      pairs[2 * (b * num_q_heads + hq) + 1] = hq;
    }
  int rc = oracle_decode_pairs(D, k_codes, k_params, k_res, k_sink, v_codes, v_params, v_res,
                               v_sink, packed_len, res_len, res_head, sink_len, q, num_q_heads,
                               pairs, np, out);
  free(pairs);
  return rc;
}
