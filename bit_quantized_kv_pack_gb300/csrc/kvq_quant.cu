// kvq_quant.cu -- quantize/pack of a prefill and the decode-step append.
//
// Rule: asymmetric uniform quantization with scale = (max - min) / (2^b - 1) and
// code = round((x - min) / scale) ("Tensor Core accelerated low-bit KV cache
// decoding" page, section 2.1), over groups of 32 consecutive head_dim values
// (InnerQ page, section 2.1).  Kernel shape: per-thread min/max over its values,
// a shuffle-xor reduction inside the group, codes packed in registers and
// written straight out (BitDecoding page, section 3.1).  Residual split: the
// last min(Nr, L) tokens stay fp16 (BitDecoding page, section 2.2), and so do
// the first min(S, L) with an attention-sink window; append follows the sliding
// recent window and leaves the sink as the prefill set it (InnerQ page,
// section 2.3).
//
// Thread mapping.  The tokens of one (sequence, KV head) are contiguous rows of
// d fp16 values, so its groups are contiguous 64-byte pieces of memory, and so
// are their outputs (4*b code bytes, one 4-byte param).  A warp takes 8
// consecutive groups: lane l holds values 8*(l%4) .. +7 of group l/4, one
// 16-byte load.  Every store of the warp is contiguous (128 or 64 bytes of codes,
// 32 bytes of params).
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kPackThreads = 256;  // 8 warps
constexpr int kPackUnroll = 4;     // independent 16-byte loads in flight per thread
constexpr int kGroupsPerIter = kPackThreads / 4;
constexpr int kGroupsPerCta = kGroupsPerIter * kPackUnroll;

// Index 0 = K, 1 = V (blockIdx.z).
struct PackArgs {
  const __half* x[2];    // element (b, h, t, j) at x + b * sb + h * sh + t * st + j
  uint8_t* codes[2];     // [B][Hkv][cap][row_bytes]
  uint32_t* params[2];   // [B][Hkv][cap][Ng]
  __half* res[2];        // [B][Hkv][Nr][d]
  __half* sink[2];       // [B][Hkv][Ns][d]
  uint8_t* modes[2];     // [B][Hkv][cap] mode bytes (hybrid caches)
  RowMap rm;             // packed token -> row (contiguous or paged)
  const int32_t* seq_lens;
  int32_t* packed_len;
  int32_t* res_len;
  int32_t* res_head;
  int32_t* sink_len;
  uint32_t* err_word;
  int Hkv, d, Ng, row_bytes, cap, Nr, Ns, Lmax;
  int ng_shift;            // log2(Ng)
  int64_t sb, sh, st;      // element strides of the input: sequence, head, token
};

// Without hybrid groups the kernel fits 40 registers, so six CTAs (1536 threads)
// share an SM and keep more loads in flight; the hybrid rule needs more (4).
template <int BITS, bool HYB>
__global__ void __launch_bounds__(kPackThreads, HYB ? 4 : 6) quantize_pack_kernel(PackArgs a) {
  const int bh = blockIdx.y;
  const int which = blockIdx.z;
  const int b = bh / a.Hkv;
  const int L = a.seq_lens[b];
  const bool bad = (L < 0 || L > a.Lmax);
  // tokens [0, ns) -> sink, [ns, ns + npk) -> packed, the last nres -> window
  const int ns = bad ? 0 : min(L, a.Ns);
  const int nres = bad ? 0 : min(L - ns, a.Nr);
  const int npk_all = bad ? 0 : L - ns - nres;
  const int npk = min(npk_all, a.cap);

  if (which == 0 && blockIdx.x == 0 && (bh % a.Hkv) == 0 && threadIdx.x == 0) {
    a.packed_len[b] = npk;
    a.res_len[b] = nres;
    a.res_head[b] = 0;
    if (a.Ns > 0) a.sink_len[b] = ns;
    if (bad) set_error(a.err_word, KVQ_ERRBIT_BADLEN);
    if (npk_all > a.cap) set_error(a.err_word, KVQ_ERRBIT_CAPACITY);
  }
  if (bad) return;

  const int64_t groups_used = (int64_t)L * a.Ng;
  const int64_t g0 = (int64_t)blockIdx.x * kGroupsPerCta;
  if (g0 >= groups_used) return;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int quad = lane & 3;
  const int h = bh % a.Hkv;
  const __half* src = a.x[which] + (int64_t)b * a.sb + (int64_t)h * a.sh;

  // CTA-uniform fast path: every group of this CTA is packed into a contiguous
  // cache (the prefill's bulk).  Addresses are 32-bit offsets from the CTA's
  // first token, and no group needs classifying.
  const int64_t g_last = min(groups_used, g0 + kGroupsPerCta) - 1;
  const int t_lo = (int)(g0 >> a.ng_shift);
  if (!a.rm.paged && t_lo >= ns && (int)(g_last >> a.ng_shift) < ns + npk) {
    const __half* xs = src + (int64_t)t_lo * a.st;
    const int64_t row_lo = (int64_t)bh * a.cap + (t_lo - ns);
    uint8_t* cbase = a.codes[which] + row_lo * a.row_bytes;
    uint32_t* pbase = a.params[which] + row_lo * a.Ng;
    const int ng_used = (int)(g_last - g0) + 1;
    {
      // One lane per group, its 32 values in four 16-byte loads: the group's
      // min/max needs no shuffle and its scale and reciprocal are worked out
      // once per 32 values; the lane stores the group's codes at once (16
      // bytes INT4, 12 bytes INT3, 8 bytes INT2) and its params.  A warp's 32 groups are whole
      // token rows (Ng divides 32), so each row's mode byte comes from one ballot.
      const int gl = warp * 32 + lane;
      const bool act = gl < ng_used;
      if (!HYB && !act) return;  // (with hybrid groups every lane takes part in the ballot)
      const int tl = gl >> a.ng_shift, g = gl & (a.Ng - 1);
      uint4 raw[4];
      if (act) {
        const uint4* p = reinterpret_cast<const uint4*>(xs + (int64_t)tl * a.st) + g * (kGroup / 8);
#pragma unroll
        for (int k = 0; k < 4; ++k) raw[k] = __ldg(p + k);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) raw[k] = make_uint4(0, 0, 0, 0);
      }
      uint32_t c[4], prm, asym;
      quantize_group32<BITS, HYB>(raw, c, prm, asym);
      if constexpr (HYB) {
        const uint32_t modes = __ballot_sync(0xffffffffu, act && asym);
        if (act && g == 0) a.modes[which][row_lo + tl] = (uint8_t)((modes >> lane) & ((1u << a.Ng) - 1u));
      }
      if (act) {
        uint8_t* dst = cbase + (uint32_t)(tl * a.row_bytes + g * (4 * BITS));
        if (BITS == 4) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
        } else if (BITS == 3) {  // four 24-bit pieces spliced into three words
          uint32_t* d3 = reinterpret_cast<uint32_t*>(dst);
          d3[0] = c[0] | (c[1] << 24);
          d3[1] = (c[1] >> 8) | (c[2] << 16);
          d3[2] = (c[2] >> 16) | (c[3] << 8);
        } else {
          *reinterpret_cast<uint2*>(dst) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        }
        pbase[(uint32_t)gl] = prm;
      }
      return;
    }
  }

  uint4 raw[kPackUnroll];
  int64_t gi[kPackUnroll];
#pragma unroll
  for (int u = 0; u < kPackUnroll; ++u) {
    gi[u] = g0 + u * kGroupsPerIter + warp * 8 + (lane >> 2);
    raw[u] = make_uint4(0, 0, 0, 0);
    if (gi[u] < groups_used) {
      const int64_t t = gi[u] >> a.ng_shift, g = gi[u] & (a.Ng - 1);
      raw[u] = __ldg(reinterpret_cast<const uint4*>(src + t * a.st + g * kGroup + quad * 8));
    }
  }

#pragma unroll
  for (int u = 0; u < kPackUnroll; ++u) {
    const bool in_range = gi[u] < groups_used;
    const int t = in_range ? (int)(gi[u] >> a.ng_shift) : 0;
    const int g = in_range ? (int)(gi[u] & (a.Ng - 1)) : 0;
    uint32_t prm, asym = 1;
    const uint32_t packed = quantize_quad<BITS>(raw[u], prm, HYB, &asym);  // all lanes take part
    // the warp's 8 groups are whole token rows (Ng divides 8): each row's mode
    // byte comes from one ballot
    const uint32_t modes = HYB ? __ballot_sync(0xffffffffu, quad == 0 && asym) : 0u;
    const bool packs = in_range && t >= ns && t - ns < npk;
    const int64_t row = packs ? a.rm.row(b, h, t - ns) : -1;
    if (packs && row < 0 && quad == 0) set_error(a.err_word, KVQ_ERRBIT_BADPAGE);
    const bool to_pack = packs && row >= 0;
    store_group_codes<BITS>(to_pack ? a.codes[which] + row * a.row_bytes + g * (4 * BITS) : nullptr,
                            packed, quad, to_pack);
    if (!in_range) continue;
    if (t < ns) {
      __half* dst = a.sink[which] + ((int64_t)bh * a.Ns + t) * a.d + g * kGroup + quad * 8;
      *reinterpret_cast<uint4*>(dst) = raw[u];
    } else if (to_pack) {
      if (quad == 0) a.params[which][row * a.Ng + g] = prm;
      if (HYB && quad == 0 && g == 0) a.modes[which][row] = mode_byte(modes, lane >> 2, a.Ng);
    } else if (!packs && t - ns >= npk_all) {
      const int j = t - ns - npk_all;  // ring slot; res_head = 0 after a prefill
      __half* dst = a.res[which] + ((int64_t)bh * a.Nr + j) * a.d + g * kGroup + quad * 8;
      *reinterpret_cast<uint4*>(dst) = raw[u];
    }
    // tokens in [cap, npk_all) are dropped (capacity error raised above)
  }
}

// One CTA per sequence; warps take (KV head, K-or-V) items.
struct AppendArgs {
  const __half* k_new;  // [B][Hkv][d]
  const __half* v_new;
  uint8_t* codes[2];
  uint32_t* params[2];
  __half* res[2];
  uint8_t* modes[2];
  RowMap rm;
  int32_t* packed_len;
  int32_t* res_len;
  int32_t* res_head;
  uint32_t* err_word;
  int Hkv, d, Ng, row_bytes, cap, Nr;
};

template <int BITS, bool HYB>
__global__ void __launch_bounds__(1024) append_kernel(AppendArgs a) {
  // The decode of the same step may start launching now; it waits for this
  // grid to finish (griddepcontrol.wait) before it reads the cache.
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const bool active = lane * 8 < a.d;
  // the new tokens do not depend on the counters: start their loads first
  // items per warp whose new token is loaded up front (fewer for the hybrid
  // quantizer, which needs the registers)
  constexpr int kMaxItems = HYB ? 2 : 4;
  uint4 newv[kMaxItems];
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int item = warp + k * nwarps;
    newv[k] = make_uint4(0, 0, 0, 0);
    if (item < 2 * a.Hkv && active) {
      const int64_t bh = (int64_t)b * a.Hkv + (item >> 1);
      const __half* nsrc = ((item & 1) ? a.v_new : a.k_new) + bh * a.d;
      newv[k] = __ldg(reinterpret_cast<const uint4*>(nsrc + lane * 8));
    }
  }
  const int pl = a.packed_len[b];
  const int rl = a.res_len[b];
  const int rh = a.res_head[b];
  const bool pack_now = (a.Nr == 0) || (rl == a.Nr);
  if (pack_now && pl >= a.cap) {
    if (threadIdx.x == 0) set_error(a.err_word, KVQ_ERRBIT_CAPACITY);
    return;
  }
  const int slot_new = (a.Nr == 0) ? 0 : (pack_now ? rh : (rh + rl) % a.Nr);

  for (int k = 0;; ++k) {
    const int item = warp + k * nwarps;
    if (item >= 2 * a.Hkv) break;  // warp-uniform
    const int which = item & 1;
    const int h = item >> 1;
    const int64_t bh = (int64_t)b * a.Hkv + h;
    uint4 nv = make_uint4(0, 0, 0, 0);
    if (k < kMaxItems) {
#pragma unroll
      for (int kk = 0; kk < kMaxItems; ++kk)
        if (kk == k) nv = newv[kk];
    } else if (active) {  // more than four items per warp: load here
      const __half* nsrc = (which ? a.v_new : a.k_new) + bh * a.d;
      nv = __ldg(reinterpret_cast<const uint4*>(nsrc + lane * 8));
    }
    __half* const res_base = which ? a.res[1] : a.res[0];
    uint8_t* const codes_base = which ? a.codes[1] : a.codes[0];
    uint32_t* const params_base = which ? a.params[1] : a.params[0];
    __half* ring_row = (a.Nr > 0) ? res_base + (bh * a.Nr + slot_new) * a.d : nullptr;
    if (pack_now) {
      uint4 oldv = nv;
      if (a.Nr > 0 && active) oldv = *reinterpret_cast<const uint4*>(ring_row + lane * 8);
      uint32_t prm, asym = 1;
      const uint32_t packed = quantize_quad<BITS>(oldv, prm, HYB, &asym);
      if (HYB) {
        const uint32_t modes = __ballot_sync(0xffffffffu, (lane & 3) == 0 && asym);
        const int64_t mrow = a.rm.row(b, h, pl);
        if (lane == 0 && mrow >= 0) (which ? a.modes[1] : a.modes[0])[mrow] = mode_byte(modes, 0, a.Ng);
      }
      const int64_t row = a.rm.row(b, h, pl);  // warp-uniform
      if (row < 0 && lane == 0) set_error(a.err_word, KVQ_ERRBIT_BADPAGE);
      const int g = lane >> 2, quad = lane & 3;
      store_group_codes<BITS>(codes_base + (row < 0 ? 0 : row) * a.row_bytes + g * (4 * BITS), packed,
                              quad, active && row >= 0);
      if (active && row >= 0 && quad == 0) params_base[row * a.Ng + g] = prm;
    }
    if (a.Nr > 0 && active) *reinterpret_cast<uint4*>(ring_row + lane * 8) = nv;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.Nr == 0) {
      a.packed_len[b] = pl + 1;
    } else if (pack_now) {
      a.packed_len[b] = pl + 1;
      a.res_head[b] = (rh + 1) % a.Nr;
    } else {
      a.res_len[b] = rl + 1;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_pack(const Dims& s, const kvq_cache_view& v, const __half* k,
                                 const __half* vv, const int32_t* seq_lens, int Lmax,
                                 const int64_t strides[3], cudaStream_t st) {
  // With Lmax == 0 one CTA per (sequence, head) still runs to write the counters.
  const int64_t groups = (int64_t)(Lmax > 0 ? Lmax : 1) * s.Ng;
  dim3 grid((unsigned)((groups + kGroupsPerCta - 1) / kGroupsPerCta), (unsigned)(s.B * s.Hkv), 2);
  PackArgs a;
  a.x[0] = k;
  a.x[1] = vv;
  a.codes[0] = v.k_codes;
  a.codes[1] = v.v_codes;
  a.params[0] = v.k_params;
  a.params[1] = v.v_params;
  a.res[0] = reinterpret_cast<__half*>(v.k_res);
  a.res[1] = reinterpret_cast<__half*>(v.v_res);
  a.sink[0] = reinterpret_cast<__half*>(v.k_sink);
  a.sink[1] = reinterpret_cast<__half*>(v.v_sink);
  a.modes[0] = v.k_mode;
  a.modes[1] = v.v_mode;
  a.rm = row_map(s, v.block_table);
  a.seq_lens = seq_lens;
  a.packed_len = v.packed_len;
  a.res_len = v.res_len;
  a.res_head = v.res_head;
  a.sink_len = v.sink_len;
  a.err_word = v.err_word;
  a.Hkv = s.Hkv;
  a.d = s.d;
  a.Ng = s.Ng;
  a.row_bytes = s.row_bytes;
  a.cap = s.cap;
  a.Nr = s.Nr;
  a.Ns = s.Ns;
  a.Lmax = Lmax;
  a.ng_shift = __builtin_ctz((unsigned)s.Ng);
  a.sb = strides[0];
  a.sh = strides[1];
  a.st = strides[2];
  if (s.bits == 4) {
    if (s.hybrid)
      quantize_pack_kernel<4, true><<<grid, kPackThreads, 0, st>>>(a);
    else
      quantize_pack_kernel<4, false><<<grid, kPackThreads, 0, st>>>(a);
  } else if (s.bits == 3) {
    if (s.hybrid)
      quantize_pack_kernel<3, true><<<grid, kPackThreads, 0, st>>>(a);
    else
      quantize_pack_kernel<3, false><<<grid, kPackThreads, 0, st>>>(a);
  } else {
    if (s.hybrid)
      quantize_pack_kernel<2, true><<<grid, kPackThreads, 0, st>>>(a);
    else
      quantize_pack_kernel<2, false><<<grid, kPackThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const Dims& s, const kvq_cache_view& v, const __half* k_new,
                          const __half* v_new, cudaStream_t st) {
  AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.codes[0] = v.k_codes;
  a.codes[1] = v.v_codes;
  a.params[0] = v.k_params;
  a.params[1] = v.v_params;
  a.res[0] = reinterpret_cast<__half*>(v.k_res);
  a.res[1] = reinterpret_cast<__half*>(v.v_res);
  a.modes[0] = v.k_mode;
  a.modes[1] = v.v_mode;
  a.rm = row_map(s, v.block_table);
  a.packed_len = v.packed_len;
  a.res_len = v.res_len;
  a.res_head = v.res_head;
  a.err_word = v.err_word;
  a.Hkv = s.Hkv;
  a.d = s.d;
  a.Ng = s.Ng;
  a.row_bytes = s.row_bytes;
  a.cap = s.cap;
  a.Nr = s.Nr;
  // one warp per (KV head, K or V) item, up to 32 warps (then more items per warp)
  const int items = 2 * s.Hkv;
  const int threads = 32 * (items < 32 ? items : 32);
  if (s.bits == 4) {
    if (s.hybrid)
      append_kernel<4, true><<<s.B, threads, 0, st>>>(a);
    else
      append_kernel<4, false><<<s.B, threads, 0, st>>>(a);
  } else if (s.bits == 3) {
    if (s.hybrid)
      append_kernel<3, true><<<s.B, threads, 0, st>>>(a);
    else
      append_kernel<3, false><<<s.B, threads, 0, st>>>(a);
  } else {
    if (s.hybrid)
      append_kernel<2, true><<<s.B, threads, 0, st>>>(a);
    else
      append_kernel<2, false><<<s.B, threads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvq
