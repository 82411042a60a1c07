// kvq_decode.cu -- decode planning (kernel choice, split count, workspace
// layout) and the dispatch between the decode kernels.  The log-sum-exp merge of
// the split partials runs at the end of each decode kernel (combine_unit).
#include <math.h>

#include <atomic>

#include "kvq_decode_common.cuh"

namespace kvq {
namespace {

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

// SM count of the current device, queried once per device (every plan needs it).
int device_sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cached[kMaxDev];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();  // clear a no-device error so it does not leak into later calls
    return 152;
  }
  if (dev >= 0 && dev < kMaxDev && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  if (dev >= 0 && dev < kMaxDev) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Testing hook of kvq_testing_wait_fault (0: off).
static std::atomic<uint32_t> g_wait_fault_us{0};
void set_testing_wait_fault_us(uint32_t us) { g_wait_fault_us.store(us, std::memory_order_relaxed); }
uint32_t testing_wait_fault_us() { return g_wait_fault_us.load(std::memory_order_relaxed); }

DecodePlan plan_decode(const kvq_cache_desc& D, int num_q_heads, int sm_count, bool step) {
  DecodePlan p;
  p.gq = num_q_heads / D.num_kv_heads;
  int64_t target, min_tokens;
  p.cps = 0;
  p.fold = 0;
  p.tile = 128;
  if (tc_supported(D, p.gq)) {
    // tensor-core kernel: 4 query heads per CTA, one wave of resident CTAs.
    // When even one packed split per (sequence, KV head) plus its fp16 splits
    // fills more than a wave, the grid runs in several waves anyway and takes
    // the 4-CTAs-per-SM variant.
    p.kernel = 1;
    p.qb = 4;
    p.nqb = 1;
    p.threads = tc_threads();
    const int64_t units1 = (int64_t)D.batch * D.num_kv_heads;
    const int64_t fp16_splits = (D.residual + D.sink + tc_residual_rows() - 1) / tc_residual_rows();
    const bool waves = units1 * (1 + (fp16_splits > 0 ? fp16_splits : (step ? 1 : 0))) >
                       (int64_t)sm_count * tc_ctas_per_sm(false);
    p.cps = tc_ctas_per_sm(waves);
    target = (int64_t)sm_count * p.cps;
    min_tokens = 256;
  } else {
    p.kernel = 0;
    p.qb = next_pow2(p.gq < 8 ? p.gq : 8);
    p.nqb = (p.gq + p.qb - 1) / p.qb;
    p.threads = 128;
    target = (int64_t)sm_count * 4;
    min_tokens = 256;
  }
  const int64_t units = (int64_t)D.batch * D.num_kv_heads * p.nqb;
  const int64_t tokens_max = (int64_t)D.capacity + D.residual + D.sink;
  // one CTA per unit short of a full wave: the previous launch's last CTA of
  // each unit (its merger) still holds a slot when this launch starts
  if (p.kernel == 1 && units * 4 <= target) target -= units;
  int64_t S = (target + units - 1) / units;
  const int64_t by_len = (tokens_max + min_tokens - 1) / min_tokens;
  if (S > by_len) S = by_len;
  if (S < 1) S = 1;
  if (S > 1024) S = 1024;
  p.splits = (int)S;
  p.splits_packed = p.splits;
  if (p.kernel == 1) {
    // the fp16 tokens (window ring slots, then sink rows) get splits of their
    // own, one per tc_residual_rows() rows (at least one in a fused step: it
    // takes the appended token)
    const int rr = tc_residual_rows();
    int sr = (D.residual + D.sink + rr - 1) / rr;
    if (step && sr < 1) sr = 1;
    // A grid of several waves gives its fp16 rows to the last packed split of
    // each (sequence, KV head) instead of CTAs of their own.
    if (p.cps == 4) {
      sr = 0;
      p.fold = 1;
    }
    const int sp = (int)S - sr > 1 ? (int)S - sr : 1;
    p.splits_packed = sp;
    p.splits = sp + sr;
    p.tile = tc_tile_tokens(D, p.cps, ((int64_t)D.capacity + sp - 1) / sp);
  }
  const int64_t nparts = units * p.splits * p.qb;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t uq = (size_t)units * p.qb;
  p.ws_cnt_off = 0;
  p.ws_seq_off = up((size_t)units * sizeof(uint32_t));
  p.ws_ref_off = up(p.ws_seq_off + (size_t)D.batch * sizeof(uint32_t));
  p.ws_flag_off = up(p.ws_ref_off + uq * sizeof(uint32_t));
  p.ws_oacc_off = up(p.ws_flag_off + (size_t)units * sizeof(uint32_t));
  p.ws_lacc_off = up(p.ws_oacc_off + uq * D.head_dim * sizeof(float));
  p.ws_ml_off = up(p.ws_lacc_off + uq * sizeof(float));
  p.ws_part_off = up(p.ws_ml_off + (size_t)nparts * sizeof(float2));
  p.ws_total = p.ws_part_off + (size_t)nparts * D.head_dim * sizeof(float);
  return p;
}

cudaError_t launch_decode(const Dims& s, const DecodePlan& p, const kvq_cache_view& v,
                          const __half* q, int Hq, void* out, void* workspace, cudaStream_t st,
                          const __half* k_new, const __half* v_new, uint32_t flags) {
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
  a.rm = row_map(s, v.block_table);
  a.k_sink = reinterpret_cast<const __half*>(v.k_sink);
  a.v_sink = reinterpret_cast<const __half*>(v.v_sink);
  a.sink_len = v.sink_len;
  a.q = q;
  a.out = out;
  a.out_f32 = (flags & KVQ_OUT_F32) ? 1 : 0;
  char* ws = reinterpret_cast<char*>(workspace);
  a.o_part = reinterpret_cast<float*>(ws + p.ws_part_off);
  a.ml_part = reinterpret_cast<float2*>(ws + p.ws_ml_off);
  a.counters = reinterpret_cast<uint32_t*>(ws + p.ws_cnt_off);
  a.seq_tickets = reinterpret_cast<uint32_t*>(ws + p.ws_seq_off);
  a.ref_max = reinterpret_cast<uint32_t*>(ws + p.ws_ref_off);
  a.fb_flag = reinterpret_cast<uint32_t*>(ws + p.ws_flag_off);
  a.o_acc = reinterpret_cast<float*>(ws + p.ws_oacc_off);
  a.l_acc = reinterpret_cast<float*>(ws + p.ws_lacc_off);
  // the fused step (tensor-core kernel only) writes the cache
  a.k_new = k_new;
  a.v_new = v_new;
  a.w_codes[0] = v.k_codes;
  a.w_codes[1] = v.v_codes;
  a.w_params[0] = v.k_params;
  a.w_params[1] = v.v_params;
  a.w_res[0] = reinterpret_cast<__half*>(v.k_res);
  a.w_res[1] = reinterpret_cast<__half*>(v.v_res);
  a.w_modes[0] = v.k_mode;
  a.w_modes[1] = v.v_mode;
  a.hybrid = s.hybrid;
  a.w_packed_len = v.packed_len;
  a.w_res_len = v.res_len;
  a.w_res_head = v.res_head;
  a.Hkv = s.Hkv;
  a.Hq = Hq;
  a.gq = p.gq;
  a.qb = p.qb;
  a.nqb = p.nqb;
  a.S = p.splits;
  a.Sp = p.splits_packed;
  a.fold = p.fold;
  a.Ns = s.Ns;
  a.cap = s.cap;
  a.Nr = s.Nr;
  a.d = s.d;
  a.row_bytes = s.row_bytes;
  a.early = (flags & KVQ_STEP_EARLY_CACHE_READ) ? 1 : 0;
  a.qk_scale_log2 = (float)(1.4426950408889634 / sqrt((double)s.d));
  const uint32_t fault_us = testing_wait_fault_us();
  a.wait_limit_us = fault_us ? fault_us : 1000000u;
  a.fault_tx = fault_us ? 16u : 0u;
  const bool step = k_new != nullptr;
  if (p.kernel == 1) return launch_decode_tc(s, p, a, st, step);
  cudaError_t e = cudaSuccess;
  if (step) e = launch_append(s, v, k_new, v_new, st);  // generic path: two launches
  if (e != cudaSuccess) return e;
  return launch_decode_generic(s, p, a, st);
}

}  // namespace kvq
