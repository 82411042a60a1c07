// kvq_api.cu -- the C ABI of libkvq.so: argument checks, launch, status codes.
// Every entry point validates on the host and launches nothing on an error.
#include <string.h>

#include "kvq_internal.cuh"

namespace {

using kvq::Dims;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

kvq_status check_desc(const kvq_cache_desc* D) {
  if (!D) return KVQ_ERR_INVALID_ARG;
  if (D->batch < 1 || D->num_kv_heads < 1 || D->capacity < 0 || D->residual < 0 ||
      D->group != kvq::kGroup || D->head_dim < 32 || D->head_dim % 32 != 0)
    return KVQ_ERR_INVALID_ARG;
  if (D->bits < 2 || D->bits > 4) return KVQ_ERR_UNSUPPORTED;
  if (D->head_dim != 32 && D->head_dim != 64 && D->head_dim != 128 && D->head_dim != 256)
    return KVQ_ERR_UNSUPPORTED;
  if (D->sink < 0 || (D->hybrid != 0 && D->hybrid != 1)) return KVQ_ERR_INVALID_ARG;
  if (D->page_size != 0 && D->page_size != kvq::kPage) return KVQ_ERR_UNSUPPORTED;
  if (D->page_size && (D->capacity % kvq::kPage != 0 || D->num_pages < 0 ||
                       (D->capacity > 0 && D->num_pages < 1)))
    return KVQ_ERR_INVALID_ARG;
  if (D->residual > 1024 || D->sink > 256) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)D->batch * D->num_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

kvq_status check_view(const kvq_cache_desc& D, const kvq_cache_view* v) {
  if (!v) return KVQ_ERR_INVALID_ARG;
  if (!v->packed_len || !v->res_len || !v->res_head || !v->err_word) return KVQ_ERR_INVALID_ARG;
  if (D.capacity > 0 && (!v->k_codes || !v->v_codes || !v->k_params || !v->v_params))
    return KVQ_ERR_INVALID_ARG;
  if (D.residual > 0 && (!v->k_res || !v->v_res)) return KVQ_ERR_INVALID_ARG;
  if (D.sink > 0 && (!v->k_sink || !v->v_sink || !v->sink_len)) return KVQ_ERR_INVALID_ARG;
  if (D.hybrid && D.capacity > 0 && (!v->k_mode || !v->v_mode)) return KVQ_ERR_INVALID_ARG;
  if (D.page_size && D.capacity > 0 && !v->block_table) return KVQ_ERR_INVALID_ARG;
  const void* a16[] = {v->k_codes, v->v_codes, v->k_params, v->v_params, v->k_res,
                       v->v_res,   v->k_sink,   v->v_sink,   v->k_mode,   v->v_mode};
  for (const void* p : a16)
    if (!aligned(p, 16)) return KVQ_ERR_MISALIGNED;
  const void* a4[] = {v->packed_len, v->res_len, v->res_head, v->err_word, v->sink_len,
                      v->block_table};
  for (const void* p : a4)
    if (!aligned(p, 4)) return KVQ_ERR_MISALIGNED;
  return KVQ_OK;
}

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

constexpr uint32_t kStepFlags = KVQ_STEP_EARLY_CACHE_READ | KVQ_OUT_F32;

// A page-locked host buffer the device addresses with the same pointer (the
// allocation registered with the driver, mapped, and the device pointer equal).
bool host_mapped(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost && at.devicePointer == p && at.hostPointer == p;
}

}  // namespace

extern "C" {

size_t kvq_cache_bytes(const kvq_cache_desc* desc, int which) {
  if (check_desc(desc) != KVQ_OK) return 0;
  const Dims s = kvq::dims_of(*desc);
  const size_t rows = (size_t)s.B * s.Hkv;
  // packed rows: every (sequence, head, slot), or every (page, head, slot) of the pool
  const size_t prow = s.page ? (size_t)s.npages * s.Hkv * s.page : rows * (size_t)s.cap;
  switch (which) {
    case KVQ_ARRAY_CODES: return prow * s.row_bytes;
    case KVQ_ARRAY_PARAMS: return prow * s.Ng * sizeof(uint32_t);
    case KVQ_ARRAY_RESIDUAL: return rows * (size_t)s.Nr * s.d * sizeof(uint16_t);
    case KVQ_ARRAY_SINK: return rows * (size_t)s.Ns * s.d * sizeof(uint16_t);
    case KVQ_ARRAY_MODE: return s.hybrid ? prow : 0;
    default: return 0;
  }
}

size_t kvq_decode_workspace_bytes(const kvq_cache_desc* desc, int32_t num_q_heads) {
  if (check_desc(desc) != KVQ_OK || num_q_heads < 1 || num_q_heads % desc->num_kv_heads) return 0;
  // the fused step's plan has at least as many splits; tickets sit at fixed offsets
  return kvq::plan_decode(*desc, num_q_heads, kvq::device_sm_count(), true).ws_total;
}

kvq_status kvq_quantize_pack_strided(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                     const void* k, const void* v, const int32_t* seq_lens,
                                     int32_t Lmax, int64_t stride_b, int64_t stride_h,
                                     int64_t stride_t, void* stream) {
  kvq_status st = check_desc(desc);
  if (st != KVQ_OK) return st;
  if ((st = check_view(*desc, view)) != KVQ_OK) return st;
  if (Lmax < 0 || !seq_lens || (Lmax > 0 && (!k || !v))) return KVQ_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_h < 0 || stride_t < 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(seq_lens, 4)) return KVQ_ERR_MISALIGNED;
  // every 8-value piece a lane loads must start on a 16-byte boundary
  if (stride_b % 8 || stride_h % 8 || stride_t % 8) return KVQ_ERR_MISALIGNED;
  const Dims s = kvq::dims_of(*desc);
  const int64_t strides[3] = {stride_b, stride_h, stride_t};
  return from_cuda(kvq::launch_quantize_pack(s, *view, static_cast<const __half*>(k),
                                             static_cast<const __half*>(v), seq_lens, Lmax, strides,
                                             static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_quantize_pack(const kvq_cache_desc* desc, const kvq_cache_view* view,
                             const void* k, const void* v, const int32_t* seq_lens,
                             int32_t Lmax, void* stream) {
  if (check_desc(desc) != KVQ_OK) return check_desc(desc);
  const int64_t d = desc->head_dim;
  return kvq_quantize_pack_strided(desc, view, k, v, seq_lens, Lmax,
                                   (int64_t)desc->num_kv_heads * Lmax * d, (int64_t)Lmax * d, d,
                                   stream);
}

kvq_status kvq_append(const kvq_cache_desc* desc, const kvq_cache_view* view, const void* k_new,
                      const void* v_new, void* stream) {
  kvq_status st = check_desc(desc);
  if (st != KVQ_OK) return st;
  if ((st = check_view(*desc, view)) != KVQ_OK) return st;
  if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return KVQ_ERR_MISALIGNED;
  const Dims s = kvq::dims_of(*desc);
  return from_cuda(kvq::launch_append(s, *view, static_cast<const __half*>(k_new),
                                      static_cast<const __half*>(v_new),
                                      static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_attention(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                const void* q, int32_t num_q_heads, void* out, void* workspace,
                                size_t ws_bytes, uint32_t flags, void* stream) {
  kvq_status st = check_desc(desc);
  if (st != KVQ_OK) return st;
  if ((st = check_view(*desc, view)) != KVQ_OK) return st;
  if (!q || !out || !workspace || num_q_heads < 1 || num_q_heads % desc->num_kv_heads ||
      (flags & ~(uint32_t)KVQ_OUT_F32))
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16)) return KVQ_ERR_MISALIGNED;
  if ((int64_t)desc->batch * num_q_heads > 2147483647LL) return KVQ_ERR_UNSUPPORTED;
  const kvq::DecodePlan p = kvq::plan_decode(*desc, num_q_heads, kvq::device_sm_count());
  if ((int64_t)desc->num_kv_heads * p.nqb > 65535) return KVQ_ERR_UNSUPPORTED;
  if (ws_bytes < p.ws_total) return KVQ_ERR_INVALID_ARG;
  const Dims s = kvq::dims_of(*desc);
  return from_cuda(kvq::launch_decode(s, p, *view, static_cast<const __half*>(q), num_q_heads, out,
                                      workspace, static_cast<cudaStream_t>(stream), nullptr,
                                      nullptr, flags));
}

kvq_status kvq_decode_step(const kvq_cache_desc* desc, const kvq_cache_view* view, const void* q,
                           int32_t num_q_heads, const void* k_new, const void* v_new, void* out,
                           void* workspace, size_t ws_bytes, uint32_t flags, void* stream) {
  kvq_status st = check_desc(desc);
  if (st != KVQ_OK) return st;
  if ((st = check_view(*desc, view)) != KVQ_OK) return st;
  if (!q || !out || !workspace || !k_new || !v_new || num_q_heads < 1 ||
      num_q_heads % desc->num_kv_heads || (flags & ~kStepFlags))
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16) || !aligned(k_new, 16) ||
      !aligned(v_new, 16))
    return KVQ_ERR_MISALIGNED;
  if ((int64_t)desc->batch * num_q_heads > 2147483647LL) return KVQ_ERR_UNSUPPORTED;
  const kvq::DecodePlan p = kvq::plan_decode(*desc, num_q_heads, kvq::device_sm_count(), true);
  if ((int64_t)desc->num_kv_heads * p.nqb > 65535) return KVQ_ERR_UNSUPPORTED;
  if (ws_bytes < p.ws_total) return KVQ_ERR_INVALID_ARG;
  const Dims s = kvq::dims_of(*desc);
  return from_cuda(kvq::launch_decode(s, p, *view, static_cast<const __half*>(q), num_q_heads, out,
                                      workspace, static_cast<cudaStream_t>(stream),
                                      static_cast<const __half*>(k_new),
                                      static_cast<const __half*>(v_new), flags));
}

namespace {
struct StepIo {
  size_t q, kv, in_bytes, out_off, total;
};
// Byte layout of the packed step input [q | k_new | v_new] and of the device
// staging area (the input, then out at a 256-byte boundary).
StepIo step_io(const kvq_cache_desc& D, int32_t num_q_heads) {
  StepIo io;
  io.q = (size_t)D.batch * num_q_heads * D.head_dim * sizeof(uint16_t);
  io.kv = (size_t)D.batch * D.num_kv_heads * D.head_dim * sizeof(uint16_t);
  io.in_bytes = io.q + 2 * io.kv;
  io.out_off = (io.in_bytes + 255) & ~(size_t)255;
  io.total = io.out_off + 2 * io.q;  // room for an fp32 out
  return io;
}
}  // namespace

size_t kvq_step_io_bytes(const kvq_cache_desc* desc, int32_t num_q_heads) {
  if (check_desc(desc) != KVQ_OK || num_q_heads < 1 || num_q_heads % desc->num_kv_heads) return 0;
  return step_io(*desc, num_q_heads).total;
}

kvq_status kvq_decode_step_host(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                const void* in_host, int32_t num_q_heads, void* out_host,
                                void* dev_io, size_t dev_io_bytes, void* workspace,
                                size_t ws_bytes, uint32_t flags, void* stream) {
  kvq_status st = check_desc(desc);
  if (st != KVQ_OK) return st;
  if (flags & KVQ_STEP_HOST_MAPPED) {
    // the step reads the input block and writes out in place, over the host link
    if (!in_host || !out_host || num_q_heads < 1 || num_q_heads % desc->num_kv_heads)
      return KVQ_ERR_INVALID_ARG;
    if (!host_mapped(in_host) || !host_mapped(out_host)) return KVQ_ERR_INVALID_ARG;
    const StepIo io = step_io(*desc, num_q_heads);
    const char* in = static_cast<const char*>(in_host);
    return kvq_decode_step(desc, view, in, num_q_heads, in + io.q, in + io.q + io.kv, out_host,
                           workspace, ws_bytes, flags & ~(uint32_t)KVQ_STEP_HOST_MAPPED, stream);
  }
  if (!in_host || !out_host || !dev_io || num_q_heads < 1 || num_q_heads % desc->num_kv_heads)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(dev_io, 256)) return KVQ_ERR_MISALIGNED;
  const StepIo io = step_io(*desc, num_q_heads);
  if (dev_io_bytes < io.total) return KVQ_ERR_INVALID_ARG;
  char* d = static_cast<char*>(dev_io);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every argument the step itself checks is checked before anything is enqueued
  const kvq::DecodePlan p = kvq::plan_decode(*desc, num_q_heads, kvq::device_sm_count(), true);
  if ((st = check_view(*desc, view)) != KVQ_OK) return st;
  if (!workspace || ws_bytes < p.ws_total || (flags & ~kStepFlags)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return KVQ_ERR_MISALIGNED;
  if (cudaMemcpyAsync(d, in_host, io.in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  // the step follows this call's own copy, not a kernel: an early cache read
  // would have nothing to overlap
  st = kvq_decode_step(desc, view, d, num_q_heads, d + io.q, d + io.q + io.kv, d + io.out_off,
                       workspace, ws_bytes, flags & ~(uint32_t)KVQ_STEP_EARLY_CACHE_READ, stream);
  if (st != KVQ_OK) return st;
  const size_t out_bytes = (flags & KVQ_OUT_F32) ? 2 * io.q : io.q;
  if (cudaMemcpyAsync(out_host, d + io.out_off, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_read_error(const kvq_cache_view* view, uint32_t* word_out, void* stream) {
  if (!view || !view->err_word) return KVQ_ERR_INVALID_ARG;
  if (!aligned(view->err_word, 4)) return KVQ_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  cudaError_t e = cudaMemcpyAsync(&w, view->err_word, sizeof(w), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(view->err_word, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  if (word_out) *word_out = w;
  if (w & KVQ_ERRBIT_TIMEOUT) kvq::noalloc_forget_layout();
  if (w & KVQ_ERRBIT_CAPACITY) return KVQ_ERR_CAPACITY;
  if (w & KVQ_ERRBIT_EMPTY) return KVQ_ERR_EMPTY;
  if (w & KVQ_ERRBIT_TIMEOUT) return KVQ_ERR_TIMEOUT;
  if (w & (KVQ_ERRBIT_BADLEN | KVQ_ERRBIT_BADPAGE)) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_MISALIGNED: return "misaligned pointer";
    case KVQ_ERR_CAPACITY: return "packed capacity exceeded";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
    case KVQ_ERR_EMPTY: return "sequence with no tokens";
    default: return "unknown status";
  }
}

int32_t kvq_version(void) { return 160; }

void kvq_testing_wait_fault(uint32_t limit_us) { kvq::set_testing_wait_fault_us(limit_us); }

}  // extern "C"
