// kvq_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain scratch memory at decode time: code that
// runs under a caching allocator it does not own, embedders whose memory is
// fixed up front, or runtimes that forbid cudaMalloc once the serving loop has
// started.  kvq_decode_attention_noalloc serves them by taking the decode's
// split partials from one file-scope device array instead of a caller buffer.
//
// The array is `static __device__`: every GPU that loads this library holds it
// (KVQ_NOALLOC_SCRATCH_BYTES) until the process exits, and every call on a
// device shares it.  The host only ever sees a stand-in for its name, so its
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, on the first call there; make that first call before any
// stream capture.  The counters and accumulators that must be zero at the start
// of a call sit at offsets that depend on the cache shape and head count, and
// every completed call leaves them zero for its own shape.  So the first call on
// a device, a call whose shape differs from the previous call's there, and the
// first call after kvq_read_error reported a timed-out wait (which may leave
// them non-zero) clear that part of the array first, with cudaMemsetAsync on the
// call's own stream (the call is then two operations on that stream).  Two calls
// whose kernels overlap on the GPU race on the array: issue them on one stream,
// or order the streams.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Shape of the zero-between-calls part of the array as the last call on each
// device left it (every completed call leaves that part zero for its own shape).
struct ZeroLayout {
  int32_t batch, num_kv_heads, head_dim, qb, nqb;
  bool operator==(const ZeroLayout& o) const {
    return batch == o.batch && num_kv_heads == o.num_kv_heads && head_dim == o.head_dim &&
           qb == o.qb && nqb == o.nqb;
  }
};
ZeroLayout g_last_layout[kMaxDevices];
bool g_has_layout[kMaxDevices] = {false};

// Device address of g_decode_scratch on the current device (looked up once).
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return KVQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

namespace kvq {

// After a timed-out wait the counters of the array on this device may be left
// non-zero: the next call clears them whatever its shape.
void noalloc_forget_layout() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_has_layout[dev] = false;
}

}  // namespace kvq

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_cache_desc* desc,
                                                   const kvq_cache_view* view, const void* q,
                                                   int32_t num_q_heads, void* out, uint32_t flags,
                                                   void* stream) {
  // Sizes are checked first so an oversized request fails without touching the device.
  const size_t need = kvq_decode_workspace_bytes(desc, num_q_heads);
  if (need == 0) return KVQ_ERR_INVALID_ARG;  // invalid description or head count
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  kvq_status st = scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  const kvq::DecodePlan p = kvq::plan_decode(*desc, num_q_heads, kvq::device_sm_count());
  const ZeroLayout lay = {desc->batch, desc->num_kv_heads, desc->head_dim, p.qb, p.nqb};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_has_layout[dev] || !(g_last_layout[dev] == lay)) {
      // everything before the partials: tickets, reference maxima, flags, accumulators
      if (cudaMemsetAsync(scratch, 0, p.ws_ml_off, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
      g_last_layout[dev] = lay;
      g_has_layout[dev] = true;
    }
  }
  return kvq_decode_attention(desc, view, q, num_q_heads, out, scratch,
                              (size_t)KVQ_NOALLOC_SCRATCH_BYTES, flags, stream);
}
