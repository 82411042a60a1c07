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
// that device current, on the first call there, which also clears the array
// once (its arrival counters must start at zero; every completed call leaves
// them at zero again); make that first call before any stream capture.  Two
// calls whose kernels overlap on the GPU race on the array: issue them on one
// stream, or order the streams.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (set up once).
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e == cudaSuccess && p != nullptr) e = cudaMemset(p, 0, KVQ_NOALLOC_SCRATCH_BYTES);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return KVQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_cache_desc* desc,
                                                   const kvq_cache_view* view, const void* q,
                                                   int32_t num_q_heads, void* out, void* stream) {
  // Sizes are checked first so an oversized request fails without touching the device.
  const size_t need = kvq_decode_workspace_bytes(desc, num_q_heads);
  if (need == 0) return KVQ_ERR_INVALID_ARG;  // invalid description or head count
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  kvq_status st = scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  return kvq_decode_attention(desc, view, q, num_q_heads, out, scratch,
                              (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
