// Decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attention needs a caller-provided device workspace (an error
// word, one counter per (batch, kv head) and the per-split partial results).
// Some callers have no way to provide one: a custom-operator or plugin
// interface that hands over only the input and output tensors, or a serving
// process whose device memory is owned entirely by another allocator, where a
// cudaMalloc is either not allowed or would stall the device.  This variant
// keeps that workspace in a fixed-size array in the library's own static
// device memory instead, and otherwise runs the very same decode path.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits.  Every call shares it, so calls whose kernels can
// overlap on the GPU (two streams, or two threads) race on it and must be
// serialized by the caller.
#include <mutex>

#include "kvq_internal.h"

namespace {

// The static scratch: error word, split counters, split partial results.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is taken once
// per device with cudaGetSymbolAddress while that device is current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_cache* cache, const void* q,
                                                   void* out, void* stream) {
  kvq_status st = kvq::check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!q || !out || ((uintptr_t)q & 15u) || ((uintptr_t)out & 15u)) {
    kvq::set_last_error("q/out must be non-NULL and 16-byte aligned");
    return KVQ_ERR_INVALID_ARG;
  }
  // the smallest workspace the decode needs (one split per head); more splits
  // are used only as far as the fixed array allows
  const size_t need = kvq_workspace_bytes(cache, 1);
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) {
    kvq::set_last_error("this cache needs more decode scratch than the static array of "
                        "KVQ_NOALLOC_SCRATCH_BYTES holds (too many batch x kv heads); "
                        "use kvq_decode_attention with a caller workspace");
    return KVQ_ERR_CAPACITY;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    kvq::set_last_error(cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  // the error word and the split counters must start at zero; the array keeps
  // whatever the previous call left, so clear them on the caller's stream
  e = cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    kvq::set_last_error(cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  return kvq_decode_attention(cache, q, out, scratch, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}

// The error word of the static scratch (its first int32), which the decode
// kernels raise when a bounded wait runs out: the caller of the entry point
// above has no pointer to it.  Reads it after the work queued on `stream`.
extern "C" kvq_status kvq_noalloc_error(int32_t* err_out, void* stream) {
  if (!err_out) {
    kvq::set_last_error("NULL argument");
    return KVQ_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    kvq::set_last_error(cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  return kvq_workspace_error(scratch, err_out, stream);
}
