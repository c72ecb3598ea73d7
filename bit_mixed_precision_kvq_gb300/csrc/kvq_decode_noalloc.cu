// kvq_decode_noalloc.cu -- kvq_decode_attention_static_ws: the decode
// entry point for callers that cannot allocate device memory.
//
// Some hosts of this library may not call cudaMalloc themselves: plug-ins
// that run inside a framework which owns every device allocation through its
// own allocator (memory obtained behind its back is invisible to its
// accounting and can make its later allocations fail), serving loops that
// must not risk the implicit device synchronisation an allocation can cause,
// and processes that reserve almost all device memory up front.  For them
// this entry point keeps the split-KV scratch (the per-chunk partial results
// that kvq_decode_attention otherwise takes as a caller-provided workspace)
// in a fixed array that is part of the library's own device image.
//
// The array is KVQ_STATIC_WS_BYTES long, is created on every GPU that loads
// the library and stays there until the process exits.  It is shared by all
// calls on a device: two calls whose kernels overlap on the GPU (different
// streams without ordering between them) race on it and may return wrong
// results.  Nothing in it needs to start at zero: each call writes every
// partial it later reads, so the previous call's leftovers are never used.
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

// The scratch itself.  In host code this name only stands for the symbol;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char kvq_static_scratch[KVQ_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex scratch_mu;
void* scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this set-up).
kvq_status scratch_address(void** out) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq_cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(scratch_mu);
  if (!scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t se = cudaGetSymbolAddress(&p, kvq_static_scratch);
    if (se != cudaSuccess) return kvq_cuda_fail(se);
    if (p == nullptr) return kvq_cuda_fail(cudaErrorInvalidSymbol);
    scratch_ptr[dev] = p;
  }
  *out = scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_static_ws(const kvq_layout* L, const void* cache,
                                                     const void* q_bf16, int32_t T,
                                                     float softmax_scale, void* out_bf16,
                                                     float* lse, void* stream) {
  const kvq_status st = kvq_check_layout(L);
  if (st != KVQ_OK) return st;
  // Layouts whose scratch does not fit the fixed array are refused before
  // any CUDA call.
  if (L->workspace_bytes > static_cast<int64_t>(KVQ_STATIC_WS_BYTES)) return KVQ_ERR_CAPACITY;
  void* ws = nullptr;
  const kvq_status sst = scratch_address(&ws);
  if (sst != KVQ_OK) return sst;
  return kvq_decode_attention(L, cache, q_bf16, T, softmax_scale, out_bf16, lse, ws,
                              KVQ_STATIC_WS_BYTES, stream);
}
