// attn_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// The scratch the backward needs (delta = rowsum(dO * O), fp32 per query row, and for a
// split GQA group the fp32 partial dK/dV) lives in a static device array owned by the
// library instead of a caller workspace. Host code may not use the array's name as a
// device address (on the host it names a host-side stand-in), so the address is looked
// up once per device with cudaGetSymbolAddress while that device is current, cached, and
// handed to the ordinary attn_bwd path.

#include <cuda_runtime.h>

#include <mutex>

#include "attn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress((void**)&ptr, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* o, const void* dout, const float* lse,
                                          void* dq, void* dk, void* dv, int B, int Hq,
                                          int Hkv, int Sq, int Skv, int D, float scale,
                                          int causal, const int32_t* kv_lens,
                                          attn_dtype_t dtype, attn_stream_t stream) {
  const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype);
  if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, scale, causal,
                  kv_lens, dtype, scratch, (size_t)ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
