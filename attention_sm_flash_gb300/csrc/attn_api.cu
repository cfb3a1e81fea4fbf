// The C ABI of libattn (declared in include/attn.h): host-side argument checks, the
// device error word, and the choice of kernel family by element type.

#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

// The device error word: kernels OR ATTN_DEVERR_* bits into it.
__device__ unsigned int g_error_word = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_addr[kMaxDevices] = {};

// The error word's device address on the current device (looked up once per device).
cudaError_t error_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_error_word);
    if (e != cudaSuccess) return e;
    g_err_addr[dev] = static_cast<unsigned int*>(ptr);
  }
  *out = g_err_addr[dev];
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

// Checks shared by the forward and the backward. Returns ATTN_OK, or the error.
attn_status_t check_common(int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                           int causal, const int32_t* kv_lens, attn_dtype_t dtype) {
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (kv_lens != nullptr && !aligned(kv_lens, 4)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // grid limits of the launch shapes: heads and batches index grid dimensions
  if (Hq > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;
  // every element offset must fit a signed 64-bit integer with room to spare
  const double elems_q = (double)B * Sq * Hq * D, elems_k = (double)B * Skv * Hkv * D;
  if (elems_q > 4.0e18 || elems_k > 4.0e18) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

namespace {

thread_local cudaError_t g_last_cuda = cudaSuccess;

}  // namespace

attn_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  g_last_cuda = e;
  return ATTN_ERR_CUDA;
}

namespace {

std::atomic<uint64_t> g_launches{0};

}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                  float scale, int causal, const int32_t* kv_lens,
                                  attn_dtype_t dtype, attn_stream_t stream) {
  attn_status_t st = check_common(B, Hq, Hkv, Sq, Skv, D, scale, causal, kv_lens, dtype);
  if (st != ATTN_OK) return st;
  if (B == 0 || Sq == 0) return ATTN_OK;  // an empty problem: nothing to compute
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (Skv > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.D = D;
  p.scale = scale; p.causal = causal; p.kv_lens = kv_lens; p.dtype = dtype;
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(dtype == ATTN_BF16 ? tc_fwd(p, s) : tf32_fwd(p, s));
}

extern "C" attn_status_t attn_fwd_paged(const void* q, const void* k_pages,
                                        const void* v_pages, const int32_t* block_table,
                                        const int32_t* seq_lens, void* o, float* lse, int B,
                                        int Hq, int Hkv, int Sq, int num_pages, int page_size,
                                        int max_pages, int D, float scale, int causal,
                                        attn_dtype_t dtype, attn_stream_t stream) {
  if (num_pages < 1 || max_pages < 1 || page_size < 1) return ATTN_ERR_INVALID_ARG;
  const long long skv = (long long)max_pages * page_size;
  if (skv > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (seq_lens != nullptr && !aligned(seq_lens, 4)) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_common(B, Hq, Hkv, Sq, (int)skv, D, scale, causal, nullptr, dtype);
  if (st != ATTN_OK) return st;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  // a power of two of at least 16 keys: a 128-key tile is then whole pages or lies inside
  // one page, and the kernel locates keys with shifts
  if (page_size < 16 || (page_size & (page_size - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
  if ((double)num_pages * page_size * Hkv * D > 4.0e18) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || lse == nullptr || k_pages == nullptr ||
      v_pages == nullptr || block_table == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(block_table, 4))
    return ATTN_ERR_INVALID_ARG;
  Problem p{};
  p.q = q; p.k = k_pages; p.v = v_pages; p.o = o; p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = (int)skv; p.D = D;
  p.scale = scale; p.causal = causal; p.kv_lens = seq_lens; p.dtype = dtype;
  p.block_table = block_table; p.num_pages = num_pages; p.page_size = page_size;
  p.max_pages = max_pages;
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(tc_fwd(p, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv,
                                                  int D, attn_dtype_t dtype) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0) return 0;
  int per = 0;
  const int n = fwd_split_count(B, Hq, Sq, Skv, dtype, &per);
  if (n <= 1) return 0;
  return fwd_split_part_bytes(n, B, Hq, Sq, D) + fwd_split_lse_bytes(n, B, Hq, Sq);
}

extern "C" attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o,
                                          float* lse, int B, int Hq, int Hkv, int Sq, int Skv,
                                          int D, float scale, int causal,
                                          const int32_t* kv_lens, attn_dtype_t dtype,
                                          void* workspace, size_t workspace_bytes,
                                          attn_stream_t stream) {
  attn_status_t st = check_common(B, Hq, Hkv, Sq, Skv, D, scale, causal, kv_lens, dtype);
  if (st != ATTN_OK) return st;
  int per = 0;
  const int n = (B > 0 && Sq > 0) ? fwd_split_count(B, Hq, Sq, Skv, dtype, &per) : 1;
  if (n <= 1)
    return attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, causal, kv_lens, dtype,
                    stream);
  if (q == nullptr || o == nullptr || lse == nullptr || k == nullptr || v == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return ATTN_ERR_WORKSPACE;
  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.D = D;
  p.scale = scale; p.causal = causal; p.kv_lens = kv_lens; p.dtype = dtype;
  p.fwd_splits = n;
  p.fwd_split_tiles = per;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        fwd_split_part_bytes(n, B, Hq, Sq, D));
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(tc_fwd(p, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                          attn_dtype_t dtype) {
  if (B <= 0 || Hq <= 0 || Sq <= 0 || Hkv <= 0 || Skv < 0 || D <= 0) return 0;
  size_t n = bwd_delta_bytes(B, Hq, Sq);
  const int parts = Skv > 0 ? bwd_split_parts(B, Hq, Hkv, Skv, dtype) : 0;
  if (parts > 0) n += 2 * bwd_partial_bytes(B, Hkv, parts, Skv, D);
  return n;
}

extern "C" attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                  const void* dout, const float* lse, void* dq, void* dk,
                                  void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                  float scale, int causal, const int32_t* kv_lens,
                                  attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                  attn_stream_t stream) {
  attn_status_t st = check_common(B, Hq, Hkv, Sq, Skv, D, scale, causal, kv_lens, dtype);
  if (st != ATTN_OK) return st;
  if (B == 0 || (Sq == 0 && Skv == 0)) return ATTN_OK;
  if (Sq == 0) {
    // no queries: every key gets zero gradient; dk, dv are still outputs
    if (dk == nullptr || dv == nullptr) return ATTN_ERR_INVALID_ARG;
    const size_t elem = dtype == ATTN_F32 ? 4 : 2;
    const size_t bytes = (size_t)B * Skv * Hkv * D * elem;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(dk, 0, bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, bytes, s);
    return from_cuda(e);
  }
  if (q == nullptr || o == nullptr || dout == nullptr || lse == nullptr || dq == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (Skv > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return ATTN_ERR_WORKSPACE;
  Problem p{};
  p.q = q; p.k = k; p.v = v; p.o_in = o; p.dout = dout; p.lse = const_cast<float*>(lse);
  p.dq = dq; p.dk = dk; p.dv = dv; p.delta = static_cast<float*>(workspace);
  p.split = Skv > 0 ? bwd_split_parts(B, Hq, Hkv, Skv, dtype) : 0;
  if (p.split) {
    uint8_t* w = static_cast<uint8_t*>(workspace) + bwd_delta_bytes(B, Hq, Sq);
    p.part_dk = reinterpret_cast<float*>(w);
    p.part_dv = reinterpret_cast<float*>(w + bwd_partial_bytes(B, Hkv, p.split, Skv, D));
  }
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.D = D;
  p.scale = scale; p.causal = causal; p.kv_lens = kv_lens; p.dtype = dtype;
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(dtype == ATTN_BF16 ? tc_bwd(p, s) : simt_bwd(p, s));
}

extern "C" attn_status_t attn_peek_device_error(uint32_t* bits, attn_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (bits != nullptr) *bits = word;
  if (word & ATTN_DEVERR_TIMEOUT) return ATTN_ERR_TIMEOUT;
  if (word & ATTN_DEVERR_LAYOUT) return ATTN_ERR_CUDA;
  if (word & (ATTN_DEVERR_KVLEN | ATTN_DEVERR_PAGE)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

extern "C" const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported configuration";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: device barrier wait timed out";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown attn status";
}

extern "C" void attn_test_inject_fault(uint32_t mask, uint32_t timeout_ms) {
  tc_set_test_fault(mask, (uint64_t)timeout_ms * 1000000ull);
}

extern "C" const char* attn_last_cuda_error(void) {
  return g_last_cuda == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda);
}

extern "C" uint64_t attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char* attn_build_info(void) {
  return "libattn sm_103a: bf16 fwd (dense, paged, split-KV) + bwd tcgen05/TMA/TMEM; fp32 "
         "fwd tcgen05 3xTF32, fp32 bwd CUDA-core";
}
