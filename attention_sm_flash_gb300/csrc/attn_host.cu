// The forward on tensors in pinned host memory (attn_fwd_host, declared in
// include/attn.h). Attention heads are independent, so the problem crosses the
// host-device link in chunks of kv heads (with their query heads): the inputs of chunk
// c + 1 are copied in while chunk c is computed and the outputs of chunk c - 1 are copied
// out. Each chunk is an ordinary attn_fwd call on a compact sub-problem, so the results
// are those of attn_fwd on the same values, bit for bit.
//
// Streams: the compute runs on the caller's stream; copies in and copies out run on two
// streams of the library's own (one pair per device, created on first use), ordered
// against the caller's stream with events, so that work the caller queued before the
// call (which may still use the workspace) finishes before the first copy, and work
// queued after it sees every output in host memory.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kSlots = 2;    // chunks in flight: one being copied in, one computed
constexpr int kMaxDev = 64;
constexpr int kChunks = 5;   // the problem is cut into about this many chunks

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t entry = nullptr;
  cudaEvent_t copied_in[kSlots] = {}, computed[kSlots] = {}, copied_out[kSlots] = {};
};
HostPipe g_pipes[kMaxDev];
std::mutex g_pipe_mu;  // held while a call queues its work (events are reused per slot)

cudaError_t pipe_for_device(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  HostPipe& hp = g_pipes[dev];
  if (!hp.ready) {
    if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int s = 0; s < kSlots; ++s) {
      if ((e = cudaEventCreateWithFlags(&hp.copied_in[s], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&hp.computed[s], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&hp.copied_out[s], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    hp.ready = true;
  }
  *out = &hp;
  return cudaSuccess;
}

// The chunking of a problem and the layout of one workspace slot.
struct HostPlan {
  int kvc = 1;         // kv heads per chunk (the last chunk may hold fewer)
  int chunks = 1;
  size_t q = 0, kv = 0, lse = 0, lens = 0;  // bytes of each region of a slot (256-aligned)
  size_t slot = 0;                          // q, k, v, o, lse, lens
};

HostPlan host_plan(int B, int Hq, int Hkv, int Sq, int Skv, int D, attn_dtype_t dtype) {
  HostPlan pl;
  const int g = Hq / Hkv;
  const size_t el = dtype == ATTN_F32 ? 4 : 2;
  pl.kvc = (Hkv + kChunks - 1) / kChunks;
  pl.chunks = (Hkv + pl.kvc - 1) / pl.kvc;
  const size_t hc = (size_t)pl.kvc * g;  // query heads per chunk
  pl.q = round256((size_t)B * Sq * hc * D * el);
  pl.kv = round256((size_t)B * Skv * pl.kvc * D * el);
  pl.lse = round256((size_t)B * hc * Sq * sizeof(float));
  pl.lens = round256((size_t)B * pl.kvc * sizeof(int32_t));
  pl.slot = 2 * pl.q + 2 * pl.kv + pl.lse + pl.lens;
  return pl;
}

// Host memory that a copy on a stream can read or write asynchronously: page-locked
// (allocated or registered with CUDA).
bool pinned(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // the failed query is not the caller's error
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                               attn_dtype_t dtype) {
  if (check_common(B, Hq, Hkv, Sq, Skv, D, 1.f, 0, nullptr, dtype) != ATTN_OK) return 0;
  if (B == 0 || Sq == 0) return 0;
  return (size_t)kSlots * host_plan(B, Hq, Hkv, Sq, Skv, D, dtype).slot;
}

extern "C" attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int Hq, int Hkv, int Sq, int Skv,
                                       int D, float scale, int causal, const int32_t* kv_lens,
                                       attn_dtype_t dtype, void* workspace,
                                       size_t workspace_bytes, attn_stream_t stream) {
  attn_status_t st = check_common(B, Hq, Hkv, Sq, Skv, D, scale, causal, kv_lens, dtype);
  if (st != ATTN_OK) return st;
  if (B == 0 || Sq == 0) return ATTN_OK;  // an empty problem: nothing to copy or compute
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (Skv > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID_ARG;
  const HostPlan pl = host_plan(B, Hq, Hkv, Sq, Skv, D, dtype);
  if (workspace == nullptr || workspace_bytes < (size_t)kSlots * pl.slot ||
      (reinterpret_cast<uintptr_t>(workspace) % 256) != 0)
    return ATTN_ERR_WORKSPACE;
  if (!pinned(q) || !pinned(o) || !pinned(lse) || (Skv > 0 && (!pinned(k) || !pinned(v))) ||
      (kv_lens != nullptr && !pinned(kv_lens)))
    return ATTN_ERR_INVALID_ARG;

  const int g = Hq / Hkv;
  const size_t el = dtype == ATTN_F32 ? 4 : 2;
  const size_t row_q = (size_t)Hq * D * el, row_kv = (size_t)Hkv * D * el;  // bytes per token
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  uint8_t* ho = static_cast<uint8_t*>(o);

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = nullptr;
  cudaError_t e = pipe_for_device(&hp);
  if (e != cudaSuccess) return from_cuda(e);
  auto fail = [](cudaError_t err) -> attn_status_t { return from_cuda(err); };
  // the caller's earlier work (which may still use the workspace) comes first
  if ((e = cudaEventRecord(hp->entry, cs)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(hp->in, hp->entry, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(hp->out, hp->entry, 0)) != cudaSuccess) return fail(e);

  for (int c = 0; c < pl.chunks; ++c) {
    const int s = c % kSlots;
    const int kv0 = c * pl.kvc;
    const int kvn = (kv0 + pl.kvc <= Hkv) ? pl.kvc : Hkv - kv0;  // kv heads of this chunk
    const int h0 = kv0 * g, hn = kvn * g;                          // its query heads
    uint8_t* slot = static_cast<uint8_t*>(workspace) + (size_t)s * pl.slot;
    uint8_t* dq = slot;
    uint8_t* dk = dq + pl.q;
    uint8_t* dv = dk + pl.kv;
    uint8_t* dout = dv + pl.kv;
    float* dlse = reinterpret_cast<float*>(dout + pl.q);
    int32_t* dlens = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(dlse) + pl.lse);
    const size_t cq = (size_t)hn * D * el, ckv = (size_t)kvn * D * el;  // bytes per token

    // in: the slot's inputs were last read by the kernel of chunk c - 2
    if (c >= kSlots && (e = cudaStreamWaitEvent(hp->in, hp->computed[s], 0)) != cudaSuccess) return fail(e);
    e = cudaMemcpy2DAsync(dq, cq, hq + (size_t)h0 * D * el, row_q, cq, (size_t)B * Sq,
                          cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && Skv > 0)
      e = cudaMemcpy2DAsync(dk, ckv, hk + (size_t)kv0 * D * el, row_kv, ckv, (size_t)B * Skv,
                            cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && Skv > 0)
      e = cudaMemcpy2DAsync(dv, ckv, hv + (size_t)kv0 * D * el, row_kv, ckv, (size_t)B * Skv,
                            cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && kv_lens != nullptr)
      e = cudaMemcpy2DAsync(dlens, (size_t)kvn * 4, kv_lens + kv0, (size_t)Hkv * 4, (size_t)kvn * 4,
                            (size_t)B, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->copied_in[s], hp->in);
    if (e != cudaSuccess) return fail(e);

    // compute: after the chunk's inputs are in and the slot's previous outputs are out
    if ((e = cudaStreamWaitEvent(cs, hp->copied_in[s], 0)) != cudaSuccess) return fail(e);
    if (c >= kSlots && (e = cudaStreamWaitEvent(cs, hp->copied_out[s], 0)) != cudaSuccess) return fail(e);
    st = attn_fwd(dq, dk, dv, dout, dlse, B, hn, kvn, Sq, Skv, D, scale, causal,
                  kv_lens != nullptr ? dlens : nullptr, dtype, stream);
    if (st != ATTN_OK) return st;
    if ((e = cudaEventRecord(hp->computed[s], cs)) != cudaSuccess) return fail(e);

    // out: O rows into their heads' columns, LSE rows into their heads' blocks
    if ((e = cudaStreamWaitEvent(hp->out, hp->computed[s], 0)) != cudaSuccess) return fail(e);
    e = cudaMemcpy2DAsync(ho + (size_t)h0 * D * el, row_q, dout, cq, cq, (size_t)B * Sq,
                          cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(lse + (size_t)h0 * Sq, (size_t)Hq * Sq * 4, dlse, (size_t)hn * Sq * 4,
                            (size_t)hn * Sq * 4, (size_t)B, cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->copied_out[s], hp->out);
    if (e != cudaSuccess) return fail(e);
  }
  // the caller's later work sees every output in host memory
  e = cudaStreamWaitEvent(cs, hp->copied_out[(pl.chunks - 1) % kSlots], 0);
  return fail(e);
}
