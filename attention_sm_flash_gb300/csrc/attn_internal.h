// Internal interface between the C ABI (attn_api.cu) and the kernel families.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

// One validated attention problem. Every pointer is a device pointer.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;            // forward output
  float* lse;         // forward output (fwd) / input (bwd)
  const void* o_in;   // backward input: the forward's O
  const void* dout;   // backward input: dO
  void* dq;
  void* dk;
  void* dv;
  float* delta;       // backward workspace: rowsum(dO * O), [B, Hq, Sq]
  float* part_dk;     // backward workspace when the GQA group is split: fp32 [B, Skv, Hkv * split, D]
  float* part_dv;
  int split;          // parts per GQA group (bwd_split_parts), 0: not split
  int B, Hq, Hkv, Sq, Skv, D;
  float scale;
  int causal;
  const int32_t* kv_lens;  // [B, Hkv] or null; [B] for a paged forward
  attn_dtype_t dtype;
  unsigned int* err;       // device error word (ATTN_DEVERR_* bits)
  // paged forward (block_table non-null): k, v are page pools [num_pages, page_size, Hkv,
  // D]; block_table [B, max_pages]; Skv = max_pages * page_size
  const int32_t* block_table;
  int num_pages, page_size, max_pages;
  // split-KV forward (fwd_splits > 1): ranges of fwd_split_tiles key tiles, partial
  // outputs in the caller's workspace
  int fwd_splits, fwd_split_tiles;
  float* o_part;   // [fwd_splits, B, Hq, Sq, D]
  float* lse_part; // [fwd_splits, B, Hq, Sq]
};

inline size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Split-KV forward: into how many key ranges each (batch, head, 128-row query block) is
// cut, and how many 128-key tiles a range holds. Short query blocks over long K/V (decode,
// a few query rows against a whole cache) give too few work items to fill the GPU. The
// split chosen minimises an estimate of the time: the rounds in which the SMs of a
// 152-SM GB300 work through the items, times an item's length in key tiles plus 3 tiles
// of fixed cost (Q load, pipeline fill and drain, partial-output store; measured on
// decode over a 32760-key cache, where 7, 11, 19 and 64 ranges per head took 130, 133,
// 136 and 167 us). Rounds matter: 40 items cut 8 ways make 320 items, 2.1 rounds, the last
// one run by 16 SMs while the rest wait; cut 7 ways, 280 items fill 2 rounds. A range
// holds at least 4 tiles. 1: no split. A pure function of the sizes, so that the workspace query and the
// launch agree.
inline int fwd_split_count(int B, int Hq, int Sq, int Skv, attn_dtype_t dtype, int* tiles_per) {
  const int tiles = (Skv + 127) / 128;
  if (tiles_per != nullptr) *tiles_per = tiles;
  if (dtype != ATTN_BF16 || B <= 0 || Hq <= 0 || Sq <= 0 || Skv <= 0) return 1;
  const long long base = (long long)B * Hq * ((Sq + 127) / 128);
  const long long sms = 152;
  if (base >= sms) return 1;
  // cost in half tiles: rounds * (2 * tiles per item + 6)
  long long best_n = 1, best = (base + sms - 1) / sms * (2LL * tiles + 6);
  for (long long n = 2; n <= tiles / 4; ++n) {
    const long long per = (tiles + n - 1) / n;
    if ((tiles + per - 1) / per != n) continue;  // the same ranges as a smaller n
    const long long cost = (base * n + sms - 1) / sms * (2 * per + 6);
    if (cost < best) {
      best = cost;
      best_n = n;
    }
  }
  if (best_n <= 1) return 1;
  const int per = (int)((tiles + best_n - 1) / best_n);
  if (tiles_per != nullptr) *tiles_per = per;
  return (tiles + per - 1) / per;
}
inline size_t fwd_split_part_bytes(int splits, int B, int Hq, int Sq, int D) {
  return round256((size_t)splits * B * Hq * Sq * D * sizeof(float));
}
inline size_t fwd_split_lse_bytes(int splits, int B, int Hq, int Sq) {
  return round256((size_t)splits * B * Hq * Sq * sizeof(float));
}

// Into how many parts the bf16 backward splits each GQA group's dK/dV work (0: not
// split). A (batch, kv head, 128-key tile) work item covers the whole group; when such
// items alone are too few to balance the GPU (under 256), each becomes `parts` items of
// Hq / Hkv / parts consecutive query heads: the fewest parts (a divisor of the group
// size) that give at least 256 items, else one item per query head. Each item writes an
// fp32 partial dK/dV to the workspace and a second kernel sums a group's partials in a
// fixed order. A pure function of the sizes, so that the workspace query and the launch
// agree.
inline int bwd_split_parts(int B, int Hq, int Hkv, int Skv, attn_dtype_t dtype) {
  if (dtype != ATTN_BF16 || Hkv <= 0 || Hq <= Hkv || Hq % Hkv != 0) return 0;
  const long long items = (long long)B * Hkv * ((Skv + 127) / 128);
  if (items >= 256) return 0;
  const int g = Hq / Hkv;
  for (int d = 2; d < g; ++d)
    if (g % d == 0 && items * d >= 256) return d;
  return g;
}
inline size_t bwd_delta_bytes(int B, int Hq, int Sq) { return round256((size_t)B * Hq * Sq * sizeof(float)); }
// one fp32 partial dK (or dV) buffer [B, Skv, Hkv * parts, D]
inline size_t bwd_partial_bytes(int B, int Hkv, int parts, int Skv, int D) {
  return round256((size_t)B * Skv * Hkv * parts * D * sizeof(float));
}

// Counts one kernel launch issued by the library (see attn_launch_count()).
void count_launches(int n);

// CUDA-core kernels (fp32 arithmetic): the fp32 backward, any D in {64, 128}.
cudaError_t simt_bwd(const Problem& p, cudaStream_t stream);
// delta = rowsum(dO * O) into p.delta (one warp per row), for the CUDA-core backward
// (the bf16 backward has a delta kernel of its own).
cudaError_t simt_delta(const Problem& p, cudaStream_t stream);

// Tensor-core (tcgen05) kernels for bf16, sm_103a. tc_fwd covers the dense, the paged
// and the split-KV forward (the latter adds the merge kernel).
cudaError_t tc_fwd(const Problem& p, cudaStream_t stream);
// The size, scale, causal, dtype and kv_lens-alignment checks shared by the entry points.
attn_status_t check_common(int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                           int causal, const int32_t* kv_lens, attn_dtype_t dtype);
// ATTN_OK for cudaSuccess; otherwise records `e` for attn_last_cuda_error() and returns
// ATTN_ERR_CUDA.
attn_status_t from_cuda(cudaError_t e);
// The fp32 forward on the tensor cores (tcgen05 kind::tf32, three-term split).
cudaError_t tf32_fwd(const Problem& p, cudaStream_t stream);
cudaError_t tc_bwd(const Problem& p, cudaStream_t stream);

// A bf16 [B, S, H, D] tensor as a 4-D TMA map (D, H, S, B) whose box is one head:
// 64 columns (128 bytes, 128-byte swizzle) x `rows` tokens. False if encoding fails.
bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int H, int D, int rows);
// Test-only: the next tensor-core forward launch injects `mask` faults and uses a
// barrier-wait limit of `timeout_ns` (0 = the default).
void tc_set_test_fault(uint32_t mask, uint64_t timeout_ns);

// Reads one valid key length on the device: clamps to [0, Skv], flags out-of-range.
__device__ __forceinline__ int load_kv_len(const int32_t* kv_lens, int b, int kvh, int Hkv,
                                           int Skv, unsigned int* err) {
  if (kv_lens == nullptr) return Skv;
  int L = __ldg(kv_lens + (int64_t)b * Hkv + kvh);
  if (L < 0 || L > Skv) {
    if (err != nullptr) atomicOr(err, ATTN_DEVERR_KVLEN);
    L = L < 0 ? 0 : Skv;
  }
  return L;
}

}  // namespace attn
