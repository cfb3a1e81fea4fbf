// CUDA-core attention backward with fp32 arithmetic (FFMA + expf): the fp32 element-type
// path of attn_bwd, which must meet a 1e-5 relative tolerance (the fp32 forward runs on
// the tensor cores with a three-term TF32 split, fwd_tf32x3.cu).
//
// Backward ("xtrain evolution.md", infra table row T14): recompute the scores from Q, K
// and LSE, delta = rowsum(dO * O), dS = P * (dP - delta); a dK/dV kernel owns its key
// rows and loops over the query heads of the GQA group (row T15: in-group sum in a fixed
// order, no atomics), and a dQ kernel owns its query rows. All sums run in a fixed
// order, so results are bitwise reproducible.
//
// Thread layout: 4 threads per row (query or key), thread t holding dimensions
// d = 4c + t, so that the 4 threads of a row read 4 consecutive shared-memory words
// and the rows of a warp read the same tile row (a broadcast): no bank conflicts.

#include <cuda_bf16.h>
#include <math_constants.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kTpr = 4;     // threads per row
constexpr int kRows = 32;   // rows per block (128 threads)
constexpr int kTile = 32;   // keys (or queries) per shared-memory tile

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float row_sum4(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Loads rows [r0, r0 + kTile) of a [.., rows, heads, D] tensor slice into shared memory
// as fp32; rows at or past `valid` are written as zeros (and never read from global).
template <typename T, int D>
__device__ __forceinline__ void load_tile(float (*dst)[D], const T* base, int64_t row_stride,
                                          int r0, int valid) {
  for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    const int row = r0 + r;
    dst[r][d] = row < valid ? to_f32(base[(int64_t)row * row_stride + d]) : 0.f;
  }
}

// delta[b, h, i] = sum_d dO[b, i, h, d] * O[b, i, h, d]; one warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(256) simt_delta_kernel(Problem p) {
  const int64_t rows = (int64_t)p.B * p.Sq * p.Hq;
  const int64_t row = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const T* O = static_cast<const T*>(p.o_in) + row * D;
  const T* dO = static_cast<const T*>(p.dout) + row * D;
  float acc = 0.f;
#pragma unroll
  for (int d = lane; d < D; d += 32) acc = fmaf(to_f32(dO[d]), to_f32(O[d]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const int h = (int)(row % p.Hq);
    const int64_t bi = row / p.Hq;  // b * Sq + i
    const int i = (int)(bi % p.Sq), b = (int)(bi / p.Sq);
    p.delta[((int64_t)b * p.Hq + h) * p.Sq + i] = acc;
  }
}

// dK, dV for kRows keys of one (b, kv head): loops over the group's query heads (in
// order) and over query tiles (in order).
template <typename T, int D>
__global__ void __launch_bounds__(kRows * kTpr)
simt_dkdv_kernel(Problem p) {
  constexpr int DPT = D / kTpr;
  __shared__ float sQ[kTile][D];
  __shared__ float sdO[kTile][D];
  __shared__ float sLse[kTile];
  __shared__ float sDel[kTile];
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = p.Hq / p.Hkv;
  const int L = load_kv_len(p.kv_lens, b, kvh, p.Hkv, p.Skv, threadIdx.x == 0 ? p.err : nullptr);
  const int r = threadIdx.x / kTpr, t = threadIdx.x % kTpr;
  const int j0 = blockIdx.x * kRows;
  const int j = j0 + r;
  const bool key_ok = j < L;
  const int64_t kv_stride = (int64_t)p.Hkv * D;
  const int64_t koff = (((int64_t)b * p.Skv + j) * p.Hkv + kvh) * D;
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);
  float kr[DPT], vr[DPT], dk[DPT], dv[DPT];
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    kr[c] = key_ok ? to_f32(K[koff + kTpr * c + t]) : 0.f;
    vr[c] = key_ok ? to_f32(V[koff + kTpr * c + t]) : 0.f;
    dk[c] = 0.f;
    dv[c] = 0.f;
  }
  // first query that sees key j0 (causal): i >= j0 - L + Sq
  int istart = 0;
  if (p.causal) istart = max(0, j0 - L + p.Sq);
  istart = (istart / kTile) * kTile;
  const bool block_has_keys = j0 < L;
  const int64_t q_stride = (int64_t)p.Hq * D;
  for (int rh = 0; rh < g && block_has_keys; ++rh) {
    const int h = kvh * g + rh;
    const T* Q = static_cast<const T*>(p.q) + ((int64_t)b * p.Sq * p.Hq + h) * D;
    const T* dO = static_cast<const T*>(p.dout) + ((int64_t)b * p.Sq * p.Hq + h) * D;
    const float* lse = p.lse + ((int64_t)b * p.Hq + h) * p.Sq;
    const float* del = p.delta + ((int64_t)b * p.Hq + h) * p.Sq;
    for (int q0 = istart; q0 < p.Sq; q0 += kTile) {
      __syncthreads();
      load_tile<T, D>(sQ, Q, q_stride, q0, p.Sq);
      load_tile<T, D>(sdO, dO, q_stride, q0, p.Sq);
      if (threadIdx.x < kTile) {
        const int i = q0 + threadIdx.x;
        sLse[threadIdx.x] = i < p.Sq ? lse[i] : -CUDART_INF_F;
        sDel[threadIdx.x] = i < p.Sq ? del[i] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int ii = 0; ii < kTile; ++ii) {
        const int i = q0 + ii;
        float ps = 0.f, pdp = 0.f;
#pragma unroll
        for (int c = 0; c < DPT; ++c) {
          ps = fmaf(kr[c], sQ[ii][kTpr * c + t], ps);
          pdp = fmaf(vr[c], sdO[ii][kTpr * c + t], pdp);
        }
        ps = row_sum4(ps);
        pdp = row_sum4(pdp);
        const float lse_i = sLse[ii];
        const bool vis = key_ok && i < p.Sq && (!p.causal || j <= i + L - p.Sq) &&
                         lse_i != -CUDART_INF_F;
        const float pij = vis ? expf(ps * p.scale - lse_i) : 0.f;
        const float ds = pij * (pdp - sDel[ii]);
#pragma unroll
        for (int c = 0; c < DPT; ++c) {
          dv[c] = fmaf(pij, sdO[ii][kTpr * c + t], dv[c]);
          dk[c] = fmaf(ds, sQ[ii][kTpr * c + t], dk[c]);
        }
      }
    }
  }
  if (j >= p.Skv) return;
  T* dK = static_cast<T*>(p.dk);
  T* dV = static_cast<T*>(p.dv);
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    dK[koff + kTpr * c + t] = from_f32<T>(dk[c] * p.scale);
    dV[koff + kTpr * c + t] = from_f32<T>(dv[c]);
  }
  (void)kv_stride;
}

// dQ for kRows query rows of one (b, h): loops over K/V tiles in order.
template <typename T, int D>
__global__ void __launch_bounds__(kRows * kTpr)
simt_dq_kernel(Problem p) {
  constexpr int DPT = D / kTpr;
  __shared__ float sK[kTile][D];
  __shared__ float sV[kTile][D];
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = p.Hq / p.Hkv, kvh = h / g;
  const int L = load_kv_len(p.kv_lens, b, kvh, p.Hkv, p.Skv, nullptr);
  const int r = threadIdx.x / kTpr, t = threadIdx.x % kTpr;
  const int i0 = blockIdx.x * kRows;
  const int i = i0 + r;
  const bool row_ok = i < p.Sq;
  const int64_t qoff = (((int64_t)b * p.Sq + i) * p.Hq + h) * D;
  const T* Q = static_cast<const T*>(p.q);
  const T* dO = static_cast<const T*>(p.dout);
  const T* K = static_cast<const T*>(p.k) + ((int64_t)b * p.Skv * p.Hkv + kvh) * D;
  const T* V = static_cast<const T*>(p.v) + ((int64_t)b * p.Skv * p.Hkv + kvh) * D;
  const int64_t kv_stride = (int64_t)p.Hkv * D;
  float qr[DPT], dor[DPT], dq[DPT];
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    qr[c] = row_ok ? to_f32(Q[qoff + kTpr * c + t]) : 0.f;
    dor[c] = row_ok ? to_f32(dO[qoff + kTpr * c + t]) : 0.f;
    dq[c] = 0.f;
  }
  const int64_t srow = ((int64_t)b * p.Hq + h) * p.Sq;
  const float lse_i = row_ok ? p.lse[srow + i] : -CUDART_INF_F;
  const float del_i = row_ok ? p.delta[srow + i] : 0.f;
  int kend = L;
  if (p.causal) kend = min(L, max(0, i0 + kRows - 1 + L - p.Sq + 1));
  for (int j0 = 0; j0 < kend; j0 += kTile) {
    __syncthreads();
    load_tile<T, D>(sK, K, kv_stride, j0, L);
    load_tile<T, D>(sV, V, kv_stride, j0, L);
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kTile; ++jj) {
      const int j = j0 + jj;
      float ps = 0.f, pdp = 0.f;
#pragma unroll
      for (int c = 0; c < DPT; ++c) {
        ps = fmaf(qr[c], sK[jj][kTpr * c + t], ps);
        pdp = fmaf(dor[c], sV[jj][kTpr * c + t], pdp);
      }
      ps = row_sum4(ps);
      pdp = row_sum4(pdp);
      const bool vis = row_ok && j < L && (!p.causal || j <= i + L - p.Sq) &&
                       lse_i != -CUDART_INF_F;
      const float pij = vis ? expf(ps * p.scale - lse_i) : 0.f;
      const float ds = pij * (pdp - del_i);
#pragma unroll
      for (int c = 0; c < DPT; ++c) dq[c] = fmaf(ds, sK[jj][kTpr * c + t], dq[c]);
    }
  }
  if (!row_ok) return;
  T* dQ = static_cast<T*>(p.dq);
#pragma unroll
  for (int c = 0; c < DPT; ++c) dQ[qoff + kTpr * c + t] = from_f32<T>(dq[c] * p.scale);
}

template <typename T, int D>
cudaError_t bwd_launch(const Problem& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.Sq * p.Hq;
  simt_delta_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.Skv > 0) {
    dim3 gk((p.Skv + kRows - 1) / kRows, p.Hkv, p.B);
    simt_dkdv_kernel<T, D><<<gk, kRows * kTpr, 0, s>>>(p);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 gq((p.Sq + kRows - 1) / kRows, p.Hq, p.B);
  simt_dq_kernel<T, D><<<gq, kRows * kTpr, 0, s>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t delta_launch(const Problem& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.Sq * p.Hq;
  simt_delta_kernel<T, D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_delta(const Problem& p, cudaStream_t s) {
  if (p.dtype == ATTN_F32) return p.D == 64 ? delta_launch<float, 64>(p, s) : delta_launch<float, 128>(p, s);
  return p.D == 64 ? delta_launch<__nv_bfloat16, 64>(p, s) : delta_launch<__nv_bfloat16, 128>(p, s);
}

cudaError_t simt_bwd(const Problem& p, cudaStream_t s) {
  if (p.dtype == ATTN_F32) return p.D == 64 ? bwd_launch<float, 64>(p, s) : bwd_launch<float, 128>(p, s);
  return p.D == 64 ? bwd_launch<__nv_bfloat16, 64>(p, s) : bwd_launch<__nv_bfloat16, 128>(p, s);
}

}  // namespace attn
